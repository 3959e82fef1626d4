"""GPU parity of the MXFP4 indexer keys (E2M1 codes with an E8M0 scale per 32
channels, 68 bytes per 128-channel key) against the oracle.

* Append: the codes and scale bytes written by csa2_quant_append equal the
  oracle's quantize_mxfp4 bit for bit, on seeded rows and on rows built to hit
  the format's edges (zero and subnormal blocks, saturation, ties, blocks whose
  scales differ by up to 2^24 within one key).
* Scoring: Full top-k sets and pools, Reindex top-k sets (paged and
  contiguous caches, ragged lengths, every padded head count) are compared
  with the oracle's scores over the decoded keys under the tie band of
  checks.check_select.  Rows with widely spread block scales make a scale
  applied to the wrong block or row change the ranking by orders of magnitude.
* A prefill chunk (Tq > 1, causal limits) and a 128K decode sequence.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
import synth  # noqa: E402
import synth.device  # noqa: E402
from checks import attended_set, check_attention, check_select  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle import formats as F  # noqa: E402
from oracle.workload import SeqRef  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import FULL, REINDEX, Workload  # noqa: E402


def dev_idx(dw, b, positions):
    c = dw.cache
    ix = torch.tensor([c.physical_row(b, int(t)) for t in positions], dtype=torch.long,
                      device="cuda")
    return (c.idx_k.index_select(0, ix).cpu().numpy()[:, :64],
            c.idx_scales.index_select(0, ix).cpu().numpy()[:, :4])


def run_full(dw, inp, k, tq=1, q_pos=None):
    wl = dw.wl
    B = wl.batch
    oi = torch.full((B, tq, k), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B, tq), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, tq, K.POOL_BLOCKS), -7, dtype=torch.int32, device="cuda")
    pc = torch.full((B, tq), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, tq, q_pos, None, B, k, oi, oc,
                 pool, pc, dw.ws)
    return oi, oc, pool, pc


def mx_workload(name, lengths, hi, page_size, seed, **kw):
    return Workload(name, len(lengths), lengths, 128, 32, hi, 128, 16, 64, 16, seed=seed,
                    page_size=page_size, outlier_frac=0.02, idx_format="mxfp4",
                    layers=[FULL, REINDEX], **kw)


@pytest.fixture(scope="module", params=[(64, 8), (0, 8), (0, 32), (128, 64)],
                ids=["paged64-hi8", "contiguous-hi8", "contiguous-hi32", "paged128-hi64"])
def mini(request):
    page, hi = request.param
    wl = mx_workload(f"mx-mini-p{page}-h{hi}", [1, 7, 64, 129, 2049, 20000], hi, page, 31 + hi)
    return wl, DeviceWorkload(wl)


def test_mx_seeded_append_bit_exact(mini):
    wl, dw = mini
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        pos = np.arange(n) if n < 3000 else np.unique(np.r_[np.arange(300), np.arange(n - 300, n),
                                                             np.random.default_rng(b).integers(0, n, 400)])
        codes, scales = dev_idx(dw, b, pos)
        rc, rs = ref.idxk_rows(pos)
        assert np.array_equal(codes, rc), b
        assert np.array_equal(scales, rs), b


@pytest.mark.parametrize("k", [1, 64, 2048])
def test_mx_full_and_reindex(mini, k):
    wl, dw = mini
    inp0, inp1 = dw.layer_inputs(0), dw.layer_inputs(1)
    oi, oc, pool, pc = run_full(dw, inp0, k)
    ri = torch.full((wl.batch, 1, k), -7, dtype=torch.int32, device="cuda")
    rcn = torch.full((wl.batch, 1), -7, dtype=torch.int32, device="cuda")
    K.index_reindex(dw.cache, inp1["q_idx"], inp1["w"], wl.idx_heads, 1, None, pool, pc, None,
                    wl.batch, k, ri, rcn, dw.ws)
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        s, ridx, rpool = ref.full(0, k)
        gi = oi[b, 0, : int(oc[b, 0])].cpu().numpy()
        check_select(gi, s, np.arange(n), k, f"mx full b={b}")
        gp = pool[b, 0, : int(pc[b, 0])].cpu().numpy()
        check_select(gp, O.block_maxima(s), np.arange(-(-n // 8)), K.POOL_BLOCKS, f"mx pool b={b}")
        s2, pos2, _ = ref.reindex(1, attended_set(gp, rpool), k)
        g2 = ri[b, 0, : int(rcn[b, 0])].cpu().numpy()
        check_select(g2, s2, pos2, k, f"mx reindex b={b}")


def edge_rows(rng, n, di=128):
    """fp32 key rows whose four blocks sit at scales up to 2^24 apart, plus rows
    that hit the format's edges."""
    x = rng.standard_normal((n, di)).astype(np.float32)
    mult = np.exp2(rng.integers(-12, 13, size=(n, di // 32))).astype(np.float32)
    x *= np.repeat(mult, 32, axis=1)
    if n >= 8:
        x[0] = 0.0                                    # all-zero key: codes 0, scales 0
        x[1, :32] = np.float32(1e-40)                 # subnormal block
        x[2, :] = 0.0
        x[2, 0], x[2, 1], x[2, 2], x[2, 3] = 7.0, -7.9, 5.0, 0.25   # saturation, ties
        x[3, 32:64] = -0.0
        x[4] *= np.float32(1e25)                      # huge scales
        x[5] *= np.float32(1e-25)                     # tiny scales
    return x


@pytest.mark.parametrize("page", [0, 64], ids=["contiguous", "paged64"])
def test_mx_spread_scales_append_and_select(page):
    lengths = [3000, 517, 8]
    wl = mx_workload(f"mx-spread-p{page}", lengths, 64, page, 41)
    dw = DeviceWorkload(wl, build_cache=False)
    rng = np.random.default_rng(41)
    keys = []
    for b, n in enumerate(lengths):
        v = dw.seq_view(b)
        ik = edge_rows(rng, n)
        kv = synth.device.gen_rows_normal(wl.seed, synth.T_KV, b, 0, n, wl.dim)
        K.quant_append(v, kv, torch.from_numpy(ik).cuda(), n, dw.ws)
        keys.append(ik)
    torch.cuda.synchronize()
    assert K.get_status(dw.ws) == 0
    inp = dw.layer_inputs(0)
    q = inp["q_idx"].cpu().numpy()
    w = inp["w"].cpu().numpy()
    for k in (1, 50, 600):
        oi, oc, pool, pc = run_full(dw, inp, k)
        assert K.get_status(dw.ws) == 0
        for b, n in enumerate(lengths):
            rc, rs = O.quantize_mxfp4(keys[b])
            codes, scales = dev_idx(dw, b, np.arange(n))
            assert np.array_equal(codes, rc) and np.array_equal(scales, rs), b
            s = O.indexer_scores_values(F.e4m3_decode(q[b, 0]).reshape(wl.idx_heads, 128),
                                        w[b, 0], O.dequantize_mxfp4(rc, rs, 128))
            gi = oi[b, 0, : int(oc[b, 0])].cpu().numpy()
            check_select(gi, s, np.arange(n), k, f"spread full b={b} k={k}")
            gp = pool[b, 0, : int(pc[b, 0])].cpu().numpy()
            check_select(gp, O.block_maxima(s), np.arange(-(-n // 8)), K.POOL_BLOCKS,
                         f"spread pool b={b}")


def test_mx_prefill_chunk_and_attention():
    T = 48
    wl = Workload("mx-prefill", 2, [9000, 300], 576, 64, 64, 128, 64, 512, 128, seed=43,
                  outlier_frac=0.01, prefill_tokens=T, idx_format="mxfp4")
    dw = DeviceWorkload(wl)
    B, k = wl.batch, wl.topk
    kv = torch.stack([synth.device.gen_rows_normal(wl.seed, synth.T_KV, b, wl.lengths[b], T,
                                                   wl.dim, dw.mult) for b in range(B)])
    ik = torch.stack([synth.device.gen_rows_normal(wl.seed, synth.T_IDXK, b, wl.lengths[b], T,
                                                   wl.idx_dim) for b in range(B)])
    K.quant_append(dw.cache, kv.contiguous(), ik.contiguous(), T, dw.ws)
    q_pos = torch.tensor([[wl.lengths[b] + t for t in range(T)] for b in range(B)],
                         dtype=torch.int32, device="cuda")
    inp = dw.layer_inputs(0, tq=T)
    oi, oc, _, _ = run_full(dw, inp, k, tq=T, q_pos=q_pos)
    out = torch.empty((B, T, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_prefill(dw.cache, inp["q"].view(torch.int16), wl.heads, T, q_pos, oi, oc, k,
                   inp["swa"], wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    for b in range(B):
        ref = SeqRef(wl, b, n=wl.lengths[b] + T)
        ref.n_prior_positions = wl.lengths[b]
        pos = np.arange(wl.lengths[b], wl.lengths[b] + T)
        codes, scales = dev_idx(dw, b, pos)
        rc, rs = ref.idxk_rows(pos)
        assert np.array_equal(codes, rc) and np.array_equal(scales, rs)
        for t in (0, 1, 17, T - 1):
            vis = wl.lengths[b] + t + 1
            s = ref.scores(0, vis, t, T)
            gi = oi[b, t, : int(oc[b, t])].cpu().numpy()
            check_select(gi, s, np.arange(vis), k, f"mx prefill b={b} t={t}")
            ridx = O.topk(s, k)
            check_attention(out[b, t].cpu().numpy(),
                            ref.attention(0, attended_set(gi, ridx), tq=t, tq_total=T),
                            f"mx prefill attention b={b} t={t}")


def test_mx_long_decode_sequence():
    wl = Workload("mx-decode-128k", 2, [131072, 4099], 576, 64, 64, 128, 64, 2048, 128,
                  seed=44, outlier_frac=0.01, idx_format="mxfp4")
    dw = DeviceWorkload(wl)
    inp = dw.layer_inputs(0)
    oi, oc, pool, pc = run_full(dw, inp, wl.topk)
    out = torch.empty((wl.batch, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_decode(dw.cache, inp["q"].view(torch.int16), wl.heads, oi.view(wl.batch, -1),
                  oc.view(wl.batch), wl.topk, inp["swa"], None, wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        s, ridx, rpool = ref.full(0, wl.topk)
        gi = oi[b, 0, : int(oc[b, 0])].cpu().numpy()
        check_select(gi, s, np.arange(n), wl.topk, f"mx decode b={b}")
        gp = pool[b, 0, : int(pc[b, 0])].cpu().numpy()
        check_select(gp, O.block_maxima(s), np.arange(-(-n // 8)), K.POOL_BLOCKS,
                     f"mx decode pool b={b}")
        check_attention(out[b].cpu().numpy(), ref.attention(0, attended_set(gi, ridx)),
                        f"mx decode attn b={b}")
