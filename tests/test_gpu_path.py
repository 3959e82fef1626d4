"""GPU parity of the whole path against the oracle on small workloads:
the tiny Full-layer decode workload, ragged/paged edge cases, Reindex and
Reuse, a short prefill chunk, and device-status error reporting.
All calls go through the C ABI (ctypes binding)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
import synth  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle import formats as F  # noqa: E402
from oracle.workload import SeqRef  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import FULL, REINDEX, REUSE, Workload, get_workload  # noqa: E402

from checks import attended_set, check_attention, check_select  # noqa: E402


def dev_rows(dw, b, positions):
    c = dw.cache
    phys = [c.physical_row(b, int(t)) for t in positions]
    ix = torch.tensor(phys, dtype=torch.long, device="cuda")
    return (c.codes.index_select(0, ix).cpu().numpy(), c.scales.index_select(0, ix).cpu().numpy(),
            c.idx_k.index_select(0, ix).cpu().numpy())


def run_full(dw, layer, k, inp, n_batch=None, batch_ids=None):
    wl = dw.wl
    B = wl.batch
    out_idx = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
    out_cnt = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, 1, K.POOL_BLOCKS), -7, dtype=torch.int32, device="cuda")
    pool_cnt = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, 1, None, batch_ids,
                 B if n_batch is None else n_batch, k, out_idx, out_cnt, pool, pool_cnt, dw.ws)
    return out_idx, out_cnt, pool, pool_cnt


def test_fp8_cast_bit_exact():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 2 ** 32, size=1 << 20, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x)]
    fin = F.e4m3_decode(np.arange(0x7F))
    mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)
    extra = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                            fin.astype(np.float32), [0.0, -0.0, 448.0, 464.0, 1e30, -1e30]])
    x = np.concatenate([x, extra, -extra]).astype(np.float32)
    xd = torch.from_numpy(x).cuda()
    out = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
    K.fp8_quant(xd, out)
    got = out.cpu().numpy()
    ref = O.fp8_cast(x)
    bad = np.nonzero(got != ref)[0]
    assert len(bad) == 0, (x[bad[:4]], got[bad[:4]], ref[bad[:4]])


@pytest.fixture(scope="module")
def tiny():
    wl = get_workload(1)
    dw = DeviceWorkload(wl)
    return wl, dw


def test_tiny_cache_bit_exact(tiny):
    wl, dw = tiny
    ref = SeqRef(wl, 0)
    pos = np.arange(wl.lengths[0])
    codes, scales, idxk = dev_rows(dw, 0, pos)
    rc, rs = ref.cache_rows(pos)
    assert np.array_equal(codes[:, : wl.dim // 2], rc)
    assert np.array_equal(scales[:, : wl.dim // 16], rs)
    assert np.array_equal(idxk[:, : wl.idx_dim], ref.idxk_rows(pos))
    assert int(dw.cache.seq_len[0]) == wl.lengths[0]
    assert K.get_status(dw.ws) == 0


def test_tiny_full_layer_end_to_end(tiny):
    wl, dw = tiny
    inp = dw.layer_inputs(0)
    oi, oc, pool, pc = run_full(dw, 0, wl.topk, inp)
    ref = SeqRef(wl, 0)
    s, ridx, rpool = ref.full(0, wl.topk)
    cnt = int(oc[0, 0])
    gi = oi[0, 0, :cnt].cpu().numpy()
    check_select(gi, s, np.arange(len(s)), wl.topk)
    npool = int(pc[0, 0])
    gp = pool[0, 0, :npool].cpu().numpy()
    bm = O.block_maxima(s)
    check_select(gp, bm, np.arange(len(bm)), K.POOL_BLOCKS, "pool")
    assert npool == len(rpool) == 256
    # attention over the GPU's own selection and the window
    out = torch.empty((1, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    q = inp["q"].view(torch.int16)
    K.attn_decode(dw.cache, q, wl.heads, oi.view(1, -1), oc.view(1), wl.topk, inp["swa"], None,
                  wl.window, 0.0, out, dw.ws)
    check_attention(out[0].cpu().numpy(), ref.attention(0, attended_set(gi, ridx)))
    assert K.get_status(dw.ws) == 0


def mini_workload(page_size=64):
    lengths = [1, 7, 64, 129, 2049, 20000]
    return Workload("mini-ragged", 6, lengths, 128, 32, 8, 64, 16, 64, 16, seed=11,
                    page_size=page_size, outlier_frac=0.02)


# Page sizes: the common 64, none, and the other layouts the indexer's
# producer handles differently: 8-32-row pages (several pages per 128-position
# tile, page-table windows shifted every few tiles), 256-row pages (two tiles
# per page) and 384-row pages (not a power of two: a division, not a shift).
@pytest.fixture(scope="module", params=[64, 0, 8, 16, 32, 256, 384],
                ids=["paged64", "contiguous", "paged8", "paged16", "paged32", "paged256", "paged384"])
def mini(request):
    wl = mini_workload(request.param)
    return wl, DeviceWorkload(wl)


def test_mini_cache_bit_exact(mini):
    wl, dw = mini
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        pos = np.arange(n) if n < 3000 else np.unique(np.r_[np.arange(200), np.arange(n - 200, n),
                                                             np.random.default_rng(b).integers(0, n, 300)])
        codes, scales, idxk = dev_rows(dw, b, pos)
        rc, rs = ref.cache_rows(pos)
        assert np.array_equal(codes[:, :64], rc) and np.array_equal(scales[:, :8], rs)
        assert np.array_equal(idxk[:, :64], ref.idxk_rows(pos))


@pytest.mark.parametrize("k", [1, 64, 2048])
def test_mini_full_reindex_reuse(mini, k):
    wl, dw = mini
    inp0 = dw.layer_inputs(0)
    oi, oc, pool, pc = run_full(dw, 0, k, inp0)
    inp1 = dw.layer_inputs(1)
    ri = torch.full((wl.batch, 1, k), -7, dtype=torch.int32, device="cuda")
    rc = torch.full((wl.batch, 1), -7, dtype=torch.int32, device="cuda")
    K.index_reindex(dw.cache, inp1["q_idx"], inp1["w"], wl.idx_heads, 1, None, pool, pc, None,
                    wl.batch, k, ri, rc, dw.ws)
    swa_cnt = torch.tensor([0, 1, 16, 16, 5, 16], dtype=torch.int32, device="cuda")
    outs = []
    for layer, (idx_t, cnt_t) in enumerate([(oi, oc), (ri, rc), (ri, rc)]):
        inp = dw.layer_inputs(layer)
        out = torch.empty((wl.batch, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
        K.attn_decode(dw.cache, inp["q"].view(torch.int16), wl.heads, idx_t.view(wl.batch, k),
                      cnt_t.view(wl.batch), k, inp["swa"], swa_cnt, wl.window, 0.0, out, dw.ws)
        outs.append(out.cpu().numpy())
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        s, ridx, rpool = ref.full(0, k)
        cnt = int(oc[b, 0])
        gi = oi[b, 0, :cnt].cpu().numpy()
        check_select(gi, s, np.arange(n), k, f"full b={b}")
        gp = pool[b, 0, : int(pc[b, 0])].cpu().numpy()
        bm = O.block_maxima(s)
        check_select(gp, bm, np.arange(len(bm)), K.POOL_BLOCKS, f"pool b={b}")
        sc = int(swa_cnt[b])
        check_attention(outs[0][b], ref.attention(0, attended_set(gi, ridx), sc), f"full attn b={b}")
        # the GPU's Reindex searched the GPU's pool (accepted above; it can
        # differ from the oracle's only among near-tied block maxima)
        upool = attended_set(gp, rpool)
        s2, pos2, r2 = ref.reindex(1, upool, k)
        g2 = ri[b, 0, : int(rc[b, 0])].cpu().numpy()
        check_select(g2, s2, pos2, k, f"reindex b={b}")
        assert set(g2.tolist()) <= set(O.pool_positions(upool, n).tolist())
        sel = attended_set(g2, r2)
        check_attention(outs[1][b], ref.attention(1, sel, sc), f"reindex attn b={b}")
        check_attention(outs[2][b], ref.attention(2, sel, sc), f"reuse attn b={b}")


def test_attention_given_indices_and_bad_index(mini):
    wl, dw = mini
    k = 300
    idx = np.full((wl.batch, k), 0, dtype=np.int32)
    cnt = np.zeros(wl.batch, dtype=np.int32)
    sets = []
    for b, n in enumerate(wl.lengths):
        sel = synth.sample_distinct(wl.seed, synth.T_PRIOR, b, n, k)
        idx[b, : len(sel)] = sel
        cnt[b] = len(sel)
        sets.append(sel)
    # sequence 5 gets one out-of-range index that must be left out
    idx[5, 10] = wl.lengths[5] + 5
    inp = dw.layer_inputs(2)
    out = torch.empty((wl.batch, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.reset_status(dw.ws)
    K.attn_decode(dw.cache, inp["q"].view(torch.int16), wl.heads, torch.from_numpy(idx).cuda(),
                  torch.from_numpy(cnt).cuda(), k, inp["swa"], None, wl.window, 0.0, out, dw.ws)
    st = K.get_status(dw.ws)
    assert st & K.DEV_BAD_INDEX
    K.reset_status(dw.ws)
    assert K.get_status(dw.ws) == 0
    o = out.cpu().numpy()
    for b in range(wl.batch):
        ref = SeqRef(wl, b)
        sel = sets[b] if b != 5 else np.delete(sets[b], 10)
        check_attention(o[b], ref.attention(2, sel), f"given idx b={b}")


def test_prefill_chunk_small():
    T = 40
    wl = Workload("mini-prefill", 2, [300, 5], 128, 32, 8, 64, 16, 32, 16, seed=12,
                  prefill_tokens=T)
    dw = DeviceWorkload(wl)
    B = wl.batch
    # append the T new tokens (positions n .. n+T-1) in one call
    kv = torch.stack([synth.device.gen_rows_normal(wl.seed, synth.T_KV, b, wl.lengths[b], T, wl.dim)
                      for b in range(B)])
    ik = torch.stack([synth.device.gen_rows_normal(wl.seed, synth.T_IDXK, b, wl.lengths[b], T, wl.idx_dim)
                      for b in range(B)])
    # sequences must share the chunk length; append per sequence through views
    for b in range(B):
        K.quant_append(dw.seq_view(b), kv[b].contiguous(), ik[b].contiguous(), T, dw.ws)
    q_pos = torch.tensor([[wl.lengths[b] + t for t in range(T)] for b in range(B)],
                         dtype=torch.int32, device="cuda")
    inp = dw.layer_inputs(0, tq=T)
    k = wl.topk
    oi = torch.full((B, T, k), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, T, q_pos, None, B, k, oi, oc,
                 None, None, dw.ws)
    out = torch.empty((B, T, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_prefill(dw.cache, inp["q"].view(torch.int16), wl.heads, T, q_pos, oi, oc, k,
                   inp["swa"], wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    o = out.cpu().numpy()
    for b in range(B):
        ref = SeqRef(wl, b, n=wl.lengths[b] + T)
        ref.n_prior_positions = wl.lengths[b]
        pos = np.arange(wl.lengths[b] + T)
        codes, scales, idxk = dev_rows(dw, b, pos)
        rc, rs = ref.cache_rows(pos)
        assert np.array_equal(codes[:, :64], rc) and np.array_equal(scales[:, :8], rs)
        for t in range(T):
            vis = wl.lengths[b] + t + 1
            s = ref.scores(0, vis, t, T)
            cnt = int(oc[b, t])
            gi = oi[b, t, :cnt].cpu().numpy()
            check_select(gi, s, np.arange(vis), k, f"prefill b={b} t={t}")
            ridx = O.topk(s, k)
            check_attention(o[b, t], ref.attention(0, attended_set(gi, ridx), tq=t, tq_total=T),
                            f"prefill attn b={b} t={t}")


def test_append_overflow_sets_status():
    wl = Workload("overflow", 1, [60], 128, 32, 8, 64, 16, 8, 16, seed=13)
    dw = DeviceWorkload(wl)
    assert wl.max_len == 124
    kv = synth.device.gen_rows_normal(wl.seed, synth.T_KV, 0, 60, 70, wl.dim)
    K.reset_status(dw.ws)
    K.quant_append(dw.cache, kv, None, 70, dw.ws)
    assert K.get_status(dw.ws) & K.DEV_OVERFLOW
    assert int(dw.cache.seq_len[0]) == wl.max_len
    K.reset_status(dw.ws)


def test_invalid_arguments_rejected():
    wl = mini_workload(0)
    dw = DeviceWorkload(wl, build_cache=False)
    inp = dw.layer_inputs(0)
    oi = torch.zeros((wl.batch, 1, 64), dtype=torch.int32, device="cuda")
    oc = torch.zeros((wl.batch, 1), dtype=torch.int32, device="cuda")
    with pytest.raises(K.Csa2Error):
        K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, 1, None, None, wl.batch,
                     4096, oi, oc, None, None, dw.ws)   # k above the cap
    with pytest.raises(K.Csa2Error):
        K.attn_decode(dw.cache, inp["q"].view(torch.int16), 65, oi.view(wl.batch, -1),
                      oc.view(-1), 64, inp["swa"], None, wl.window, 0.0,
                      torch.empty(1, device="cuda"), dw.ws)  # more than 64 heads


def test_attention_with_large_queries(tiny):
    """Heads whose |q| reach 2^14 and beyond take the scaled f16 copy; the
    output must still match the oracle (which uses the bf16 values exactly)."""
    wl, dw = tiny
    inp = dw.layer_inputs(0)
    q = inp["q"].clone()                                   # bf16 [1, 1, H, D]
    scale = torch.ones(wl.heads, dtype=torch.float32, device="cuda")
    scale[0], scale[3], scale[7] = 2.0 ** 15, 2.0 ** 20, 2.0 ** -20
    q = (q.float() * scale.view(1, 1, -1, 1)).to(torch.bfloat16)
    n = wl.lengths[0]
    idx = torch.arange(0, n, n // wl.topk, dtype=torch.int32, device="cuda")[: wl.topk].view(1, -1)
    cnt = torch.tensor([wl.topk], dtype=torch.int32, device="cuda")
    out = torch.empty((1, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_decode(dw.cache, q.view(torch.int16), wl.heads, idx, cnt, wl.topk, inp["swa"], None,
                  wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    ref = SeqRef(wl, 0)
    qb = q.view(torch.int16).cpu().numpy().view(np.uint16).reshape(wl.heads, wl.dim)
    rows = np.concatenate([ref.dequant_rows(idx.cpu().numpy()[0]),
                           O.swa_rows_decode(ref.inputs(0)["swa"][: wl.window])])
    expect = O.sparse_attention(F.bf16_bits_to_f64(qb), rows)
    check_attention(out[0].cpu().numpy(), expect, "large queries")
