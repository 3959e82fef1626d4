"""GPU parity of the encoder's m = 2 cache (two source positions per entry,
combined by the per-channel softmax of their compression logits, then RoPE at
the entry position and FP4) against the oracle.

* Codes and scales bit-exact on seeded caches (contiguous and paged, ragged
  entry counts) and on logits built to hit the weight rule's edges: equal
  logits, differences of +-0, tiny, large and beyond the e^-80 cut.
* A decode append of one entry per sequence through csa2_quant_append_pairs.
* The rest of the path is the same over entries: a Full layer and its
  attention on a compressed cache against the oracle.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
import synth  # noqa: E402
from checks import attended_set, check_attention, check_select  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle.workload import SeqRef  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import Workload  # noqa: E402


def dev_rows(dw, b, positions):
    c = dw.cache
    ix = torch.tensor([c.physical_row(b, int(t)) for t in positions], dtype=torch.long,
                      device="cuda")
    return c.codes.index_select(0, ix).cpu().numpy(), c.scales.index_select(0, ix).cpu().numpy()


def enc_workload(lengths, page, seed=51, **kw):
    return Workload(f"enc-pairs-p{page}", len(lengths), lengths, 576, 64, 64, 128, 64, 512, 128,
                    seed=seed, outlier_frac=0.01, page_size=page, compress=2, **kw)


@pytest.fixture(scope="module", params=[0, 64], ids=["contiguous", "paged64"])
def enc(request):
    wl = enc_workload([1, 777, 20000], request.param)
    return wl, DeviceWorkload(wl)


def test_pairs_cache_bit_exact(enc):
    wl, dw = enc
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        pos = np.arange(n) if n < 2000 else np.unique(np.r_[np.arange(500), np.arange(n - 500, n),
                                                             np.random.default_rng(b).integers(0, n, 500)])
        codes, scales = dev_rows(dw, b, pos)
        rc, rs = ref.cache_rows(pos)
        assert np.array_equal(codes[:, : wl.dim // 2], rc), b
        assert np.array_equal(scales[:, : wl.dim // 16], rs), b
        assert int(dw.cache.seq_len[b]) == n


def test_pairs_full_layer_and_attention(enc):
    wl, dw = enc
    B, k = wl.batch, wl.topk
    inp = dw.layer_inputs(0)
    oi = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, 1, None, None, B, k, oi, oc,
                 None, None, dw.ws)
    out = torch.empty((B, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_decode(dw.cache, inp["q"].view(torch.int16), wl.heads, oi.view(B, k), oc.view(B), k,
                  inp["swa"], None, wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        s, ridx, _ = ref.full(0, k)
        gi = oi[b, 0, : int(oc[b, 0])].cpu().numpy()
        check_select(gi, s, np.arange(n), k, f"pairs full b={b}")
        check_attention(out[b].cpu().numpy(), ref.attention(0, attended_set(gi, ridx)),
                        f"pairs attention b={b}")


def test_pairs_decode_append_one_entry():
    wl = enc_workload([300, 41], 0, seed=52, extra_capacity=8)
    dw = DeviceWorkload(wl)
    kvs, zs, iks = [], [], []
    for b, n in enumerate(wl.lengths):
        kv, z = dw.pair_sources(b, n, 1)
        kvs.append(kv)
        zs.append(z)
        iks.append(synth.device.gen_rows_normal(wl.seed, synth.T_IDXK, b, n, 1, wl.idx_dim))
    K.quant_append_pairs(dw.cache, torch.stack(kvs).contiguous(), torch.stack(zs).contiguous(),
                         torch.stack(iks).contiguous(), 1, dw.ws)
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        assert int(dw.cache.seq_len[b]) == n + 1
        ref = SeqRef(wl, b, n=n + 1)
        codes, scales = dev_rows(dw, b, [n - 1, n])
        rc, rs = ref.cache_rows([n - 1, n])
        assert np.array_equal(codes[:, : wl.dim // 2], rc) and np.array_equal(scales[:, :36], rs)


@pytest.mark.parametrize("T", [64, 320], ids=["cluster-kernel", "streaming-kernel"])
def test_pairs_logit_edges_bit_exact(T):
    """Source rows with hand-built logits: equal, +-0 differences, tiny, around
    the 80 cut, huge; compared with the oracle's compress + quantise.  64
    entries go through the small-append kernel, 320 through the streaming
    kernel (rows staged in shared memory)."""
    wl = enc_workload([T], 0, seed=53)
    dw = DeviceWorkload(wl, build_cache=False)
    rng = np.random.default_rng(53)
    D = wl.dim
    x = (rng.standard_normal((2 * T, D)) * 3).astype(np.float32)
    z0 = (rng.standard_normal((T, D)) * 4).astype(np.float32)
    diffs = np.array([0.0, -0.0, 1e-7, -1e-7, 1e-3, 79.9, 80.0, 80.1, -80.2, 200.0, -1e30, 0.5],
                     dtype=np.float32)
    d = diffs[rng.integers(0, len(diffs), size=(T, D))]
    d[:4] = (rng.standard_normal((4, D)) * 10).astype(np.float32)   # and plain random rows
    z1 = (z0 + d).astype(np.float32)
    z = np.empty((2 * T, D), dtype=np.float32)
    z[0::2], z[1::2] = z0, z1
    ik = synth.device.gen_rows_normal(wl.seed, synth.T_IDXK, 0, 0, T, wl.idx_dim)
    K.quant_append_pairs(dw.cache, torch.from_numpy(x).cuda(), torch.from_numpy(z).cuda(), ik, T,
                         dw.ws)
    assert K.get_status(dw.ws) == 0
    ref = SeqRef(wl, 0)
    rc, rs = O.quant_append_rows(O.compress_pairs(x, z), np.arange(T), ref.cos, ref.sin,
                                 wl.rope_dim)
    codes, scales = dev_rows(dw, 0, np.arange(T))
    assert np.array_equal(codes[:, : D // 2], rc)
    assert np.array_equal(scales[:, : D // 16], rs)
