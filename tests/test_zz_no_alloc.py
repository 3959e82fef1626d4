"""GPU test of csa2_index_full_noalloc, the index_full variant whose scratch is
a fixed array inside the library.  Two calls in a row (different inputs,
batch subsets and k, so the second finds the first one's leftovers in the
shared array) must return exactly what csa2_index_full returns with a caller
workspace; a request larger than the array is rejected before any launch.
Collected last so that it also runs after every other GPU test."""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import Workload  # noqa: E402


def outputs(n_rows, k):
    dev = "cuda"
    return dict(
        out_idx=torch.full((n_rows, 1, k), -7, dtype=torch.int32, device=dev),
        out_cnt=torch.full((n_rows, 1), -7, dtype=torch.int32, device=dev),
        pool=torch.full((n_rows, 1, K.POOL_BLOCKS), -7, dtype=torch.int32, device=dev),
        pool_cnt=torch.full((n_rows, 1), -7, dtype=torch.int32, device=dev),
    )


def host(o):
    return {name: t.cpu().numpy() for name, t in o.items()}


def test_noalloc_matches_index_full_twice():
    lengths = [9000, 131072, 300, 70001]
    wl = Workload("noalloc", 4, lengths, 128, 32, 64, 128, 16, 2048, 128, seed=31,
                  page_size=64)
    dw = DeviceWorkload(wl)
    B = wl.batch
    calls = [
        # (layer, batch subset or None, k)
        (0, None, 2048),
        (1, [2, 1, 3], 500),
    ]
    for layer, subset, k in calls:
        inp = dw.layer_inputs(layer)
        ids = None if subset is None else torch.tensor(subset, dtype=torch.int32, device="cuda")
        n_batch = B if subset is None else len(subset)
        ref, got = outputs(B, k), outputs(B, k)
        K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, 1, None, ids, n_batch, k,
                     ref["out_idx"], ref["out_cnt"], ref["pool"], ref["pool_cnt"], dw.ws)
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        K.index_full_noalloc(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, 1, None, ids,
                             n_batch, k, got["out_idx"], got["out_cnt"], got["pool"],
                             got["pool_cnt"], status)
        torch.cuda.synchronize()
        assert K.get_status(dw.ws) == 0
        assert int(status.item()) == 0
        r, g = host(ref), host(got)
        rows = list(range(B)) if subset is None else subset
        for b in rows:
            n = min(k, lengths[b])
            assert r["out_cnt"][b, 0] == n
            assert r["pool_cnt"][b, 0] == min(K.POOL_BLOCKS, -(-lengths[b] // 8))
        for name in r:
            assert np.array_equal(r[name], g[name]), (layer, name)


def test_noalloc_rejects_requests_larger_than_its_scratch():
    wl = Workload("noalloc-big", 4, [1000] * 4, 128, 32, 4, 32, 16, 64, 16, seed=32)
    dw = DeviceWorkload(wl)
    inp = dw.layer_inputs(0)
    o = outputs(4, 64)
    big = K.Csa2Cache.from_buffer_copy(dw.cache.struct)
    big.max_len = 1 << 21      # four rows of 2^21 positions need about 38 MB of scratch
    r = K._index_full_noalloc(ctypes.byref(big), K._ptr(inp["q_idx"]), K._ptr(inp["w"]), 4, 1,
                              None, None, 4, 64, K._ptr(o["out_idx"]), K._ptr(o["out_cnt"]),
                              None, None, None, K._stream(None))
    assert r == K.CSA2_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (o["out_cnt"] == -7).all()                 # nothing was launched
    # one row of the same cache fits
    o1 = outputs(4, 64)
    ids = torch.tensor([0], dtype=torch.int32, device="cuda")
    K.index_full_noalloc(dw.cache, inp["q_idx"], inp["w"], 4, 1, None, ids, 1, 64,
                         o1["out_idx"], o1["out_cnt"], None, None, None)
    torch.cuda.synchronize()
    assert int(o1["out_cnt"][0, 0]) == 64
