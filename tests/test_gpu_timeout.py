"""The kernels' bounded waits, made to run out on an ordinary launch.

Every mbarrier wait of the indexer is bounded by the GPU's global timer.
With the limit set to 1 ns (csa2_set_wait_limit), waits give up at once: the
kernel must stop its pipeline, wait for the copies and MMAs it has already
started, free its tensor memory, return, and report CSA2_DEV_TIMEOUT in the
workspace status word.  The next call with the default limit, on the same
workspace, must then give the oracle's selections again.  No GPU is made to
fault or hang: the waits return and the kernels exit.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle.workload import SeqRef  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import Workload  # noqa: E402

from checks import check_select  # noqa: E402


def run_full(dw, inp, k):
    wl = dw.wl
    B = wl.batch
    oi = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, 1, K.POOL_BLOCKS), -7, dtype=torch.int32, device="cuda")
    pc = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, 1, None, None, B, k, oi, oc,
                 pool, pc, dw.ws)
    return oi, oc, pool, pc


def test_wait_timeout_reported_then_next_call_correct():
    wl = Workload("timeout", 4, [131072, 65536, 40000, 3000], 576, 64, 64, 128, 64, 2048, 128,
                  seed=81, outlier_frac=0.01)
    dw = DeviceWorkload(wl)
    inp = dw.layer_inputs(0)
    k = wl.topk
    K.reset_status(dw.ws)
    try:
        K.set_wait_limit(1)
        run_full(dw, inp, k)
        torch.cuda.synchronize()
    finally:
        K.set_wait_limit(0)
    st = K.get_status(dw.ws)
    assert st & K.DEV_TIMEOUT, f"status {st:#x}: no wait gave up"
    K.reset_status(dw.ws)
    oi, oc, pool, pc = run_full(dw, inp, k)
    torch.cuda.synchronize()
    assert K.get_status(dw.ws) == 0
    for b, n in enumerate(wl.lengths):
        ref = SeqRef(wl, b)
        s, ridx, rpool = ref.full(0, k)
        check_select(oi[b, 0, : int(oc[b, 0])].cpu().numpy(), s, np.arange(n), k, f"topk b={b}")
        check_select(pool[b, 0, : int(pc[b, 0])].cpu().numpy(), O.block_maxima(s),
                     np.arange(-(-n // 8)), K.POOL_BLOCKS, f"pool b={b}")
