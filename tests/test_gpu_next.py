"""GPU parity of the multi-query forms of the path.

* Multi-query decode (a 5-token speculative verify): five draft tokens are
  appended to every sequence, and each is scored, selected and attended
  causally, up to and including its own position.  Shapes are those of the
  128K decode workload with three sequences.
* Pool-aware prefill: a chunk of new tokens whose Full layer gives every
  query its own pool of blocks (exact), then a Reindex layer in which every
  query searches only its own pool, then attention over the Reindex
  selection.

Selections are compared as sets with the tie band of checks.check_select;
every attention row is compared, over the oracle's selection or, where the
GPU's differs from it only among near-ties, over the GPU's accepted one
(checks.attended_set)."""
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
from oracle.workload import SeqRef  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import FULL, REINDEX, Workload  # noqa: E402


def append_chunk(dw, T):
    """Append T new tokens to every sequence (positions n_b .. n_b+T-1)."""
    wl = dw.wl
    kv = torch.stack([synth.device.gen_rows_normal(wl.seed, synth.T_KV, b, wl.lengths[b], T,
                                                   wl.dim, dw.mult) for b in range(wl.batch)])
    ik = torch.stack([synth.device.gen_rows_normal(wl.seed, synth.T_IDXK, b, wl.lengths[b], T,
                                                   wl.idx_dim) for b in range(wl.batch)])
    K.quant_append(dw.cache, kv.contiguous(), ik.contiguous(), T, dw.ws)
    return torch.tensor([[wl.lengths[b] + t for t in range(T)] for b in range(wl.batch)],
                        dtype=torch.int32, device="cuda")


def test_verify5_multi_query_decode():
    T = 5
    wl = Workload("verify5-b3", 3, [131072, 20000, 3000], 576, 64, 64, 128, 64, 2048, 128,
                  seed=5, outlier_frac=0.01, prefill_tokens=T)
    dw = DeviceWorkload(wl)
    B, k = wl.batch, wl.topk
    q_pos = append_chunk(dw, T)
    inp = dw.layer_inputs(0, tq=T)
    oi = torch.full((B, T, k), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, T, q_pos, None, B, k, oi, oc,
                 None, None, dw.ws)
    out = torch.empty((B, T, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_prefill(dw.cache, inp["q"].view(torch.int16), wl.heads, T, q_pos, oi, oc, k,
                   inp["swa"], wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    o, oi_h, oc_h = out.cpu().numpy(), oi.cpu().numpy(), oc.cpu().numpy()
    for b in range(B):
        ref = SeqRef(wl, b, n=wl.lengths[b] + T)
        ref.n_prior_positions = wl.lengths[b]
        for t in range(T):
            vis = wl.lengths[b] + t + 1
            s = ref.scores(0, vis, t, T)
            gi = oi_h[b, t, : oc_h[b, t]]
            assert oc_h[b, t] == min(k, vis)
            check_select(gi, s, np.arange(vis), k, f"verify5 top-k b={b} t={t}")
            ridx = O.topk(s, k)
            check_attention(o[b, t], ref.attention(0, attended_set(gi, ridx), tq=t, tq_total=T),
                            f"verify5 attention b={b} t={t}")


def test_pool_aware_prefill_full_then_reindex():
    T = 32
    wl = Workload("pool-prefill-b2", 2, [30000, 9000], 576, 64, 64, 128, 64, 2048, 128,
                  seed=6, outlier_frac=0.01, prefill_tokens=T, layers=[FULL, REINDEX])
    dw = DeviceWorkload(wl)
    B, k = wl.batch, wl.topk
    q_pos = append_chunk(dw, T)
    full_in, re_in = dw.layer_inputs(0, tq=T), dw.layer_inputs(1, tq=T)
    # Full layer: per-query top-k and per-query pools
    oi = torch.full((B, T, k), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, T, K.POOL_BLOCKS), -7, dtype=torch.int32, device="cuda")
    pcnt = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, full_in["q_idx"], full_in["w"], wl.idx_heads, T, q_pos, None, B, k,
                 oi, oc, pool, pcnt, dw.ws)
    # Reindex layer: every query searches its own pool
    oi2 = torch.full((B, T, k), -7, dtype=torch.int32, device="cuda")
    oc2 = torch.full((B, T), -7, dtype=torch.int32, device="cuda")
    K.index_reindex(dw.cache, re_in["q_idx"], re_in["w"], wl.idx_heads, T, q_pos, pool, pcnt,
                    None, B, k, oi2, oc2, dw.ws)
    out = torch.empty((B, T, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_prefill(dw.cache, re_in["q"].view(torch.int16), wl.heads, T, q_pos, oi2, oc2, k,
                   re_in["swa"], wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    h = {n: v.cpu().numpy() for n, v in dict(oi=oi, oc=oc, pool=pool, pcnt=pcnt, oi2=oi2,
                                               oc2=oc2, out=out).items()}
    rng = np.random.default_rng(6)
    for b in range(B):
        ref = SeqRef(wl, b, n=wl.lengths[b] + T)
        ref.n_prior_positions = wl.lengths[b]
        for t in sorted(set([0, 1, T - 1] + rng.choice(T, 5, replace=False).tolist())):
            vis = wl.lengths[b] + t + 1
            s, ridx, rpool = ref.full(0, k, n=vis, tq=t, tq_total=T)
            gi = h["oi"][b, t, : h["oc"][b, t]]
            check_select(gi, s, np.arange(vis), k, f"prefill full top-k b={b} t={t}")
            gp = h["pool"][b, t, : h["pcnt"][b, t]]
            assert np.array_equal(gp, rpool), f"per-query pool b={b} t={t}"
            # the pools agree exactly, so the oracle's Reindex uses its own pool
            s2, pos, ridx2 = ref.reindex(1, rpool, k, n=vis, tq=t, tq_total=T)
            gi2 = h["oi2"][b, t, : h["oc2"][b, t]]
            assert h["oc2"][b, t] == min(k, len(pos))
            check_select(gi2, s2, pos, k, f"prefill reindex top-k b={b} t={t}")
            check_attention(h["out"][b, t],
                            ref.attention(1, attended_set(gi2, ridx2), tq=t, tq_total=T),
                            f"prefill reindex attention b={b} t={t}")
