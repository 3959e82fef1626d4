"""GPU selection edge cases: massive exact ties in the indexer scores (few
distinct key rows), all-equal scores, a tied pool boundary split over the
CTAs of a cluster, and a sequence long enough that the
pool is chosen through two levels of block groups.  The indexer-key bytes
are written directly into the cache by the test (the same bytes feed the
oracle), so ties are exact on both sides and the sets must match exactly:
ranking is by score, then by lower position."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle import formats as F  # noqa: E402
from synth.device import DeviceWorkload  # noqa: E402
from synth.workloads import Workload  # noqa: E402


def run_index(dw, q_codes, w, k):
    wl = dw.wl
    B = wl.batch
    oi = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
    oc = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    pool = torch.full((B, 1, K.POOL_BLOCKS), -7, dtype=torch.int32, device="cuda")
    pc = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, torch.from_numpy(q_codes).cuda(), torch.from_numpy(w).cuda(),
                 wl.idx_heads, 1, None, None, B, k, oi, oc, pool, pc, dw.ws)
    assert K.get_status(dw.ws) == 0
    return oi.cpu().numpy(), oc.cpu().numpy(), pool.cpu().numpy(), pc.cpu().numpy()


def write_idx_rows(dw, b, rows_codes):
    c = dw.cache
    n = rows_codes.shape[0]
    base = b * c.max_len
    c.idx_k[base:base + n, : rows_codes.shape[1]] = torch.from_numpy(rows_codes).cuda()


def test_ties_and_equal_scores():
    lengths = [5000, 20000, 3000, 40000]
    wl = Workload("ties", 4, lengths, 128, 32, 8, 32, 16, 1024, 16, seed=21)
    dw = DeviceWorkload(wl)
    rng = np.random.default_rng(21)
    hi, di = wl.idx_heads, wl.idx_dim
    q = F.e4m3_encode(rng.standard_normal((wl.batch, 1, hi, di)).astype(np.float32))
    w = rng.random((wl.batch, 1, hi)).astype(np.float32)
    distinct = F.e4m3_encode(rng.standard_normal((4, di)).astype(np.float32))
    patterns = [
        np.arange(lengths[0]) % 3 == 0,                       # two distinct rows
        np.arange(lengths[1]) % 4,                            # four distinct rows
        np.zeros(lengths[2], dtype=np.int64),                 # one row: all equal
        (np.arange(lengths[3]) * 7919) % 2,                   # two rows, scattered
    ]
    rows = []
    for b, pat in enumerate(patterns):
        r = distinct[np.asarray(pat, dtype=np.int64)]
        write_idx_rows(dw, b, r)
        rows.append(r)
    torch.cuda.synchronize()
    for k in (1, 1000, 1024):
        oi, oc, pool, pc = run_index(dw, q, w, k)
        for b in range(wl.batch):
            s = O.indexer_scores(q[b, 0], w[b, 0], rows[b])
            ridx, rpool = O.full_select(s, k)
            assert oc[b, 0] == len(ridx)
            assert np.array_equal(oi[b, 0, : oc[b, 0]], ridx), (b, k)
            assert pc[b, 0] == len(rpool)
            assert np.array_equal(pool[b, 0, : pc[b, 0]], rpool), (b, k)


def test_tied_boundary_split_across_cluster():
    """Equal block maxima on the pool boundary held by three CTAs of a row's
    cluster and taken in part (the first `remaining` of them by position),
    with the blocks above the boundary held by a fourth CTA.  Every CTA must
    agree on every CTA's share: the pool slots of the first CTA are filled
    from its peers' selections, and the top-k that follows (all its keys in
    one tie as well) is split the same way."""
    nb = 11164
    wl = Workload("split-ties", 1, [nb * 8], 128, 32, 4, 32, 16, 2048, 16, seed=23)
    dw = DeviceWorkload(wl)
    rng = np.random.default_rng(23)
    hi, di = wl.idx_heads, wl.idx_dim
    q = F.e4m3_encode(rng.standard_normal((1, 1, hi, di)).astype(np.float32))
    w = rng.random((1, 1, hi)).astype(np.float32)
    cand = F.e4m3_encode(rng.standard_normal((16, di)).astype(np.float32))
    sc = O.indexer_scores(q[0, 0], w[0, 0], cand)
    order = np.argsort(-sc, kind="stable")
    top, mid, low = cand[order[0]], cand[order[8]], cand[order[15]]
    s_top, s_mid, s_low = sc[order[0]], sc[order[8]], sc[order[15]]
    assert s_top > s_mid * 1.01 and s_mid > 0 and s_mid > s_low * 1.01 + 1e-6
    blk = np.full(nb, 2)                 # below the boundary
    blk[0:50] = 1                        # on the boundary: 50 + 50 + 3000 blocks,
    blk[3072:3122] = 1                   # of which the first 100 are taken
    blk[6144:9144] = 1
    blk[9216:] = 0                       # above the boundary: 1948 blocks
    rows = np.stack([top, mid, low])[np.repeat(blk, 8)]
    write_idx_rows(dw, 0, rows)
    torch.cuda.synchronize()
    s = O.indexer_scores(q[0, 0], w[0, 0], rows)
    for k in (1, 1024, 2048):
        oi, oc, pool, pc = run_index(dw, q, w, k)
        ridx, rpool = O.full_select(s, k)
        assert pc[0, 0] == len(rpool) == K.POOL_BLOCKS
        assert np.array_equal(pool[0, 0, : pc[0, 0]], rpool), k
        assert oc[0, 0] == len(ridx)
        assert np.array_equal(oi[0, 0, : oc[0, 0]], ridx), k


def test_two_level_pool_long_sequence():
    n = 1_300_000  # more blocks than one selection holds, and more groups of 8
    wl = Workload("long", 1, [n], 128, 32, 4, 32, 16, 2048, 16, seed=22)
    dw = DeviceWorkload(wl, chunk_rows=1 << 18)
    rng = np.random.default_rng(22)
    q = F.e4m3_encode(rng.standard_normal((1, 1, 4, 32)).astype(np.float32))
    w = rng.random((1, 1, 4)).astype(np.float32)
    oi, oc, pool, pc = run_index(dw, q, w, 2048)
    from oracle.workload import SeqRef
    ref = SeqRef(wl, 0)
    s = O.indexer_scores(q[0, 0], w[0, 0], ref.idxk_all(n))
    ridx, rpool = O.full_select(s, 2048)
    from checks import check_select
    check_select(oi[0, 0, : oc[0, 0]], s, np.arange(n), 2048, "topk two-level")
    bm = O.block_maxima(s)
    check_select(pool[0, 0, : pc[0, 0]], bm, np.arange(len(bm)), 2048, "pool two-level")
