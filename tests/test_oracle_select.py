"""Pins of the oracle's indexer scores, top-k, block pool and Reindex (CPU)."""
import json
import os
from fractions import Fraction

import numpy as np

import synth
from oracle import csa2 as O
from oracle import formats as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "byte_model.json")))


def rand_e4m3(rng, shape):
    return F.e4m3_encode(rng.standard_normal(shape).astype(np.float32))


def exact_score(qc, w, kc):
    """sum_h w_h * max(0, q_h . k) in exact rational arithmetic."""
    hi, di = qc.shape
    s = Fraction(0)
    for h in range(hi):
        dot = sum(Fraction(float(F.e4m3_decode(qc[h, d]))) * Fraction(float(F.e4m3_decode(kc[d])))
                  for d in range(di))
        s += Fraction(float(w[h])) * max(dot, Fraction(0))
    return s


def test_indexer_one_head_is_relu_dot():
    rng = np.random.default_rng(1)
    q = rand_e4m3(rng, (1, 32))
    k = rand_e4m3(rng, (40, 32))
    s = O.indexer_scores(q, np.ones(1, dtype=np.float32), k)
    for t in range(40):
        assert Fraction(float(s[t])) == exact_score(q, np.ones(1), k[t])   # exact in fp64


def test_indexer_many_heads_brute_force():
    rng = np.random.default_rng(2)
    q = rand_e4m3(rng, (4, 16))
    w = rng.random(4).astype(np.float32)
    k = rand_e4m3(rng, (30, 16))
    s = O.indexer_scores(q, w, k)
    for t in range(30):
        ref = exact_score(q, w, k[t])
        assert abs(Fraction(float(s[t])) - ref) <= abs(ref) * Fraction(1, 2 ** 50)
    # weights are per head, not per channel: permuting heads with their
    # weights leaves scores unchanged, permuting weights alone does not
    perm = np.array([2, 0, 3, 1])
    assert np.allclose(O.indexer_scores(q[perm], w[perm], k), s, rtol=1e-15)
    assert not np.allclose(O.indexer_scores(q, w[perm], k), s, rtol=1e-6)


def test_topk_brute_force_with_ties():
    rng = np.random.default_rng(3)
    for n in (1, 7, 64, 500):
        s = rng.integers(0, 12, n).astype(np.float64)      # many exact ties
        for k in (1, 5, 64, 600):
            got = O.topk(s, k)
            ref = sorted(sorted(range(n), key=lambda t: (-s[t], t))[:k])
            assert got.tolist() == ref


def test_block_maxima_partial_block():
    s = np.arange(21, dtype=np.float64)[::-1].copy()
    bm = O.block_maxima(s)
    assert bm.tolist() == [20.0, 12.0, 4.0]
    assert O.block_maxima(np.array([3.0])).tolist() == [3.0]


def test_pool_brute_force_and_caps():
    rng = np.random.default_rng(4)
    n = 20000
    s = rng.integers(0, 5000, n).astype(np.float64)
    idx, pool = O.full_select(s, 2048)
    nb = -(-n // 8)
    bm = [max(s[8 * b:min(8 * b + 8, n)]) for b in range(nb)]
    ref = sorted(sorted(range(nb), key=lambda b: (-bm[b], b))[:2048])
    assert pool.tolist() == ref
    assert len(pool) == GOLD["pool_blocks"]["value"]
    assert len(O.pool_positions(pool, n)) <= GOLD["pool_positions_max"]["value"]
    assert GOLD["pool_blocks"]["value"] * GOLD["block_positions"]["value"] == \
        GOLD["pool_positions_max"]["value"]
    # short sequence: every block is in the pool
    idx2, pool2 = O.full_select(s[:100], 64)
    assert pool2.tolist() == list(range(13))


def test_topk_lies_inside_pool():
    """Top-k positions (k <= pool size) always lie inside the block pool: each
    of the pool's blocks holds a position at least as high as its block max."""
    rng = np.random.default_rng(5)
    for trial in range(20):
        n = int(rng.integers(1, 40000))
        s = rng.standard_normal(n) if trial % 2 else rng.integers(0, 50, n).astype(np.float64)
        k = int(rng.integers(1, 2049))
        idx, pool = O.full_select(s, k)
        assert set(idx.tolist()) <= set(O.pool_positions(pool, n).tolist())
        assert len(idx) == min(k, n)
        assert set(O.topk(s, k).tolist()) <= set(O.topk(s, k + 1).tolist())


def test_reindex_with_full_query_equals_full_when_pool_covers_all():
    rng = np.random.default_rng(6)
    n, hi, di = 2048, 4, 32
    q = rand_e4m3(rng, (hi, di))
    w = rng.random(hi).astype(np.float32)
    k = rand_e4m3(rng, (n, di))
    s = O.indexer_scores(q, w, k)
    idx, pool = O.full_select(s, 64)
    assert len(pool) == n // 8
    r = O.reindex_select(q, w, lambda pos: k[pos], pool, n, 64)
    assert r.tolist() == idx.tolist()


def test_reindex_stays_inside_pool():
    rng = np.random.default_rng(7)
    n, hi, di = 40000, 4, 32
    k = rand_e4m3(rng, (n, di))
    q1, q2 = rand_e4m3(rng, (hi, di)), rand_e4m3(rng, (hi, di))
    w = rng.random(hi).astype(np.float32)
    _, pool = O.full_select(O.indexer_scores(q1, w, k), 2048)
    r = O.reindex_select(q2, w, lambda pos: k[pos], pool, n, 512)
    pp = set(O.pool_positions(pool, n).tolist())
    assert set(r.tolist()) <= pp and len(r) == 512
    # brute force over the pool
    pos = np.array(sorted(pp))
    s2 = O.indexer_scores(q2, w, k[pos])
    ref = sorted(pos[sorted(range(len(pos)), key=lambda i: (-s2[i], pos[i]))[:512]].tolist())
    assert r.tolist() == ref


def test_scored_position_counts_of_the_pages():
    g = GOLD["decoder_indexer_positions_at_1m"]
    n, p = g["n"], g["pool"]
    # one Full scan over N plus four Reindex scans over the pool
    full_scan = len(O.block_maxima(np.zeros(n))) * O.BLOCK
    assert full_scan == n
    assert n + (g["indexers"] - 1) * p == g["value"]
    assert round(n / p) == GOLD["reindex_ratio_at_1m"]["value"]
    assert O.POOL_BLOCKS * O.BLOCK == p
