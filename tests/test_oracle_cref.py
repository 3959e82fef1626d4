"""The C++ restatement of the oracle (oracle/cref.cpp) pinned against the
numpy oracle (oracle/csa2.py, itself pinned by the other test_oracle_*
files) on seeded inputs: bit for bit where the definition decides bytes or
ids (FP4 codes and scales, E4M3 decoding, block maxima, top-k and the pool),
within fp64 rounding where the summation order is free (indexer scores,
attention).  CPU only."""
import numpy as np
import pytest

from oracle import cref as C
from oracle import csa2 as O
from oracle import formats as F


@pytest.fixture(scope="module", autouse=True)
def built():
    C.build()


def finite_e4m3_codes(rng, shape):
    c = rng.integers(0, 256, size=shape).astype(np.uint8)
    return np.where((c & 0x7F) == 0x7F, c ^ 0x01, c).astype(np.uint8)   # no NaN codes


def edge_rows(rng, n, d):
    """Rows whose 16-channel groups reach the FP4 format's corners: zero and
    -0 groups, scales at every binade incl. E4M3 subnormals and saturation,
    values on and one ulp around every E2M1 rounding midpoint."""
    rows = (rng.standard_normal((n, d)) * 3).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    for r in range(n):
        for g in range(d // 16):
            kind = (r * 7 + g) % 6
            s = np.float32(2.0 ** rng.integers(-12, 10)) * np.float32(rng.choice([1.0, 1.125, 1.875]))
            if kind == 0:
                v = np.zeros(16, np.float32) * (-1 if r % 2 else 1)
            elif kind == 1:                                  # midpoints, nudged
                m = mids[rng.integers(0, 7, 14)] * s
                m = np.where(rng.random(14) < 0.3, np.nextafter(m, np.float32(np.inf)), m)
                m = np.where(rng.random(14) < 0.3, np.nextafter(m, np.float32(0)), m)
                v = np.concatenate([[6 * s, -6 * s], m]).astype(np.float32)
            elif kind == 2:                                  # saturating scales
                v = (rng.uniform(-1, 1, 16) * np.float32(3000.0)).astype(np.float32)
            elif kind == 3:                                  # subnormal E4M3 scales
                v = (rng.uniform(-1, 1, 16) * np.float32(6 * 2.0 ** -8)).astype(np.float32)
            else:
                continue
            rows[r, 16 * g:16 * g + 16] = v
    return rows


def test_hardware_threads():
    assert C.threads() >= 1


def test_quant_append_rows_bit_exact():
    rng = np.random.default_rng(5)
    n, d, r = 96, 576, 64
    kv = edge_rows(rng, n, d)
    pos = rng.integers(0, 4096, n)
    ang = rng.uniform(-np.pi, np.pi, (4096, r // 2))
    cos, sin = np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)
    c1, s1 = C.quant_append_rows(kv, pos, cos, sin, r)
    c0, s0 = O.quant_append_rows(kv, pos, cos, sin, r)
    assert np.array_equal(c1, c0) and np.array_equal(s1, s0)
    assert (s0 == 0x7E).any() and (s0 == 0).any() and ((s0 > 0) & (s0 < 8)).any()
    c1, s1 = C.quant_append_rows(kv, pos, cos, sin, 0)           # no RoPE slice
    c0, s0 = O.quant_append_rows(kv, pos, cos, sin, 0)
    assert np.array_equal(c1, c0) and np.array_equal(s1, s0)


def test_encoders_on_bit_patterns():
    """The C++ encoders equal the numpy ones on every fp32 bit pattern of a
    few dense ranges (around 0, the E2M1 midpoints, the E4M3 subnormal and
    saturation edges) and on random patterns; NaN patterns give 0xFF."""
    rng = np.random.default_rng(11)
    starts = [0, 0x80000000, 0x3E800000 - 4096, 0x3F400000 - 4096, 0x40A00000 - 4096,
              0x3B000000 - 4096, 0x43E00000 - 4096, 0x7F800000 - 4096]
    for first in starts:
        e2, e4 = C.encode_range(first, 8192)
        x = (np.arange(first, first + 8192, dtype=np.uint64) & 0xFFFFFFFF).astype(
            np.uint32).view(np.float32)
        ok = ~np.isnan(x)
        assert np.array_equal(e2[ok], F.e2m1_encode(x[ok]))
        assert np.array_equal(e4[ok], F.e4m3_encode(x[ok]))
        assert np.all(e2[~ok] == 0xFF) and np.all(e4[~ok] == 0xFF)
    bits = rng.integers(0, 2 ** 32, 20000, dtype=np.uint64)
    for b in bits[:200]:
        e2, e4 = C.encode_range(int(b), 1)
        x = np.array([int(b)], np.uint32).view(np.float32)
        if not np.isnan(x[0]):
            assert e2[0] == F.e2m1_encode(x)[0] and e4[0] == F.e4m3_encode(x)[0]


def test_compress_pairs_bit_exact():
    """The m = 2 pair combination, logits at the exponential's edges
    (equal, +-0 apart, tiny, around the -80 cut, huge) and random."""
    rng = np.random.default_rng(13)
    t, d = 64, 576
    x = (rng.standard_normal((2 * t, d)) * 3).astype(np.float32)
    z0 = (rng.standard_normal((t, d)) * 4).astype(np.float32)
    diffs = np.array([0.0, -0.0, 1e-7, -1e-7, 1e-3, 79.9, 80.0, 80.1, -80.2, 200.0, -1e30, 0.5],
                     np.float32)
    dd = diffs[rng.integers(0, len(diffs), (t, d))]
    dd[:8] = (rng.standard_normal((8, d)) * 10).astype(np.float32)
    z = np.empty((2 * t, d), np.float32)
    z[0::2], z[1::2] = z0, (z0 + dd).astype(np.float32)
    assert np.array_equal(C.compress_pairs(x, z), O.compress_pairs(x, z))


def test_e4m3_decode_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    assert np.array_equal(C.e4m3_decode(codes), F.e4m3_decode(codes), equal_nan=True)


@pytest.mark.parametrize("hi,di,n", [(1, 128, 777), (64, 128, 5000), (8, 64, 1031)])
def test_indexer_scores(hi, di, n):
    rng = np.random.default_rng(hi * 1000 + n)
    q = finite_e4m3_codes(rng, hi * di)
    k = finite_e4m3_codes(rng, (n, di))
    w = rng.standard_normal(hi).astype(np.float32)
    s0 = O.indexer_scores(q, w, k)
    s1 = C.indexer_scores(q, w, k)
    # the head sum may round in any order: both lie within the summation
    # bound hi * eps * sum_h |w_h relu(q_h . k_t)| of the exact value
    dots = F.e4m3_decode(k).reshape(n, di) @ F.e4m3_decode(q).reshape(hi, di).T
    mag = np.maximum(dots, 0.0) @ np.abs(w.astype(np.float64))
    assert np.all(np.abs(s1 - s0) <= 2 * hi * np.finfo(np.float64).eps * mag)
    if hi == 1:     # one head, w = 1: max(0, q.k), whose fp64 sum is exact in any order
        w1 = np.ones(1, np.float32)
        assert np.array_equal(C.indexer_scores(q, w1, k), O.indexer_scores(q, w1, k))
    # the split over threads changes nothing
    assert np.array_equal(C.indexer_scores(q, w, k, nthreads=1), s1)


def test_indexer_scores_mxfp4():
    rng = np.random.default_rng(9)
    hi, di, n = 16, 128, 2000
    q = finite_e4m3_codes(rng, hi * di)
    w = rng.standard_normal(hi).astype(np.float32)
    x = (rng.standard_normal((n, di)) * np.exp2(rng.integers(-6, 6, (n, 1)))).astype(np.float32)
    codes, scales = O.quantize_mxfp4(x)
    s0 = O.indexer_scores_values(F.e4m3_decode(q).reshape(hi, di), w,
                                 O.dequantize_mxfp4(codes, scales, di))
    s1 = C.indexer_scores_mx(q, w, codes, scales, di)
    k = O.dequantize_mxfp4(codes, scales, di)
    dots = np.abs(k) @ np.abs(F.e4m3_decode(q).reshape(hi, di)).T
    mag = dots @ np.abs(w.astype(np.float64))
    assert np.all(np.abs(s1 - s0) <= 2 * (hi + di) * np.finfo(np.float64).eps * mag)


@pytest.mark.parametrize("n,k", [(1, 4), (37, 5), (1000, 64), (5003, 2048), (70000, 2048)])
def test_topk_block_maxima_and_pool(n, k):
    rng = np.random.default_rng(n)
    s = rng.integers(0, 50, n).astype(np.float64)        # many equal scores
    assert np.array_equal(C.topk(s, k), O.topk(s, k))
    assert np.array_equal(C.block_maxima(s), O.block_maxima(s))
    i1, p1 = C.full_select(s, k)
    i0, p0 = O.full_select(s, k)
    assert np.array_equal(i1, i0) and np.array_equal(p1, p0)
    ids = np.sort(rng.choice(10 * n, n, replace=False))  # explicit ids (pool positions)
    assert np.array_equal(C.topk(s, k, ids=ids), O.topk(s, k, ids=ids))


def test_dequantize_fp4():
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 256, (50, 288)).astype(np.uint8)
    scales = finite_e4m3_codes(rng, (50, 36))
    assert np.array_equal(C.dequantize_fp4(codes, scales, 576),
                          O.dequantize_fp4(codes, scales, 576))


@pytest.mark.parametrize("n", [0, 1, 300, 2176])
def test_sparse_attention(n):
    rng = np.random.default_rng(n + 1)
    h, d = 64, 576
    q = rng.standard_normal((h, d))
    rows = rng.standard_normal((n, d)) * 2
    o0 = O.sparse_attention(q, rows)
    o1 = C.sparse_attention(q, rows)
    assert np.allclose(o1, o0, rtol=1e-11, atol=1e-13)
    assert np.array_equal(C.sparse_attention(q, rows, nthreads=1), o1)
