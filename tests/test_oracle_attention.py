"""Pins of the oracle's dequantisation and sparse attention (CPU)."""
import math

import numpy as np

import synth
from oracle import csa2 as O
from oracle import formats as F


def naive_attention(q, rows, scale):
    """Two-pass softmax with Python loops: max, then exp-sum and weighted sum."""
    h, d = len(q), len(q[0])
    out = []
    for i in range(h):
        logits = [scale * sum(q[i][c] * r[c] for c in range(d)) for r in rows]
        m = max(logits)
        e = [math.exp(v - m) for v in logits]
        z = sum(e)
        out.append([sum(e[j] * rows[j][c] for j in range(len(rows))) / z for c in range(d)])
    return np.array(out)


def test_dense_equivalence_small():
    rng = np.random.default_rng(1)
    q = rng.standard_normal((3, 16))
    rows = rng.standard_normal((11, 16))
    got = O.sparse_attention(q, rows)
    ref = naive_attention(q.tolist(), rows.tolist(), 1 / 4)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_selecting_everything_equals_dense_over_cache_and_window():
    cos, sin = synth.rope_table(64, 8, 10000.0)
    kv = synth.normal_block(3, 1, (40, 32))
    codes, scales = O.quant_append_rows(kv, np.arange(40), cos, sin, 8)
    swa = O.fp8_cast(synth.normal_block(3, 2, (6, 32)))
    xh = O.dequantize_fp4(codes, scales, 32)
    q = synth.normal_block(3, 3, (4, 32)).astype(np.float64)
    idx, _ = O.full_select(np.random.default_rng(0).random(40), 100)   # k >= N: all rows
    rows = np.concatenate([xh[idx], O.swa_rows_decode(swa)])
    got = O.sparse_attention(q, rows)
    ref = naive_attention(q.tolist(), np.concatenate([xh, O.swa_rows_decode(swa)]).tolist(),
                          1 / math.sqrt(32))
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_single_row_equal_logits_and_shift():
    rng = np.random.default_rng(2)
    rows = rng.standard_normal((1, 8))
    q = rng.standard_normal((2, 8))
    assert np.allclose(O.sparse_attention(q, rows), np.repeat(rows, 2, 0), rtol=0, atol=1e-15)
    rows = rng.standard_normal((9, 8))
    assert np.allclose(O.sparse_attention(np.zeros((2, 8)), rows), rows.mean(0)[None].repeat(2, 0))
    # a constant channel adds the same amount to every logit: other channels
    # are unchanged and the constant channel comes out as the constant
    q = rng.standard_normal((3, 8))
    q2 = np.concatenate([q, np.full((3, 1), 5.0)], 1)
    rows2 = np.concatenate([rows, np.ones((9, 1))], 1)
    a = O.sparse_attention(q, rows, scale=0.3)
    b = O.sparse_attention(q2, rows2, scale=0.3)
    assert np.allclose(b[:, :8], a, rtol=1e-12) and np.allclose(b[:, 8], 1.0)
    assert np.array_equal(O.sparse_attention(q, np.zeros((0, 8))), np.zeros((3, 8)))


def test_union_softmax_is_log_sum_exp_merge():
    """One softmax over selected rows + window == merge of two partial softmaxes."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((5, 12))
    a, b = rng.standard_normal((7, 12)), rng.standard_normal((4, 12)) * 3
    sc = 0.4
    whole = O.sparse_attention(q, np.concatenate([a, b]), scale=sc)
    def part(rows):
        lg = sc * q @ rows.T
        m = lg.max(1, keepdims=True)
        p = np.exp(lg - m)
        return p @ rows, p.sum(1, keepdims=True), m
    oa, la, ma = part(a)
    ob, lb, mb = part(b)
    m = np.maximum(ma, mb)
    merged = (oa * np.exp(ma - m) + ob * np.exp(mb - m)) / (la * np.exp(ma - m) + lb * np.exp(mb - m))
    assert np.allclose(whole, merged, rtol=1e-12)
    # and it differs from averaging the two partial outputs
    assert not np.allclose(whole, (oa / la + ob / lb) / 2, rtol=1e-3)


def test_default_scale_is_inverse_sqrt_dim():
    rng = np.random.default_rng(4)
    q, rows = rng.standard_normal((2, 36)), rng.standard_normal((5, 36))
    assert np.allclose(O.sparse_attention(q, rows), O.sparse_attention(q, rows, 1 / 6))
    assert not np.allclose(O.sparse_attention(q, rows), O.sparse_attention(q, rows, 1 / 36))


def test_dequantize_matches_group_scaling():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, (3, 16), dtype=np.uint8)
    scales = F.e4m3_encode(rng.random((3, 2)).astype(np.float32) + 0.01)
    x = O.dequantize_fp4(codes, scales, 32)
    for r in range(3):
        for c in range(32):
            nib = (codes[r, c // 2] >> (4 * (c % 2))) & 0xF
            assert x[r, c] == F.e2m1_decode(nib) * F.e4m3_decode(scales[r, c // 16])


def test_prefill_swa_band_rows_brute_force():
    """The SWA band of a prefill chunk: row r holds position p0-(W-1)+r, and
    query tq (position p0+tq) must see exactly the positions q with
    0 <= q <= p0+tq and p0+tq-q < W.  Checked by walking every position,
    including chunks that start before W-1 (p0 < W-1: negative band rows)."""
    for W in (1, 2, 5, 16):
        for p0 in (0, 1, 3, W - 2, W - 1, W, 40):
            if p0 < 0:
                continue
            T = 7
            band_pos = [p0 - (W - 1) + r for r in range(T + W - 1)]
            for tq in range(T):
                p = p0 + tq
                want = [q for q in range(0, p + 1) if p - q < W]
                got = [band_pos[r] for r in O.swa_band_rows(p0, tq, W)]
                assert got == want, (W, p0, tq, got, want)
