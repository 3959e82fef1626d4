"""Pins of the oracle's m = 2 pair compression (CPU only).

Reading pinned here: a compressed entry is the per-channel softmax-weighted
sum of its two source rows, weights from the compression logits Z
("DeepSeek-V4.1-Flash" knowledge note, symbol table and "Causal
Encoder-Decoder"; "Inside DeepSeek V4.1 Flash", "CSA2: reuse memory and reuse
selection independently").  Expectations come from fp64 and exact arithmetic,
closed forms and symmetries, never from the oracle's own formula.
"""
import math

import numpy as np

import synth
from oracle import csa2 as O


def ulps(got, ref):
    ref32 = np.asarray(ref, dtype=np.float64).astype(np.float32)
    return np.abs(np.asarray(got, dtype=np.float64) - np.asarray(ref, dtype=np.float64)) / \
        np.spacing(np.abs(ref32)).astype(np.float64)


def test_exponential_within_a_few_ulp():
    x = np.concatenate([np.linspace(-80, 0, 400001), -np.logspace(-30, 1.9, 20001)]).astype(np.float32)
    got = O.exp_neg_f32(x)
    assert ulps(got, np.exp(x.astype(np.float64))).max() <= 4.0
    assert O.exp_neg_f32(np.float32(0.0)) == 1.0
    assert O.exp_neg_f32(np.float32(-80.5)) == 0.0
    # the range-reduction constants are ln 2 split exactly
    assert float(O.LN2_HI) * 4096 == 2839.0
    assert abs(float(O.LN2_HI) + float(O.LN2_LO) - math.log(2.0)) <= float(np.spacing(O.LN2_LO)) / 2


def test_equal_logits_give_the_exact_mean():
    x = synth.normal_block(31, 1, (2, 576))
    z = np.full((2, 576), 0.375, dtype=np.float32)
    c = O.compress_pairs(x, z)
    assert np.array_equal(c[0], (x[0].astype(np.float64) * 0.5 + x[1].astype(np.float64) * 0.5)
                          .astype(np.float32))


def test_weights_match_fp64_softmax_and_sum_to_one():
    rng = np.random.default_rng(5)
    z0 = (rng.standard_normal(100000) * 6).astype(np.float32)
    z1 = (rng.standard_normal(100000) * 6).astype(np.float32)
    w0, w1 = O.pair_weights(z0, z1)
    a, b = z0.astype(np.float64), z1.astype(np.float64)
    m = np.maximum(a, b)
    r0 = np.exp(a - m) / (np.exp(a - m) + np.exp(b - m))
    r1 = 1.0 - r0
    # d = z1 - z0 is rounded once in fp32: allow that on top of a few ulp
    d_err = np.abs((z1 - z0).astype(np.float64) - (b - a))
    assert np.all(np.abs(w0 - r0) <= 4 * np.spacing(np.float32(1.0)) + d_err)
    assert np.all(np.abs(w1 - r1) <= 4 * np.spacing(np.float32(1.0)) + d_err)
    s = w0.astype(np.float64) + w1.astype(np.float64)
    assert np.all(np.abs(s - 1.0) <= 2 * np.spacing(np.float32(1.0)))


def test_swapping_the_pair_swaps_the_weights():
    rng = np.random.default_rng(6)
    x = synth.normal_block(31, 2, (2, 4096))
    z = (rng.standard_normal((2, 4096)) * 3).astype(np.float32)
    c = O.compress_pairs(x, z)
    c_sw = O.compress_pairs(x[::-1].copy(), z[::-1].copy())
    assert np.array_equal(c, c_sw)


def test_far_apart_logits_select_one_row():
    x = synth.normal_block(31, 3, (4, 64))
    z = np.zeros((4, 64), dtype=np.float32)
    z[1] = 200.0                    # pair 0: row 1 wins outright
    z[2] = 90.0                     # pair 1: row 2 wins (e^-90 is below the cut)
    c = O.compress_pairs(x, z)
    assert np.array_equal(c[0], x[1]) and np.array_equal(c[1], x[2])


def test_compressed_row_against_fp64_convex_combination():
    rng = np.random.default_rng(7)
    x = synth.normal_block(31, 4, (512, 128)) * np.float32(3.0)
    z = (rng.standard_normal((512, 128)) * 2).astype(np.float32)
    c = O.compress_pairs(x, z).astype(np.float64)
    a, b = z[0::2].astype(np.float64), z[1::2].astype(np.float64)
    p0 = 1.0 / (1.0 + np.exp(b - a))
    ref = p0 * x[0::2] + (1.0 - p0) * x[1::2]
    mag = np.abs(x[0::2]).astype(np.float64) + np.abs(x[1::2])
    assert np.all(np.abs(c - ref) <= 1e-6 * mag + 1e-30)
    # a convex combination stays between its two rows
    lo = np.minimum(x[0::2], x[1::2]).astype(np.float64)
    hi = np.maximum(x[0::2], x[1::2]).astype(np.float64)
    assert np.all(c >= lo - 1e-6 * mag) and np.all(c <= hi + 1e-6 * mag)
