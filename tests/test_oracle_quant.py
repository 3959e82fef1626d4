"""Pins of the oracle's RoPE and FP4 quantisation step (CPU only)."""
import json
import math
import os
from fractions import Fraction

import numpy as np

import synth
from oracle import csa2 as O
from oracle import formats as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "byte_model.json")))


def test_rope_position_zero_is_identity_bitwise():
    cos, sin = synth.rope_table(16, 64, 10000.0)
    x = synth.normal_block(5, 1, (4, 576))
    y = O.rope_rotate(x, np.zeros(4, dtype=np.int64), cos, sin, 64)
    assert np.array_equal(y.view(np.uint32), x.view(np.uint32))


def test_rope_zero_dims_and_passthrough():
    cos, sin = synth.rope_table(100, 32, 10000.0)
    x = synth.normal_block(5, 2, (3, 128))
    pos = np.array([3, 50, 99])
    y = O.rope_rotate(x, pos, cos, sin, 32)
    assert np.array_equal(y[:, :96], x[:, :96])
    assert np.array_equal(O.rope_rotate(x, pos, cos, sin, 0), x)


def test_rope_pairs_rotate_like_complex_multiplication():
    R, D, n = 32, 128, 64
    cos, sin = synth.rope_table(5000, R, 10000.0)
    x = synth.normal_block(9, 3, (n, D))
    pos = np.arange(n) * 77
    y = O.rope_rotate(x, pos, cos, sin, R)
    z = (x[:, D - R::2].astype(np.float64) + 1j * x[:, D - R + 1::2].astype(np.float64))
    w = cos[pos].astype(np.float64) + 1j * sin[pos].astype(np.float64)
    ref = z * w
    err0 = np.abs(y[:, D - R::2] - ref.real)
    err1 = np.abs(y[:, D - R + 1::2] - ref.imag)
    scale = np.abs(z) * np.abs(w)
    assert np.all(err0 <= 4 * 2 ** -24 * scale + 1e-30)
    assert np.all(err1 <= 4 * 2 ** -24 * scale + 1e-30)


def test_rope_unit_vectors_and_norm():
    R, D = 8, 32
    cos, sin = synth.rope_table(64, R, 10000.0)
    for i in range(R // 2):
        x = np.zeros((1, D), dtype=np.float32)
        x[0, D - R + 2 * i] = 1.0
        y = O.rope_rotate(x, np.array([37]), cos, sin, R)
        assert y[0, D - R + 2 * i] == cos[37, i] and y[0, D - R + 2 * i + 1] == sin[37, i]
        others = np.delete(y[0], [D - R + 2 * i, D - R + 2 * i + 1])
        assert np.all(others == 0)
    x = synth.normal_block(1, 4, (50, D))
    y = O.rope_rotate(x, np.arange(50), cos, sin, R)
    nx = np.hypot(x[:, D - R::2].astype(np.float64), x[:, D - R + 1::2].astype(np.float64))
    ny = np.hypot(y[:, D - R::2].astype(np.float64), y[:, D - R + 1::2].astype(np.float64))
    assert np.allclose(nx, ny, rtol=4 * 2 ** -24, atol=0)


def test_rope_table_matches_closed_form():
    cos, sin = synth.rope_table(3000, 64, 10000.0)
    for p in (0, 1, 17, 2999):
        for i in (0, 5, 31):
            a = p * 10000.0 ** (-2.0 * i / 64)
            assert abs(cos[p, i] - math.cos(a)) <= 2 ** -24
            assert abs(sin[p, i] - math.sin(a)) <= 2 ** -24


def test_quant_zero_group_and_nibble_order():
    y = np.zeros((1, 32), dtype=np.float32)
    codes, scales = O.quantize_fp4(y)
    assert np.all(codes == 0) and np.all(scales == 0)
    y[0, 0] = 3.0       # element 0 -> low nibble of byte 0
    y[0, 17] = -6.0     # element 17 -> high nibble of byte 8, group 1
    codes, scales = O.quantize_fp4(y)
    assert codes[0, 0] & 0xF == 7 and codes[0, 0] >> 4 == 0     # 3.0 / 0.5 = 6 -> code 7
    assert codes[0, 8] >> 4 == 15 and codes[0, 8] & 0xF == 0    # -6 / 1 -> -6
    assert F.e4m3_decode(scales[0, :2]).tolist() == [0.5, 1.0]


def test_quant_power_of_two_groups_exact():
    for e in range(-6, 8):
        y = np.zeros((1, 16), dtype=np.float32)
        grid = np.array([6, -3, 1.5, 0.5, -4, 2] + [0] * 10, dtype=np.float32)
        y[0] = np.float32(2.0 ** e) * grid
        codes, scales = O.quantize_fp4(y)
        assert F.e4m3_decode(scales)[0, 0] == 2.0 ** e
        xh = O.dequantize_fp4(codes, scales, 16)
        assert np.array_equal(xh[0], y[0].astype(np.float64))


def test_quant_saturation():
    y = np.full((1, 16), 5000.0, dtype=np.float32)
    y[0, 1] = -3000.0
    y[0, 2] = 10.0
    codes, scales = O.quantize_fp4(y)
    assert scales[0, 0] == 0x7E                      # 448
    c = np.concatenate([codes[0] & 0xF, codes[0] >> 4])
    assert codes[0, 0] & 0xF == 7 and codes[0, 0] >> 4 == 15
    xh = O.dequantize_fp4(codes, scales, 16)
    assert xh[0, 0] == 2688.0 and xh[0, 1] == -2688.0
    assert xh[0, 2] == 0.0                            # 10/448 rounds to 0
    assert len(c) == 16


def test_quant_error_bound_and_sign():
    y = synth.normal_block(11, 1, (512, 576), chan_mult=synth.outlier_multipliers(1, 576, 0.01))
    codes, scales = O.quantize_fp4(y)
    xh = O.dequantize_fp4(codes, scales, 576)
    s = np.repeat(F.e4m3_decode(scales), 16, axis=1)
    q = np.abs(y.astype(np.float64)) / s
    h = np.where(q < 2, 0.25, np.where(q < 4, 0.5, 1.0))
    assert np.all(np.abs(y - xh) <= s * h)
    # negative values that round to zero keep the sign bit (code 8)
    nib = np.empty((512, 576), dtype=np.uint8)
    nib[:, 0::2] = codes & 0xF
    nib[:, 1::2] = codes >> 4
    tiny_neg = (y < 0) & (q <= 0.25)
    assert np.all(nib[tiny_neg] == 8)
    assert np.all(np.sign(xh[xh != 0]) == np.sign(y[xh != 0]))


def test_range_bound_never_saturates_scale():
    # normalised KV values stay below about 22.6 (= sqrt(512)); amax/6 is then
    # far inside E4M3, so no second global scale is needed
    bound = GOLD["normalised_range_bound"]["value"]
    assert abs(bound - math.sqrt(512)) < 0.05
    y = np.linspace(-bound, bound, 16 * 100, dtype=np.float32).reshape(100, 16)
    _, scales = O.quantize_fp4(y)
    assert np.all(scales < 0x7E) and F.e4m3_decode(scales).max() <= bound / 6 * 1.07


def test_byte_model_matches_pages():
    assert F.fp4_entry_bytes(512) == GOLD["main_kv_entry_bytes_512"]["value"]
    assert F.fp4_entry_bytes(128, group=32) == GOLD["indexer_entry_bytes_mxfp4_128"]["value"]
    ent = F.fp4_entry_bytes(512) + F.fp4_entry_bytes(128, group=32)
    assert ent == GOLD["global_entry_bytes"]["value"]
    per_tok = Fraction(3, 2) * ent + 1 * ent
    assert per_tok == GOLD["entries_per_token"]["value"] * ent == GOLD["bytes_per_token"]["value"]
    total = per_tok * 10 ** 6
    assert total / 10 ** 6 == GOLD["bytes_at_1m_tokens_decimal_mb"]["value"]
    assert round(total / 2 ** 20) == GOLD["bytes_at_1m_tokens_mib_approx"]["value"]
    assert F.fp4_entry_bytes(576) == 324 and F.fp4_entry_bytes(128) == 72


def test_quant_append_rows_composes():
    cos, sin = synth.rope_table(100, 64, 10000.0)
    x = synth.normal_block(2, 1, (8, 576))
    pos = np.arange(8) + 40
    a = O.quant_append_rows(x, pos, cos, sin, 64)
    b = O.quantize_fp4(O.rope_rotate(x, pos, cos, sin, 64))
    assert all(np.array_equal(u, v) for u, v in zip(a, b))
