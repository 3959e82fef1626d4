"""Pins of the oracle's MXFP4 indexer-key format and its scores (CPU only).

The format: E2M1 values with one E8M0 scale per 32 channels, 68 bytes per
128-channel key ("Inside DeepSeek V4.1 Flash: CED, CSA2 and the 890-Byte KV
Cache", sections "Reconstructing the 890-byte cache budget" and "How the
derived numbers were built").  The scale rule is the OCP Microscaling one:
2^(floor(log2 amax) - 2).  Each pin derives its expectation another way than
the oracle does (from fp32 bit fields, exact rationals, closed-form grids).
"""
import json
import os
from fractions import Fraction

import numpy as np

import synth
from oracle import csa2 as O
from oracle import formats as F

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "byte_model.json")))
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e8m0_codes_are_fp32_exponent_fields():
    codes = np.arange(1, 255)
    v = F.e8m0_decode(codes)
    bits = v.astype(np.float32).view(np.uint32)
    assert np.array_equal(bits >> 23, codes)          # sign 0, biased exponent = code
    assert np.array_equal(bits & 0x7FFFFF, np.zeros_like(codes))
    assert F.e8m0_decode(127) == 1.0
    assert F.e8m0_decode(0) == 2.0 ** -127
    assert np.isnan(F.e8m0_decode(255))


def test_entry_bytes_match_pages():
    assert F.mxfp4_entry_bytes(128) == GOLD["indexer_entry_bytes_mxfp4_128"]["value"]
    assert (F.fp4_entry_bytes(512) + F.mxfp4_entry_bytes(128)
            == GOLD["global_entry_bytes"]["value"])


def test_scale_code_from_fp32_bit_fields():
    x = synth.normal_block(21, 1, (64, 128)) * np.float32(3.7)
    x[3, :32] *= np.float32(1e-30)                    # small blocks
    x[5, 32:64] *= np.float32(1e30)                   # large blocks
    _, s = O.quantize_mxfp4(x)
    amax = np.abs(x.reshape(64, 4, 32)).max(axis=-1).astype(np.float32)
    biased = (amax.view(np.uint32) >> 23).astype(np.int64)  # floor(log2 amax) + 127
    assert np.array_equal(s.astype(np.int64), np.maximum(biased - 2, 0))


def test_grid_values_round_trip_exactly():
    rng = np.random.default_rng(3)
    n = 40
    k = rng.integers(-20, 20, size=(n, 4))
    mags = rng.choice(GRID, size=(n, 4, 32))
    mags[:, :, 7] = rng.choice([4.0, 6.0], size=(n, 4))   # a value in the top binade
    sign = rng.choice([-1.0, 1.0], size=(n, 4, 32))
    x = (sign * mags * np.exp2(k)[..., None]).reshape(n, 128).astype(np.float32)
    codes, s = O.quantize_mxfp4(x)
    assert np.array_equal(s.astype(np.int64), k + 127)
    assert np.array_equal(O.dequantize_mxfp4(codes, s, 128), x.astype(np.float64))


def test_saturation_between_six_and_eight_times_the_scale():
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 0] = 7.0
    x[0, 1] = -7.9
    x[0, 2] = 5.0                                     # tie between 4 and 6 -> even code (4)
    x[0, 3] = 0.25                                    # tie between 0 and 0.5 -> 0
    codes, s = O.quantize_mxfp4(x)
    assert s[0, 0] == 127                             # floor(log2 7.9) - 2 = 0
    v = O.dequantize_mxfp4(codes, s, 128)[0]
    assert v[0] == 6.0 and v[1] == -6.0 and v[2] == 4.0 and v[3] == 0.0


def test_packing_low_nibble_first():
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 0], x[0, 1] = 1.0, -6.0                       # amax 6 -> scale 1
    codes, s = O.quantize_mxfp4(x)
    assert s[0, 0] == 127
    assert codes[0, 0] == (0x2 | (0xF << 4))


def test_zero_and_tiny_blocks():
    x = np.zeros((2, 128), dtype=np.float32)
    x[0, 40] = -0.0
    x[1, :32] = np.float32(1e-40)                     # fp32 subnormal
    codes, s = O.quantize_mxfp4(x)
    assert s[0].tolist() == [0, 0, 0, 0]
    assert s[1, 0] == 0
    assert np.all(O.dequantize_mxfp4(codes, s, 128) == 0.0)
    # the sign bit of -0.0 is copied into its nibble (channel 40 = low nibble of byte 20)
    assert codes[0, 20] == 0x08


def test_error_bound_of_the_grid():
    x = synth.normal_block(22, 2, (256, 128)) * np.float32(5.0)
    codes, s = O.quantize_mxfp4(x)
    v = O.dequantize_mxfp4(codes, s, 128)
    scale = np.repeat(F.e8m0_decode(s), 32, axis=1)
    y = np.abs(x.astype(np.float64)) / scale          # in units of the scale
    half_step = np.where(y <= 2.0, 0.25, np.where(y <= 4.0, 0.5, 1.0))
    bound = np.where(y > 6.0, y - 6.0, half_step) * scale
    assert np.all(np.abs(v - x) <= bound)
    assert np.all(y < 8.0)                            # the rule never needs more than 8x


def _rational_key(codes_row, scales_row):
    """Exact key values: E2M1 magnitude table and a 2^(code-127) per block, as Fractions."""
    out = []
    for c in range(128):
        nib = (int(codes_row[c // 2]) >> (4 * (c % 2))) & 0xF
        mag = Fraction(GRID[nib & 7]).limit_denominator(2)
        val = -mag if nib & 8 else mag
        e = int(scales_row[c // 32]) - 127
        out.append(val * (Fraction(2) ** e))
    return out


def test_scores_one_head_equal_exact_relu_dot():
    x = synth.normal_block(23, 3, (12, 128))
    x[:, 32:64] *= np.float32(1000.0)                 # blocks at different scales
    x[:, 96:] *= np.float32(0.001)
    codes, s = O.quantize_mxfp4(x)
    q = synth.normal_block(23, 4, (1, 128))
    qc = O.fp8_cast(q)
    got = O.indexer_scores_values(F.e4m3_decode(qc).reshape(1, 128), np.array([1.0]),
                                  O.dequantize_mxfp4(codes, s, 128))
    qv = [Fraction(float(v)) for v in F.e4m3_decode(qc).ravel()]
    for t in range(12):
        kv = _rational_key(codes[t], s[t])
        dot = sum(a * b for a, b in zip(qv, kv))
        mag = float(sum(abs(a * b) for a, b in zip(qv, kv)))
        # every product is exact in fp64; only the 128-term fp64 sum rounds
        assert abs(got[t] - float(max(dot, Fraction(0)))) <= 128 * 2.0 ** -53 * mag


def test_scores_heads_and_weights():
    x = synth.normal_block(24, 5, (20, 128))
    codes, s = O.quantize_mxfp4(x)
    k = O.dequantize_mxfp4(codes, s, 128)
    q = F.e4m3_decode(O.fp8_cast(synth.normal_block(24, 6, (4, 128))))
    w = np.array([0.5, -1.25, 2.0, 0.0])
    got = O.indexer_scores_values(q.reshape(4, 128), w, k)
    for t in range(20):
        ref = sum(float(w[h]) * max(0.0, float(np.dot(q.reshape(4, 128)[h], k[t])))
                  for h in range(4))
        assert abs(got[t] - ref) <= 1e-12 * max(1.0, abs(ref))
