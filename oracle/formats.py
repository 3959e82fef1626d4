"""Element formats of the FP4 main-KV cache and the FP8 operands (oracle side).

Formats named by the pages:

* main KV: E2M1 values with one E4M3 scale per 16 channels, no second global
  scale -- "DeepSeek-V4.1-Flash: Pushing the Limits of KV Cache Compression"
  (knowledge note), section "FP4 main KV: trade precision for bytes, not for a
  new GEMM"; "Inside DeepSeek V4.1 Flash: CED, CSA2 and the 890-Byte KV Cache",
  section "Reconstructing the 890-byte cache budget".
* SWA window and indexer operands: FP8 (E4M3), same sections.
* indexer key, MXFP4 form: E2M1 values with one E8M0 scale per 32 channels
  (128 x 4/8 + 128/32 = 68 bytes per entry) -- "Inside DeepSeek V4.1 Flash",
  sections "Reconstructing the 890-byte cache budget" and "How the derived
  numbers were built".

The bit layouts are those of the OCP 8-bit floating point specification
(E4M3 "FN": bias 7, no infinities, S.1111.111 is NaN, largest finite 448) and
of the OCP Microscaling specification (E2M1: bias 1, magnitudes
0, 0.5, 1, 1.5, 2, 3, 4, 6; E8M0: the power of two 2^(code - 127), code 255
is NaN).

Encoders are written as the definition of rounding: among all finite values
of the format pick the nearest one; on an exact tie pick the one whose code
is even; values beyond the largest finite magnitude give that magnitude
(saturation).  The sign bit is copied from the input, so -0.0 and negative
values that round to zero keep the sign bit.  Non-finite inputs are outside
the contract.
"""
from __future__ import annotations

import numpy as np

# E2M1 magnitudes indexed by the 3-bit magnitude code (exponent:mantissa).
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E4M3_MAX = 448.0
E2M1_MAX = 6.0


def e2m1_decode(codes) -> np.ndarray:
    """4-bit codes (0..15, sign in bit 3) -> float64 values."""
    c = np.asarray(codes, dtype=np.int64)
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c >> 3) & 1, -mag, mag)


def e4m3_magnitude(code7) -> np.ndarray:
    """Magnitude of a 7-bit E4M3 code (exponent 4 bits, mantissa 3 bits)."""
    c = np.asarray(code7, dtype=np.int64)
    e = (c >> 3) & 0xF
    m = c & 7
    sub = m.astype(np.float64) * 2.0 ** -9            # e == 0: m/8 * 2^(1-7)
    nor = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    return np.where(e == 0, sub, nor)


def e4m3_decode(codes) -> np.ndarray:
    """8-bit E4M3 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    c = np.asarray(codes, dtype=np.int64)
    mag = e4m3_magnitude(c & 0x7F)
    mag = np.where((c & 0x7F) == 0x7F, np.nan, mag)
    return np.where((c >> 7) & 1, -mag, mag)


# Sorted finite non-negative magnitudes and their codes (codes are monotone).
_E4M3_FINITE = e4m3_magnitude(np.arange(0x7F))      # codes 0..126


def _nearest_code(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of the increasing ``table``; ties -> even index.

    Magnitudes above the last entry map to the last index (saturation).
    """
    mag = np.asarray(mag, dtype=np.float64)
    hi = np.searchsorted(table, mag, side="left")      # first table >= mag
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_lo = np.abs(mag - table[lo])
    d_hi = np.abs(table[hi] - mag)
    pick = np.where(d_lo < d_hi, lo, hi)
    tie = d_lo == d_hi
    pick = np.where(tie, np.where(lo % 2 == 0, lo, hi), pick)
    pick = np.where(mag >= table[-1], len(table) - 1, pick)
    return pick.astype(np.int64)


def e2m1_encode(x) -> np.ndarray:
    """fp32 values -> 4-bit E2M1 codes (uint8 0..15), RNE, saturating."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x.astype(np.float64))
    code = _nearest_code(mag, E2M1_MAGNITUDES)
    sign = np.signbit(x).astype(np.int64)
    return (code | (sign << 3)).astype(np.uint8)


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> 8-bit E4M3 codes, RNE, saturating at +-448."""
    x = np.asarray(x, dtype=np.float32)
    mag = np.abs(x.astype(np.float64))
    code = _nearest_code(mag, _E4M3_FINITE)
    sign = np.signbit(x).astype(np.int64)
    return (code | (sign << 7)).astype(np.uint8)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def fp4_entry_bytes(dim: int, group: int = 16, scale_bytes: int = 1) -> int:
    """Algorithmic bytes of one FP4 cache entry: dim/2 codes + one scale per group."""
    return dim // 2 + (dim // group) * scale_bytes


E8M0_BIAS = 127


def e8m0_decode(codes) -> np.ndarray:
    """8-bit E8M0 scale codes -> float64 powers of two 2^(code - 127) (NaN for 255)."""
    c = np.asarray(codes, dtype=np.int64)
    v = np.ldexp(1.0, c - E8M0_BIAS)
    return np.where(c == 255, np.nan, v)


def mxfp4_entry_bytes(dim: int, block: int = 32) -> int:
    """Algorithmic bytes of one MXFP4 row: dim/2 codes + one E8M0 byte per block."""
    return dim // 2 + dim // block
