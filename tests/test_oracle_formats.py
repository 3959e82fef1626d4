"""Pins of the oracle's element formats (E2M1, E4M3) against closed forms,
exhaustive brute force in exact rational arithmetic, and torch's own E4M3
dtype.  CPU only."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import formats as F


def e2m1_closed_form(code):
    s = -1 if code & 8 else 1
    e = (code >> 1) & 3
    m = code & 1
    mag = Fraction(m, 2) if e == 0 else Fraction(2) ** (e - 1) * (1 + Fraction(m, 2))
    return s * mag


def e4m3_closed_form(code):
    s = -1 if code & 0x80 else 1
    e = (code >> 3) & 0xF
    m = code & 7
    if (code & 0x7F) == 0x7F:
        return None
    mag = Fraction(m, 8) * Fraction(1, 64) if e == 0 else Fraction(2) ** (e - 7) * (1 + Fraction(m, 8))
    return s * mag


def test_e2m1_decode_all_codes():
    got = F.e2m1_decode(np.arange(16))
    for c in range(16):
        assert Fraction(got[c]) == e2m1_closed_form(c), c
    # the eight magnitudes of the OCP MX E2M1 element type
    assert sorted(set(abs(x) for x in got)) == [0, 0.5, 1, 1.5, 2, 3, 4, 6]


def test_e4m3_decode_all_codes_closed_form_and_torch():
    got = F.e4m3_decode(np.arange(256))
    ref_t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        cf = e4m3_closed_form(c)
        if cf is None:
            assert np.isnan(got[c]) and np.isnan(ref_t[c])
        else:
            assert Fraction(got[c]) == cf, c
            assert got[c] == ref_t[c], c
    assert np.nanmax(got) == 448.0 and np.nanmin(got) == -448.0


def _brute_nearest(x, codes, decode):
    """Exact nearest finite code with ties to the even code; saturating."""
    xf = Fraction(float(x))
    best = None
    for c in codes:
        v = decode(c)
        if v is None:
            continue
        d = abs(xf - v)
        key = (d, c % 2)  # smaller distance, then even code
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def test_e2m1_encode_brute_force_midpoints_and_neighbours():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    vals = []
    for m in mids + [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 7.0, 1e9]:
        f = np.float32(m)
        vals += [f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(np.inf))]
    vals = np.array(vals + [-v for v in vals], dtype=np.float32)
    got = F.e2m1_encode(vals)
    for x, g in zip(vals, got):
        mag = _brute_nearest(abs(x), range(8), lambda c: e2m1_closed_form(c))
        exp = mag | (8 if np.signbit(x) else 0)
        assert g == exp, (x, g, exp)
    # the midpoint rule spelled out: ties go to the even code
    table = {0.25: 0, 0.75: 2, 1.25: 2, 1.75: 4, 2.5: 4, 3.5: 6, 5.0: 6, 7.0: 7}
    for x, c in table.items():
        assert F.e2m1_encode(np.float32(x)) == c


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2 ** 32, size=400000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= 464.0)]
    # every midpoint between neighbouring finite codes and its two neighbours
    fin = F.e4m3_decode(np.arange(0x7F))
    mids = ((fin[:-1] + fin[1:]) / 2).astype(np.float32)
    extra = np.concatenate([mids, np.nextafter(mids, np.float32(0)),
                            np.nextafter(mids, np.float32(np.inf)), fin.astype(np.float32)])
    x = np.concatenate([x, extra, -extra]).astype(np.float32)
    got = F.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(got != ref)[0]
    assert len(bad) == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_e4m3_encode_brute_force_sample():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(300) * np.exp2(rng.integers(-12, 10, 300))).astype(np.float32)
    got = F.e4m3_encode(x)
    for xi, g in zip(x, got):
        mag = _brute_nearest(abs(xi), range(0x7F), lambda c: e4m3_closed_form(c))
        assert g == (mag | (0x80 if np.signbit(xi) else 0)), xi


def test_round_trip_and_saturation():
    c4 = np.arange(16)
    assert np.array_equal(F.e2m1_encode(F.e2m1_decode(c4).astype(np.float32)) & 0xF, c4 & 0xF)
    # -0.0 keeps the sign bit
    assert F.e2m1_encode(np.float32(-0.0)) == 8
    c8 = np.array([c for c in range(256) if (c & 0x7F) != 0x7F])
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(c8).astype(np.float32)), c8)
    assert F.e4m3_encode(np.float32(1e30)) == 0x7E
    assert F.e4m3_encode(np.float32(-1e30)) == 0xFE
    assert F.e4m3_encode(np.float32(470.0)) == 0x7E   # beyond the top midpoint
    assert F.e2m1_encode(np.float32(100.0)) == 7
    assert F.e2m1_encode(np.float32(-100.0)) == 15


def test_encoders_monotone():
    x = np.linspace(-500, 500, 200001, dtype=np.float32)
    v = F.e4m3_decode(F.e4m3_encode(x))
    assert np.all(np.diff(v) >= 0)
    x = np.linspace(-8, 8, 20001, dtype=np.float32)
    v = F.e2m1_decode(F.e2m1_encode(x))
    assert np.all(np.diff(v) >= 0)


def test_bf16_bits():
    x = torch.randn(1000).to(torch.bfloat16)
    got = F.bf16_bits_to_f64(x.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(got, x.double().numpy())
