"""The append kernels' shortcut for E2M1(fl(y / s)), checked by brute force
in fp32 on the host (no GPU): the code of q' = fl(y * fl(1 / s)) equals the
code of the correctly rounded quotient fl(y / s) for every value the kernels'
boundary test lets through.  The test flags q' when its low 21 mantissa bits
are within 16 of a multiple of 2^21, i.e. q' within a few ulps of a value
with at most three significant bits, which includes every E2M1 rounding
boundary (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5); flagged groups take the
quotients.  Inputs: every E4M3 scale, values on and up to 40 ulps around
every boundary times the scale, and random values."""
import numpy as np

from oracle import formats as F


def flagged(qp):
    bits = qp.view(np.uint32).astype(np.uint64)
    return ((bits + 8) & 0x1FFFFF) <= 16


def test_product_code_equals_quotient_code_unless_flagged():
    rng = np.random.default_rng(17)
    codes = np.arange(1, 0x7F, dtype=np.uint8)                # every positive E4M3 scale
    s_all = F.e4m3_decode(codes).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 0.5, 1.0, 6.0], np.float32)
    s = np.repeat(s_all, len(mids) * 81)
    t = np.tile(np.repeat(mids, 81), len(s_all))
    base = (t * s).astype(np.float32).view(np.int32).astype(np.int64)
    off = np.tile(np.arange(-40, 41), len(s_all) * len(mids))
    y = (base + off).astype(np.int32).view(np.float32)
    y = np.concatenate([y, -y, (rng.standard_normal(200000) * 6).astype(np.float32)])
    s = np.concatenate([s, s, s_all[rng.integers(0, len(s_all), 200000)]])
    s = s * np.float32(1.0)
    exact = (y / s).astype(np.float32)                        # correctly rounded (IEEE)
    qp = (y * (np.float32(1.0) / s).astype(np.float32)).astype(np.float32)
    differ = F.e2m1_encode(exact) != F.e2m1_encode(qp)
    assert differ.any(), "the inputs never reach a boundary"
    assert not np.any(differ & ~flagged(qp))
