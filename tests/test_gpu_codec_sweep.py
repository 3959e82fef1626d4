"""The hardware conversions the append kernels use (cvt.rn.satfinite
.e2m1x2.f32 and .e4m3x2.f32, through csrc/codec.cuh) equal the oracle's
E2M1 and E4M3 encoders (round to nearest, ties to the even code, saturating,
sign kept) on every fp32 bit pattern but the NaNs, in both lanes of the
packed result.  The oracle side is its C++ restatement (oracle/cref.cpp),
itself pinned against the numpy codecs in tests/test_oracle_cref.py."""
import ctypes
import os
import subprocess

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from oracle import cref as C  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))


def sweep_lib():
    out_dir = os.path.join(HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "libcodec_sweep.so")
    subprocess.run(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "cuda", "codec_sweep.cu"),
                    "-o", so], check=True)
    lib = ctypes.CDLL(so)
    lib.codec_sweep.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p,
                                ctypes.c_void_p]
    lib.codec_sweep.restype = ctypes.c_int
    return lib


def test_hardware_conversions_equal_the_oracle_on_every_fp32():
    lib = sweep_lib()
    C.build()
    chunk = 1 << 28
    e2d = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    e4d = torch.empty(chunk, dtype=torch.int16, device="cuda")
    checked = 0
    for first in range(0, 1 << 32, chunk):
        assert lib.codec_sweep(first, chunk, e2d.data_ptr(), e4d.data_ptr()) == 0
        torch.cuda.synchronize()
        g2 = e2d.cpu().numpy()
        g4 = e4d.cpu().numpy().view(np.uint16)
        o2, o4 = C.encode_range(first, chunk)
        nan = o2 == 0xFF
        assert np.array_equal(np.where(nan, 0xFF, g2 & 0xF), o2), hex(first)
        assert np.array_equal(np.where(nan, 0xFF, g2 >> 4), np.where(nan, 0xFF, o2 ^ 8)), hex(first)
        assert np.array_equal(np.where(nan, 0xFF, g4 & 0xFF), o4), hex(first)
        assert np.array_equal(np.where(nan, 0xFF, g4 >> 8), np.where(nan, 0xFF, o4 ^ 0x80)), \
            hex(first)
        checked += int((~nan).sum())
    assert checked == (1 << 32) - 2 * ((1 << 23) - 1)      # every non-NaN pattern
