"""CPU checks of the C-ABI library: it builds, loads without a GPU, exports
every function include/csa2.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    path = g._builder().build(verbose=False)
    return ctypes.CDLL(path)


def declared_functions():
    text = open(os.path.join(ROOT, "include", "csa2.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    import fp4_kv_cache_rope_gb300 as K
    assert sorted(K.EXPORTED) == names


def test_host_validation_without_gpu(lib):
    import fp4_kv_cache_rope_gb300 as K
    c = K.Csa2Cache()
    assert K.workspace_size(c, 1, 64) == 0                 # all-zero description
    c = K.Csa2Cache(2, 576, 64, 128, 0, 0, 1024, 0, 16, 288, 32, 48, 48, 128, None, 64, 80, 96)
    assert K.workspace_size(c, 2, 64) > 0
    assert K.workspace_size(c, 2, 65) == 0                 # more than 64 heads
    bad = K.Csa2Cache.from_buffer_copy(c)
    bad.dim = 100                                          # not a multiple of 64
    assert K.workspace_size(bad, 2, 64) == 0
    bad = K.Csa2Cache.from_buffer_copy(c)
    bad.scale_stride = 40                                  # < round_up(36, 16)
    assert K.workspace_size(bad, 2, 64) == 0
    bad = K.Csa2Cache.from_buffer_copy(c)
    bad.page_size = 24                                     # divides neither way into 128
    assert K.workspace_size(bad, 2, 64) == 0
    # null pointers and out-of-range k are rejected before any launch
    r = K._index_full(ctypes.byref(c), None, None, 64, 1, None, None, 2, 64, None, None, None,
                      None, None, None)
    assert r == K.CSA2_ERR_INVALID
    r = K._index_full(ctypes.byref(c), 16, 16, 64, 1, None, None, 2, 4096, 16, 16, None, None,
                      16, None)
    assert r == K.CSA2_ERR_INVALID
    r = K._attn_decode(ctypes.byref(c), 16, 65, 16, 16, 64, 16, None, 128, 0.0, 16, 16, None)
    assert r == K.CSA2_ERR_INVALID
    # the layer-grouped attention: 1..MAX_ATTN_LAYERS layers, every pointer given
    P = ctypes.c_void_p * 9
    ptrs = P(*([16] * 9))
    for n in (0, K.MAX_ATTN_LAYERS + 1):
        r = K._attn_decode_layers(ctypes.byref(c), n, ptrs, 64, 16, 16, 64, ptrs, None, 128, 0.0,
                                  ptrs, 16, None)
        assert r == K.CSA2_ERR_INVALID
    holes = P(16, None, *([16] * 7))
    r = K._attn_decode_layers(ctypes.byref(c), 2, holes, 64, 16, 16, 64, ptrs, None, 128, 0.0,
                              ptrs, 16, None)
    assert r == K.CSA2_ERR_INVALID
    r = K._attn_decode_layers(ctypes.byref(c), 2, ptrs, 64, 16, 16, 64, ptrs, None, 128, 0.0,
                              holes, 16, None)
    assert r == K.CSA2_ERR_INVALID
    # layers x rows beyond the grid's y extent (65,535) is refused on the host
    big = K.Csa2Cache.from_buffer_copy(c)
    big.batch = 16384
    r = K._attn_decode_layers(ctypes.byref(big), 4, ptrs, 64, 16, 16, 64, ptrs, None, 128, 0.0,
                              ptrs, 16, None)
    assert r == K.CSA2_ERR_INVALID
    assert K.entry_bytes(512) == 288 and K.entry_bytes(576) == 324
    assert K.status_string(K.CSA2_ERR_INVALID) == "invalid argument"


def test_cache_struct_layout_matches_header(tmp_path):
    """The ctypes description and the C struct agree field by field (gcc)."""
    import shutil
    import subprocess
    import fp4_kv_cache_rope_gb300 as K
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    names = [f[0] for f in K.Csa2Cache._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "csa2.h"\nint main(void){\n'
                   + "".join(f'printf("%zu\\n", offsetof(csa2_cache, {n}));\n' for n in names)
                   + 'printf("%zu\\n", sizeof(csa2_cache));\nreturn 0;}\n')
    exe = tmp_path / "layout"
    subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], check=True, capture_output=True,
                                          text=True).stdout.split()]
    want = [getattr(K.Csa2Cache, n).offset for n in names] + [ctypes.sizeof(K.Csa2Cache)]
    assert got == want


def test_mxfp4_key_description_checks(lib):
    import fp4_kv_cache_rope_gb300 as K
    base = K.Csa2Cache(2, 576, 64, 128, 0, 0, 1024, 0, 256, 288, 512, 48, 1024, 64, None, 64,
                       80, 96, K.IDX_MXFP4, 2048, 4)
    assert K.workspace_size(base, 2, 64) > 0
    for field, value in [("idx_dim", 64),            # MXFP4 keys are 128 channels
                         ("idxk_stride", 48),        # not a multiple of 32
                         ("idx_k", 1024 + 16),       # not 32-byte aligned
                         ("idx_scales", None),
                         ("idx_scales", 2048 + 4),   # not 16-byte aligned
                         ("idx_scale_stride", 8),
                         ("max_len", 1022),          # contiguous rows need max_len % 4 == 0
                         ("idx_format", 2)]:
        bad = K.Csa2Cache.from_buffer_copy(base)
        setattr(bad, field, value)
        assert K.workspace_size(bad, 2, 64) == 0, field
