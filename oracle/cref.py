"""The C++ restatement of the oracle (``oracle/cref.cpp``), through ctypes.

Test infrastructure, like the rest of ``oracle/``: only the tests, the smoke
check and the bench's CPU-baseline legs use it.  It computes the same
definitions as ``oracle/csa2.py`` in plain loops, one thread per host core,
and is pinned against that module by ``tests/test_oracle_cref.py``.

``build()`` compiles ``oracle/libcref.so`` with the host C++ compiler
(``-ffp-contract=off``: every float operation one rounding).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "cref.cpp")
LIB = os.path.join(HERE, "libcref.so")
FLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
         "-pthread"]

_lib = None


def build(force: bool = False) -> str:
    """Compile libcref.so if it is missing or older than its source."""
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        tmp = LIB + ".tmp"
        subprocess.run(["g++", *FLAGS, SRC, "-o", tmp], check=True)
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(LIB)
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        L.cref_hardware_threads.restype = ctypes.c_int
        L.cref_quant_append_rows.argtypes = [P, P, I64, I32, P, P, I32, P, P]
        L.cref_encode_range.argtypes = [ctypes.c_uint64, I64, P, P, I32]
        L.cref_compress_pairs.argtypes = [P, P, I64, I32, P]
        L.cref_index_scores.argtypes = [P, P, I32, I32, P, I64, I64, P, I32]
        L.cref_index_scores_mx.argtypes = [P, P, I32, I32, P, I64, P, I64, I64, P, I32]
        L.cref_block_maxima.argtypes = [P, I64, P]
        L.cref_topk.argtypes = [P, P, I64, I64, P]
        L.cref_topk.restype = I64
        L.cref_dequant_fp4.argtypes = [P, I64, P, I64, I64, I32, P]
        L.cref_decode_e4m3.argtypes = [P, I64, P]
        L.cref_attention.argtypes = [P, I32, I32, P, I64, D, P, I32]
        for f in (L.cref_quant_append_rows, L.cref_encode_range, L.cref_compress_pairs,
                  L.cref_index_scores,
                  L.cref_index_scores_mx,
                  L.cref_block_maxima, L.cref_dequant_fp4, L.cref_decode_e4m3,
                  L.cref_attention):
            f.restype = None
        _lib = L
    return _lib


def threads() -> int:
    """Host threads the multi-threaded functions use: one per core."""
    return int(lib().cref_hardware_threads())


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def quant_append_rows(kv, pos, cos_tab, sin_tab, rope_dim):
    """As ``csa2.quant_append_rows``: (codes [n, D/2], scales [n, D/16])."""
    kv = _c(kv, np.float32)
    n, d = kv.shape
    pos = _c(pos, np.int64)
    cos_tab, sin_tab = _c(cos_tab, np.float32), _c(sin_tab, np.float32)
    codes = np.zeros((n, d // 2), np.uint8)
    scales = np.zeros((n, d // 16), np.uint8)
    lib().cref_quant_append_rows(_p(kv), _p(pos), n, d, _p(cos_tab), _p(sin_tab), rope_dim,
                                 _p(codes), _p(scales))
    return codes, scales


def compress_pairs(kv, z):
    """As ``csa2.compress_pairs``: source rows [2T, D] and logits [2T, D] ->
    T compressed rows (fp32)."""
    kv, z = _c(kv, np.float32), _c(z, np.float32)
    t2, d = kv.shape
    out = np.zeros((t2 // 2, d), np.float32)
    lib().cref_compress_pairs(_p(kv), _p(z), t2 // 2, d, _p(out))
    return out


def encode_range(first, n, nthreads=None):
    """E2M1 and E4M3 codes of the fp32 values with bit patterns first ..
    first + n - 1 (uint8 [n] each; 0xFF for NaN patterns)."""
    e2 = np.empty(n, np.uint8)
    e4 = np.empty(n, np.uint8)
    lib().cref_encode_range(first, n, _p(e2), _p(e4), nthreads or threads())
    return e2, e4


def indexer_scores(q_codes, w, k_codes, nthreads=None):
    """As ``csa2.indexer_scores``: one query's E4M3 codes [Hi * di], weights
    [Hi] and E4M3 key rows [n, di] -> fp64 scores [n]."""
    w = _c(w, np.float32)
    hi = len(w)
    q = _c(q_codes, np.uint8).reshape(-1)
    di = q.size // hi
    k = np.asarray(k_codes, dtype=np.uint8).reshape(-1, di)
    if not k.flags.c_contiguous:
        k = np.ascontiguousarray(k)
    out = np.zeros(k.shape[0], np.float64)
    lib().cref_index_scores(_p(q), _p(w), hi, di, _p(k), di, k.shape[0], _p(out),
                            nthreads or threads())
    return out


def indexer_scores_mx(q_codes, w, k_codes, k_scales, dim, nthreads=None):
    """Scores against MXFP4 key rows (codes [n, dim/2], E8M0 scales [n, >= dim/32])."""
    w = _c(w, np.float32)
    hi = len(w)
    q = _c(q_codes, np.uint8).reshape(-1)
    k = _c(np.asarray(k_codes, np.uint8)[:, : dim // 2], np.uint8)
    s = _c(np.asarray(k_scales, np.uint8)[:, : dim // 32], np.uint8)
    out = np.zeros(k.shape[0], np.float64)
    lib().cref_index_scores_mx(_p(q), _p(w), hi, dim, _p(k), dim // 2, _p(s), dim // 32,
                               k.shape[0], _p(out), nthreads or threads())
    return out


def block_maxima(scores):
    s = _c(scores, np.float64)
    out = np.zeros(-(-len(s) // 8), np.float64)
    lib().cref_block_maxima(_p(s), len(s), _p(out))
    return out


def topk(scores, k, ids=None):
    """As ``csa2.topk``: the k best ids by (score desc, id asc), ascending."""
    s = _c(scores, np.float64)
    k = min(int(k), len(s))
    if k <= 0:
        return np.zeros(0, np.int64)
    out = np.zeros(k, np.int64)
    idp = None
    if ids is not None:
        ids = _c(ids, np.int64)
        idp = _p(ids)
    lib().cref_topk(_p(s), idp, len(s), k, _p(out))
    return out


def full_select(scores, k, pool_blocks=2048):
    """As ``csa2.full_select``: (top-k positions, pool block ids), ascending."""
    bm = block_maxima(scores)
    return topk(scores, k), topk(bm, min(pool_blocks, len(bm)))


def dequantize_fp4(codes, scales, dim):
    c = _c(np.asarray(codes, np.uint8)[:, : dim // 2], np.uint8)
    s = _c(np.asarray(scales, np.uint8)[:, : dim // 16], np.uint8)
    out = np.zeros((c.shape[0], dim), np.float64)
    lib().cref_dequant_fp4(_p(c), dim // 2, _p(s), dim // 16, c.shape[0], dim, _p(out))
    return out


def e4m3_decode(codes):
    c = _c(codes, np.uint8)
    out = np.zeros(c.shape, np.float64)
    lib().cref_decode_e4m3(_p(c), c.size, _p(out))
    return out


def sparse_attention(q, rows, scale=None, nthreads=None):
    """As ``csa2.sparse_attention``: q fp64 [H, D], rows fp64 [n, D]."""
    q = _c(q, np.float64)
    rows = _c(rows, np.float64).reshape(-1, q.shape[1])
    h, d = q.shape
    if scale is None or scale <= 0:
        scale = 1.0 / math.sqrt(d)
    out = np.zeros((h, d), np.float64)
    lib().cref_attention(_p(q), h, d, _p(rows), rows.shape[0], float(scale), _p(out),
                         nthreads or threads())
    return out
