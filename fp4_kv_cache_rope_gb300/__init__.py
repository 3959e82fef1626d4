"""Python binding of libcsa2 (CSA2 sparse attention over an FP4 global KV cache).

Argument marshalling only: every step of the path runs in the CUDA kernels of
``libcsa2.so`` behind the C ABI declared in ``include/csa2.h``.  Tensors are
passed as ``torch.Tensor`` (device memory) and the current torch CUDA stream
is used unless a stream is given.  There is no CPU fallback: importing this
module fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcsa2.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`"
    )

_lib = ctypes.CDLL(LIB_PATH)

CSA2_OK, CSA2_ERR_INVALID, CSA2_ERR_CUDA, CSA2_ERR_UNSUPPORTED, CSA2_ERR_TIMEOUT, CSA2_ERR_DEVICE = range(6)
DEV_BAD_INDEX, DEV_BAD_PAGE, DEV_OVERFLOW, DEV_TIMEOUT, DEV_BAD_POOL, DEV_BAD_ALIGN = (
    0x1, 0x2, 0x4, 0x8, 0x10, 0x20)
MAX_TOPK = 2048
POOL_BLOCKS = 2048
BLOCK = 8

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class Csa2Cache(ctypes.Structure):
    _fields_ = [
        ("batch", _i32), ("dim", _i32), ("rope_dim", _i32), ("idx_dim", _i32),
        ("page_size", _i32), ("max_pages_per_seq", _i32), ("max_len", _i32), ("num_pages", _i32),
        ("kv_codes", _p), ("code_stride", _i64),
        ("kv_scales", _p), ("scale_stride", _i64),
        ("idx_k", _p), ("idxk_stride", _i64),
        ("page_table", _p), ("seq_len", _p),
        ("rope_cos", _p), ("rope_sin", _p),
        ("idx_format", _i32), ("idx_scales", _p), ("idx_scale_stride", _i64),
    ]


IDX_E4M3, IDX_MXFP4 = 0, 1


def _sig(name, args, res=_i32):
    f = getattr(_lib, name)
    f.argtypes = args
    f.restype = res
    return f


_CP = ctypes.POINTER(Csa2Cache)
_workspace_size = _sig("csa2_workspace_size", [_CP, _i32, _i32], ctypes.c_size_t)
_entry_bytes = _sig("csa2_entry_bytes", [_i32], _i64)
_fp8_quant = _sig("csa2_fp8_quant", [_p, _i64, _p, _p])
_quant_append = _sig("csa2_quant_append", [_CP, _p, _p, _i32, _p, _p])
_quant_append_pairs = _sig("csa2_quant_append_pairs", [_CP, _p, _p, _p, _i32, _p, _p])
_index_full = _sig("csa2_index_full", [_CP, _p, _p, _i32, _i32, _p, _p, _i32, _i32,
                                       _p, _p, _p, _p, _p, _p])
_index_full_noalloc = _sig("csa2_index_full_noalloc", [_CP, _p, _p, _i32, _i32, _p, _p, _i32,
                                                       _i32, _p, _p, _p, _p, _p, _p])
NOALLOC_SCRATCH_BYTES = 32 * 1024 * 1024
_index_reindex = _sig("csa2_index_reindex", [_CP, _p, _p, _i32, _i32, _p, _p, _p, _p, _i32,
                                             _i32, _p, _p, _p, _p])
_attn_decode = _sig("csa2_attn_decode", [_CP, _p, _i32, _p, _p, _i32, _p, _p, _i32,
                                         ctypes.c_float, _p, _p, _p])
_attn_decode_layers = _sig("csa2_attn_decode_layers", [_CP, _i32, _p, _i32, _p, _p, _i32, _p, _p,
                                                       _i32, ctypes.c_float, _p, _p, _p])
_attn_prefill = _sig("csa2_attn_prefill", [_CP, _p, _i32, _i32, _p, _p, _p, _i32, _p, _i32,
                                           ctypes.c_float, _p, _p, _p])
_get_status = _sig("csa2_get_status", [_p, ctypes.POINTER(ctypes.c_uint32), _p])
_reset_status = _sig("csa2_reset_status", [_p, _p])
_status_string = _sig("csa2_status_string", [_i32], ctypes.c_char_p)
_set_launch_events = _sig("csa2_set_launch_events", [_i32, _p, _p])
_set_wait_limit = _sig("csa2_set_wait_limit", [ctypes.c_uint64])
KERNEL_QUANT, KERNEL_INDEXER, KERNEL_SELECT, KERNEL_ATTENTION = 0, 1, 2, 3

EXPORTED = ["csa2_workspace_size", "csa2_entry_bytes", "csa2_fp8_quant", "csa2_quant_append",
            "csa2_index_full", "csa2_index_reindex", "csa2_attn_decode", "csa2_attn_prefill",
            "csa2_get_status", "csa2_reset_status", "csa2_status_string",
            "csa2_set_launch_events", "csa2_index_full_noalloc", "csa2_quant_append_pairs",
            "csa2_set_wait_limit", "csa2_attn_decode_layers"]


class Csa2Error(RuntimeError):
    pass


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(code, what):
    if code != CSA2_OK:
        raise Csa2Error(f"{what}: {status_string(code)} ({code})")
    return code


def status_string(code: int) -> str:
    return _status_string(int(code)).decode()


def entry_bytes(dim: int) -> int:
    return int(_entry_bytes(dim))


def workspace_size(cache: "Cache | Csa2Cache", max_rows: int, heads: int) -> int:
    c = cache.struct if isinstance(cache, Cache) else cache
    return int(_workspace_size(ctypes.byref(c), max_rows, heads))


def fp8_quant(x, out, stream=None):
    """fp32 -> E4M3 codes (RNE, saturating at 448, sign copied)."""
    _check(_fp8_quant(_ptr(x), x.numel(), _ptr(out), _stream(stream)), "csa2_fp8_quant")


def quant_append(cache, kv, idx_k_in, T, ws, stream=None):
    _check(_quant_append(ctypes.byref(cache.struct), _ptr(kv), _ptr(idx_k_in), T, _ptr(ws),
                         _stream(stream)), "csa2_quant_append")


def quant_append_pairs(cache, kv, z, idx_k_in, T, ws, stream=None):
    """Append T entries per sequence, each compressed from 2 source rows (m = 2)."""
    _check(_quant_append_pairs(ctypes.byref(cache.struct), _ptr(kv), _ptr(z), _ptr(idx_k_in), T,
                               _ptr(ws), _stream(stream)), "csa2_quant_append_pairs")


def index_full(cache, q_idx, w, hi, tq, q_pos, batch_ids, n_batch, k, out_idx, out_cnt,
               pool_blocks, pool_cnt, ws, stream=None):
    _check(_index_full(ctypes.byref(cache.struct), _ptr(q_idx), _ptr(w), hi, tq, _ptr(q_pos),
                       _ptr(batch_ids), n_batch, k, _ptr(out_idx), _ptr(out_cnt),
                       _ptr(pool_blocks), _ptr(pool_cnt), _ptr(ws), _stream(stream)),
           "csa2_index_full")


def index_full_noalloc(cache, q_idx, w, hi, tq, q_pos, batch_ids, n_batch, k, out_idx, out_cnt,
                       pool_blocks, pool_cnt, status, stream=None):
    """index_full for callers that may not allocate device memory: the scratch
    is a fixed array inside the library; ``status`` (a 4-byte device tensor or
    None) receives the call's device status word."""
    _check(_index_full_noalloc(ctypes.byref(cache.struct), _ptr(q_idx), _ptr(w), hi, tq,
                               _ptr(q_pos), _ptr(batch_ids), n_batch, k, _ptr(out_idx),
                               _ptr(out_cnt), _ptr(pool_blocks), _ptr(pool_cnt), _ptr(status),
                               _stream(stream)), "csa2_index_full_noalloc")


def index_reindex(cache, q_idx, w, hi, tq, q_pos, pool_blocks, pool_cnt, batch_ids, n_batch, k,
                  out_idx, out_cnt, ws, stream=None):
    _check(_index_reindex(ctypes.byref(cache.struct), _ptr(q_idx), _ptr(w), hi, tq, _ptr(q_pos),
                          _ptr(pool_blocks), _ptr(pool_cnt), _ptr(batch_ids), n_batch, k,
                          _ptr(out_idx), _ptr(out_cnt), _ptr(ws), _stream(stream)),
           "csa2_index_reindex")


def attn_decode(cache, q, heads, idx, cnt, kcap, swa, swa_cnt, window, softmax_scale, out, ws,
                stream=None):
    _check(_attn_decode(ctypes.byref(cache.struct), _ptr(q), heads, _ptr(idx), _ptr(cnt), kcap,
                        _ptr(swa), _ptr(swa_cnt), window, float(softmax_scale), _ptr(out),
                        _ptr(ws), _stream(stream)), "csa2_attn_decode")


MAX_ATTN_LAYERS = 8


def attn_decode_layers(cache, qs, heads, idx, cnt, kcap, swas, swa_cnt, window, softmax_scale,
                       outs, ws, stream=None):
    """csa2_attn_decode_layers: qs, swas, outs are sequences of one tensor per
    layer (the host pointer arrays are built here)."""
    n = len(qs)
    if not 1 <= n <= MAX_ATTN_LAYERS or len(outs) != n or len(swas) != n:
        raise Csa2Error("csa2_attn_decode_layers: 1..%d layers, one q, swa and out each"
                        % MAX_ATTN_LAYERS)
    arr = ctypes.c_void_p * n
    qa, sa, oa = arr(*[_ptr(x) for x in qs]), arr(*[_ptr(x) for x in swas]), arr(*[_ptr(x) for x in outs])
    _check(_attn_decode_layers(ctypes.byref(cache.struct), n, ctypes.cast(qa, ctypes.c_void_p),
                               heads, _ptr(idx), _ptr(cnt), kcap, ctypes.cast(sa, ctypes.c_void_p),
                               _ptr(swa_cnt), window, float(softmax_scale),
                               ctypes.cast(oa, ctypes.c_void_p), _ptr(ws), _stream(stream)),
           "csa2_attn_decode_layers")


def attn_prefill(cache, q, heads, tq, q_pos, idx, cnt, kcap, swa, window, softmax_scale, out, ws,
                 stream=None):
    _check(_attn_prefill(ctypes.byref(cache.struct), _ptr(q), heads, tq, _ptr(q_pos), _ptr(idx),
                         _ptr(cnt), kcap, _ptr(swa), window, float(softmax_scale), _ptr(out),
                         _ptr(ws), _stream(stream)), "csa2_attn_prefill")


def set_launch_events(family, begin=None, end=None):
    """Bracket the family's main kernel with torch.cuda.Event records (or stop)."""
    b = begin.cuda_event if begin is not None else None
    e = end.cuda_event if end is not None else None
    _check(_set_launch_events(family, b, e), "csa2_set_launch_events")


def set_wait_limit(ns: int = 0):
    """Limit of the kernels' bounded on-chip waits in ns (0 = the 2 s default)."""
    _check(_set_wait_limit(int(ns)), "csa2_set_wait_limit")


def get_status(ws, stream=None) -> int:
    v = ctypes.c_uint32(0)
    code = _get_status(_ptr(ws), ctypes.byref(v), _stream(stream))
    if code not in (CSA2_OK, CSA2_ERR_DEVICE):
        _check(code, "csa2_get_status")
    return int(v.value)


def reset_status(ws, stream=None):
    _check(_reset_status(_ptr(ws), _stream(stream)), "csa2_reset_status")


class Cache:
    """Device storage of one shared global cache plus its C description.

    Row strides are the smallest multiples of 16 bytes that hold a row:
    codes D/2, scales round_up(D/16, 16), indexer key di (E4M3).  With
    ``idx_format=IDX_MXFP4`` (di = 128) the indexer key is 64 code bytes per
    row and a separate array holds its 4 E8M0 scale bytes per row.
    """

    def __init__(self, batch, dim, rope_dim, idx_dim, max_len, rope_cos, rope_sin,
                 page_size=0, page_table=None, num_pages=0, device="cuda",
                 idx_format=IDX_E4M3):
        import torch
        self.batch, self.dim, self.rope_dim, self.idx_dim = batch, dim, rope_dim, idx_dim
        self.max_len, self.page_size = max_len, page_size
        self.idx_format = idx_format
        self.code_stride = (dim // 2 + 15) // 16 * 16
        self.scale_stride = (dim // 16 + 15) // 16 * 16
        if idx_format == IDX_MXFP4:
            self.idxk_stride = (idx_dim // 2 + 31) // 32 * 32
            self.idx_scale_stride = idx_dim // 32
        else:
            self.idxk_stride = (idx_dim + 15) // 16 * 16
            self.idx_scale_stride = 0
        if page_size:
            self.num_pages = num_pages
            rows = num_pages * page_size
            self.page_table = page_table.to(device=device, dtype=torch.int32).contiguous()
            self.max_pages = self.page_table.shape[1]
        else:
            self.num_pages = 0
            rows = batch * max_len
            self.page_table = None
            self.max_pages = 0
        self.rows = rows
        self.codes = torch.zeros((rows, self.code_stride), dtype=torch.uint8, device=device)
        self.scales = torch.zeros((rows, self.scale_stride), dtype=torch.uint8, device=device)
        self.idx_k = torch.zeros((rows, self.idxk_stride), dtype=torch.uint8, device=device)
        self.idx_scales = (torch.zeros((rows, self.idx_scale_stride), dtype=torch.uint8,
                                       device=device) if idx_format == IDX_MXFP4 else None)
        self.seq_len = torch.zeros(batch, dtype=torch.int32, device=device)
        self.rope_cos = rope_cos.to(device=device, dtype=torch.float32).contiguous()
        self.rope_sin = rope_sin.to(device=device, dtype=torch.float32).contiguous()
        self.struct = Csa2Cache(
            batch, dim, rope_dim, idx_dim, page_size, self.max_pages, max_len, self.num_pages,
            self.codes.data_ptr(), self.code_stride, self.scales.data_ptr(), self.scale_stride,
            self.idx_k.data_ptr(), self.idxk_stride,
            self.page_table.data_ptr() if self.page_table is not None else None,
            self.seq_len.data_ptr(), self.rope_cos.data_ptr(), self.rope_sin.data_ptr(),
            idx_format, self.idx_scales.data_ptr() if self.idx_scales is not None else None,
            self.idx_scale_stride)

    def physical_row(self, b, t):
        """Host mirror of the row mapping (for reading rows back in tests)."""
        if not self.page_size:
            return b * self.max_len + t
        pt = self.page_table_host()
        return int(pt[b, t // self.page_size]) * self.page_size + t % self.page_size

    def page_table_host(self):
        if not hasattr(self, "_pt_host"):
            self._pt_host = self.page_table.cpu().numpy()
        return self._pt_host

    def workspace(self, max_rows, heads):
        import torch
        n = workspace_size(self, max_rows, heads)
        if n == 0:
            raise Csa2Error("invalid cache description")
        ws = torch.zeros(n, dtype=torch.uint8, device=self.codes.device)
        return ws
