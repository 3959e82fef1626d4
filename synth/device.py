"""GPU side of the seeded input generator, and the device copy of a workload.

``gen_normal`` / ``gen_uniform`` produce on the GPU the same bits as
``synth.normal`` / ``synth.uniform`` on the host (they call the twin kernels
in ``synth_gpu.cu``).  ``DeviceWorkload`` lays a workload out in device
memory through the public calls of the CUDA path (cache rows are appended
with ``quant_append``; FP8 operands are made with ``fp8_quant``).  Nothing
here computes any step of the method itself.

Flat index convention (shared with the host generator): position t of
sequence b is logical row (b << 21) + t, so the values of a cache row do not
depend on the cache capacity or its paging.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

from . import (LAYER_STRIDE, NORMAL_TABLE, T_IDXK, T_KV, T_Z, T_PAGE, T_POOL, T_PRIOR, T_Q, T_QIDX,
               T_SWA, T_W, outlier_multipliers, permutation, rope_table, sample_distinct,
               stream_key)
from .host import (ROW_SHIFT, host_layer_inputs, host_rows_normal,  # noqa: F401
                   supplied_pool, supplied_prior)
from .workloads import FULL, REINDEX, REUSE, Workload

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libsynth.so")


def build():
    src = os.path.join(HERE, "synth_gpu.cu")
    if os.path.exists(LIB) and os.path.getmtime(LIB) > os.path.getmtime(src):
        return LIB
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared",
           "-Xcompiler", "-fPIC", "-o", LIB, src]
    subprocess.run(cmd, check=True, capture_output=True)
    return LIB


_lib = None


def _get():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build()
        _lib = ctypes.CDLL(LIB)
        _lib.synth_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                           ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.c_int32, ctypes.c_void_p]
        _lib.synth_fill_uniform.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                            ctypes.c_int64, ctypes.c_void_p]
    return _lib


_tables = {}


def _table(device):
    import torch
    if device not in _tables:
        _tables[device] = torch.from_numpy(NORMAL_TABLE).to(device)
    return _tables[device]


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def gen_normal(shape, seed, tensor_id, start=0, chan_mult=None, device="cuda"):
    import torch
    out = torch.empty(shape, dtype=torch.float32, device=device)
    mult = None
    period = 1
    if chan_mult is not None:
        mult = torch.as_tensor(np.asarray(chan_mult, dtype=np.float32), device=device)
        period = mult.numel()
    r = _get().synth_fill_normal(out.data_ptr(), out.numel(), stream_key(seed, tensor_id), start,
                                 _table(device).data_ptr(),
                                 mult.data_ptr() if mult is not None else None, period, _stream())
    if r:
        raise RuntimeError(f"synth_fill_normal failed: {r}")
    return out


def gen_uniform(shape, seed, tensor_id, start=0, device="cuda"):
    import torch
    out = torch.empty(shape, dtype=torch.float32, device=device)
    r = _get().synth_fill_uniform(out.data_ptr(), out.numel(), stream_key(seed, tensor_id), start,
                                  _stream())
    if r:
        raise RuntimeError(f"synth_fill_uniform failed: {r}")
    return out


def gen_rows_normal(seed, tensor_id, b, t0, n, width, chan_mult=None, device="cuda"):
    """Rows t0..t0+n of sequence b of a [*, width] normal tensor."""
    start = ((b << ROW_SHIFT) + t0) * width
    return gen_normal((n, width), seed, tensor_id, start, chan_mult, device)


def page_table_for(wl: Workload):
    """Seeded random physical page ids: [B, max_pages] int32, -1 where unused."""
    ps = wl.page_size
    max_pages = -(-wl.max_len // ps)
    need = [-(-min(wl.max_len, n + 64 + max(wl.prefill_tokens, 0) + wl.extra_capacity) // ps)
            for n in wl.lengths]
    need = [min(max_pages, x) for x in need]
    total = int(sum(need))
    perm = permutation(wl.seed, T_PAGE, total)
    pt = np.full((wl.batch, max_pages), -1, dtype=np.int32)
    o = 0
    for b, k in enumerate(need):
        pt[b, :k] = perm[o:o + k]
        o += k
    return pt, total


class DeviceWorkload:
    """A workload's cache and per-layer inputs in device memory."""

    def __init__(self, wl: Workload, device="cuda", build_cache=True, chunk_rows=1 << 16):
        import torch
        import fp4_kv_cache_rope_gb300 as K
        self.wl, self.device, self.K = wl, device, K
        self.mult = outlier_multipliers(wl.seed, wl.dim, wl.outlier_frac) if wl.outlier_frac else None
        cos, sin = rope_table(wl.max_len, wl.rope_dim, wl.theta)
        self.rope_cos, self.rope_sin = cos, sin
        idx_format = K.IDX_MXFP4 if wl.idx_format == "mxfp4" else K.IDX_E4M3
        if wl.page_size:
            pt, npages = page_table_for(wl)
            self.page_table_np = pt
            self.cache = K.Cache(wl.batch, wl.dim, wl.rope_dim, wl.idx_dim, wl.max_len,
                                 torch.from_numpy(cos), torch.from_numpy(sin),
                                 page_size=wl.page_size, page_table=torch.from_numpy(pt),
                                 num_pages=npages, device=device, idx_format=idx_format)
        else:
            self.page_table_np = None
            self.cache = K.Cache(wl.batch, wl.dim, wl.rope_dim, wl.idx_dim, wl.max_len,
                                 torch.from_numpy(cos), torch.from_numpy(sin), device=device,
                                 idx_format=idx_format)
        rows = max(wl.batch * max(1, wl.prefill_tokens), wl.batch)
        self.ws = self.cache.workspace(rows, wl.heads)
        if build_cache:
            self.fill_cache(chunk_rows)

    # ---- cache -------------------------------------------------------------
    def seq_view(self, b):
        """A one-sequence view of the cache (C description only)."""
        import fp4_kv_cache_rope_gb300 as K
        c = self.cache
        s = K.Csa2Cache.from_buffer_copy(c.struct)
        s.batch = 1
        if c.page_size:
            s.page_table = c.page_table.data_ptr() + 4 * b * c.max_pages
        else:
            s.kv_codes = c.codes.data_ptr() + b * c.max_len * c.code_stride
            s.kv_scales = c.scales.data_ptr() + b * c.max_len * c.scale_stride
            s.idx_k = c.idx_k.data_ptr() + b * c.max_len * c.idxk_stride
            if c.idx_scales is not None:
                s.idx_scales = c.idx_scales.data_ptr() + b * c.max_len * c.idx_scale_stride
        s.seq_len = c.seq_len.data_ptr() + 4 * b
        view = type("View", (), {})()
        view.struct = s
        return view

    def fill_cache(self, chunk_rows=1 << 16):
        """Append entries 0..N_b-1 of every sequence through quant_append (or,
        for an m = 2 cache, quant_append_pairs over source rows 0..2N_b-1)."""
        wl = self.wl
        for b, n in enumerate(wl.lengths):
            v = self.seq_view(b)
            for t0 in range(0, n, chunk_rows):
                m = min(chunk_rows, n - t0)
                ik = gen_rows_normal(wl.seed, T_IDXK, b, t0, m, wl.idx_dim, None, self.device)
                if wl.compress == 2:
                    kv, z = self.pair_sources(b, t0, m)
                    self.K.quant_append_pairs(v, kv, z, ik, m, self.ws)
                else:
                    kv = gen_rows_normal(wl.seed, T_KV, b, t0, m, wl.dim, self.mult, self.device)
                    self.K.quant_append(v, kv, ik, m, self.ws)
        import torch
        torch.cuda.synchronize()

    def pair_sources(self, b, e0, m):
        """Source rows 2e0..2(e0+m)-1 of sequence b and their compression logits."""
        wl = self.wl
        kv = gen_rows_normal(wl.seed, T_KV, b, 2 * e0, 2 * m, wl.dim, self.mult, self.device)
        z = gen_rows_normal(wl.seed, T_Z, b, 2 * e0, 2 * m, wl.dim, None, self.device) * 2.0
        return kv, z

    def new_token_inputs(self, step_positions):
        """fp32 main-KV and indexer-key rows of the next token of every sequence."""
        import torch
        wl = self.wl
        kv = torch.stack([gen_rows_normal(wl.seed, T_KV, b, int(p), 1, wl.dim, self.mult,
                                          self.device)[0]
                          for b, p in enumerate(step_positions)])
        ik = torch.stack([gen_rows_normal(wl.seed, T_IDXK, b, int(p), 1, wl.idx_dim, None,
                                          self.device)[0]
                          for b, p in enumerate(step_positions)])
        return kv, ik

    # ---- per-layer inputs ----------------------------------------------------
    def layer_inputs(self, layer, tq=1):
        """Query-side inputs of one layer: q_idx (E4M3), w, q (bf16), swa (E4M3)."""
        import torch
        wl = self.wl
        off = LAYER_STRIDE * layer
        B, Hi, di, H, D, W = wl.batch, wl.idx_heads, wl.idx_dim, wl.heads, wl.dim, wl.window
        qf = gen_normal((B, tq, Hi, di), wl.seed, T_QIDX + off, device=self.device)
        q_idx = torch.empty(qf.shape, dtype=torch.uint8, device=self.device)
        self.K.fp8_quant(qf, q_idx)
        w = gen_uniform((B, tq, Hi), wl.seed, T_W + off, device=self.device)
        q = gen_normal((B, tq, H, D), wl.seed, T_Q + off, device=self.device).to(torch.bfloat16)
        swa_rows = (tq + W - 1) if tq > 1 else W
        sf = gen_normal((B, swa_rows, D), wl.seed, T_SWA + off, chan_mult=self.mult,
                        device=self.device)
        swa = torch.empty(sf.shape, dtype=torch.uint8, device=self.device)
        self.K.fp8_quant(sf, swa)
        return dict(q_idx=q_idx, w=w, q=q, swa=swa, q_f32=qf, swa_f32=sf)
