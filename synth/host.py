"""Host side of the seeded input generator: rows and per-layer inputs of a
workload as numpy arrays, with the same bits as the device generator in
``synth.device``.  Seeded generators only (no arithmetic of the method); the
oracle reads its inputs through this module.
"""
from __future__ import annotations

import numpy as np

from . import (LAYER_STRIDE, T_POOL, T_PRIOR, T_Q, T_QIDX, T_SWA, T_W, outlier_multipliers,
               sample_distinct)
from .workloads import Workload

# position t of sequence b is logical row (b << ROW_SHIFT) + t
ROW_SHIFT = 21


def host_rows_normal(seed, tensor_id, b, positions, width, chan_mult=None):
    """Host copy of rows ``positions`` of sequence b (same bits as the device)."""
    from . import normal_rows
    rows = (np.int64(b) << ROW_SHIFT) + np.asarray(positions, dtype=np.int64)
    return normal_rows(seed, tensor_id, rows, width, chan_mult)


def host_layer_inputs(wl: Workload, layer, b, tq=1):
    """Host copy (fp32 / bf16 as float) of sequence b's query-side inputs."""
    import torch
    from . import normal_block, uniform_block
    off = LAYER_STRIDE * layer
    Hi, di, H, D, W = wl.idx_heads, wl.idx_dim, wl.heads, wl.dim, wl.window
    mult = outlier_multipliers(wl.seed, wl.dim, wl.outlier_frac) if wl.outlier_frac else None
    qf = normal_block(wl.seed, T_QIDX + off, (tq, Hi, di), start=b * tq * Hi * di)
    w = uniform_block(wl.seed, T_W + off, (tq, Hi), start=b * tq * Hi)
    q = normal_block(wl.seed, T_Q + off, (tq, H, D), start=b * tq * H * D)
    qb = torch.from_numpy(q).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    swa_rows = (tq + W - 1) if tq > 1 else W
    sf = normal_block(wl.seed, T_SWA + off, (swa_rows, D), start=b * swa_rows * D, chan_mult=mult)
    return dict(q_idx_f32=qf, w=w, q_bf16=qb, swa_f32=sf)


def supplied_pool(wl: Workload, b, n):
    """Pool given to a Reindex sequence of the ragged workload (sorted block ids)."""
    nb = -(-n // 8)
    return sample_distinct(wl.seed, T_POOL, b, nb, 2048)


def supplied_prior(wl: Workload, b, n):
    """Prior index set given to a Reuse sequence of the ragged workload."""
    return sample_distinct(wl.seed, T_PRIOR, b, n, min(wl.topk, n))
