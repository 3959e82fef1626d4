"""Seeded synthetic inputs for the CSA2 FP4-KV-cache hot path.

This module is shared by the oracle side and the CUDA side of every test and
benchmark, so it holds none of the method's arithmetic: no RoPE, no FP4/FP8
codec, no scoring, selection or attention.  It holds

* one counter-based random stream (SplitMix64, Steele/Lea/Flood 2014, the
  64-bit finaliser published with ``java.util.SplittableRandom``),
* a 65,536-entry table of standard-normal quantiles used to turn 16 random
  bits into an N(0,1) sample by table lookup,
* the shapes of the five workloads (dataclasses in ``workloads``).

Every value is a pure function of ``(seed, tensor id, flat index)``: any slice
of any tensor can be regenerated on any core, and the GPU generator in
``synth_gpu.cu`` produces the same bits because it does the same integer
operations and reads the same table.
"""
from __future__ import annotations

import statistics

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB

# Tensor ids: one independent stream per logical input tensor.
T_KV = 1          # main-KV rows before RoPE, fp32 [B, max_len, D]
T_IDXK = 2        # indexer keys before the FP8 cast, fp32 [B, max_len, di]
T_QIDX = 3        # indexer queries before the FP8 cast, fp32 [B, Tq, Hi, di]
T_W = 4           # indexer head weights, U(0,1) fp32 [B, Tq, Hi]
T_Q = 5           # attention queries (taken as post-RoPE), bf16 [B, Tq, H, D]
T_SWA = 6         # SWA window rows before the FP8 cast, fp32
T_OUTLIER = 7     # channel permutation that picks outlier channels
T_LEN = 8         # ragged sequence lengths
T_PAGE = 9        # physical page permutation
T_MODE = 10       # per-sequence layer mode
T_POOL = 11       # supplied pools for Reindex sequences
T_PRIOR = 12      # supplied prior indices for Reuse sequences
T_NEWKV = 13      # the new token's main-KV row appended each decode step
T_NEWIDXK = 14    # the new token's indexer key appended each decode step
T_Z = 15          # compression logits of encoder source rows (m = 2), N(0,1) x 2, fp32
LAYER_STRIDE = 100  # tensor id offset between layers of one CSA2 group


def _mix64_int(x: int) -> int:
    z = (x + GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, tensor_id: int) -> int:
    """64-bit key of one tensor's stream."""
    return _mix64_int(((seed & 0xFFFFFFFF) << 32) ^ (tensor_id & 0xFFFFFFFF))


def mix64(x: np.ndarray) -> np.ndarray:
    """SplitMix64 finaliser applied element-wise to a uint64 array."""
    with np.errstate(over="ignore"):
        z = x + np.uint64(GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
        return z ^ (z >> np.uint64(31))


def hashes(key: int, index: np.ndarray) -> np.ndarray:
    """Raw 64-bit draws of stream ``key`` at the given flat indices."""
    with np.errstate(over="ignore"):
        return mix64(np.uint64(key) + index.astype(np.uint64))


def _normal_table() -> np.ndarray:
    nd = statistics.NormalDist()
    q = [nd.inv_cdf((i + 0.5) / 65536.0) for i in range(65536)]
    return np.asarray(q, dtype=np.float64).astype(np.float32)


NORMAL_TABLE = _normal_table()


def normal(seed: int, tensor_id: int, index: np.ndarray) -> np.ndarray:
    """N(0,1) fp32 samples: the quantile at the top 16 bits of each draw."""
    h = hashes(stream_key(seed, tensor_id), index)
    return NORMAL_TABLE[(h >> np.uint64(48)).astype(np.int64)]


def uniform(seed: int, tensor_id: int, index: np.ndarray) -> np.ndarray:
    """U[0,1) fp32 samples with 24 random bits (exact in fp32)."""
    h = hashes(stream_key(seed, tensor_id), index)
    u24 = ((h >> np.uint64(40)) & np.uint64(0xFFFFFF)).astype(np.float32)
    return u24 * np.float32(2.0 ** -24)


def normal_block(seed, tensor_id, shape, start=0, chan_mult=None):
    """A contiguous block of a normal tensor, flat indices start..start+prod(shape).

    ``chan_mult`` (length = last dim) multiplies each channel (1.0 or 8.0 for
    the outlier channels, an exact power-of-two scaling).
    """
    n = int(np.prod(shape))
    idx = np.arange(start, start + n, dtype=np.int64)
    x = normal(seed, tensor_id, idx).reshape(shape)
    if chan_mult is not None:
        x = x * np.asarray(chan_mult, dtype=np.float32)
    return x


def normal_rows(seed, tensor_id, row_ids, width, chan_mult=None):
    """Rows ``row_ids`` (flat row numbers) of a [*, width] normal tensor."""
    row_ids = np.asarray(row_ids, dtype=np.int64)
    idx = row_ids[:, None] * width + np.arange(width, dtype=np.int64)[None, :]
    x = normal(seed, tensor_id, idx.reshape(-1)).reshape(len(row_ids), width)
    if chan_mult is not None:
        x = x * np.asarray(chan_mult, dtype=np.float32)
    return x


def uniform_block(seed, tensor_id, shape, start=0):
    n = int(np.prod(shape))
    idx = np.arange(start, start + n, dtype=np.int64)
    return uniform(seed, tensor_id, idx).reshape(shape)


def permutation(seed: int, tensor_id: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n) (argsort of the draws, ties by index)."""
    h = hashes(stream_key(seed, tensor_id), np.arange(n, dtype=np.int64))
    return np.argsort(h, kind="stable").astype(np.int64)


def outlier_multipliers(seed: int, dim: int, frac: float) -> np.ndarray:
    """Per-channel multiplier: 8.0 on round(frac*dim) seeded channels, else 1.0."""
    m = np.ones(dim, dtype=np.float32)
    n_out = int(round(frac * dim))
    if n_out:
        m[permutation(seed, T_OUTLIER, dim)[:n_out]] = 8.0
    return m


def sample_distinct(seed: int, tensor_id: int, salt: int, n: int, count: int) -> np.ndarray:
    """``count`` distinct values of range(n), sorted ascending (smallest draws)."""
    key = stream_key(seed, tensor_id) ^ (salt * 0x100000001B3 & MASK64)
    h = hashes(key, np.arange(n, dtype=np.int64))
    count = min(count, n)
    pick = np.argpartition(h, count - 1)[:count] if count < n else np.arange(n)
    return np.sort(pick).astype(np.int32)


def rope_table(max_len: int, rope_dim: int, theta: float):
    """cos/sin table [max_len, rope_dim/2] in fp32, angles taken in fp64.

    The table is an input of the path (callers build it once, as serving
    stacks do for rotary caches); frequency i is theta**(-2i/rope_dim).
    """
    half = rope_dim // 2
    if half == 0:
        z = np.zeros((max_len, 0), dtype=np.float32)
        return z, z.copy()
    i = np.arange(half, dtype=np.float64)
    inv = theta ** (-2.0 * i / rope_dim)
    ang = np.arange(max_len, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


from .workloads import WORKLOADS, Workload, get_workload  # noqa: E402,F401
