"""The five workload shapes of the CSA2 FP4-KV hot path (sizes only).

Each workload is a dataclass; ``materialise_*`` helpers in the tests and in
``bench.py`` turn one into tensors through the seeded streams of ``synth``.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

FULL, REINDEX, REUSE = 0, 1, 2
MODE_NAMES = {FULL: "full", REINDEX: "reindex", REUSE: "reuse"}


@dataclass
class Workload:
    name: str
    batch: int
    lengths: list            # visible global entries per sequence before the step
    dim: int                 # D (main-KV width, all channels stored FP4)
    rope_dim: int            # R, the last R channels are rotated
    idx_heads: int           # Hi
    idx_dim: int             # di
    heads: int               # H (attention query heads, one shared KV head)
    topk: int                # k
    window: int              # W (SWA rows)
    seed: int
    theta: float = 10000.0
    outlier_frac: float = 0.0
    page_size: int = 0       # 0 = contiguous rows per sequence
    layers: list = field(default_factory=lambda: [FULL])  # modes of one CSA2 group
    modes: list | None = None   # per-sequence mode (ragged mixed decode)
    prefill_tokens: int = 0  # T new tokens appended and queried (prefill chunk)
    pool_blocks: int = 2048  # pool capacity in 8-position blocks
    extra_capacity: int = 0  # positions reserved for tokens appended by decode steps
    idx_format: str = "e4m3"  # indexer-key storage: "e4m3" (1 B/channel) or "mxfp4"
    compress: int = 1        # m: source positions per main-KV entry (2 for encoder caches);
                             # lengths count entries

    @property
    def max_len(self) -> int:
        m = int(max(self.lengths)) + max(self.prefill_tokens, 0) + 64 + self.extra_capacity
        if self.idx_format == "mxfp4":   # whole 16-byte runs of 4-byte scale rows
            m = (m + 7) // 8 * 8
        return m

    def entry_bytes(self) -> int:
        return self.dim // 2 + self.dim // 16

    def idx_entry_bytes(self) -> int:
        """Algorithmic indexer-key bytes per position."""
        if self.idx_format == "mxfp4":
            return self.idx_dim // 2 + self.idx_dim // 32
        return self.idx_dim


def _ragged_lengths(seed: int, batch: int, lo: int, hi: int) -> list:
    from . import T_LEN, uniform
    u = uniform(seed, T_LEN, np.arange(batch, dtype=np.int64)).astype(np.float64)
    a, b = math.log(lo), math.log(hi)
    return [int(math.floor(math.exp(a + (b - a) * x))) for x in u]


def _modes(seed: int, batch: int) -> list:
    from . import T_MODE, hashes, stream_key
    h = hashes(stream_key(seed, T_MODE), np.arange(batch, dtype=np.int64))
    return [int(x % np.uint64(3)) for x in h]


def get_workload(i: int) -> Workload:
    """Workload number i (1..9)."""
    if i == 1:
        return Workload("tiny-full-decode-b1-n2048-d128", 1, [2048], 128, 32, 4, 32,
                        16, 64, 128, seed=0)
    if i == 2:
        return Workload("full-decode-b32-n131072-d576", 32, [131072] * 32, 576, 64, 64, 128,
                        64, 2048, 128, seed=1, outlier_frac=0.01)
    if i == 3:
        return Workload("group-full-reindex-reuse-b16-n1048576-d576", 16, [1048576] * 16,
                        576, 64, 64, 128, 64, 2048, 128, seed=2, outlier_frac=0.01,
                        layers=[FULL, REINDEX, REUSE])
    if i == 4:
        return Workload("prefill-t4096-after-n262144-d576", 1, [262144], 576, 64, 64, 128,
                        64, 2048, 128, seed=3, prefill_tokens=4096)
    if i == 5:
        lens = _ragged_lengths(4, 64, 8192, 1048576)
        return Workload("ragged-mixed-decode-b64-paged64-d576", 64, lens, 576, 64, 64, 128,
                        64, 2048, 128, seed=4, outlier_frac=0.01, page_size=64,
                        modes=_modes(4, 64))
    if i == 6:
        # multi-query decode: a 5-token speculative verify per sequence (each
        # draft token appended, queried causally up to itself)
        return Workload("verify5-decode-b32-n131072-d576", 32, [131072] * 32, 576, 64, 64, 128,
                        64, 2048, 128, seed=5, outlier_frac=0.01, prefill_tokens=5)
    if i == 7:
        # pool-aware prefill: a chunk whose Full layer gives every query its own
        # pool of blocks, followed by a Reindex layer over those pools
        return Workload("pool-prefill-t256-after-n65536-d576", 2, [65536] * 2, 576, 64, 64, 128,
                        64, 2048, 128, seed=6, outlier_frac=0.01, prefill_tokens=256,
                        layers=[FULL, REINDEX])
    if i == 8:
        # the 128K decode step with the indexer keys stored as MXFP4 (68 bytes
        # per position instead of 128)
        return Workload("full-decode-b32-n131072-d576-mxfp4-keys", 32, [131072] * 32, 576, 64, 64,
                        128, 64, 2048, 128, seed=1, outlier_frac=0.01, idx_format="mxfp4")
    if i == 9:
        # one decode token through the whole model's 38 CSA2 layers (synth.model:
        # three encoder caches of m = 2 entries, one decoder cache); lengths
        # count tokens
        return Workload("model-decode-38-layers-b32-n131072-d576", 32, [131072] * 32, 576, 64, 64,
                        128, 64, 2048, 128, seed=7, outlier_frac=0.01)
    raise ValueError(f"no workload {i}")


WORKLOADS = {i: get_workload for i in range(1, 8)}
