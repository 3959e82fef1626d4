"""Oracle view of a workload: the reference result of one sequence (or one
query row) computed from the seeded host inputs of ``synth`` with the oracle's
own codecs and steps.  Test infrastructure only; imports nothing from the
CUDA path.
"""
from __future__ import annotations

import numpy as np

import synth
from synth.host import host_layer_inputs, host_rows_normal
from synth.workloads import Workload

from . import cref as CR
from . import csa2 as O
from . import formats as F


class SeqRef:
    """Reference quantities of sequence ``b`` of workload ``wl``."""

    def __init__(self, wl: Workload, b: int, n: int | None = None, cos=None, sin=None,
                 cpp: bool = False):
        # cpp: the arithmetic steps (FP4 append, scores, selection,
        # dequantisation, attention) through the C++ restatement
        # (oracle/cref.cpp) instead of numpy; the inputs are the same
        self.cpp = cpp
        self.wl, self.b = wl, b
        self.n = wl.lengths[b] if n is None else n
        self.mult = (synth.outlier_multipliers(wl.seed, wl.dim, wl.outlier_frac)
                     if wl.outlier_frac else None)
        if cos is None:
            cos, sin = synth.rope_table(wl.max_len, wl.rope_dim, wl.theta)
        self.cos, self.sin = cos, sin
        self._idxk = None
        self._idxk_n = 0
        self._inputs = {}

    # ---- cache contents ----------------------------------------------------
    def cache_rows(self, positions):
        """(codes, scales) the cache must hold at ``positions`` (entries; for an
        m = 2 cache each entry compresses source rows 2j and 2j+1)."""
        positions = np.asarray(positions, dtype=np.int64)
        if getattr(self.wl, "compress", 1) == 2:
            src = np.stack([2 * positions, 2 * positions + 1], axis=1).reshape(-1)
            x = host_rows_normal(self.wl.seed, synth.T_KV, self.b, src, self.wl.dim, self.mult)
            z = host_rows_normal(self.wl.seed, synth.T_Z, self.b, src, self.wl.dim) * np.float32(2.0)
            x = (CR if self.cpp else O).compress_pairs(x, z)
        else:
            x = host_rows_normal(self.wl.seed, synth.T_KV, self.b, positions, self.wl.dim, self.mult)
        qa = CR.quant_append_rows if self.cpp else O.quant_append_rows
        return qa(x, positions, self.cos, self.sin, self.wl.rope_dim)

    @property
    def mx_keys(self):
        return getattr(self.wl, "idx_format", "e4m3") == "mxfp4"

    def idxk_rows(self, positions):
        """Stored indexer-key bytes at ``positions``: E4M3 codes, or for MXFP4
        keys the pair (E2M1 codes, E8M0 scales)."""
        x = host_rows_normal(self.wl.seed, synth.T_IDXK, self.b, positions, self.wl.idx_dim)
        return O.quantize_mxfp4(x) if self.mx_keys else O.fp8_cast(x)

    def idxk_all(self, n=None):
        n = self.n if n is None else n
        if self._idxk is None or self._idxk_n < n:
            self._idxk = self.idxk_rows(np.arange(n))
            self._idxk_n = n
        if self.mx_keys:
            return self._idxk[0][:n], self._idxk[1][:n]
        return self._idxk[:n]

    def _scores_of(self, inp, tq, keys):
        """Scores of query ``tq`` against stored keys (either format)."""
        if self.cpp:
            if self.mx_keys:
                return CR.indexer_scores_mx(inp["q_idx"][tq], inp["w"][tq], keys[0], keys[1],
                                            self.wl.idx_dim)
            return CR.indexer_scores(inp["q_idx"][tq], inp["w"][tq], keys)
        if self.mx_keys:
            q = F.e4m3_decode(inp["q_idx"][tq]).reshape(self.wl.idx_heads, -1)
            return O.indexer_scores_values(
                q, inp["w"][tq], O.dequantize_mxfp4(keys[0], keys[1], self.wl.idx_dim))
        return O.indexer_scores(inp["q_idx"][tq], inp["w"][tq], keys)

    def dequant_rows(self, positions):
        codes, scales = self.cache_rows(positions)
        return (CR if self.cpp else O).dequantize_fp4(codes, scales, self.wl.dim)

    # ---- one layer ---------------------------------------------------------
    def inputs(self, layer, tq=1):
        if (layer, tq) not in self._inputs:
            h = host_layer_inputs(self.wl, layer, self.b, tq)
            h["q_idx"] = O.fp8_cast(h["q_idx_f32"])
            h["swa"] = O.fp8_cast(h["swa_f32"])
            self._inputs[(layer, tq)] = h
        return self._inputs[(layer, tq)]

    def scores(self, layer, n=None, tq=0, tq_total=1):
        inp = self.inputs(layer, tq_total)
        n = self.n if n is None else n
        return self._scores_of(inp, tq, self.idxk_all(n))

    def full(self, layer, k, n=None, tq=0, tq_total=1):
        s = self.scores(layer, n, tq, tq_total)
        idx, pool = (CR if self.cpp else O).full_select(s, k)
        return s, idx, pool

    def reindex(self, layer, pool, k, n=None, tq=0, tq_total=1):
        """Reindex query tq of layer `layer` over the positions of `pool`
        visible below n."""
        inp = self.inputs(layer, tq_total)
        n = self.n if n is None else n
        pos = O.pool_positions(pool, n)
        if self._idxk is not None and self._idxk_n >= n:
            kp = ((self._idxk[0][pos], self._idxk[1][pos]) if self.mx_keys
                  else self._idxk[pos])
        else:
            kp = self.idxk_rows(pos)
        s = self._scores_of(inp, tq, kp)
        return s, pos, (CR if self.cpp else O).topk(s, k, ids=pos)

    def attention(self, layer, idx, swa_count=None, tq=0, tq_total=1, scale=None):
        """Decode attention (tq_total == 1) or prefill row tq."""
        inp = self.inputs(layer, tq_total)
        wl = self.wl
        q = synth_bf16_to_f64(inp["q_bf16"][tq])
        rows = [self.dequant_rows(np.asarray(idx))] if len(idx) else [np.zeros((0, wl.dim))]
        swa_decode = CR.e4m3_decode if self.cpp else O.swa_rows_decode
        if tq_total == 1:
            wc = wl.window if swa_count is None else swa_count
            rows.append(swa_decode(inp["swa"][:wc]))
        else:
            band = O.swa_band_rows(self.n_prior_positions, tq, wl.window)
            rows.append(swa_decode(inp["swa"][band]))
        return (CR if self.cpp else O).sparse_attention(q, np.concatenate(rows), scale)

    n_prior_positions = 0


def synth_bf16_to_f64(bits):
    from .formats import bf16_bits_to_f64
    return bf16_bits_to_f64(bits)
