"""Synthetic inputs of a whole-model CSA2 decode: three encoder caches of
m = 2 entries and one decoder cache, the per-layer query-side inputs, and the
rows each decode token appends.  Seeded generators only (no arithmetic of the
method): the tests and bench.py feed the same tensors to the CUDA path and,
through oracle.workload.SeqRef, to the oracle.
"""
from __future__ import annotations

from dataclasses import replace

from .workloads import Workload


def model_workloads(base: Workload) -> list:
    """The four cache workloads of a model whose sequences hold base.lengths
    tokens: encoder caches 0..2 (entries = tokens // 2, m = 2) and the decoder
    cache 3 (entries = tokens).  Each cache draws its own rows (its own seed);
    layer l's query-side inputs come from the workload of the cache it reads."""
    out = []
    for g in range(3):
        out.append(replace(base, name=f"{base.name}-enc{g}", seed=base.seed * 16 + 1 + g,
                           lengths=[n // 2 for n in base.lengths], compress=2,
                           extra_capacity=base.extra_capacity // 2 + 8))
    out.append(replace(base, name=f"{base.name}-dec", seed=base.seed * 16 + 4, compress=1))
    return out


class ModelInputs:
    """Device caches, workspaces and inputs of a whole-model decode."""

    def __init__(self, base: Workload, device="cuda"):
        import torch
        from fp4_kv_cache_rope_gb300.schedule import layer_plan
        from .device import DeviceWorkload, gen_rows_normal
        from . import T_IDXK
        self.base = base
        self.wls = model_workloads(base)
        self.dws = [DeviceWorkload(wl, device=device) for wl in self.wls]
        self.plan = layer_plan()
        self.inputs = {}
        for p in self.plan:
            inp = self.dws[p.cache].layer_inputs(p.layer)
            inp["q"] = inp["q"].view(torch.int16)
            self.inputs[p.layer] = inp
        B = base.batch
        self.out = {p.layer: torch.empty((B, base.heads, base.dim), dtype=torch.float32,
                                         device=device) for p in self.plan}
        self._gen_rows = gen_rows_normal
        self._t_idxk = T_IDXK

    @property
    def caches(self):
        return [dw.cache for dw in self.dws]

    @property
    def workspaces(self):
        return [dw.ws for dw in self.dws]

    def token_inputs(self, positions):
        """Rows appended by the decode token at token positions[b] (all of one
        parity): the decoder entry, and for an odd position the pair
        (positions - 1, positions) of each encoder cache."""
        import torch
        dec = self.dws[3]
        kv, ik = dec.new_token_inputs(positions)
        B = self.base.batch
        dec_in = (kv.view(B, 1, -1).contiguous(), ik.view(B, 1, -1).contiguous())
        odd = [p % 2 for p in positions]
        assert len(set(odd)) == 1, "a batch decodes tokens of one parity"
        enc_in = None
        if odd[0]:
            enc_in = []
            for g in range(3):
                dw, wl = self.dws[g], self.wls[g]
                kvs, zs, iks = [], [], []
                for b, p in enumerate(positions):
                    e = p // 2
                    kv2, z2 = dw.pair_sources(b, e, 1)
                    kvs.append(kv2)
                    zs.append(z2)
                    iks.append(self._gen_rows(wl.seed, self._t_idxk, b, e, 1, wl.idx_dim))
                enc_in.append((torch.stack(kvs).contiguous(), torch.stack(zs).contiguous(),
                               torch.stack(iks).contiguous()))
        return dec_in, enc_in
