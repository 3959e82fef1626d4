"""GPU parity of the whole-model CSA2 decode schedule: two decode tokens (the
second completes a pair, so every encoder cache gains an m = 2 entry) through
the 38 CSA2 layers, every layer checked against the oracle:

* Full layers (2, 8, 14 on the encoder caches, 20 on the decoder cache):
  top-k sets and, for layer 20, the pool;
* Reindex layers (24, 28, 32, 36) over layer 20's pool;
* every layer's attention output (Full, Reindex and the 30 Reuse layers, each
  with its own query and window over its group's selection), where the GPU's
  selection equals the oracle's.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
from checks import attended_set, check_attention, check_select  # noqa: E402
from fp4_kv_cache_rope_gb300.schedule import FULL, REINDEX, DecodeSchedule  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle.workload import SeqRef  # noqa: E402
from synth.model import ModelInputs  # noqa: E402
from synth.workloads import Workload, get_workload  # noqa: E402


def run_two_tokens(base, per_launch=None):
    """Two decode tokens (n even, then n + 1 completing a pair) through the 38
    CSA2 layers; returns the model inputs and the schedule after the second.
    per_launch: layers per attention launch (None: as many as fill the SMs)."""
    m = ModelInputs(base)
    sch = DecodeSchedule(m.caches, m.workspaces, base.heads, base.idx_heads, base.topk,
                         base.window, per_launch)
    n = list(base.lengths)
    for step in range(2):
        pos = [x + step for x in n]
        dec_in, enc_in = m.token_inputs(pos)
        assert (enc_in is not None) == (step == 1)
        sch.append(dec_in[0], dec_in[1], enc_in)
        sch.layers(m.inputs, m.out)
    torch.cuda.synchronize()
    for dw in m.dws:
        assert K.get_status(dw.ws) == 0
    return m, sch


def check_layers(base, m, sch, seqs):
    """Every layer of the second token for sequences `seqs`: selections and
    pools against the oracle's scores, and attention of every layer (over the
    oracle's selection, or the GPU's accepted one where they differ among
    near-ties).  Returns (compared, total)."""
    k = base.topk
    n = list(base.lengths)
    idx = {h: t.cpu().numpy() for h, t in sch.idx.items()}
    cnt = {h: t.cpu().numpy() for h, t in sch.cnt.items()}
    pool, pcnt = sch.pool.cpu().numpy(), sch.pool_cnt.cpu().numpy()
    compared = total = 0
    for b in seqs:
        entries = [(n[b] + 2) // 2] * 3 + [n[b] + 2]
        refs = [SeqRef(wl, b, n=entries[c]) for c, wl in enumerate(m.wls)]
        for c in range(4):
            assert int(m.caches[c].seq_len[b]) == entries[c]
        sel = {}
        rpool = None
        for p in sch.plan:
            ref = refs[p.cache]
            nvis = entries[p.cache]
            if p.mode == FULL:
                s, ridx, rp = ref.full(p.layer, k, n=nvis)
                gi = idx[p.layer][b, : cnt[p.layer][b]]
                check_select(gi, s, np.arange(nvis), k, f"layer {p.layer} b={b}")
                if p.cache == 3:
                    gp = pool[b, 0, : pcnt[b, 0]]
                    check_select(gp, O.block_maxima(s), np.arange(-(-nvis // 8)), K.POOL_BLOCKS,
                                 f"pool b={b}")
                    rpool = attended_set(gp, rp)
                sel[p.layer] = (gi, ridx)
            elif p.mode == REINDEX:
                gi = idx[p.layer][b, : cnt[p.layer][b]]
                s2, pos2, ridx = ref.reindex(p.layer, rpool, k, n=nvis)
                check_select(gi, s2, pos2, k, f"layer {p.layer} b={b}")
                sel[p.layer] = (gi, ridx)
            gi, ridx = sel[p.selection]
            total += 1
            check_attention(m.out[p.layer][b].cpu().numpy(),
                            ref.attention(p.layer, attended_set(gi, ridx)),
                            f"attention layer {p.layer} b={b}")
            compared += 1
    return compared, total


@pytest.mark.parametrize("per_launch", [None, 1, 4])
def test_two_decode_tokens_through_all_layers(per_launch):
    """One layer per attention launch, four, and as many as the group holds
    (None: six encoder layers, four decoder layers per launch at B = 2)."""
    base = Workload("model-mini", 2, [3000, 520], 128, 32, 8, 64, 16, 64, 16, seed=61,
                    outlier_frac=0.02, extra_capacity=8)
    m, sch = run_two_tokens(base, per_launch)
    compared, total = check_layers(base, m, sch, range(base.batch))
    assert compared == total == 38 * base.batch


def test_whole_model_at_full_size():
    """The bench's whole-model workload (B = 32 sequences of 131,072 tokens):
    two decode tokens through all 38 layers, sequences 0 and 31 checked, in
    the bench's launch configuration (four layers per attention launch on 152
    SMs)."""
    base = get_workload(9)
    base.extra_capacity = 8
    m, sch = run_two_tokens(base)
    compared, total = check_layers(base, m, sch, (0, base.batch - 1))
    assert compared == total == 38 * 2
