"""GPU parity at the full sizes of the benchmark workloads, in the launch
configuration bench.py times:

* 128K-context Full-layer decode (B = 32): cache bytes of sequences 0 and 31
  and 1% of the other rows bit-exact; top-k and pool of all 32 sequences;
  attention of all 32 sequences;
* the same decode with MXFP4 indexer keys: key codes and block scales of
  sequences 0 and 31 and 1% of the other rows bit-exact; top-k, pool and
  attention of sequences 0, 9, 22, 31;
* 1M-context Full -> Reindex -> Reuse group (B = 16): sequences 0, 7, 15;
* ragged paged mixed-mode decode (B = 64): 8 sequences covering the modes;
* prefill chunk of 4,096 tokens after 262,144: 64 sampled query rows (the
  first 16, the last 16 and 32 random) and every appended row.

Every checked attention row is compared: over the oracle's selection when the
GPU's equals it, else over the GPU's selection once it has passed the
tie-band check (``checks.attended_set``).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import fp4_kv_cache_rope_gb300 as K  # noqa: E402
import synth  # noqa: E402
from oracle import csa2 as O  # noqa: E402
from oracle.workload import SeqRef  # noqa: E402
from synth.device import DeviceWorkload, gen_rows_normal, supplied_pool, supplied_prior  # noqa: E402
from synth.workloads import FULL, REINDEX, REUSE, get_workload  # noqa: E402

from checks import attended_set, check_attention, check_select  # noqa: E402


def dev_rows(dw, b, positions):
    c = dw.cache
    phys = [c.physical_row(b, int(t)) for t in positions]
    ix = torch.tensor(phys, dtype=torch.long, device="cuda")
    return (c.codes.index_select(0, ix).cpu().numpy(), c.scales.index_select(0, ix).cpu().numpy(),
            c.idx_k.index_select(0, ix).cpu().numpy())


def alloc_outputs(B, k, tq=1):
    return (torch.full((B, tq, k), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, tq), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, tq, K.POOL_BLOCKS), -7, dtype=torch.int32, device="cuda"),
            torch.full((B, tq), -7, dtype=torch.int32, device="cuda"))


def full_layer_checks(wl, dw, seqs, layer=0):
    B, k = wl.batch, wl.topk
    inp = dw.layer_inputs(layer)
    oi, oc, pool, pc = alloc_outputs(B, k)
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, 1, None, None, B, k, oi, oc,
                 pool, pc, dw.ws)
    out = torch.empty((B, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_decode(dw.cache, inp["q"].view(torch.int16), wl.heads, oi.view(B, k), oc.view(B), k,
                  inp["swa"], None, wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    o = out.cpu().numpy()
    refs = {}
    for b in seqs:
        ref = SeqRef(wl, b)
        s, ridx, rpool = ref.full(layer, k)
        n = ref.n
        gi = oi[b, 0, : int(oc[b, 0])].cpu().numpy()
        check_select(gi, s, np.arange(n), k, f"topk b={b}")
        bm = O.block_maxima(s)
        gp = pool[b, 0, : int(pc[b, 0])].cpu().numpy()
        check_select(gp, bm, np.arange(len(bm)), K.POOL_BLOCKS, f"pool b={b}")
        check_attention(o[b], ref.attention(layer, attended_set(gi, ridx)), f"attention b={b}")
        refs[b] = (ref, ridx, rpool, gi, gp)
    return refs, (oi, oc, pool, pc)


@pytest.fixture(scope="module")
def w2():
    wl = get_workload(2)
    return wl, DeviceWorkload(wl)


def test_w2_cache_bytes(w2):
    wl, dw = w2
    rng = np.random.default_rng(2)
    for b in range(wl.batch):
        n = wl.lengths[b]
        pos = np.arange(n) if b in (0, wl.batch - 1) else np.sort(rng.choice(n, n // 100, replace=False))
        codes, scales, idxk = dev_rows(dw, b, pos)
        ref = SeqRef(wl, b)
        rc, rs = ref.cache_rows(pos)
        assert np.array_equal(codes[:, : wl.dim // 2], rc), b
        assert np.array_equal(scales[:, : wl.dim // 16], rs), b
        assert np.array_equal(idxk[:, : wl.idx_dim], ref.idxk_rows(pos)), b


def test_w2_full_layer_all_sequences(w2):
    wl, dw = w2
    full_layer_checks(wl, dw, range(wl.batch))


@pytest.fixture(scope="module")
def w8():
    wl = get_workload(8)
    return wl, DeviceWorkload(wl)


def test_w8_mxfp4_key_bytes(w8):
    """MXFP4 indexer keys of the 128K decode (B = 32): E2M1 codes and E8M0
    block scales of sequences 0 and 31 in full, 1% of the other rows."""
    wl, dw = w8
    rng = np.random.default_rng(8)
    c = dw.cache
    for b in range(wl.batch):
        n = wl.lengths[b]
        pos = np.arange(n) if b in (0, wl.batch - 1) else np.sort(rng.choice(n, n // 100, replace=False))
        ix = torch.tensor([c.physical_row(b, int(t)) for t in pos], dtype=torch.long, device="cuda")
        codes = c.idx_k.index_select(0, ix).cpu().numpy()
        scales = c.idx_scales.index_select(0, ix).cpu().numpy()
        rc, rs = SeqRef(wl, b).idxk_rows(pos)
        assert np.array_equal(codes[:, : wl.idx_dim // 2], rc), b
        assert np.array_equal(scales[:, : wl.idx_dim // O.MX_BLOCK], rs), b


def test_w8_mxfp4_full_layer_sampled_sequences(w8):
    wl, dw = w8
    full_layer_checks(wl, dw, (0, 9, 22, wl.batch - 1))


def test_w3_group_full_reindex_reuse():
    wl = get_workload(3)
    dw = DeviceWorkload(wl)
    B, k = wl.batch, wl.topk
    seqs = (0, 7, 15)
    refs, (oi, oc, pool, pc) = full_layer_checks(wl, dw, seqs, 0)
    inp1 = dw.layer_inputs(1)
    ri = torch.full((B, 1, k), -7, dtype=torch.int32, device="cuda")
    rc = torch.full((B, 1), -7, dtype=torch.int32, device="cuda")
    K.index_reindex(dw.cache, inp1["q_idx"], inp1["w"], wl.idx_heads, 1, None, pool, pc, None, B,
                    k, ri, rc, dw.ws)
    outs = {}
    for L in (1, 2):
        inp = dw.layer_inputs(L)
        out = torch.empty((B, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
        K.attn_decode(dw.cache, inp["q"].view(torch.int16), wl.heads, ri.view(B, k), rc.view(B), k,
                      inp["swa"], None, wl.window, 0.0, out, dw.ws)
        outs[L] = out.cpu().numpy()
    assert K.get_status(dw.ws) == 0
    for b in seqs:
        ref, ridx, rpool, gi, gp = refs[b]
        # the GPU's Reindex searched the GPU's pool, which check_select accepted
        s2, pos2, r2 = ref.reindex(1, attended_set(gp, rpool), k)
        g2 = ri[b, 0, : int(rc[b, 0])].cpu().numpy()
        check_select(g2, s2, pos2, k, f"reindex b={b}")
        sel = attended_set(g2, r2)
        check_attention(outs[1][b], ref.attention(1, sel), f"reindex attention b={b}")
        check_attention(outs[2][b], ref.attention(2, sel), f"reuse attention b={b}")


def test_w5_ragged_paged_mixed_modes():
    wl = get_workload(5)
    dw = DeviceWorkload(wl)
    B, k = wl.batch, wl.topk
    modes = wl.modes
    full_ids = [b for b in range(B) if modes[b] == FULL]
    re_ids = [b for b in range(B) if modes[b] == REINDEX]
    ru_ids = [b for b in range(B) if modes[b] == REUSE]
    assert full_ids and re_ids and ru_ids
    idx = torch.zeros((B, 1, k), dtype=torch.int32)
    cnt = torch.zeros((B, 1), dtype=torch.int32)
    pool = torch.zeros((B, 1, K.POOL_BLOCKS), dtype=torch.int32)
    pcnt = torch.zeros((B, 1), dtype=torch.int32)
    for b in re_ids:
        pb = supplied_pool(wl, b, wl.lengths[b])
        pool[b, 0, : len(pb)] = torch.from_numpy(pb)
        pcnt[b, 0] = len(pb)
    for b in ru_ids:
        pr = supplied_prior(wl, b, wl.lengths[b])
        idx[b, 0, : len(pr)] = torch.from_numpy(pr)
        cnt[b, 0] = len(pr)
    idx, cnt, pool, pcnt = idx.cuda(), cnt.cuda(), pool.cuda(), pcnt.cuda()
    inp = [dw.layer_inputs(L) for L in range(3)]
    fid = torch.tensor(full_ids, dtype=torch.int32, device="cuda")
    rid = torch.tensor(re_ids, dtype=torch.int32, device="cuda")
    K.index_full(dw.cache, inp[0]["q_idx"], inp[0]["w"], wl.idx_heads, 1, None, fid, len(full_ids),
                 k, idx, cnt, None, None, dw.ws)
    K.index_reindex(dw.cache, inp[1]["q_idx"], inp[1]["w"], wl.idx_heads, 1, None, pool, pcnt, rid,
                    len(re_ids), k, idx, cnt, dw.ws)
    out = torch.empty((B, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_decode(dw.cache, inp[2]["q"].view(torch.int16), wl.heads, idx.view(B, k), cnt.view(B), k,
                  inp[2]["swa"], None, wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    o = out.cpu().numpy()
    picks = full_ids[:3] + re_ids[:3] + ru_ids[:2]
    for b in picks:
        ref = SeqRef(wl, b)
        n = ref.n
        pos = np.unique(np.r_[np.arange(64), np.arange(n - 64, n)])
        codes, scales, idxk = dev_rows(dw, b, pos)
        rc_, rs_ = ref.cache_rows(pos)
        assert np.array_equal(codes[:, : wl.dim // 2], rc_) and np.array_equal(scales[:, :36], rs_)
        g = idx[b, 0, : int(cnt[b, 0])].cpu().numpy()
        if modes[b] == FULL:
            s, ridx, _ = ref.full(0, k)
            check_select(g, s, np.arange(n), k, f"full b={b}")
        elif modes[b] == REINDEX:
            s2, pos2, ridx = ref.reindex(1, supplied_pool(wl, b, n), k)
            check_select(g, s2, pos2, k, f"reindex b={b}")
        else:
            ridx = supplied_prior(wl, b, n)
            assert np.array_equal(g, ridx)
        check_attention(o[b], ref.attention(2, attended_set(g, ridx)),
                        f"attention b={b} mode={modes[b]}")


def test_w4_prefill_sampled_rows():
    wl = get_workload(4)
    dw = DeviceWorkload(wl)
    B, T, k = wl.batch, wl.prefill_tokens, wl.topk
    n0 = wl.lengths[0]
    kv = gen_rows_normal(wl.seed, synth.T_KV, 0, n0, T, wl.dim)
    ik = gen_rows_normal(wl.seed, synth.T_IDXK, 0, n0, T, wl.idx_dim)
    K.quant_append(dw.cache, kv, ik, T, dw.ws)
    q_pos = (torch.arange(T, dtype=torch.int32, device="cuda") + n0).view(1, T)
    inp = dw.layer_inputs(0, tq=T)
    oi, oc, _, _ = alloc_outputs(B, k, T)
    K.index_full(dw.cache, inp["q_idx"], inp["w"], wl.idx_heads, T, q_pos, None, B, k, oi, oc,
                 None, None, dw.ws)
    out = torch.empty((B, T, wl.heads, wl.dim), dtype=torch.float32, device="cuda")
    K.attn_prefill(dw.cache, inp["q"].view(torch.int16), wl.heads, T, q_pos, oi, oc, k, inp["swa"],
                   wl.window, 0.0, out, dw.ws)
    assert K.get_status(dw.ws) == 0
    ref = SeqRef(wl, 0, n=n0 + T)
    ref.n_prior_positions = n0
    pos = np.arange(n0, n0 + T)
    codes, scales, idxk = dev_rows(dw, 0, pos)
    rc_, rs_ = ref.cache_rows(pos)
    assert np.array_equal(codes[:, : wl.dim // 2], rc_) and np.array_equal(scales[:, :36], rs_)
    assert np.array_equal(idxk[:, : wl.idx_dim], ref.idxk_rows(pos))
    # the first 16, the last 16 and 32 random query rows of the chunk
    rng = np.random.default_rng(4)
    middle = np.arange(16, T - 16)
    rows = sorted(set(range(16)) | set(range(T - 16, T)) |
                  set(rng.choice(middle, 32, replace=False).tolist()))
    assert len(rows) == 64
    ref.idxk_all(n0 + T)      # decode the whole key plane once
    o_all = out[0].cpu().numpy()
    for tq in rows:
        vis = n0 + tq + 1
        s = ref.scores(0, vis, tq, T)
        gi = oi[0, tq, : int(oc[0, tq])].cpu().numpy()
        check_select(gi, s, np.arange(vis), k, f"prefill topk t={tq}")
        ridx = O.topk(s, k)
        check_attention(o_all[tq], ref.attention(0, attended_set(gi, ridx), tq=tq, tq_total=T),
                        f"prefill attention t={tq}")
