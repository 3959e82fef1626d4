"""Benchmark of the CSA2 decode layer-step on GB300 (one JSON line on stdout).

A step is one pass of the whole path over the batch: append the new token's
main-KV and indexer-key rows (RoPE + FP4 quantisation), score and select
(Full: every visible position; Reindex: the pool), and attend over the
selected FP4 rows plus the FP8 window.  The default workload is the
128K-context Full-layer decode (B = 32, N = 131,072, D = 576, k = 2,048).

  python bench.py [--steps K] [--warmup W] [--workload 1..8] [--impl reference]

Workloads (synth/workloads.py): 1 tiny, 2 the 128K decode (default), 3 a CSA2
group (Full + Reindex + Reuse) at 1M, 4 a 4,096-token prefill chunk, 5 ragged
mixed-mode paged decode, 6 a 5-token verify, 7 pool-aware prefill, 8 the 128K
decode with MXFP4 indexer keys.

`value` is layer-steps/s with inputs resident in HBM: the K steps' C-ABI
calls are captured once into a CUDA graph, which is replayed between CUDA
events (`--eager` issues every call from the host instead).  `e2e` repeats
the steps through the same calls with each step's inputs copied from pinned
host memory and the attention output read back (on copy streams that
overlap the compute, double buffered), also as a graph (the eager figure is
reported beside it).  `roofline` is for the indexer kernel (the dominant one),
timed live with CUDA events around each of its launches.  Under torchrun
every rank runs an independent replica (the path does not shard: one GPU per
problem); the JSON line reports the whole job.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HBM_FALLBACK_GBS = 6800.0
EVENT_EVERY = 25  # timed steps per sampled pair of kernel events
# DRAM bytes (read + write) per visible position of indexer_kernel<64,128,false>,
# from one ncu capture of that kernel on 8 of the 32 sequences of the 128K
# decode workload (134.49 MB read + 4.41 MB written for 1,048,592 positions;
# the indexer summary under profiles/).  Scaled to a launch by its visible
# positions; must be re-measured whenever the kernel changes.
INDEXER_TRAFFIC_B_PER_POS = 138.904064e6 / 1048592
# The same figure for the MXFP4-key indexer (71.47 MB read + 0.73 MB written for
# the same 1,048,592 positions; profiles/indexer_kernel_mxfp4-decode-b8-n131072.md).
MX_INDEXER_TRAFFIC_B_PER_POS = 72.197888e6 / 1048592


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return HBM_FALLBACK_GBS, "fallback"


_FP8_PEAK = None


def measure_fp8_peak(n=8192, reps=10, sustain_s=2.0):
    """Dense FP8 (E4M3 x E4M3, fp32 accumulate) tensor throughput of this GPU,
    measured with the library GEMM (torch._scaled_mm, n^3): the best of `reps`
    timed calls (burst) and the mean over about `sustain_s` seconds of back to
    back calls (sustained), in TFLOP/s."""
    import torch
    a = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn)
    b = torch.randn(n, n, device="cuda").to(torch.float8_e4m3fn).t()
    one = torch.ones((), device="cuda", dtype=torch.float32)
    mm = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
    for _ in range(3):
        mm()
    torch.cuda.synchronize()
    flop = 2.0 * n ** 3
    best = 0.0
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        mm()
        e1.record()
        torch.cuda.synchronize()
        best = max(best, flop / (e0.elapsed_time(e1) * 1e-3) / 1e12)
    iters = max(1, int(sustain_s * best * 1e12 / flop))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        mm()
    e1.record()
    torch.cuda.synchronize()
    sustained = flop * iters / (e0.elapsed_time(e1) * 1e-3) / 1e12
    del a, b
    torch.cuda.empty_cache()
    return best, sustained


def fp8_peak():
    """Dense FP8 tensor peak for a kernel timed inside a long step: the
    sustained figure of measure_fp8_peak (measured once per run); without it,
    the measured bf16 burst figure times the nominal fp8/bf16 ratio."""
    global _FP8_PEAK
    if _FP8_PEAK is None:
        try:
            burst, sustained = measure_fp8_peak()
            _FP8_PEAK = (sustained, f"measured in this run: torch._scaled_mm e4m3 8192^3 "
                                    f"sustained {sustained:.0f} TFLOP/s (burst {burst:.0f})")
        except Exception as exc:
            try:
                with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
                    p = json.load(f)
                _FP8_PEAK = (2.0 * float(p["bf16_tflops"]),
                             f"measured bf16 x nominal fp8/bf16 ratio ({type(exc).__name__})")
            except Exception:
                _FP8_PEAK = (2.0 * 1900.0, "fallback bf16 x nominal fp8/bf16 ratio")
    return _FP8_PEAK


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


def max_over_ranks(ms, world, device="cuda"):
    """The slowest rank's time: every rank runs an independent replica, and
    the job's throughput is the units of all ranks over this time."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms):
    """Whole-job units per second for `world` replicas that took `ms` (max over ranks)."""
    return world * units_per_rank / (ms * 1e-3)


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------- workloads
def build_run(wid, extra_capacity, batch=None):
    import torch
    import fp4_kv_cache_rope_gb300 as K
    from synth.device import DeviceWorkload, supplied_pool, supplied_prior
    from synth.workloads import FULL, REINDEX, REUSE, get_workload

    wl = get_workload(wid)
    if batch:                            # smaller batch of the same shapes (profiling)
        wl.batch = batch
        wl.lengths = list(wl.lengths)[:batch]
        if wl.modes is not None:
            wl.modes = list(wl.modes)[:batch]
        wl.name = wl.name + "-first" + str(batch)
    T = max(1, wl.prefill_tokens)         # tokens appended and queried per sequence per step
    wl.extra_capacity = extra_capacity * T
    dw = DeviceWorkload(wl)
    B, k = wl.batch, wl.topk
    layers = wl.layers if wl.modes is None else [FULL]
    n_in = len(layers) if wl.modes is None else 3
    inputs = [dw.layer_inputs(L, tq=T) for L in range(n_in)]
    n0 = torch.tensor(wl.lengths, dtype=torch.int32, device="cuda")
    if wl.prefill_tokens:
        from synth import T_IDXK, T_KV
        from synth.device import gen_rows_normal
        new_kv = torch.stack([gen_rows_normal(wl.seed, T_KV, b, wl.lengths[b], T, wl.dim, dw.mult)
                              for b in range(B)]).contiguous()
        new_idx = torch.stack([gen_rows_normal(wl.seed, T_IDXK, b, wl.lengths[b], T, wl.idx_dim)
                               for b in range(B)]).contiguous()
    else:
        new_kv, new_idx = dw.new_token_inputs(wl.lengths)
        new_kv = new_kv.view(B, 1, wl.dim).contiguous()
        new_idx = new_idx.view(B, 1, wl.idx_dim).contiguous()
    st = dict(wl=wl, dw=dw, K=K, inputs=inputs, n0=n0, new_kv=new_kv, new_idx=new_idx, T=T)
    if wl.prefill_tokens:
        # query positions of step i (counted from the last reset): n_b + i*T + t
        base = torch.tensor(wl.lengths, dtype=torch.int32).view(1, B, 1)
        steps_i = torch.arange(extra_capacity, dtype=torch.int32).view(-1, 1, 1) * T
        st["q_pos_all"] = (base + steps_i + torch.arange(T, dtype=torch.int32).view(1, 1, T)).to("cuda")
    st["idx"] = [torch.zeros((B, T, k), dtype=torch.int32, device="cuda") for _ in range(3)]
    st["cnt"] = [torch.zeros((B, T), dtype=torch.int32, device="cuda") for _ in range(3)]
    st["pool"] = torch.zeros((B, T, K.POOL_BLOCKS), dtype=torch.int32, device="cuda")
    st["pool_cnt"] = torch.zeros((B, T), dtype=torch.int32, device="cuda")
    out_shape = (B, T, wl.heads, wl.dim) if wl.prefill_tokens else (B, wl.heads, wl.dim)
    st["out"] = [torch.empty(out_shape, dtype=torch.float32, device="cuda") for _ in range(3)]
    if wl.modes is not None:
        modes = wl.modes
        full_ids = [b for b in range(B) if modes[b] == FULL]
        re_ids = [b for b in range(B) if modes[b] == REINDEX]
        ru_ids = [b for b in range(B) if modes[b] == REUSE]
        st["full_ids"] = torch.tensor(full_ids, dtype=torch.int32, device="cuda")
        st["re_ids"] = torch.tensor(re_ids, dtype=torch.int32, device="cuda")
        pool = torch.zeros((B, 1, K.POOL_BLOCKS), dtype=torch.int32)
        pcnt = torch.zeros((B, 1), dtype=torch.int32)
        for b in re_ids:
            pb = supplied_pool(wl, b, wl.lengths[b])
            pool[b, 0, : len(pb)] = torch.from_numpy(pb)
            pcnt[b, 0] = len(pb)
        idx = torch.zeros((B, 1, k), dtype=torch.int32)
        cnt = torch.zeros((B, 1), dtype=torch.int32)
        for b in ru_ids:
            pr = supplied_prior(wl, b, wl.lengths[b])
            idx[b, 0, : len(pr)] = torch.from_numpy(pr)
            cnt[b, 0] = len(pr)
        st["pool"].copy_(pool)
        st["pool_cnt"].copy_(pcnt)
        st["idx"][0].copy_(idx)
        st["cnt"][0].copy_(cnt)
        st["counts"] = dict(full=len(full_ids), reindex=len(re_ids), reuse=len(ru_ids))
    torch.cuda.synchronize()
    return st


def append_roofline(wl, rows, ms, peak):
    """Algorithmic bytes of one quant_append launch of `rows` rows (read the
    fp32 row, the fp32 indexer key and the position's cos/sin row of the
    rotary table; write the FP4 codes, the E4M3 scales and the indexer key)
    over its event-timed duration, against the measured HBM peak."""
    per_row = (wl.dim * 4 + wl.idx_dim * 4 + wl.rope_dim * 4 + wl.dim // 2 + wl.dim // 16
               + wl.idx_entry_bytes())
    b = rows * per_row
    gbs = b / (ms * 1e-3) / 1e9 if ms > 0 else None
    return {"rows_per_launch": rows, "bytes_per_launch": b, "launch_us": ms * 1e3,
            "achieved_gbs": gbs, "peak": peak, "unit": "GB/s",
            "frac": gbs / peak if gbs else None}


def append_launches(wl, T):
    """Kernel launches of one quant_append of T tokens per sequence."""
    groups = wl.batch * T * (wl.dim + wl.idx_dim) // 16
    return 1 if groups <= 8 * 512 else 2


def index_launches(rows):
    """Kernel launches of one index call over `rows` query rows."""
    return 2 if rows <= 1024 else 3


def arm(K, family, pair):
    """Brackets the next launches of a kernel family with the CUDA events of
    `pair` (None disarms)."""
    if pair is not None:
        K.set_launch_events(family, pair[0], pair[1])


def disarm(K, family, pair):
    if pair is not None:
        K.set_launch_events(family)


def step_multi_query(st, i, ev=None, ev_attn=None, ev_more=None):
    """One step of a multi-query workload: T new tokens per sequence appended,
    then every layer of the chunk (Full, optionally Reindex over the Full
    layer's per-query pools) indexed and attended for all T queries."""
    K, wl, dw, ins, T = st["K"], st["wl"], st["dw"], st["inputs"], st["T"]
    B, k, ws, c = wl.batch, wl.topk, dw.ws, dw.cache
    q_pos = st["q_pos_buf"] if "q_pos_buf" in st else st["q_pos_all"][i]
    em = ev_more or {}
    arm(K, K.KERNEL_QUANT, em.get("append"))
    K.quant_append(c, st["new_kv"], st["new_idx"], T, ws)
    disarm(K, K.KERNEL_QUANT, em.get("append"))
    launches = append_launches(wl, T)
    reindex = len(wl.layers) > 1
    if ev is not None:
        K.set_launch_events(K.KERNEL_INDEXER, ev[0], ev[1])
    arm(K, K.KERNEL_SELECT, em.get("select"))
    K.index_full(c, ins[0]["q_idx"], ins[0]["w"], wl.idx_heads, T, q_pos, None, B, k,
                 st["idx"][0], st["cnt"][0], st["pool"] if reindex else None,
                 st["pool_cnt"] if reindex else None, ws)
    disarm(K, K.KERNEL_SELECT, em.get("select"))
    if ev is not None:
        K.set_launch_events(K.KERNEL_INDEXER)
    launches += index_launches(B * T)
    if reindex:
        K.index_reindex(c, ins[1]["q_idx"], ins[1]["w"], wl.idx_heads, T, q_pos, st["pool"],
                        st["pool_cnt"], None, B, k, st["idx"][1], st["cnt"][1], ws)
        launches += index_launches(B * T)
    for L in range(len(wl.layers)):
        sel = 0 if L == 0 else 1
        if ev_attn is not None and L == 0:
            K.set_launch_events(K.KERNEL_ATTENTION, ev_attn[0], ev_attn[1])
        K.attn_prefill(c, ins[L]["q"].view(st["q_dtype"]), wl.heads, T, q_pos, st["idx"][sel],
                       st["cnt"][sel], k, ins[L]["swa"], wl.window, 0.0, st["out"][L], ws)
        if ev_attn is not None and L == 0:
            K.set_launch_events(K.KERNEL_ATTENTION)
        launches += 1
    return launches


def step(st, ev=None, ev_attn=None, i=0, ev_more=None):
    """One layer-step (or one CSA2 group step for the group workload)."""
    K, wl, dw, ins = st["K"], st["wl"], st["dw"], st["inputs"]
    if wl.prefill_tokens:
        return step_multi_query(st, i, ev, ev_attn, ev_more)
    B, k, ws, c = wl.batch, wl.topk, dw.ws, dw.cache
    em = ev_more or {}
    arm(K, K.KERNEL_QUANT, em.get("append"))
    K.quant_append(c, st["new_kv"], st["new_idx"], 1, ws)
    disarm(K, K.KERNEL_QUANT, em.get("append"))
    launches = 1  # quant_append (one cluster launch that also advances seq_len)
    if ev is not None:
        K.set_launch_events(K.KERNEL_INDEXER, ev[0], ev[1])
    if wl.modes is None:
        # Full layer (layer 0); the group workload adds Reindex and Reuse
        arm(K, K.KERNEL_SELECT, em.get("select"))
        K.index_full(c, ins[0]["q_idx"], ins[0]["w"], wl.idx_heads, 1, None, None, B, k,
                     st["idx"][0], st["cnt"][0], st["pool"], st["pool_cnt"], ws)
        disarm(K, K.KERNEL_SELECT, em.get("select"))
        if ev is not None:
            K.set_launch_events(K.KERNEL_INDEXER)
        launches += 2
        if ev_attn is not None:
            K.set_launch_events(K.KERNEL_ATTENTION, ev_attn[0], ev_attn[1])
        K.attn_decode(c, ins[0]["q"].view(st["q_dtype"]), wl.heads, st["idx"][0].view(B, k),
                      st["cnt"][0].view(B), k, ins[0]["swa"], None, wl.window, 0.0, st["out"][0], ws)
        if ev_attn is not None:
            K.set_launch_events(K.KERNEL_ATTENTION)
        launches += st["attn_launches"]
        if len(wl.layers) > 1:
            K.index_reindex(c, ins[1]["q_idx"], ins[1]["w"], wl.idx_heads, 1, None, st["pool"],
                            st["pool_cnt"], None, B, k, st["idx"][1], st["cnt"][1], ws)
            launches += 2
            for L in (1, 2):
                K.attn_decode(c, ins[L]["q"].view(st["q_dtype"]), wl.heads, st["idx"][1].view(B, k),
                              st["cnt"][1].view(B), k, ins[L]["swa"], None, wl.window, 0.0,
                              st["out"][L], ws)
                launches += st["attn_launches"]
    else:
        nf, nr = st["counts"]["full"], st["counts"]["reindex"]
        if nf:
            arm(K, K.KERNEL_SELECT, em.get("select"))
            K.index_full(c, ins[0]["q_idx"], ins[0]["w"], wl.idx_heads, 1, None, st["full_ids"],
                         nf, k, st["idx"][0], st["cnt"][0], None, None, ws)
            disarm(K, K.KERNEL_SELECT, em.get("select"))
            launches += 2
        if ev is not None:
            K.set_launch_events(K.KERNEL_INDEXER)
        if nr:
            K.index_reindex(c, ins[1]["q_idx"], ins[1]["w"], wl.idx_heads, 1, None, st["pool"],
                            st["pool_cnt"], st["re_ids"], nr, k, st["idx"][0], st["cnt"][0], ws)
            launches += 2
        if ev_attn is not None:
            K.set_launch_events(K.KERNEL_ATTENTION, ev_attn[0], ev_attn[1])
        K.attn_decode(c, ins[2]["q"].view(st["q_dtype"]), wl.heads, st["idx"][0].view(B, k),
                      st["cnt"][0].view(B), k, ins[2]["swa"], None, wl.window, 0.0, st["out"][0], ws)
        if ev_attn is not None:
            K.set_launch_events(K.KERNEL_ATTENTION)
        launches += st["attn_launches"]
    return launches


def layers_per_step(wl):
    return len(wl.layers) if wl.modes is None else 1


def indexer_flops_per_launch(wl, n_at):
    """FP8 tensor flops of the Full indexer launch of a multi-query step:
    2 * Hi * di per (query, visible position); query t of sequence b sees
    n_b + t + 1 positions once its chunk is appended (n_at = lengths before)."""
    T = wl.prefill_tokens
    vis = sum(n * T + T * (T + 1) // 2 for n in n_at)
    return 2 * wl.idx_heads * wl.idx_dim * vis


def indexer_bytes_per_launch(wl, n_at):
    """Algorithmic bytes of the (first) indexer launch of a step: every scored
    position's indexer key (di bytes in E4M3; di/2 + di/32 in MXFP4)."""
    kb = wl.idx_entry_bytes()
    if wl.prefill_tokens:
        return sum(n + wl.prefill_tokens for n in n_at) * kb
    if wl.modes is None:
        return sum(n_at) * kb
    return sum(n for n, m in zip(n_at, wl.modes) if m == 0) * kb


def roofline_bytes_per_step(wl, n_at):
    """Roofline bytes of one step: indexer keys read + gathered FP4 entries
    (D/2 + D/16 B) + FP8 window rows, per layer of the step."""
    e = wl.dim // 2 + wl.dim // 16
    kb = wl.idx_entry_bytes()
    total = 0
    if wl.prefill_tokens:  # keys read once per layer, gathers per query
        T = wl.prefill_tokens
        for L, mode in enumerate(wl.layers):
            for n in n_at:
                if mode == 0:
                    total += (n + T) * kb
                else:
                    total += T * min(2048, -(-(n + T) // 8)) * 8 * kb
                total += T * (min(wl.topk, n + T) * e) + (T + wl.window - 1) * wl.dim
        return total
    for L, mode in enumerate(wl.layers if wl.modes is None else [None]):
        for b, n in enumerate(n_at):
            m = mode if mode is not None else wl.modes[b]
            if m == 0:
                total += n * kb
            elif m == 1:
                total += min(2048, -(-n // 8)) * 8 * kb
            total += min(wl.topk, n) * e + wl.window * wl.dim
    return total


# ------------------------------------------------------------- CPU baseline
ORACLE_FORM = ("the C++ oracle (oracle/cref.cpp: fp64 loops, one thread per core, pinned "
               "against the numpy oracle); the seeded inputs come from the numpy generators")
def cpu_baseline(wl, per_piece_s=2.0, target_s=10.0, max_rounds=200):
    """The oracle on the host cores over one bounded sample of the workload's
    layer-step: the pieces of oracle_plan (the same plan the reference arm
    times), run in rounds until about target_s of CPU work is sampled, each
    piece's mean time weighted by the share of the step it stands for."""
    pieces, layers, text = oracle_plan(wl, per_piece_s)
    times = [[] for _ in pieces]
    total, rounds = 0.0, 0
    while rounds < max_rounds and (rounds == 0 or total < target_s):
        for j, (run, _w) in enumerate(pieces):
            t0 = time.perf_counter()
            run()
            dt = time.perf_counter() - t0
            times[j].append(dt)
            total += dt
        rounds += 1
    step_s = sum(w * statistics.mean(t) for (_, w), t in zip(pieces, times))
    from oracle import cref as CR
    return {"value": layers / step_s, "unit": "layer-steps/s", "cores": CR.threads(),
            "kind": "oracle",
            "sample": f"{text}; the {len(pieces)} pieces run in {rounds} rounds, {ORACLE_FORM}",
            "seconds_sampled": total}


def _score_fn(wl, inp, ik, tq=0):
    """Oracle indexer scores (the C++ restatement, one thread per core) of
    query row tq against key positions [lo, hi)."""
    from oracle import cref as CR

    def score(lo, hi):
        if wl.idx_format == "mxfp4":
            return CR.indexer_scores_mx(inp["q_idx"][tq], inp["w"][tq], ik[0][lo:hi],
                                        ik[1][lo:hi], wl.idx_dim)
        return CR.indexer_scores(inp["q_idx"][tq], inp["w"][tq], ik[lo:hi])
    return score


def _slices(score, n, per_step_s):
    """Cut the scoring of n positions into slices of about per_step_s each."""
    probe_n = min(n, 8192)
    t0 = time.perf_counter()
    score(0, probe_n)
    per_pos = (time.perf_counter() - t0) / max(1, probe_n)
    m = max(1, min(256, math.ceil(per_pos * n / per_step_s)))
    cuts = [n * j // m for j in range(m + 1)]
    return [(lambda lo=cuts[j], hi=cuts[j + 1]: score(lo, hi)) for j in range(m)]


def oracle_plan(wl, per_step_s):
    """One layer-step of workload `wl` on the oracle, as bounded pieces.

    Returns (pieces, layers, text): pieces is a list of (callable, weight),
    and one step of the workload takes sum(weight * time of the piece).  A
    Full scan is cut into slices of positions (a position's score depends
    on its own key only), each about per_step_s of CPU time; the rest of a
    sequence's work (append, selection, dequantisation, attention) is one
    piece.  Sequences of one kind are represented by one of them, weighted
    by their number (or, for Full scans of ragged lengths, by their summed
    length).  Inputs are prepared outside the pieces."""
    import numpy as np
    import synth
    from oracle import cref as CR
    from oracle.formats import bf16_bits_to_f64
    from oracle.workload import SeqRef as SeqRefNumpy
    from synth.host import host_rows_normal, supplied_pool, supplied_prior
    from synth.workloads import FULL, REINDEX, REUSE
    B, k = wl.batch, wl.topk
    CR.build()

    def SeqRef(*a, **kw):   # every arithmetic step through the C++ oracle
        return SeqRefNumpy(*a, cpp=True, **kw)

    if wl.name.startswith("model-"):
        run = model_oracle_sample(wl, 0, wl.lengths[0])
        return [(run, B)], 38, (f"sequence 0's 38 CSA2 layers of one decode token (4 Full and 4 "
                                f"Reindex scans, selections, 38 attentions), weight {B}")

    def decode_parts(b, n, layer):
        ref = SeqRef(wl, b, n=n)
        ik = ref.idxk_all(n)
        inp = ref.inputs(layer)
        score = _score_fn(wl, inp, ik)
        s_full = score(0, n)
        newrow = host_rows_normal(wl.seed, synth.T_KV, b, [n], wl.dim, ref.mult)
        q64 = bf16_bits_to_f64(inp["q_bf16"][0])
        swa_codes = inp["swa"][: wl.window]

        def tail():
            CR.quant_append_rows(newrow, np.array([n]), ref.cos, ref.sin, wl.rope_dim)
            idx, pool = CR.full_select(s_full, k)
            return CR.sparse_attention(q64, np.concatenate([ref.dequant_rows(idx),
                                                            CR.e4m3_decode(swa_codes)]))
        return ref, score, s_full, tail

    def attend(ref, layer, idx, tq=0, tq_total=1):
        return lambda: ref.attention(layer, idx, tq=tq, tq_total=tq_total)

    if wl.prefill_tokens:
        # one query row of the chunk stands for all T: its scan slices are
        # weighted by the chunk's summed visible length over its own, its
        # selection + attention by T; the chunk's append is one more piece
        T = wl.prefill_tokens
        n0 = wl.lengths[0]
        tm = T // 2
        ref = SeqRef(wl, 0, n=n0 + T)
        ref.n_prior_positions = n0
        ik = ref.idxk_all(n0 + T)
        inp = ref.inputs(0, T)
        vis = n0 + tm + 1
        score = _score_fn(wl, inp, ik, tm)
        s_full = score(0, vis)
        rows = host_rows_normal(wl.seed, synth.T_KV, 0, np.arange(n0, n0 + T), wl.dim, ref.mult)
        total_vis = sum(n * T + T * (T + 1) // 2 for n in wl.lengths)
        pieces = [(f, total_vis / vis) for f in _slices(score, vis, per_step_s)]

        def tail():
            idx, pool = CR.full_select(s_full, k)
            return ref.attention(0, idx, tq=tm, tq_total=T)
        pieces.append((tail, B * T))
        pieces.append((lambda: CR.quant_append_rows(rows, np.arange(n0, n0 + T), ref.cos, ref.sin,
                                                    wl.rope_dim), B))
        return pieces, len(wl.layers), (
            f"query row {tm} of the {T}-token chunk: its scan of {vis} positions in "
            f"{len(pieces) - 2} slices weighted by the chunk's summed visible length, its "
            f"selection + attention weighted by {B * T}; the chunk's append as one piece"
            + ("; Reindex layers are not timed" if len(wl.layers) > 1 else ""))

    if wl.modes is None:
        n = wl.lengths[0]
        ref, score, s_full, tail = decode_parts(0, n, 0)
        pieces = [(f, B) for f in _slices(score, n, per_step_s)] + [(tail, B)]
        text = (f"sequence 0 of {B}: its Full scan of {n} positions in {len(pieces) - 1} slices, "
                f"then append + select + dequantise + attend; each piece weighted by {B}")
        if len(wl.layers) > 1:   # the group: Reindex over the Full layer's pool, then Reuse
            idx, pool = CR.full_select(s_full, k)
            _, _, r_idx = ref.reindex(1, pool, k)

            def reindex():
                _, _, ri = ref.reindex(1, pool, k)
                return ref.attention(1, ri)
            pieces += [(reindex, B), (attend(ref, 2, r_idx), B)]
            text += "; its Reindex (score the pool, select, attend) and Reuse (attend), weight " \
                    f"{B} each"
        return pieces, len(wl.layers), text

    # ragged mixed modes: one sequence per mode stands for all of its mode
    lens, modes = wl.lengths, wl.modes
    full = [b for b in range(B) if modes[b] == FULL]
    rei = [b for b in range(B) if modes[b] == REINDEX]
    reu = [b for b in range(B) if modes[b] == REUSE]
    pieces, parts = [], []
    if full:
        mean = sum(lens[b] for b in full) / len(full)
        bf = min(full, key=lambda b: abs(lens[b] - mean))
        ref, score, s_full, tail = decode_parts(bf, lens[bf], 0)
        w = sum(lens[b] for b in full) / lens[bf]
        sl = _slices(score, lens[bf], per_step_s)
        pieces += [(f, w) for f in sl] + [(tail, len(full))]
        parts.append(f"Full: sequence {bf} ({lens[bf]} positions) scanned in {len(sl)} slices "
                     f"weighted by the Full sequences' summed length over its own, its tail "
                     f"weighted by {len(full)}")
    if rei:
        br = rei[0]
        ref = SeqRef(wl, br)
        pool = supplied_pool(wl, br, lens[br])

        def reindex():
            _, _, ri = ref.reindex(1, pool, k)
            return ref.attention(2, ri)
        pieces.append((reindex, len(rei)))
        parts.append(f"Reindex: sequence {br} (score its pool, select, attend), weight {len(rei)}")
    if reu:
        bu = reu[0]
        ref = SeqRef(wl, bu)
        pieces.append((attend(ref, 2, supplied_prior(wl, bu, lens[bu])), len(reu)))
        parts.append(f"Reuse: sequence {bu} (attend), weight {len(reu)}")
    return pieces, 1, "; ".join(parts)


def reference_arm(args, budget_s=90.0):
    """The oracle on the host cores.  Step i runs piece i mod P of the
    workload's layer-step (oracle_plan), with the pieces sized (and a short
    piece repeated within its step) so that the warm-up and timed steps
    together take about budget_s whatever --steps is.  `value` is
    layer-steps/s from each piece's mean time and weight; `ms_per_step` is
    the measured wall time of one timed step."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from synth.workloads import get_workload
    wl = get_workload(args.workload)
    per_step = budget_s / max(1, args.steps + args.warmup)
    pieces, layers, text = oracle_plan(wl, per_step)
    # a piece shorter than the per-step share runs several times per step
    reps = []
    for j, (run, _w) in enumerate(pieces):
        t0 = time.perf_counter()
        run()
        reps.append(max(1, min(1000, int(per_step / max(time.perf_counter() - t0, 1e-6)))))
    for i in range(args.warmup):
        pieces[i % len(pieces)][0]()
    times = [[] for _ in pieces]
    t_all = time.perf_counter()
    for i in range(args.steps):
        j = i % len(pieces)
        for _ in range(reps[j]):
            t0 = time.perf_counter()
            pieces[j][0]()
            times[j].append(time.perf_counter() - t0)
    dt = time.perf_counter() - t_all
    missing = [j for j, t in enumerate(times) if not t]
    for j in missing:  # fewer steps than pieces: time the rest once, outside the step count
        t0 = time.perf_counter()
        pieces[j][0]()
        times[j].append(time.perf_counter() - t0)
    step_s = sum(w * statistics.mean(t) for (_, w), t in zip(pieces, times))
    value = layers / step_s
    sample = (f"step i = piece i mod {len(pieces)} of one layer-step, run "
              f"{'/'.join(str(r) for r in reps)} times per step (piece by piece): {text}; "
              f"{ORACLE_FORM}")
    from oracle import cref as CR
    cpu = {"value": value, "unit": "layer-steps/s", "cores": CR.threads(), "kind": "oracle",
           "sample": sample}
    line = {"impl": "reference",
            "metric": ("CSA2 decode layer-steps/s (achieved HBM GB/s vs GB300 peak in roofline)"
                       if not wl.prefill_tokens else
                       f"CSA2 multi-query layer-steps/s ({wl.prefill_tokens} tokens per sequence "
                       f"per step)"),
            "value": value, "unit": "layer-steps/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / max(1, args.steps) * 1e3,
            "layer_step_ms_estimated": step_s / layers * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": wl.name, "batch": wl.batch, "ctx": max(wl.lengths),
                       "topk": wl.topk, "window": wl.window, "dim": wl.dim,
                       "idx_heads": wl.idx_heads, "heads": wl.heads, "parallelism": "single",
                       "launch": "host oracle",
                       "tokens_per_step": wl.batch * max(1, wl.prefill_tokens)},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "layer-steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "timed_s": dt}
    print(json.dumps(line), flush=True)


# ------------------------------------------------- whole-model decode step
def model_oracle_sample(base, b, positions_n):
    """One sequence of one model decode token on the oracle: the 38 CSA2
    layers (4 Full scans, 4 Reindex scans, 38 attentions) over caches holding
    positions_n tokens.  Inputs are prepared untimed; returns the timed work."""
    from oracle.workload import SeqRef
    from fp4_kv_cache_rope_gb300.schedule import FULL, REINDEX, layer_plan
    from synth.model import model_workloads
    wls = model_workloads(base)
    entries = [positions_n // 2] * 3 + [positions_n]
    refs = [SeqRef(wl, b, n=entries[c], cpp=True) for c, wl in enumerate(wls)]
    plan = layer_plan()
    for p in plan:
        refs[p.cache].inputs(p.layer)
    for r in refs:
        r.idxk_all()

    def run():
        sel, pool = {}, None
        for p in plan:
            ref = refs[p.cache]
            if p.mode == FULL:
                s, idx, pl = ref.full(p.layer, base.topk)
                sel[p.layer] = idx
                if p.cache == 3:
                    pool = pl
            elif p.mode == REINDEX:
                sel[p.layer] = ref.reindex(p.layer, pool, base.topk)[2]
            ref.attention(p.layer, sel[p.selection])
    return run


def model_bench(args):
    """bench.py --workload 9: one decode token per sequence through the
    model's 38 CSA2 layers per step (fp4_kv_cache_rope_gb300.schedule)."""
    import torch
    import fp4_kv_cache_rope_gb300 as K
    from fp4_kv_cache_rope_gb300.schedule import REUSE, DecodeSchedule
    from synth.model import ModelInputs
    from synth.workloads import get_workload
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    base = get_workload(9)
    if args.batch:
        base.batch = args.batch
        base.lengths = base.lengths[: args.batch]
        base.name += "-first" + str(args.batch)
    base.extra_capacity = args.steps + args.warmup + 16
    m = ModelInputs(base)
    sch = DecodeSchedule(m.caches, m.workspaces, base.heads, base.idx_heads, base.topk,
                         base.window)
    B, n0 = base.batch, list(base.lengths)
    tok = [m.token_inputs([n + par for n in n0]) for par in (0, 1)]   # even / odd token rows
    starts = [c.seq_len.clone() for c in m.caches]
    layers_per = len(sch.plan)

    def reset():
        for c, s0 in zip(m.caches, starts):
            c.seq_len.copy_(s0)
        for w in m.workspaces:
            K.reset_status(w)
        torch.cuda.synchronize()

    # kernel events in a second replay of the timed steps, >= 8 per kernel
    every = max(1, min(EVENT_EVERY, args.steps // 8))
    sampled = lambda i: i % every == every // 2
    watch = {(20, "index"): K.KERNEL_INDEXER, (2, "index"): K.KERNEL_INDEXER,
             (24, "index"): K.KERNEL_INDEXER}
    # one attention launch of each launch size (layers per launch), the
    # decoder's first launch (layers 20..) among them
    attn_key = {}
    for c in sorted(sch.chunks, key=lambda c: c[0].layer != 20):
        attn_key.setdefault(len(c), (c[0].layer, "attention"))
    for key in attn_key.values():
        watch[key] = K.KERNEL_ATTENTION
    n_ev = sum(1 for i in range(args.steps) if sampled(i))
    evs = {key: [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(max(n_ev, 1))] for key in watch}
    for lst in evs.values():
        for a, b in lst:
            a.record()
            b.record()
    torch.cuda.synchronize()

    def one_step(i, inputs=None, out=None, token=None, take=False, j=0):
        dec, enc = token if token is not None else tok[i % 2]
        sch.append(dec[0], dec[1], enc)

        def hook(p, phase, before):
            key = (p.layer, phase)
            if take and key in watch:
                if before:
                    K.set_launch_events(watch[key], *evs[key][j])
                else:
                    K.set_launch_events(watch[key])
        sch.layers(inputs or m.inputs, out or m.out, hook if take else None)
        return sch.launches(enc is not None)

    def run_steps(n, with_events=False):
        cnt = 0
        for i in range(n):
            take = with_events and sampled(i)
            cnt += one_step(i, take=take, j=i // every)
        return cnt

    reset()
    run_steps(args.warmup)
    reset()
    graph = graph_ev = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            launches = run_steps(args.steps)
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev, capture_error_mode="thread_local"):
            run_steps(args.steps, True)
        reset()
        graph_ev.replay()
        reset()
        graph.replay()
        torch.cuda.synchronize()
        reset()
    clocks = ClockSampler(local)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t0.record()
    if graph is not None:
        graph.replay()
    else:
        launches = run_steps(args.steps)
    t1.record()
    torch.cuda.synchronize()
    time.sleep(0.1)
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    status = [K.get_status(w) for w in m.workspaces]
    reset()                           # the kernel-timing replay of the same steps
    if graph_ev is not None:
        graph_ev.replay()
    else:
        run_steps(args.steps, True)
    torch.cuda.synchronize()
    status = [s0 | K.get_status(w) for s0, w in zip(status, m.workspaces)]
    us = {f"{l}:{ph}": statistics.mean(a.elapsed_time(b) for a, b in evs[(l, ph)][:n_ev]) * 1e3
          for (l, ph) in watch}
    value = job_throughput(layers_per * args.steps, world, ms)
    # the dominant kernel: the attention launches (len(sch.chunks) per step,
    # each over one to several layers) against 8 indexer launches; attention
    # flops = 4 H (k + W) D per sequence and layer; the roofline is taken on
    # the decoder's first launch (layers 20..)
    dec_chunk = next(c for c in sch.chunks if c[0].layer == 20)
    attn_flops = 4.0 * base.heads * (base.topk + base.window) * base.dim * B * len(dec_chunk)
    attn_us = us["20:attention"]
    attn_step_us = sum(us["%d:attention" % attn_key[len(c)][0]] for c in sch.chunks)
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tf_peak, tf_kind = float(json.load(f)["bf16_tflops_sustained"]), "measured (sustained)"
    except Exception:
        tf_peak, tf_kind = 1700.0, "fallback (sustained)"
    ach = attn_flops / (attn_us * 1e-6) / 1e12
    idx_total = us["20:index"] + 3 * us["2:index"] + 4 * us["24:index"]
    roofline = {"bound": "tensor", "kernel": "attention_kernel", "achieved": ach, "peak": tf_peak,
                "unit": "TFLOP/s", "frac": ach / tf_peak, "traffic": None, "peak_source": tf_kind,
                "flops_per_launch": attn_flops, "launch_us": attn_us,
                "layers_per_launch": len(dec_chunk),
                "share_of_step": attn_step_us / (ms / args.steps * 1e3),
                "timed_launches": n_ev,
                "sampling": f"CUDA events around the attention launch of layers "
                            f"{dec_chunk[0].layer}-{dec_chunk[-1].layer} of every {every}th step, "
                            f"in a second replay of the {args.steps} timed steps"}
    del graph, graph_ev

    # ---- e2e through the API: per step the appended rows and every layer's
    # query-side inputs are copied from pinned host memory, and the last
    # layer's output is read back; copies on two streams, double buffered.
    modes = {p.layer: p.mode for p in sch.plan}
    need = lambda L: ("q", "swa") if modes[L] == REUSE else ("q", "swa", "q_idx", "w")
    host = {}
    for L, inp in m.inputs.items():
        for name in need(L):
            host[(L, name)] = inp[name].cpu().pin_memory()
    for par in (0, 1):
        dec, enc = tok[par]
        host[("dec", par, 0)], host[("dec", par, 1)] = dec[0].cpu().pin_memory(), dec[1].cpu().pin_memory()
        if enc is not None:
            for g in range(3):
                for r in range(3):
                    host[("enc", g, r)] = enc[g][r].cpu().pin_memory()
    bufs = []
    for _ in range(2):
        dev_inputs = {L: {n: torch.empty_like(inp[n]) for n in need(L)}
                      for L, inp in m.inputs.items()}
        dev_dec = [torch.empty_like(t) for t in tok[0][0]]
        dev_enc = [tuple(torch.empty_like(t) for t in tok[1][1][g]) for g in range(3)]
        out = {L: (torch.empty_like(o) if L == 39 else o) for L, o in m.out.items()}
        bufs.append((dev_inputs, dev_dec, dev_enc, out, torch.empty(m.out[39].shape).pin_memory()))
    h2d_even = sum(t.numel() * t.element_size() for k_, t in host.items()
                   if k_[0] not in ("dec", "enc") or (k_[0] == "dec" and k_[1] == 0))
    h2d_odd = sum(t.numel() * t.element_size() for k_, t in host.items()
                  if k_[0] not in ("dec", "enc") or (k_[0] == "dec" and k_[1] == 1) or k_[0] == "enc")
    d2h = m.out[39].numel() * 4
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    e_steps = max(args.steps // 4, 10)
    pool = [torch.cuda.Event() for _ in range(3 * e_steps + 6)]
    for e in pool:
        e.record()
    torch.cuda.synchronize()

    def e2e_steps(n):
        comp = torch.cuda.current_stream()
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        in_ready, comp_done, out_done = pool[0:n], pool[n:2 * n], pool[2 * n:3 * n]

        def issue_h2d(i):
            di, dd, de, _, _ = bufs[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])
                for L, inp in di.items():
                    for name, t in inp.items():
                        t.copy_(host[(L, name)], non_blocking=True)
                par = i % 2
                dd[0].copy_(host[("dec", par, 0)], non_blocking=True)
                dd[1].copy_(host[("dec", par, 1)], non_blocking=True)
                if par:
                    for g in range(3):
                        for r in range(3):
                            de[g][r].copy_(host[("enc", g, r)], non_blocking=True)
                in_ready[i].record(s_in)

        issue_h2d(0)
        for i in range(n):
            if i + 1 < n:
                issue_h2d(i + 1)
            di, dd, de, out, pinned = bufs[i % 2]
            comp.wait_event(in_ready[i])
            if i >= 2:
                comp.wait_event(out_done[i - 2])
            one_step(i, inputs=di, out=out, token=((dd[0], dd[1]), de if i % 2 else None))
            comp_done[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                pinned.copy_(out[39], non_blocking=True)
                out_done[i].record(s_out)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)

    def timed(fn):
        reset()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        return job_throughput(layers_per * e_steps, world, max_over_ranks(e0.elapsed_time(e1), world))

    reset()
    e2e_steps(2)
    e2e_eager = timed(lambda: e2e_steps(e_steps))
    e2e_graph, e2e_note = None, None
    if not args.eager:
        try:
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, capture_error_mode="thread_local"):
                e2e_steps(e_steps)
            reset()
            g2.replay()
            e2e_graph = timed(g2.replay)
            del g2
        except Exception as exc:
            e2e_note = f"graph capture of the copies failed: {type(exc).__name__}: {exc}"[:200]
            torch.cuda.synchronize()
    e2e_value = e2e_graph if e2e_graph is not None else e2e_eager

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        run = model_oracle_sample(base, 0, n0[0])
        t = time.perf_counter()
        run()
        dt = time.perf_counter() - t
        cpu = {"value": layers_per / (dt * B), "unit": "layer-steps/s", "cores": os.cpu_count(),
               "kind": "oracle",
               "sample": f"sequence 0 of {B}: its 38 CSA2 layers of one decode token (4 Full and "
                         f"4 Reindex scans, selections, 38 attentions) in numpy fp64, scaled to "
                         f"the batch", "seconds_per_sequence": dt}
    if rank == 0:
        line = {
            "metric": "CSA2 decode layer-steps/s, whole-model schedule (38 CSA2 layers per token)",
            "value": value, "unit": "layer-steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3/e2m1 storage; fp8 and f16 tensor-core MMA, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": base.name, "batch": B, "ctx_tokens": max(n0),
                       "encoder_entries": max(n0) // 2, "topk": base.topk, "window": base.window,
                       "layers_per_step": layers_per,
                       "model_steps_per_s": value / layers_per,
                       "parallelism": "replicas" if world > 1 else "single",
                       "launch": "eager" if args.eager else "cuda_graph",
                       "l2": "inputs exceed L2 (four caches of 1-2 GB)"},
            "roofline": roofline,
            "kernels_us": {"decoder_full_indexer": us["20:index"],
                           "encoder_full_indexer": us["2:index"],
                           "reindex_indexer": us["24:index"],
                           "attention_launch": {"layers %d-%d" % (c[0].layer, c[-1].layer):
                                                us["%d:attention" % c[0].layer]
                                                for c in sch.chunks
                                                if (c[0].layer, "attention") in watch},
                           "attention_launches_per_step": len(sch.chunks),
                           "indexers_per_step": idx_total, "attention_per_step": attn_step_us},
            "e2e": {"value": e2e_value, "unit": "layer-steps/s",
                    "h2d_bytes_per_step": (h2d_even + h2d_odd) / 2, "d2h_bytes_per_step": d2h,
                    "steps": e_steps, "cuda_graph": e2e_graph is not None, "eager_value": e2e_eager,
                    "copies": "per step: appended rows and every layer's query-side inputs in, "
                              "the last layer's output back, on two copy streams",
                    **({"note": e2e_note} if e2e_note else {})},
            "gpu_launches": launches,
            "clocks": clk,
            "device_status": status,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


# -------------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-budget", type=float, default=90.0,
                    help="--impl reference: seconds of oracle work over warm-up + timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batch", type=int, default=0, help="use only the first B sequences")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from the host instead of replaying a CUDA graph")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return reference_arm(args, args.ref_budget)
    if args.workload == 9:
        return model_bench(args)

    import numpy as np
    import torch
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    from synth.workloads import get_workload
    T_chunk = max(1, get_workload(args.workload).prefill_tokens)
    if T_chunk >= 64:  # long chunks: a bounded number of steps keeps the cache in range
        args.steps = min(args.steps, 64)
    st = build_run(args.workload, args.steps + args.warmup + 16, args.batch or None)
    wl, K = st["wl"], st["K"]
    st["q_dtype"] = torch.int16
    st["attn_launches"] = 1  # split-K partials are merged inside the attention kernel
    B = wl.batch

    def reset():
        st["dw"].cache.seq_len.copy_(st["n0"])
        K.reset_status(st["dw"].ws)
        torch.cuda.synchronize()

    # ---- device-resident timed loop
    # `value` comes from the K timed steps with nothing else in them.  The
    # per-kernel times come from a second replay of the same K steps in which
    # the indexer and attention launches of every `every`-th step are
    # bracketed by CUDA events (an event node between two kernels costs GPU
    # time and stops the next launch from overlapping the previous kernel's
    # tail), at least 8 launches of each whatever K is.
    every = max(1, min(EVENT_EVERY, args.steps // 8))

    def sampled(i):
        return i % every == every // 2

    def run_steps(n, evs=None, evas=None, state=None, evms=None):
        count = 0
        for i in range(n):
            j = i // every
            take = evs is not None and sampled(i)
            count += step(state or st, evs[j] if take else None, evas[j] if take else None, i,
                          evms[j] if take and evms is not None else None)
        return count

    reset()
    run_steps(args.warmup)            # eager warm-up: loads every kernel before any capture
    reset()
    n_start = list(wl.lengths)
    n_ev = sum(1 for i in range(args.steps) if sampled(i))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(max(n_ev, 1))]
    eva = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(max(n_ev, 1))]
    evm = [{key: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for key in ("append", "select")} for _ in range(max(n_ev, 1))]
    for a, b in ev + eva + [pr for d in evm for pr in d.values()]:   # torch creates the CUDA event on the first record
        a.record()
        b.record()
    torch.cuda.synchronize()
    graph = graph_ev = None
    if not args.eager:
        # The K timed steps, unrolled into one CUDA graph; a second graph of
        # the same steps carries the sampled kernel events (external records,
        # i.e. event nodes timed on every replay).
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, capture_error_mode="thread_local"):
            launches = run_steps(args.steps)
        graph_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_ev, capture_error_mode="thread_local"):
            run_steps(args.steps, ev, eva, evms=evm)
        reset()
        graph_ev.replay()             # warm-up replays (untimed)
        reset()
        graph.replay()
        torch.cuda.synchronize()
        reset()
    t_begin, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_begin.record()
    if graph is not None:
        graph.replay()
    else:
        launches = run_steps(args.steps)
    t_end.record()
    torch.cuda.synchronize()
    time.sleep(0.1)
    clk = clocks.stop()
    ms = t_begin.elapsed_time(t_end)
    ms = max_over_ranks(ms, world)
    status = K.get_status(st["dw"].ws)
    # the kernel-timing replay of the same steps
    reset()
    if graph_ev is not None:
        graph_ev.replay()
    else:
        run_steps(args.steps, ev, eva, evms=evm)
    torch.cuda.synchronize()
    status |= K.get_status(st["dw"].ws)
    idx_ms = [a.elapsed_time(b) for a, b in ev[:n_ev]]
    attn_ms = [a.elapsed_time(b) for a, b in eva[:n_ev]]
    app_ms = [d["append"][0].elapsed_time(d["append"][1]) for d in evm[:n_ev]]
    sel_ms = [d["select"][0].elapsed_time(d["select"][1]) for d in evm[:n_ev]]
    # bytes of the sampled indexer launches (visible length grows by T per step)
    T = st["T"]
    if wl.prefill_tokens:
        before = lambda i: [n + i * T for n in n_start]  # lengths before step i's append
        idx_bytes = [indexer_bytes_per_launch(wl, before(i)) for i in range(args.steps) if sampled(i)]
        roof_bytes = [roofline_bytes_per_step(wl, before(i)) for i in range(args.steps)]
    else:
        idx_bytes = [indexer_bytes_per_launch(wl, [n + i + 1 for n in n_start])
                     for i in range(args.steps) if sampled(i)]
        roof_bytes = [roofline_bytes_per_step(wl, [n + i + 1 for n in n_start])
                      for i in range(args.steps)]
    ach = sum(idx_bytes) / (sum(idx_ms) * 1e-3) / 1e9
    traffic = None
    if wl.idx_heads == 64 and wl.idx_dim == 128 and not wl.prefill_tokens:
        per_pos = (MX_INDEXER_TRAFFIC_B_PER_POS if wl.idx_format == "mxfp4"
                   else INDEXER_TRAFFIC_B_PER_POS)
        if per_pos is not None:
            traffic = per_pos * statistics.mean(idx_bytes) / wl.idx_entry_bytes()
    peak, peak_kind = peaks()
    if wl.prefill_tokens:
        # T query rows per sequence against the same keys: the indexer is a
        # dense FP8 contraction, reported against the tensor peak
        flops = [indexer_flops_per_launch(wl, before(i)) for i in range(args.steps) if sampled(i)]
        tf_ach = sum(flops) / (sum(idx_ms) * 1e-3) / 1e12
        tf_peak, tf_kind = fp8_peak()
        roofline = {"bound": "tensor", "kernel": "indexer_kernel", "achieved": tf_ach,
                    "peak": tf_peak, "unit": "TFLOP/s", "frac": tf_ach / tf_peak,
                    "traffic": None, "peak_source": tf_kind,
                    "flops_per_launch": statistics.mean(flops)}
    else:
        roofline = {"bound": "hbm", "kernel": "indexer_kernel", "achieved": ach, "peak": peak,
                    "unit": "GB/s", "frac": ach / peak, "traffic": traffic,
                    "peak_source": peak_kind, "bytes_per_launch": statistics.mean(idx_bytes)}
    roofline.update({"launch_us": statistics.mean(idx_ms) * 1e3, "timed_launches": len(idx_ms),
                     "sampling": f"CUDA events around the launches of every {every}th step, in a "
                                 f"second replay of the {args.steps} timed steps"})
    ms_step = ms / args.steps
    value = job_throughput(layers_per_step(wl) * args.steps, world, ms)
    path_gbs = sum(roof_bytes) / (ms * 1e-3) / 1e9
    del graph, graph_ev

    # ---- end-to-end through the C ABI with host buffers.  Every step copies
    # its inputs from pinned host memory and reads its attention output back.
    # The copies run on their own streams with double-buffered device tensors,
    # so step i+1's inputs and step i's outputs move while step i computes.
    reset()
    ins = st["inputs"]
    keys = [("new_kv", st["new_kv"]), ("new_idx", st["new_idx"])]
    if wl.prefill_tokens:  # the step's query positions are an input too
        keys.append(("q_pos", st["q_pos_all"][0]))
        host_qpos = st["q_pos_all"].cpu().pin_memory()
    for L, d in enumerate(ins):
        for name in ("q_idx", "w", "q", "swa"):
            keys.append((f"{name}{L}", d[name]))
    host = {name: t.cpu().pin_memory() for name, t in keys}
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    nl = layers_per_step(wl)
    bufs = []
    for _ in range(2):
        dev = {name: torch.empty_like(t) for name, t in keys}
        sb = dict(st)
        sb["new_kv"], sb["new_idx"] = dev["new_kv"], dev["new_idx"]
        if wl.prefill_tokens:
            sb["q_pos_buf"] = dev["q_pos"]
        sb["inputs"] = [{n: dev[f"{n}{L}"] for n in ("q_idx", "w", "q", "swa")}
                        for L in range(len(ins))]
        sb["out"] = [torch.empty_like(o) for o in st["out"]]
        pinned = [torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in st["out"][:nl]]
        bufs.append((dev, sb, pinned))
    d2h = sum(o.numel() * o.element_size() for o in bufs[0][2])
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    e_steps = max(args.steps // 4, 20)
    pool = [torch.cuda.Event() for _ in range(3 * e_steps + 6)]
    for e in pool:  # create the CUDA events before any capture
        e.record()
    torch.cuda.synchronize()

    def e2e_steps(n):
        comp = torch.cuda.current_stream()
        s_in.wait_stream(comp)
        s_out.wait_stream(comp)
        in_ready, comp_done, out_done = pool[0:n], pool[n:2 * n], pool[2 * n:3 * n]

        def issue_h2d(i):
            dev = bufs[i % 2][0]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[i - 2])  # buffer i % 2 was read by step i-2
                for name in host:
                    src = host_qpos[i] if name == "q_pos" else host[name]
                    dev[name].copy_(src, non_blocking=True)
                in_ready[i].record(s_in)

        issue_h2d(0)
        for i in range(n):
            if i + 1 < n:
                issue_h2d(i + 1)
            sb, pinned = bufs[i % 2][1], bufs[i % 2][2]
            comp.wait_event(in_ready[i])
            if i >= 2:
                comp.wait_event(out_done[i - 2])  # outputs of step i-2 were read back
            step(sb, i=i)
            comp_done[i].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[i])
                for o, src in zip(pinned, sb["out"]):
                    o.copy_(src, non_blocking=True)
                out_done[i].record(s_out)
        comp.wait_stream(s_in)
        comp.wait_stream(s_out)

    def timed(fn):
        reset()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        torch.cuda.synchronize()
        e_ms = e0.elapsed_time(e1)
        e_ms = max_over_ranks(e_ms, world)
        return job_throughput(layers_per_step(wl) * e_steps, world, e_ms)

    reset()
    e2e_steps(3)
    e2e_eager = timed(lambda: e2e_steps(e_steps))
    e2e_graph, e2e_note = None, None
    if not args.eager:
        try:
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, capture_error_mode="thread_local"):
                e2e_steps(e_steps)
            reset()
            g2.replay()
            e2e_graph = timed(g2.replay)
            del g2
        except Exception as exc:   # report the eager figure and why
            e2e_note = f"graph capture of the copies failed: {type(exc).__name__}: {exc}"[:200]
            torch.cuda.synchronize()
    e2e_value = e2e_graph if e2e_graph is not None else e2e_eager

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)
        # the oracle's wall time per layer-step and the path bytes it covers per second
        per_layer_step = statistics.mean(roof_bytes) / layers_per_step(wl)
        cpu["ms_per_layer_step"] = 1e3 / cpu["value"]
        cpu["path_gbs"] = cpu["value"] * per_layer_step / 1e9
    if rank == 0:
        line = {
            "metric": ("CSA2 decode layer-steps/s (achieved HBM GB/s vs GB300 peak in roofline)"
                       if not wl.prefill_tokens else
                       f"CSA2 multi-query layer-steps/s ({T} tokens per sequence per step)"),
            "value": value, "unit": "layer-steps/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3/e2m1 storage; fp8 and f16 tensor-core MMA, f32 accumulate",
            "data": "synthetic",
            "config": {"workload": wl.name, "batch": B, "ctx": max(n_start), "topk": wl.topk,
                       "window": wl.window, "dim": wl.dim, "idx_heads": wl.idx_heads,
                       "heads": wl.heads, "parallelism": "replicas" if world > 1 else "single",
                       "launch": "eager" if args.eager else "cuda_graph",
                       "tokens_per_step": B * T,
                       "l2": f"inputs exceed L2 ({roof_bytes[0] / 1e6:.0f} MB read per step)"},
            "roofline": roofline,
            "path_hbm": {"bytes_per_step": statistics.mean(roof_bytes), "achieved_gbs": path_gbs,
                         "frac": path_gbs / peak},
            "kernels_us": {"indexer": statistics.mean(idx_ms) * 1e3,
                           "attention": statistics.mean(attn_ms) * 1e3,
                           "select": statistics.mean(sel_ms) * 1e3,
                           "append": statistics.mean(app_ms) * 1e3},
            "append": append_roofline(wl, B * st["T"], statistics.mean(app_ms), peak),
            "e2e": {"value": e2e_value, "unit": "layer-steps/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e_steps,
                    "cuda_graph": e2e_graph is not None, "eager_value": e2e_eager,
                    "copies": "per step, on two copy streams overlapping the compute "
                              "(double-buffered device inputs and outputs)",
                    **({"note": e2e_note} if e2e_note else {})},
            "gpu_launches": launches,
            "clocks": clk,
            "device_status": status,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
