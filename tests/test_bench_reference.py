"""bench.py --impl reference: the oracle arm prints one JSON line with the
GPU arm's metric, unit and config keys, times every piece of a layer-step,
reports the measured wall time per step, and stays within its time budget,
for decode, multi-query and ragged mixed-mode workloads."""
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_ref(*args):
    t0 = time.time()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--ref-budget", "4", *args], capture_output=True, text=True,
                         timeout=600, cwd=ROOT)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [x for x in out.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0]), time.time() - t0


def test_reference_arm_line_on_the_tiny_decode():
    d, wall = run_ref("--workload", "1", "--steps", "40", "--warmup", "3")
    assert d["impl"] == "reference"
    assert d["metric"].startswith("CSA2 decode layer-steps/s")
    assert d["unit"] == "layer-steps/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["e2e"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    for key in ("workload", "batch", "ctx", "topk", "window", "dim", "idx_heads", "heads"):
        assert key in d["config"], key
    assert d["steps"] == 40 and d["warmup"] == 3
    assert wall < 300


def test_reference_arm_multi_query_workload():
    d, wall = run_ref("--workload", "6", "--steps", "3", "--warmup", "0")
    assert d["impl"] == "reference" and "unavailable" not in d
    assert d["metric"].startswith("CSA2 multi-query layer-steps/s")
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["layer_step_ms_estimated"] > 0
    assert d["config"]["tokens_per_step"] == 32 * 5
    assert wall < 300


def test_reference_arm_ragged_mixed_modes():
    d, wall = run_ref("--workload", "5", "--steps", "4", "--warmup", "0")
    assert d["impl"] == "reference" and d["value"] > 0
    sample = d["cpu_baseline"]["sample"]
    assert "Full:" in sample and "Reindex:" in sample and "Reuse:" in sample
    assert wall < 400


def test_cpu_baseline_times_the_cpp_oracle():
    """The GPU arm's cpu_baseline: the C++ oracle's pieces in rounds until
    the target time is sampled; cores = the oracle's thread count."""
    sys.path.insert(0, ROOT)
    import bench
    from oracle import cref
    from synth.workloads import get_workload
    r = bench.cpu_baseline(get_workload(1), target_s=0.3)
    assert r["kind"] == "oracle" and r["unit"] == "layer-steps/s" and r["value"] > 0
    assert r["cores"] == cref.threads()
    assert r["seconds_sampled"] >= 0.3
    assert "C++ oracle" in r["sample"] and "rounds" in r["sample"]
