"""bench.py's host-only parts on the CPU: the reference arm (the FP64 oracle
timed on a bounded sample) prints the contract's JSON line, other ranks of a
multi-rank launch print nothing, and the per-step sample shrinks to a causal
prefix when a whole document would overrun its time budget."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_bench(args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    r = run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "2", "--warmup", "3"])
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    assert j["impl"] == "reference" and j["value"] > 0 and j["steps"] == 2
    assert j["unit"] == "TFLOP/s" and j["higher_is_better"] is True
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["value"] == j["value"]
    assert j["e2e"] == {"value": j["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}


def test_reference_arm_other_ranks_are_silent():
    r = run_bench(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3",
                   "--gpus", "2"], env={"RANK": "1", "LOCAL_RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_cpu_baseline_prefix_sample():
    sys.path.insert(0, ROOT)
    import bench
    from precision_causal_attention_block_gb300 import workloads as W
    w = W.fixed4x4096()
    cb = bench.cpu_baseline(w, budget_s=0.3)
    assert cb["value"] > 0 and "causal prefix" in cb["sample"]
    full = bench.cpu_baseline(W.tiny(), budget_s=5.0)
    assert full["value"] > 0 and "document(s)" in full["sample"]
