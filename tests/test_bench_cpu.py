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


def test_profiled_traffic_only_for_unchanged_sources(tmp_path, monkeypatch):
    """The roofline line's DRAM traffic comes from a profile summary only while
    the kernel sources it lists hash to the recorded digest; any change to
    them turns it into null (a figure measured on other code)."""
    import hashlib
    import shutil
    sys.path.insert(0, ROOT)
    import bench
    from precision_causal_attention_block_gb300 import workloads as W
    csrc = tmp_path / "precision_causal_attention_block_gb300" / "csrc"
    shutil.copytree(os.path.join(ROOT, "precision_causal_attention_block_gb300", "csrc"), csrc)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    w = W.tiny()
    srcs = ["attn_bwd.cu", "ptx.cuh"]
    h = hashlib.sha256()
    for s in srcs:
        h.update((csrc / s).read_bytes())
    name = f"{bench.bwd_kernel_name(w, False)}_{w.name.replace('_', '', 1)}.md"
    prof = tmp_path / "profiles" / name
    prof.write_text("# summary\n\n    traffic_bytes_per_launch: 123456\n"
                    f"    sources: {' '.join(srcs)}\n    sources_sha256: {h.hexdigest()}\n")
    assert bench.profiled_traffic(w, False) == 123456
    # no summary for the mixed path's kernel
    assert bench.profiled_traffic(w, True) is None
    # a changed source invalidates the figure
    (csrc / "ptx.cuh").write_text((csrc / "ptx.cuh").read_text() + "\n// changed\n")
    assert bench.profiled_traffic(w, False) is None
