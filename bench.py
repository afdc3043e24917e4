#!/usr/bin/env python
"""Throughput of the MXFP8 causal attention training call (quantise Q, K, V
-> work list -> forward -> quantise dO with D -> backward) on synthetic packed
inputs, printed as one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload long131072]

The default workload is the largest single-GPU configuration: one causal
document of 131,072 tokens, 32 heads of dimension 64 (MXFP8).

A step is one whole training call over one batch resident in HBM.  FLOPs use
the causal convention 7 * H * d * sum(L^2) (forward 4, backward 10, over the
L^2/2 visible pairs).  With N > 1 (torchrun) every rank runs its own replica
of the workload on its own GPU (weak scaling, no collective on the data path);
the value is the sum over ranks of the work divided by the slowest rank's time.
``--impl reference`` times the FP64 CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_BF16_TFLOPS = 1900.0     # profiling recipe fallback (burst)
FALLBACK_BF16_SUSTAINED = 1700.0
FALLBACK_HBM_GBS = 6800.0
FP8_OVER_BF16 = 2.0               # nominal dense FP8 / BF16 ratio (4.5 / 2.25 PFLOP/s)
L2_FLUSH_BYTES = 256 << 20
STRUCTURE_NOTE = {"rms": "per-head RMS drawn in [0.5, 2]",
                  "outlier20pct1": "1% of channels x20",
                  "outlier16x2": "2 of 64 channels x16", "plain": "no structure"}


def peaks():
    """FP8 tensor peak = the measured BF16 burst GEMM rate x the nominal FP8 /
    BF16 ratio: the roofline kernel is timed alone (one launch of well under a
    second), so the burst figure applies; HBM = the measured copy bandwidth."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        bf16 = p.get("bf16_tflops") or p.get("bf16_tflops_sustained")
        return {"fp8_tflops": float(bf16) * FP8_OVER_BF16, "hbm_gbs": float(p.get("hbm_gbs")),
                "source": "of measured (bf16 burst x nominal fp8/bf16 ratio 2)"}
    return {"fp8_tflops": FALLBACK_BF16_TFLOPS * FP8_OVER_BF16, "hbm_gbs": FALLBACK_HBM_GBS,
            "source": "of fallback (bf16 burst x nominal fp8/bf16 ratio 2)"}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def reduce_max(values, device):
    """Element-wise maximum over ranks (the slowest rank sets the time)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_throughput(flops_per_step, steps, world, slowest_ms):
    """Whole-job TFLOP/s: every rank ran its own replica of the step."""
    return world * flops_per_step * steps / (slowest_ms * 1e-3) / 1e12


def bwd_kernel_name(w, nvfp4):
    return ("attn_bwd128_kernel" if w.d == 128 and not nvfp4 else
            "attn_bwd_kernel_d64_nvfp4" if nvfp4 else f"attn_bwd_kernel_d{w.d}")


def profiled_traffic(w, nvfp4):
    """DRAM bytes per launch of the backward kernel from the committed ncu
    summary of this workload, if the kernel's sources are unchanged since the
    capture (else None)."""
    import hashlib
    import re
    path = os.path.join(ROOT, "profiles",
                        f"{bwd_kernel_name(w, nvfp4)}_{w.name.replace('_', '', 1)}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    t = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    srcs = re.search(r"sources:\s*(.+)", text)
    sha = re.search(r"sources_sha256:\s*([0-9a-f]+)", text)
    if not (t and srcs and sha):
        return None
    h = hashlib.sha256()
    for f in srcs.group(1).split():
        h.update(open(os.path.join(ROOT, "precision_causal_attention_block_gb300", "csrc", f),
                      "rb").read())
    return int(t.group(1)) if h.hexdigest() == sha.group(1) else None


def make_workload(name):
    from precision_causal_attention_block_gb300 import workloads as W
    return W.WORKLOADS[name]()


def run_ours(args, rank, world, local):
    import torch

    from precision_causal_attention_block_gb300 import build as B
    from precision_causal_attention_block_gb300 import flamia as fl
    from precision_causal_attention_block_gb300 import workloads as W

    if not os.path.exists(B.LIB) and rank == 0:
        B.build()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        if not os.path.exists(B.LIB):
            B.build()
        dist.barrier()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = make_workload(args.workload)
    x = W.make_inputs_bf16(w)
    hkv = args.kv_heads or w.H
    if hkv != w.H:  # grouped-query attention: the first hkv heads of K and V
        x["k"], x["v"] = x["k"][:, :hkv].contiguous(), x["v"][:, :hkv].contiguous()
    xd = {n: t.to(dev) for n, t in x.items()}
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    call = fl.TrainingCall(w.T, w.H, w.d, cu, w.sm_scale, nvfp4_qk=args.nvfp4,
                           hadamard=args.hadamard, causal=not args.noncausal, H_kv=hkv,
                           deterministic_dq=args.deterministic, dq_accum=args.dq_accum,
                           schedule=args.schedule, ds_rows=args.ds_rows,
                           token_scales=args.token_scales, bwd_ctas=args.bwd_ctas, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        call.forward(xd["q"], xd["k"], xd["v"])
        call.backward(xd["do"])

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    call.check_status()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # ---------------- device-resident timed region (per-step events, L2 flushed between)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    evb = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    barrier()
    torch.cuda.synchronize(dev)
    launches0 = fl.flamia_debug_launch_count()
    with ClockSampler(local) as clocks:
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            ev[i][0].record(stream)
            call.forward(xd["q"], xd["k"], xd["v"])
            flamia_quant_do = fl.flamia_quantize_tokenblock
            flamia_quant_do(xd["do"], call.cu, call.dout, call.fmt_do, o=call.o, D=call.D,
                            dev_status=call.status)
            evb[i][0].record(stream)
            fl.flamia_attn_bwd_gqa(call.q, call.k, call.v, call.dout, call.D, call.lse, call.cu,
                                   call.T, call.H, call.H_kv, call.d, call.scale, call.wl,
                                   call.dq, call.dk, call.dv, call.ws, call.bwd_flags,
                                   dev_status=call.status)
            evb[i][1].record(stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
    launches = fl.flamia_debug_launch_count() - launches0
    barrier()
    call.check_status()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    bwd_ms = [a.elapsed_time(b) for a, b in evb]
    total_ms = sum(step_ms)

    # ---------------- end to end through host buffers (pinned), copies timed
    # Every step copies its inputs from pinned host memory and its outputs
    # (O, dQ, dK, dV) back.  The copies of one step overlap the compute of the
    # neighbouring steps: two sets of device buffers alternate, host-to-device
    # copies run on one stream, the call on another, device-to-host copies on
    # a third, ordered by events (a data-loader pipeline).  The inputs are
    # larger than L2 and arrive by copy every step, so L2 is not flushed.
    hx = {n: t.pin_memory() for n, t in x.items()}
    hcu = torch.tensor(w.cu_seqlens, dtype=torch.int32).pin_memory()
    calls = [call, fl.TrainingCall(w.T, w.H, w.d, torch.empty_like(cu), w.sm_scale,
                                   nvfp4_qk=args.nvfp4, hadamard=args.hadamard,
                                   causal=not args.noncausal, H_kv=hkv,
                                   deterministic_dq=args.deterministic, dq_accum=args.dq_accum,
                                   schedule=args.schedule, ds_rows=args.ds_rows,
                                   token_scales=args.token_scales, bwd_ctas=args.bwd_ctas,
                                   device=dev)]
    xin = [xd, {n: torch.empty_like(t) for n, t in xd.items()}]
    outs = lambda c: (c.o, c.dq, c.dk, c.dv)
    hout = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs(c)] for c in calls]
    h2d = sum(t.numel() * t.element_size() for t in hx.values()) + cu.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in outs(call))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def e2e_step(i):
        k = i & 1
        c = calls[k]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_cmp[k])  # the slot's previous call has read its inputs
            c.cu.copy_(hcu, non_blocking=True)
            for n in xin[k]:
                xin[k][n].copy_(hx[n], non_blocking=True)
            ev_in[k].record(s_in)
        stream.wait_event(ev_in[k])
        if i >= 2:
            stream.wait_event(ev_out[k])  # the slot's previous outputs have been copied out
        c.forward(xin[k]["q"], xin[k]["k"], xin[k]["v"])
        c.backward(xin[k]["do"])
        ev_cmp[k].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_cmp[k])
            for hdst, src in zip(hout[k], outs(c)):
                hdst.copy_(src, non_blocking=True)
            ev_out[k].record(s_out)

    # untimed warm-up of both buffer sets (first use of the second call and of
    # the pinned output buffers), then the timed steps
    for i in range(2):
        e2e_step(i)
    s_out.wait_stream(stream)
    torch.cuda.synchronize(dev)
    barrier()
    e_start.record(s_in)
    for i in range(2, 2 + args.steps):
        e2e_step(i)
    s_out.wait_stream(stream)
    e_end.record(s_out)
    torch.cuda.synchronize(dev)
    barrier()
    for c in calls:
        c.check_status()
    e2e_ms = e_start.elapsed_time(e_end)
    # the host link alone: the same copies with no compute (one step's inputs
    # in, its outputs out, on the copy streams), averaged over 3 steps
    c_start, c_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    c_start.record(s_in)
    for i in range(3):
        with torch.cuda.stream(s_in):
            for n in xin[0]:
                xin[0][n].copy_(hx[n], non_blocking=True)
        with torch.cuda.stream(s_out):
            for hdst, src in zip(hout[1], outs(calls[1])):
                hdst.copy_(src, non_blocking=True)
    s_in.wait_stream(s_out)
    c_end.record(s_in)
    torch.cuda.synchronize(dev)
    copy_ms = c_start.elapsed_time(c_end) / 3

    breakdown = stage_breakdown(call, xd, stream, flush, w)

    # causal: the visible half of the pairs; non-causal: all L^2 pairs
    pair_factor = 2.0 if args.noncausal else 1.0
    flops = w.causal_flops() * pair_factor
    bwd_flops = 5.0 * w.H * w.d * w.sum_sq_len * pair_factor  # 10 * H * d * L^2 / 2
    res = {"total_ms": total_ms, "e2e_ms": e2e_ms, "bwd_ms": sum(bwd_ms) / len(bwd_ms),
           "clocks": clocks.summary()}
    if world > 1:
        res["total_ms"], res["e2e_ms"], res["bwd_ms"] = reduce_max(
            [total_ms, e2e_ms, res["bwd_ms"]], dev)
    if rank != 0:
        return None
    pk = peaks()
    ms_step = res["total_ms"] / args.steps
    value = job_throughput(flops, args.steps, world, res["total_ms"])
    e2e_value = job_throughput(flops, args.steps, world, res["e2e_ms"])
    achieved = bwd_flops / (res["bwd_ms"] * 1e-3) / 1e12
    line = {
        "metric": "MXFP8 causal attn fwd+bwd TFLOP/s incl. quant; % of GB300 FP8 tensor peak",
        "value": round(value, 3),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 (mxfp8 operands, f32 accumulate)",
        "data": "synthetic (seeded bf16 normals, %s)" % STRUCTURE_NOTE.get(w.structure, w.structure),
        "config": {"workload": w.name, "T": w.T, "H": w.H, "d": w.d, "docs": w.ndocs,
                   "qk_product": "nvfp4 (mixed path)" if args.nvfp4 else "mxfp8",
                   "qk_rotation": "hadamard" if args.hadamard else "none",
                   "mask": "none (non-causal)" if args.noncausal else "causal",
                   "kv_heads": hkv,
                   "dq_sum": "ordered (deterministic)" if args.deterministic else "atomic",
                   "dq_accumulator": args.dq_accum,
                   "schedule": args.schedule,
                   "bwd_ctas": args.bwd_ctas,
                   "ds_exponents": "query row" if (args.ds_rows or args.token_scales)
                   else "32x32 block",
                   "operand_scales": "per token" if args.token_scales else "32-token block",
                   "flops_per_step": flops, "l2": "flushed (256 MB write) before every step",
                   "parallelism": f"replicas x{world}"},
        "pct_of_fp8_peak": round(100.0 * value / world / pk["fp8_tflops"], 2),
        "roofline": {"kernel": "flamia_attn_bwd (memset + %s + short-document kernel + dq convert)"
                               % (("attn_bwd_pair_kernel (CTA pairs)" if args.bwd_ctas == "pair"
                                   else "attn_bwd128_kernel") if w.d == 128 and not args.nvfp4
                                  else "attn_bwd_kernel<64, nvfp4>" if args.nvfp4
                                  else "attn_bwd_kernel<64>"),
                     "bound": "tensor", "achieved": round(achieved, 2),
                     "peak": pk["fp8_tflops"], "unit": "TFLOP/s",
                     "frac": round(achieved / pk["fp8_tflops"], 4),
                     "peak_source": pk["source"],
                     "traffic": None if (args.hadamard or args.noncausal or hkv != w.H or
                                         args.deterministic or args.dq_accum != "fp32" or
                                         args.schedule != "dynamic" or args.ds_rows or
                                         args.token_scales or
                                         (args.bwd_ctas == "pair" and w.d == 128))
                     else profiled_traffic(w, args.nvfp4),
                     "traffic_unit": "bytes per launch of the attention kernel (ncu, DRAM read + write)"},
        "e2e": {"value": round(e2e_value, 3), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "copies": "overlapped with compute: 2 buffer sets, copy-in / call / copy-out "
                          "streams ordered by events; 2 untimed warm-up steps",
                "copy_only_ms_per_step": round(copy_ms, 4)},
        "gpu_launches": launches,
        "gpu_launches_counted": "the library's own launch counter read around the timed steps",
        "breakdown": breakdown,
        "clocks": res["clocks"],
    }
    line["ds_rounded_to_zero"] = ds_zero_stats(w, xd, args, hkv, dev)
    if not args.no_stress:
        line["scheduling_stress"] = stress_stats(dev, stream, flush)
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    return line


def ds_zero_stats(w, xd, args, hkv, dev):
    """One untimed training call with the dS rounded-to-zero diagnostic: the
    fraction of the nonzero dS entries (pairs the queries see) whose E4M3 code
    under the 32x32 block exponent is zero (review page, sec. 3.3; the
    pages' dS-scale ablation: 0.4% with their scale, 29% with an oversized
    one)."""
    import torch

    from precision_causal_attention_block_gb300 import flamia as fl
    if args.deterministic or args.dq_accum != "fp32" or args.bwd_ctas == "pair":
        return None
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    call = fl.TrainingCall(w.T, w.H, w.d, cu, w.sm_scale, nvfp4_qk=args.nvfp4,
                           hadamard=args.hadamard, causal=not args.noncausal, H_kv=hkv,
                           schedule=args.schedule, ds_rows=args.ds_rows,
                           token_scales=args.token_scales, ds_zero_count=True, device=dev)
    call(xd["q"], xd["k"], xd["v"], xd["do"])
    torch.cuda.synchronize(dev)
    call.check_status()
    nz, z = call.ds_zero_counts()
    del call
    return {"nonzero": nz, "zero": z, "fraction": z / nz if nz else 0.0}


def stress_stats(dev, stream, flush, reps=5):
    """The scheduling-stress shape (131,072 one-token documents, 16 heads of
    dimension 128): work-list build time, the call's time, and its peak device
    memory, the growth of torch's max_memory_allocated from before the call's
    buffers are allocated to the end of one call (inputs resident beforehand
    and reported apart)."""
    import torch

    from precision_causal_attention_block_gb300 import flamia as fl
    from precision_causal_attention_block_gb300 import workloads as W

    w = W.onetoken131072()
    xd = {n: t.to(dev) for n, t in W.make_inputs_bf16(w).items()}
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device=dev)
    torch.cuda.synchronize(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    base = torch.cuda.memory_allocated(dev)
    call = fl.TrainingCall(w.T, w.H, w.d, cu, w.sm_scale, device=dev)
    call(xd["q"], xd["k"], xd["v"], xd["do"])
    torch.cuda.synchronize(dev)
    peak = torch.cuda.max_memory_allocated(dev) - base
    call.check_status()
    times, wl = [], []
    for _ in range(reps):
        flush.fill_(3)
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        fl.flamia_build_worklist(call.cu, call.T, call.wl, dev_status=call.status)
        b.record(stream)
        call(xd["q"], xd["k"], xd["v"], xd["do"])
        c.record(stream)
        torch.cuda.synchronize(dev)
        wl.append(a.elapsed_time(b))
        times.append(b.elapsed_time(c))
    call.check_status()
    inputs = sum(t.numel() * t.element_size() for t in xd.values())
    return {"workload": w.name, "worklist_us": round(1e3 * statistics.median(wl), 2),
            "call_ms": round(statistics.median(times), 4),
            "peak_memory_GB": round(peak / 1e9, 3),
            "peak_memory": "max_memory_allocated growth over buffer allocation + one call",
            "inputs_GB": round(inputs / 1e9, 3)}


def profile_calls(args):
    """Only the training call, `args.steps` times after `args.warmup` untimed
    ones, for profiler captures (ncu): no timing, no extra measurements."""
    import torch

    from precision_causal_attention_block_gb300 import build as B
    from precision_causal_attention_block_gb300 import flamia as fl
    from precision_causal_attention_block_gb300 import workloads as W

    if not os.path.exists(B.LIB):
        B.build()
    w = make_workload(args.workload)
    xd = {n: t.cuda() for n, t in W.make_inputs_bf16(w).items()}
    cu = torch.tensor(w.cu_seqlens, dtype=torch.int32, device="cuda")
    call = fl.TrainingCall(w.T, w.H, w.d, cu, w.sm_scale, nvfp4_qk=args.nvfp4,
                           hadamard=args.hadamard, causal=not args.noncausal,
                           deterministic_dq=args.deterministic, dq_accum=args.dq_accum,
                           schedule=args.schedule, ds_rows=args.ds_rows,
                           token_scales=args.token_scales, bwd_ctas=args.bwd_ctas)
    for _ in range(args.warmup + args.steps):
        call(xd["q"], xd["k"], xd["v"], xd["do"])
    torch.cuda.synchronize()
    call.check_status()
    print(json.dumps({"profiled_calls": args.steps, "workload": w.name}))


def stage_breakdown(call, xd, stream, flush, w, reps=10):
    """Device time of each stage of the call (median of reps, L2 flushed before
    each), the quantiser's HBM throughput and the sum of the call's buffer sizes (the
    measured peak memory is the scheduling-stress entry's)."""
    import torch

    from precision_causal_attention_block_gb300 import flamia as fl

    stages = {
        "quantize_q_ms": lambda: fl.flamia_quantize_tokenblock(xd["q"], call.cu, call.q,
                                                               call.fmt_qk,
                                                               dev_status=call.status),
        "quantize_qkv_ms": lambda: fl.flamia_quantize_qkv(xd["q"], xd["k"], xd["v"], call.cu,
                                                          call.q, call.k, call.v, call.fmt_qk,
                                                          dev_status=call.status),
        "worklist_ms": lambda: fl.flamia_build_worklist(call.cu, call.T, call.wl,
                                                        dev_status=call.status),
        "fwd_ms": lambda: fl.flamia_attn_fwd_gqa(call.q, call.k, call.v, call.cu, call.T, call.H,
                                                 call.H_kv, call.d, call.scale, call.wl, call.o,
                                                 call.lse, call.flags, dev_status=call.status),
        "quantize_do_ms": lambda: fl.flamia_quantize_tokenblock(
            xd["do"], call.cu, call.dout, call.fmt_do, o=call.o, D=call.D,
            dev_status=call.status),
        "bwd_ms": lambda: fl.flamia_attn_bwd_gqa(call.q, call.k, call.v, call.dout, call.D,
                                                 call.lse, call.cu, call.T, call.H, call.H_kv,
                                                 call.d, call.scale, call.wl, call.dq, call.dk,
                                                 call.dv, call.ws, call.bwd_flags,
                                                 dev_status=call.status),
    }
    out = {}
    for name, fn in stages.items():
        times = []
        for _ in range(reps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        out[name] = round(statistics.median(times), 4)
    elems = w.T * w.H * w.d
    qbytes = elems * 3 + w.T * w.H + (elems // 2 + elems // 16 if call.fmt_qk & 0xF else 0)
    out["quantize_q_GBps"] = round(qbytes / (out["quantize_q_ms"] * 1e-3) / 1e9, 1)
    kv = w.T * call.H_kv * w.d
    kbytes = kv * 3 + w.T * call.H_kv + (kv // 2 + kv // 16 if call.fmt_qk & 0xF else 0)
    out["quantize_qkv_GBps"] = round((qbytes + kbytes + kv * 3 + w.T * call.H_kv) /
                                     (out["quantize_qkv_ms"] * 1e-3) / 1e9, 1)
    out["worklist_us"] = round(out["worklist_ms"] * 1e3, 2)
    bufs = [call.q.codes, call.q.scales, call.k.codes, call.k.scales, call.v.codes,
            call.v.scales, call.dout.codes, call.dout.scales, call.wl, call.ws, call.o, call.lse,
            call.D, call.dq, call.dk, call.dv]
    bufs += [t for t in (call.q.nvfp4_codes, call.q.nvfp4_scales, call.k.nvfp4_codes,
                         call.k.nvfp4_scales) if t is not None]
    out["call_buffers_GB"] = round(sum(t.numel() * t.element_size() for t in bufs) / 1e9, 3)
    return out


def cpu_baseline(w, budget_s=20.0, x=None):
    """The FP64 oracle as it stands, on a bounded sample of the workload:
    whole documents of the first head until about budget_s of CPU time, or,
    when one document would take longer than the budget, a causal prefix of
    the first document (its rows see exactly the keys the whole document
    gives them), sized from a short untimed calibration run.  FLOPs are
    counted with the same causal convention (7 d L^2 per document and head)."""
    from oracle import flamia_oracle as O
    from precision_causal_attention_block_gb300 import workloads as W

    if x is None:
        x = W.make_inputs_bf16(w)
    cu = list(w.cu_seqlens)
    docs = [(cu[b], cu[b + 1]) for b in range(len(cu) - 1) if cu[b + 1] > cu[b]]

    def run(s, e):
        sl = [x[n][s:e][:, [0]].double().numpy() for n in ("q", "k", "v", "do")]
        O.attention(*sl, [0, e - s], w.sm_scale)

    s0, e0 = docs[0]
    L = e0 - s0
    if L > 512:  # would the first document alone overrun the budget?
        t = time.perf_counter()
        run(s0, s0 + 512)
        est = (time.perf_counter() - t) * (L / 512) ** 2
        if est > budget_s:
            L = max(64, min(L, int(L * (budget_s / est) ** 0.5) // 32 * 32))
    t0 = time.perf_counter()
    flops = 0.0
    if L < e0 - s0:
        run(s0, s0 + L)
        flops = 7.0 * w.d * L ** 2
        what = f"the first {L} tokens of document 0 (a causal prefix)"
    else:
        n = 0
        for s, e in docs:
            run(s, e)
            flops += 7.0 * w.d * (e - s) ** 2
            n += 1
            if time.perf_counter() - t0 > budget_s:
                break
        what = f"{n} document(s)"
    dt = time.perf_counter() - t0
    return {"value": round(flops / dt / 1e12, 9), "unit": "TFLOP/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{what} of head 0 of {w.name}, fp64 numpy, {dt:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    from precision_causal_attention_block_gb300 import workloads as W
    w = make_workload(args.workload)
    x = W.make_inputs_bf16(w)
    for _ in range(args.warmup):
        pass  # the oracle has no warm-up state
    # about two minutes of oracle work in all, whatever the step count
    t0 = time.perf_counter()
    samples = [cpu_baseline(w, budget_s=max(0.5, 120.0 / max(1, args.steps)), x=x)
               for _ in range(args.steps)]
    dt = time.perf_counter() - t0
    value = statistics.median(s["value"] for s in samples)
    cb = dict(samples[0])
    cb["value"] = value
    return {
        "impl": "reference",
        "metric": "MXFP8 causal attn fwd+bwd TFLOP/s incl. quant; % of GB300 FP8 tensor peak",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(1000 * dt / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded bf16 normals)",
        "config": {"workload": w.name, "T": w.T, "H": w.H, "d": w.d, "docs": w.ndocs},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="long131072")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stress", action="store_true",
                    help="skip the one-token-document work-list / peak-memory measurement")
    ap.add_argument("--profile-calls", action="store_true",
                    help="run only the training call (for ncu), no timing and no JSON line")
    ap.add_argument("--nvfp4", action="store_true",
                    help="mixed path: QK^T from NVFP4 copies of Q and K (head dim 64)")
    ap.add_argument("--hadamard", action="store_true",
                    help="Q and K rotated by the Hadamard matrix in the quantiser")
    ap.add_argument("--kv-heads", type=int, default=0,
                    help="grouped-query attention: K / V heads (dividing the query heads)")
    ap.add_argument("--noncausal", action="store_true",
                    help="every query sees its whole document (FLOPs: all L^2 pairs)")
    ap.add_argument("--dq-accum", default="fp32",
                    choices=["fp32", "fp16_sequence", "fp16_causal"],
                    help="dQ accumulator: float32, or FP16 behind a sequence-wide / causal prescale")
    ap.add_argument("--schedule", default="dynamic", choices=["dynamic", "rule", "static"],
                    help="work distribution of the persistent kernels (rule: the pages' choice, "
                         "dynamic for causal calls, static for non-causal ones unless the "
                         "longest document is at least 4x the average)")
    ap.add_argument("--ds-rows", action="store_true",
                    help="dQ's dS operand with one exponent per (query row, 32-key block)")
    ap.add_argument("--token-scales", action="store_true",
                    help="per-token operand scales (one exponent per token, folded into the "
                         "opposite operand; with query-row dS exponents)")
    ap.add_argument("--bwd-ctas", default="rule", choices=["rule", "one", "pair"],
                    help="head dim 128: backward items of one 128-key CTA or of a CTA pair "
                         "splitting 256 keys (rule: the library's choice by shape)")
    ap.add_argument("--deterministic", action="store_true",
                    help="dQ partials added in a fixed key-tile order (bitwise reproducible)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    rank, world, local = dist_env()
    if args.profile_calls:
        return profile_calls(args)
    line = run_reference(args, rank, world) if args.impl == "reference" else \
        run_ours(args, rank, world, local)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
