#!/usr/bin/env python
"""Benchmark of the sink-aware varlen attention forward on GB300.

Default workload: the vision-tower window block at 16384 tokens (4 packed
sequences of 4096), 16 MHA heads, head dim 80, symmetric window 64, KEY0_BIAS
sinks -- the window-attention call whose H100 cost the MiMo sinks pull
request quotes.  One step = one call of the C-ABI entry point (all of the
forward runs inside its kernel).  Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the CPU oracle as the reference arm

Timing: W untimed warm-up calls, then K calls bracketed by a barrier and
torch.cuda.synchronize(); each call is also bracketed by CUDA events on the
launching stream for the kernel's own duration.  Several input sets rotate so
that the inputs touched between two calls exceed the 129 MB L2.  SM clocks and
throttle reasons are sampled with nvidia-smi during the timed region.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attention_head_sinks_gb300 import workloads as W  # noqa: E402

MODE_NAMES = {0: "NONE", 1: "KEY0_BIAS", 2: "NULL_LOGIT"}
L2_BYTES = 129 * 1024 * 1024
# The pages' cost of the same call on H100 (FA varlen + post-hoc key-0 sink
# correction, 16384 tokens, 16 heads, head dim 80, window 64): 0.289 ms.
PAGES_H100_US = {"vision_window_16384tok": 289.0, "vision_window_4096tok": 248.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------------------------
# workloads: inputs, algorithmic bytes / flops, and the call
# ----------------------------------------------------------------------------
def window_case(name):
    if name == "vision_window_16384tok":
        return W.vision_window(16384, W.SINK_KEY0_BIAS)
    if name == "vision_window_4096tok":
        return W.vision_window(4096, W.SINK_KEY0_BIAS)
    if name == "gqa_window_16384tok":
        return W.gqa_window(W.SINK_KEY0_BIAS)
    raise SystemExit("unknown workload %s" % name)


WORKLOADS = ["vision_window_16384tok", "vision_window_4096tok",
             "gqa_window_16384tok"]


def window_counts(c):
    """Algorithmic bytes (q, o once; k, v once per KV head; LSE) and flops
    (4 * D per live (row, key, head) triple) of one window call."""
    T, hq, d = c.q.shape
    hkv = c.k.shape[1]
    nbytes = 2 * T * hq * d * 2 + 2 * T * hkv * d * 2 + hq * T * 4
    cu = c.cu_seqlens.astype(np.int64)
    live = 0
    for b in range(len(cu) - 1):
        n = int(cu[b + 1] - cu[b])
        i = np.arange(n)
        lo = np.maximum(0, i - c.window_left)
        hi = np.minimum(n - 1, i + c.window_right)
        live += int((hi - lo + 1).sum())
    flops = 4 * d * live * hq
    return nbytes, flops


def window_config(c, name):
    T, hq, d = c.q.shape
    return {"workload": name, "tokens": int(T), "seqs": int(len(c.cu_seqlens) - 1),
            "q_heads": int(hq), "kv_heads": int(c.k.shape[1]), "head_dim": int(d),
            "window": int(c.window_left), "sink_mode": MODE_NAMES[c.mode]}


class WindowRunner:
    kernel_prefix = "window_fwd_kernel"

    def __init__(self, c, nsets):
        import torch
        self.c = c
        self.torch = torch
        dev = torch.device("cuda")
        self.sets = []
        for _ in range(nsets):
            q, k, v = (W.to_torch(x).to(dev) for x in (c.q, c.k, c.v))
            out = torch.empty_like(q)
            lse = torch.empty((c.q.shape[1], c.q.shape[0]), dtype=torch.float32,
                              device=dev)
            self.sets.append((q, k, v, out, lse))
        self.cu = torch.from_numpy(c.cu_seqlens).to(dev)
        self.sinks = torch.from_numpy(c.sinks).to(dev)
        self.set_bytes = sum(t.numel() * t.element_size() for t in self.sets[0])

    def call(self, i, mode=None):
        import attention_head_sinks_gb300 as sa
        q, k, v, out, lse = self.sets[i % len(self.sets)]
        c = self.c
        sa.sa_varlen_window_fwd(q, k, v, self.cu, c.window_left, c.window_right,
                                self.sinks, c.mode if mode is None else mode,
                                c.scale, out=out, lse=lse)

    def e2e(self, steps):
        """Per step: pinned host inputs -> device, the call, out + LSE -> pinned
        host.  Returns (us per step, h2d bytes, d2h bytes)."""
        import attention_head_sinks_gb300 as sa
        torch = self.torch
        c = self.c
        host_in = [W.to_torch(x).pin_memory() for x in (c.q, c.k, c.v)] + \
            [torch.from_numpy(c.cu_seqlens).pin_memory(),
             torch.from_numpy(c.sinks).pin_memory()]
        dev_in = [torch.empty_like(h, device="cuda") for h in host_in]
        q, k, v, out, lse = self.sets[0]
        host_out = [torch.empty_like(out, device="cpu").pin_memory(),
                    torch.empty_like(lse, device="cpu").pin_memory()]
        h2d = sum(h.numel() * h.element_size() for h in host_in)
        d2h = sum(h.numel() * h.element_size() for h in host_out)

        def step():
            for d_, h_ in zip(dev_in, host_in):
                d_.copy_(h_, non_blocking=True)
            sa.sa_varlen_window_fwd(dev_in[0], dev_in[1], dev_in[2], dev_in[3],
                                    c.window_left, c.window_right, dev_in[4],
                                    c.mode, c.scale, out=out, lse=lse)
            host_out[0].copy_(out, non_blocking=True)
            host_out[1].copy_(lse, non_blocking=True)

        for _ in range(3):
            step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            step()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / steps, h2d, d2h


# ----------------------------------------------------------------------------
# measurement helpers
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
               "sw_power_cap")

    def __init__(self, gpu_id):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100", "-i", gpu_id],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.REASONS, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid():
    import torch
    try:
        return "GPU-" + str(torch.cuda.get_device_properties(
            torch.cuda.current_device()).uuid)
    except Exception:
        return str(torch.cuda.current_device())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


def kernel_source_hash(path):
    with open(os.path.join(ROOT, path), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:12]


def recorded_traffic(workload, src_hash):
    """DRAM bytes per launch from an ncu capture summarised in
    profiles/dram_traffic.txt, valid only for the same kernel source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        f = line.split()
        if len(f) >= 3 and not line.startswith("#") and f[0] == workload \
                and f[1] == src_hash:
            return int(float(f[2]))
    return None


# ----------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ----------------------------------------------------------------------------
def oracle_window_sample(c, rows):
    from oracle import sa_oracle
    t0 = time.perf_counter()
    sa_oracle.window_fwd(c.q, c.k, c.v, c.cu_seqlens, c.window_left,
                         c.window_right, c.sinks, c.mode, c.scale, rows=rows)
    return time.perf_counter() - t0


def cpu_baseline(c, budget_s=10.0):
    from oracle import sa_oracle
    T = c.q.shape[0]
    rows = min(T, 512)
    dt = oracle_window_sample(c, (0, rows))
    # grow the sample to ~budget_s of CPU work, bounded by the whole call
    want = int(rows * budget_s / max(dt, 1e-6))
    rows2 = int(min(T, max(rows, want)))
    dt2 = oracle_window_sample(c, (0, rows2))
    us = dt2 * 1e6 * T / rows2
    return {"value": round(us, 1), "unit": "us/call", "cores": sa_oracle.num_threads(),
            "kind": "oracle",
            "sample": "%d of %d query tokens (all heads), fp64 C oracle with OpenMP; "
                      "scaled to one call" % (rows2, T)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from oracle import sa_oracle
    c = window_case(args.workload)
    T = c.q.shape[0]
    rows = max(1, T // 128)            # each step: 1/128 of the call
    starts = [(i * rows) % T for i in range(args.steps + args.warmup)]
    for s in starts[:args.warmup]:
        oracle_window_sample(c, (s, min(T, s + rows)))
    t0 = time.perf_counter()
    for s in starts[args.warmup:]:
        oracle_window_sample(c, (s, min(T, s + rows)))
    dt = time.perf_counter() - t0
    us_call = dt * 1e6 / max(args.steps, 1) * (T / rows)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(us_call, 1),
        "unit": "us/call", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3 / max(args.steps, 1), 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic", "config": window_config(c, args.workload),
        "cpu_baseline": {"value": round(us_call, 1), "unit": "us/call",
                         "cores": sa_oracle.num_threads(), "kind": "oracle",
                         "sample": "each step %d of %d query tokens (all heads); "
                                   "value scaled to one call" % (rows, T)},
        "e2e": {"value": round(us_call, 1), "unit": "us/call",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


METRIC = "attn fwd us/call (achieved HBM GB/s as % of GB300 roofline)"


# ----------------------------------------------------------------------------
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="vision_window_16384tok", choices=WORKLOADS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()

    c = window_case(args.workload)
    nbytes, flops = window_counts(c)
    runner = WindowRunner(c, nsets=1)
    nsets = max(2, -(-3 * L2_BYTES // runner.set_bytes))
    runner = WindowRunner(c, nsets=nsets)

    for i in range(args.warmup):
        runner.call(i)
    barrier()

    # sink cost: the same kernel with sinks disabled, timed the same way
    def timed(mode, steps, sampler=None):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        e0.record()
        for i in range(steps):
            starts[i].record()
            runner.call(i, mode)
            ends[i].record()
        e1.record()
        barrier()
        total_ms = e0.elapsed_time(e1)
        per = [s.elapsed_time(e) * 1000.0 for s, e in zip(starts, ends)]
        return total_ms, per

    sampler = ClockSampler(gpu_uuid())
    total_ms, per = timed(c.mode, args.steps)
    clocks = sampler.stop()
    total_none, per_none = timed(W.SINK_NONE, max(args.steps // 4, 10))

    step_ms = total_ms / args.steps
    if dist is not None:
        t = torch.tensor([step_ms], device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms = float(t.item())
    kern_us = statistics.mean(per)
    kern_us_none = statistics.mean(per_none)

    e2e_us, h2d, d2h = runner.e2e(args.e2e_steps)
    err = None
    import attention_head_sinks_gb300 as sa
    err = sa.sa_device_error()

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return

    hbm_peak, tf_peak, peak_src = measured_peaks()
    achieved = nbytes / (kern_us * 1e-6) / 1e9
    src_hash = kernel_source_hash("attention_head_sinks_gb300/csrc/window_fwd.cu")
    value_us = step_ms * 1000.0 / world
    cfg = window_config(c, args.workload)
    cfg.update({"global_batch": world, "parallelism": "replicas x%d" % world,
                "l2": "%d rotating input sets (%.0f MB) > 129 MB L2" %
                      (nsets, nsets * runner.set_bytes / 1e6)})
    line = {
        "metric": METRIC,
        "value": round(value_us, 3),
        "unit": "us/call",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 5),
        "higher_is_better": False,
        "scaling": "weak",
        "vs_baseline": (round(value_us / PAGES_H100_US[args.workload], 4)
                        if args.workload in PAGES_H100_US else None),
        "dtype": "bf16",
        "data": "synthetic",
        "config": cfg,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1),
                     "peak": hbm_peak, "unit": "GB/s",
                     "frac": round(achieved / hbm_peak, 4),
                     "traffic": recorded_traffic(args.workload, src_hash),
                     "peak_source": peak_src, "alg_bytes": nbytes,
                     "kernel_us": round(kern_us, 3)},
        "tensor": {"alg_tflops": round(flops / (kern_us * 1e-6) / 1e12, 2),
                   "frac_of_peak": round(flops / (kern_us * 1e-6) / 1e12 / tf_peak, 4)},
        "sink_cost": round(kern_us / kern_us_none - 1.0, 4),
        "kernel_us_sinks_disabled": round(kern_us_none, 3),
        "e2e": {"value": round(e2e_us, 2), "unit": "us/call",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "device_error": err,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(c)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
