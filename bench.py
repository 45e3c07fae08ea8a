"""Benchmark: attention forward TFLOP/s and fraction of the GB300 bf16 tensor
peak, per score-to-weight map, on one GPU (or N independent replicas).

Workload: B=16, h=16, T=4096, dk=dv=128, bf16, causal (the mid-size causal
layer on which the Yat target is set), seeded synthetic inputs.  One step is
one Yat forward through the C ABI: one cattn_forward call, which zeroes its
control words, takes the key norms (the norm prologue) and runs the fused
kernel and the near-key pass.  The prologue and the fused forward are also
timed apart (cattn_key_norms, then cattn_forward with the norms marked
ready).  softmax and s^tau are timed on the same inputs in the same run.  FLOPs per forward:
2*B*h*Tq*Tk*(dk+dv), halved for causal.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 oracle on
the host cores on bounded samples of the same workload instead.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd TFLOP/s and % of GB300 bf16 tensor peak per variant, 1 GPU"
WORKLOAD = "cfg3"
FALLBACK_TFLOPS = 1900.0
# NVIDIA's nominal dense bf16 figure for one GB300 (no sparsity): every
# tensor-core fraction is also reported against it, beside the measured
# cuBLAS peak that the roofline uses
DATASHEET_TFLOPS = 2250.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-workload table (every config, every map)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override B (small cases for profiler captures; not a bench line)")
    return ap.parse_args()


def workload(batch=None):
    from softmax_free_attention_gb300 import workloads
    w = workloads.WORKLOADS[WORKLOAD]
    return w.scaled(B=batch) if batch else w


def config_block(w, extra=None):
    cfg = {"workload": f"{w.name}: B={w.B} h={w.h} hkv={w.hkv} Tq={w.Tq} Tk={w.Tk} "
                       f"dk={w.dk} dv={w.dv} {w.dtype} {'causal' if w.causal else 'non-causal'}",
           "B": w.B, "h": w.h, "hkv": w.hkv, "Tq": w.Tq, "Tk": w.Tk, "dk": w.dk, "dv": w.dv,
           "causal": w.causal, "step": "Yat forward, one cattn_forward call (norm prologue + fused tcgen05 kernel + near-key pass)",
           "l2": "inputs larger than L2 (q,k,v = 768 MiB bf16 vs 129 MB L2); no flush needed",
           "flops_per_step": w.flops()}
    if extra:
        cfg.update(extra)
    return cfg


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0.0)), "measured"
    except Exception:
        return FALLBACK_TFLOPS, 1700.0, "fallback"


def measured_hbm_gbs():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def host_cpu():
    """Model name and clock of the host cores (lscpu, else /proc/cpuinfo and
    sysfs); missing fields are None."""
    model, vendor, mhz = None, None, None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            key, _, val = ln.partition(":")
            key, val = key.strip(), val.strip()
            if key == "Model name" and not model:
                model = val
            elif key == "Vendor ID" and not vendor:
                vendor = val
            elif key == "CPU max MHz" and val:
                mhz = float(val)
    except Exception:
        pass
    if model and vendor and vendor not in model:
        model = f"{vendor} {model}"
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for ln in f:
                    if ln.lower().startswith("model name"):
                        model = ln.split(":", 1)[1].strip()
                        break
        except Exception:
            pass
    if mhz is None:
        try:
            with open("/sys/devices/system/cpu/cpu0/cpufreq/cpuinfo_max_freq") as f:
                mhz = int(f.read().strip()) / 1000.0
        except Exception:
            pass
    return model, mhz


KERNEL_SOURCES = ("fwd_tc.cu", "maps.cuh", "ptx.cuh", "kernels.h")
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "fwd_kernel_yat_b4_full.md")


def kernel_source_hash():
    """Hash of the sources the fused kernel is compiled from."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "softmax_free_attention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(batch=None):
    """DRAM bytes per launch of the fused Yat kernel on the benchmark workload
    (at `batch` if given: every tensor scales with it), from the committed
    ncu summary, if it was captured on the current kernel sources; otherwise
    None.  The summary holds `source_hash:`, the per-launch DRAM bytes of the
    captured (smaller) case and the factor that scales it to the benchmark
    workload."""
    try:
        with open(TRAFFIC_SUMMARY) as f:
            text = f.read()
        fields = dict(re.findall(r"^- (\w+): `([^`]+)`", text, flags=re.M))
        if fields.get("source_hash") != kernel_source_hash():
            return None
        full = float(fields["dram_bytes_per_launch"]) * float(fields["scale_to_workload"])
        if batch:
            from softmax_free_attention_gb300 import workloads
            full *= batch / workloads.WORKLOADS[WORKLOAD].B
        return full
    except Exception:
        return None


def max_over_ranks(x, world, device):
    """Max of a per-rank float over all ranks (the slowest rank's time)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step, steps, seconds, world):
    """Whole-job throughput: every rank runs the same workload (weak scaling)."""
    return world * flops_per_step * steps / seconds / 1e12


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, flag in zip(names, parts[5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        busy = [s for s in sm if mx and s > 0.3 * mx] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_oracle_sample(w, inputs, target_seconds, seed=0, cap_rows=None):
    """Time the fp64 oracle on a bounded random sample of query rows.

    Rows are drawn uniformly over (batch, head, t); each (batch, head) pair is
    widened to fp64 separately.  Returns (TFLOP/s, seconds, rows, threads).
    """
    import torch

    import oracle

    threads = os.cpu_count() or 1
    rng = np.random.default_rng(seed)
    pairs = [(int(b), int(hh)) for b, hh in zip(rng.integers(0, w.B, 8), rng.integers(0, w.h, 8))]
    kw_all = {"yat": dict(b=inputs["yat_b"], eps=inputs["yat_eps"])}
    prepared = []
    for (b, hh) in pairs:
        g = hh // (w.h // w.hkv)
        prepared.append((b, hh, inputs["q"][b:b + 1, hh:hh + 1].to(torch.float64).numpy(),
                         inputs["k"][b:b + 1, g:g + 1].to(torch.float64).numpy(),
                         inputs["v"][b:b + 1, g:g + 1].to(torch.float64).numpy()))

    def run(rows_per_pair):
        flops, t0 = 0.0, time.perf_counter()
        for (b, hh, q, k, v) in prepared:
            rows = rng.integers(0, w.Tq, rows_per_pair)
            keys = (rows + 1) if w.causal else np.full_like(rows, w.Tk)
            flops += float(np.sum(2.0 * keys * (w.dk + w.dv)))
            oracle.forward("yat", q, k, v, b=kw_all["yat"]["b"][hh:hh + 1],
                           eps=kw_all["yat"]["eps"][hh:hh + 1], causal=w.causal,
                           scale=w.scale, rows=rows, nthreads=threads)
        return flops, time.perf_counter() - t0

    rows_per_pair = max(1, threads // 2)
    f, t = run(rows_per_pair)  # calibration: grow the sample until it takes a measurable time
    while t < 0.25 * target_seconds:
        rows_per_pair = max(rows_per_pair + 1, int(rows_per_pair * min(8.0, target_seconds / max(t, 1e-3))))
        if cap_rows and rows_per_pair >= cap_rows:
            rows_per_pair = cap_rows
            break
        f, t = run(rows_per_pair)
    rows_per_pair = max(1, int(rows_per_pair * target_seconds / max(t, 1e-3)))
    if cap_rows:
        rows_per_pair = min(rows_per_pair, cap_rows)
    f, t = run(rows_per_pair)
    return f / t / 1e12, t, rows_per_pair * 8, threads


def oracle_full_runs(variants=("yat", "softmax")):
    """The fp64 oracle over every row of the two small workloads (the fp32
    char-level shapes and the bf16 char-level GPT shapes): wall time and
    TFLOP/s by the metric's FLOP count."""
    import oracle
    from softmax_free_attention_gb300 import workloads
    res = {}
    for name in ("cfg1_f32", "cfg2_s1"):
        w = workloads.WORKLOADS[name]
        inp = workloads.generate(w)
        for variant in variants:
            kw = {"yat": dict(b=inp["yat_b"], eps=inp["yat_eps"]), "softmax": {},
                  "stau": dict(eps=inp["stau_eps"], tau=inp["tau"])}[variant]
            t0 = time.perf_counter()
            oracle.forward(variant, inp["q"], inp["k"], inp["v"], causal=w.causal, scale=w.scale,
                           nthreads=os.cpu_count() or 1, **kw)
            dt = time.perf_counter() - t0
            res[f"{name}/{variant}"] = {"s": dt, "tflops": w.flops() / dt / 1e12}
    return res


def per_config_table(dev, peak_burst, hbm_gbs, reps=20):
    """Every workload and map through cattn_forward on device-resident inputs:
    the whole call (Yat with its key-norm prologue) captured once in a CUDA
    graph and replayed, CUDA events over `reps` replays, so that the time is
    the device's and not the Python binding's.  The bound is the larger of
    the tensor time (metric FLOP / measured bf16 peak) and the HBM time
    (q, k, v read once, out and telemetry written once / measured copy
    bandwidth); frac = bound / measured time.  fp32 runs as three tf32 passes
    on the tensor cores, where the bf16 tensor bound does not apply: reported
    against the HBM time."""
    import torch

    from softmax_free_attention_gb300 import attention, workloads
    table = {}
    for name, w in workloads.WORKLOADS.items():
        inp = workloads.generate(w)
        q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
        par = {"yat": dict(b=torch.as_tensor(inp["yat_b"], device=dev),
                           eps=torch.as_tensor(inp["yat_eps"], device=dev)),
               "softmax": {},
               "stau": dict(eps=torch.as_tensor(inp["stau_eps"], device=dev),
                            tau=torch.as_tensor(inp["tau"], device=dev))}
        out = torch.empty((w.B, w.h, w.Tq, w.dv), dtype=q.dtype, device=dev)
        mass = torch.empty((w.B, w.h, w.Tq), dtype=torch.float32, device=dev)
        mx = torch.empty_like(mass)
        esz = q.element_size()
        hbm_bytes = ((q.numel() + k.numel() + v.numel() + out.numel()) * esz
                     + 2 * mass.numel() * 4)
        hbm_us = hbm_bytes / (hbm_gbs * 1e9) * 1e6
        tensor_us = w.flops() / (peak_burst * 1e12) * 1e6 if w.dtype == "bf16" else 0.0
        row = {}
        for variant in ("yat", "softmax", "stau"):
            prob = attention.make_problem(q, k, v, causal=w.causal, scale=w.scale)
            need = attention.workspace_bytes(variant, prob)
            ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
            f = lambda: attention.forward(variant, q, k, v, causal=w.causal, scale=w.scale,
                                          out=out, row_mass=mass, row_max=mx, workspace=ws,
                                          **par[variant])
            try:
                s = torch.cuda.Stream(dev)
                s.wait_stream(torch.cuda.current_stream(dev))
                with torch.cuda.stream(s):
                    for _ in range(3):
                        f()
                torch.cuda.current_stream(dev).wait_stream(s)
                torch.cuda.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    f()
                for _ in range(3):
                    g.replay()
                torch.cuda.synchronize()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                for _ in range(reps):
                    g.replay()
                b.record()
                torch.cuda.synchronize()
                us = a.elapsed_time(b) * 1e3 / reps
                bound_us = max(hbm_us, tensor_us)
                row[variant] = {"us": us, "tflops": w.flops() / (us * 1e-6) / 1e12,
                                "bound": "tensor" if tensor_us >= hbm_us else "hbm",
                                "bound_us": bound_us, "frac": bound_us / us}
                del g
            except Exception as e:  # reported, never fatal for the line
                row[variant] = {"unavailable": f"{type(e).__name__}: {e}"[:160]}
        assert attention.check_status() == 0
        table[name] = {"shape": f"B={w.B} h={w.h} hkv={w.hkv} Tq={w.Tq} Tk={w.Tk} dk={w.dk} "
                                f"dv={w.dv} {w.dtype} {'causal' if w.causal else 'non-causal'}",
                       "hbm_us": hbm_us, "tensor_us": tensor_us, **row}
        del q, k, v, out, mass, mx, inp
        torch.cuda.empty_cache()
    return table


def sdpa_context(q, k, v, w, flops, steps):
    """Time torch.nn.functional.scaled_dot_product_attention (softmax, the
    backend torch picks) on the benchmark's inputs, for context beside the
    library's softmax map.  Any failure is reported, not raised."""
    import torch
    import torch.nn.functional as F
    try:
        if w.hkv != w.h:
            return {"unavailable": "grouped kv heads"}
        f = lambda: F.scaled_dot_product_attention(q, k, v, is_causal=w.causal, scale=w.scale)
        for _ in range(3):
            f()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(steps):
            f()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / steps
        return {"kernel_ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                "what": "torch scaled_dot_product_attention, softmax, same inputs (context only)"}
    except Exception as e:  # context only: the benchmark line does not depend on it
        return {"unavailable": f"{type(e).__name__}: {e}"[:200]}


def reference_arm(args):
    """The fp64 oracle on the host cores, as the reference arm."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from softmax_free_attention_gb300 import workloads
    w = workload(args.batch)
    inputs = workloads.generate(w)
    per_step = max(1.0, min(6.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, inputs, per_step / 4)
    vals, secs, rows_total, threads = [], 0.0, 0, 1
    for s in range(args.steps):
        v, t, rows, threads = cpu_oracle_sample(w, inputs, per_step, seed=100 + s)
        vals.append(v)
        secs += t
        rows_total += rows
    value = statistics.mean(vals)
    sample = (f"{rows_total} query rows drawn uniformly from 8 (batch, head) pairs of {w.name}, "
              f"Yat map, fp64, over {args.steps} steps")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * secs / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(w, {"step": "fp64 oracle on a bounded row sample"}),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist

    from softmax_free_attention_gb300 import attention, build, native, workloads

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        build.build()
    if world > 1:
        dist.barrier()
    native.load()

    w = workload(args.batch)
    inputs_host = workloads.generate(w)
    q, k, v = (inputs_host[n].to(dev) for n in ("q", "k", "v"))
    yb = torch.as_tensor(inputs_host["yat_b"], device=dev)
    ye = torch.as_tensor(inputs_host["yat_eps"], device=dev)
    se = torch.as_tensor(inputs_host["stau_eps"], device=dev)
    tau = torch.as_tensor(inputs_host["tau"], device=dev)
    prob = attention.make_problem(q, k, v, causal=w.causal, scale=w.scale)
    ws = torch.empty(attention.workspace_bytes("yat", prob), dtype=torch.uint8, device=dev)
    out = torch.empty((w.B, w.h, w.Tq, w.dv), dtype=q.dtype, device=dev)
    mass = torch.empty((w.B, w.h, w.Tq), dtype=torch.float32, device=dev)
    mx = torch.empty_like(mass)

    def yat_step():
        # one cattn_forward call that takes the key norms itself
        attention.forward("yat", q, k, v, b=yb, eps=ye, causal=w.causal, scale=w.scale,
                          out=out, row_mass=mass, row_max=mx, workspace=ws)

    def yat_split_step(ev):
        # the same forward as two calls, timed apart: the norm prologue
        # (cattn_key_norms), then the fused forward with the norms marked ready
        ev[0].record()
        attention.key_norms(q, k, v, ws, causal=w.causal, scale=w.scale)
        ev[1].record()
        attention.forward("yat", q, k, v, b=yb, eps=ye, causal=w.causal, scale=w.scale,
                          out=out, row_mass=mass, row_max=mx, workspace=ws, norms_ready=True)
        ev[2].record()

    def variant_step(variant):
        kw = {"softmax": {}, "stau": dict(eps=se, tau=tau)}[variant]
        attention.forward(variant, q, k, v, causal=w.causal, scale=w.scale, out=out,
                          row_mass=mass, row_max=mx, **kw)

    # ---- headline: K Yat steps
    for _ in range(max(3, args.warmup)):
        yat_step()
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        start.record()
        for s in range(args.steps):
            yat_step()
        stop.record()
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = start.elapsed_time(stop)
    elapsed_ms = max_over_ranks(elapsed_ms, world, dev)
    # the norm prologue and the fused forward timed apart (outside the
    # headline's timed region)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for s in range(args.steps):
        yat_split_step(evs[s])
    torch.cuda.synchronize()
    norms_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    fwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    assert attention.check_status() == 0
    ms_per_step = elapsed_ms / args.steps
    flops = w.flops()
    value = job_tflops(flops, args.steps, elapsed_ms * 1e-3, world)

    peak_burst, peak_sust, peak_kind = measured_peaks()

    # ---- per-variant forward timing on the same inputs
    per_variant = {}
    fwd_tflops = flops / (fwd_ms * 1e-3) / 1e12
    step_tflops = flops / (ms_per_step * 1e-3) / 1e12
    per_variant["yat"] = {"tflops": step_tflops,
                          "kernel_tflops": fwd_tflops, "kernel_ms": fwd_ms,
                          "norm_prologue_ms": norms_ms,
                          "frac_of_peak": fwd_tflops / peak_burst,
                          "frac_of_datasheet_peak": fwd_tflops / DATASHEET_TFLOPS,
                          "step_frac_of_peak": step_tflops / peak_burst,
                          "step_frac_of_datasheet_peak": step_tflops / DATASHEET_TFLOPS}
    for variant in ("softmax", "stau"):
        for _ in range(3):
            variant_step(variant)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            variant_step(variant)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        tf = flops / (ms * 1e-3) / 1e12
        per_variant[variant] = {"tflops": tf, "kernel_ms": ms, "frac_of_peak": tf / peak_burst,
                                "frac_of_datasheet_peak": tf / DATASHEET_TFLOPS}
    assert attention.check_status() == 0
    per_variant["yat_over_softmax"] = per_variant["yat"]["tflops"] / per_variant["softmax"]["tflops"]
    per_variant["yat_kernel_over_softmax"] = (per_variant["yat"]["kernel_tflops"]
                                              / per_variant["softmax"]["tflops"])

    # ---- tau* of the s^tau map from the same scores: one S = QK^T pass plus
    # per-score ln phi statistics (SFU-bound), not part of the step above
    tau_prob = attention.make_problem(q, k, k, causal=w.causal, scale=w.scale)
    tau_ws = torch.empty(int(native.load().cattn_tau_star_workspace_bytes(ctypes.byref(tau_prob))),
                         dtype=torch.uint8, device=dev)
    for _ in range(3):
        attention.tau_star(q, k, se, causal=w.causal, scale=w.scale, workspace=tau_ws)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        attention.tau_star(q, k, se, causal=w.causal, scale=w.scale, workspace=tau_ws)
    b.record()
    torch.cuda.synchronize()
    assert attention.check_status() == 0
    tau_ms = a.elapsed_time(b) / args.steps
    qk_flops = flops * w.dk / (w.dk + w.dv)
    per_variant["tau_star"] = {"kernel_ms": tau_ms, "qk_tflops": qk_flops / (tau_ms * 1e-3) / 1e12,
                               "scores_per_s": qk_flops / (2 * w.dk) / (tau_ms * 1e-3)}

    # ---- the map's row statistics on the same inputs: the second pass
    # (cattn_row_stats: entropy, fraction below 1e-6, top-10 mass) and the
    # forward with the entropy accumulated online (cattn_forward_entropy)
    for variant in ("yat", "softmax", "stau"):
        kw = {"yat": dict(b=yb, eps=ye), "softmax": {}, "stau": dict(eps=se, tau=tau)}[variant]
        _, m_s, _ = attention.forward(variant, q, k, v, causal=w.causal, scale=w.scale, **kw)
        need = attention.workspace_bytes(variant, prob)
        ws_v = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        f_stats = lambda: attention.row_stats(variant, q, k, m_s, causal=w.causal, scale=w.scale,
                                              **kw)
        f_ent = lambda: attention.forward_entropy(variant, q, k, v, causal=w.causal, scale=w.scale,
                                                  workspace=ws_v, **kw)
        for name, f in (("row_stats_ms", f_stats), ("forward_entropy_ms", f_ent)):
            for _ in range(3):
                f()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(max(3, args.steps // 2)):
                f()
            b.record()
            torch.cuda.synchronize()
            per_variant[variant][name] = a.elapsed_time(b) / max(3, args.steps // 2)
        del m_s, ws_v
    assert attention.check_status() == 0

    # ---- backward of each map on the same inputs (not part of the step above):
    # the row-sum pass (Yat, s^tau), the dK/dV pass and the dQ pass; FLOPs
    # counted as 2.5 forward passes (the five products S, dP, dV, dK, dQ)
    dout = workloads.grad_output(w, device=dev)
    bwd_ws = None
    for variant in ("yat", "softmax", "stau"):
        kw = {"yat": dict(b=yb, eps=ye), "softmax": {}, "stau": dict(eps=se, tau=tau)}[variant]
        o_b, m_b, _ = attention.forward(variant, q, k, v, causal=w.causal, scale=w.scale, **kw)
        bprob = attention.make_problem(q, k, v, causal=w.causal, scale=w.scale)
        need = int(native.load().cattn_backward_workspace_bytes(attention.variant_id(variant),
                                                                 ctypes.byref(bprob)))
        if bwd_ws is None or bwd_ws.numel() < need:
            bwd_ws = torch.empty(need, dtype=torch.uint8, device=dev)
        for _ in range(3):
            attention.backward(variant, q, k, v, o_b, dout, m_b, causal=w.causal, scale=w.scale,
                               workspace=bwd_ws, **kw)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            attention.backward(variant, q, k, v, o_b, dout, m_b, causal=w.causal, scale=w.scale,
                               workspace=bwd_ws, **kw)
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / args.steps
        tf = 2.5 * flops / (ms * 1e-3) / 1e12
        per_variant[variant]["backward"] = {"kernel_ms": ms, "tflops": tf,
                                            "frac_of_peak": tf / peak_burst}
        del o_b, m_b
    assert attention.check_status() == 0
    del dout, bwd_ws

    # ---- end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        pinned = {n: inputs_host[n].pin_memory() for n in ("q", "k", "v")}
        h2d = sum(t.numel() * t.element_size() for t in pinned.values())
        # the caller's pinned outputs, reused every step
        host_out = dict(out=torch.empty((w.B, w.h, w.Tq, w.dv), dtype=q.dtype, pin_memory=True),
                        row_mass=torch.empty((w.B, w.h, w.Tq), pin_memory=True),
                        row_max=torch.empty((w.B, w.h, w.Tq), pin_memory=True))
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        attention.forward("yat", pinned["q"], pinned["k"], pinned["v"], b=yb.cpu(), eps=ye.cpu(),
                          causal=w.causal, scale=w.scale, **host_out)  # warm-up
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        n_e2e = max(2, min(args.steps, 5))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            attention.forward("yat", pinned["q"], pinned["k"], pinned["v"], b=yb.cpu(),
                              eps=ye.cpu(), causal=w.causal, scale=w.scale, **host_out)
        torch.cuda.synchronize()
        e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, dev)
        e2e = {"value": job_tflops(flops, 1, e2e_s, world), "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "pipeline": f"cattn_forward_host: {min(w.B, attention.HOST_CHUNKS)} batch "
                           "chunks; copies in, kernels and copies out on three streams"}

    # ---- CPU baseline: the oracle on the host cores, bounded sample
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        val, secs, rows, threads = cpu_oracle_sample(w, inputs_host, 12.0)
        model, mhz = host_cpu()
        cpu = {"value": val, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": f"{rows} random query rows from 8 (batch, head) pairs of {w.name}, "
                         f"Yat map, fp64 ({secs:.1f} s)",
               "cpu_model": model, "cpu_max_mhz": mhz if mhz else "not exposed by the host",
               "full_runs": oracle_full_runs()}

    # ---- every workload and map, device-resident, graph-replayed calls
    hbm_gbs, hbm_kind = measured_hbm_gbs()
    configs = None
    if not args.no_configs and args.batch is None:
        configs = per_config_table(dev, peak_burst, hbm_gbs)

    # ---- context only, last: torch's own scaled_dot_product_attention
    # (softmax) on the same device inputs; not part of the step, never the
    # headline, and run after every figure the line depends on
    per_variant["sdpa_context"] = sdpa_context(q, k, v, w, flops, args.steps)

    achieved = fwd_tflops
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_burst, "unit": "TFLOP/s",
                "frac": achieved / peak_burst, "traffic": recorded_traffic(w.B),
                "peak_kind": f"{peak_kind} bf16 burst (cuBLAS)",
                "frac_of_datasheet_peak": achieved / DATASHEET_TFLOPS,
                "datasheet_peak": DATASHEET_TFLOPS,
                "kernel": "cattn::tc::fwd_kernel<Yat,128,128>"}
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_block(w), "per_variant": per_variant,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "per_config": configs, "hbm_peak_gbs": {"value": hbm_gbs, "kind": hbm_kind},
            "clocks": clocks.summary(), "gpu_launches": 3 * args.steps,
            "peak_sustained_tflops": peak_sust}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
