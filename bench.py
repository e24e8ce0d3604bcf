#!/usr/bin/env python3
"""Benchmark of the attention hot path: one step = fa_fwd + fa_bwd over one synthetic batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Prints ONE JSON line (rank 0).  `value` is the whole-job throughput in TFLOP/s with inputs
resident in HBM: (forward + backward FLOPs of every rank) / (max over ranks of the device time
of K back-to-back steps), FLOPs counted as 4*B*H*L^2*D per forward (halved when causal) and 2.5x
that per backward.  Every kernel launch is bracketed by CUDA events on the launching stream, so
the per-kernel durations behind the roofline are measured live over the same timed region.
`e2e` is the same metric through the same API with pinned host buffers: each step copies
q, k, v, dO host->device and o, lse, dq, dk, dv device->host inside the timed region.

`--impl reference` times the fp64 CPU oracle (the only other implementation of this path) on
the host cores, one bounded sample of the workload per step.  Under torchrun with N > 1 each
rank runs its own replica of the workload on its own GPU (no data-path collective; weak
scaling); only rank 0 runs the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention fwd/bwd TFLOP/s (bf16, 1×GB300) and % of dense BF16 tensor peak"
DEFAULT_WORKLOAD = "train_B8_L4096"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
KERNELS = ("fa_fwd", "bwd_pre", "bwd_dkdv", "bwd_dq")
KERNEL_SOURCES = {"fa_fwd": "fa_fwd.cu", "bwd_pre": "fa_bwd_pre.cu",
                  "bwd_dkdv": "fa_bwd_dkdv.cu", "bwd_dq": "fa_bwd_dq.cu"}


# ---------------------------------------------------------------------------------------
# Distributed plumbing (timing only: a barrier and a max over ranks; no data-path collective)
# ---------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(x: float, device) -> float:
    """Max of a scalar over ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, device) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------------------
# Peaks, clocks, profile traffic
# ---------------------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str, period_ms: int = 100):
        self.gpu_id = gpu_id
        self.period_ms = period_ms
        self.proc = None
        self.error = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", str(self.period_ms), "-i", self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                         text=True)
        except OSError as e:
            self.error = str(e)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "error": self.error or "nvidia-smi unavailable"}
        time.sleep(self.period_ms / 1000.0)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_selector(dev) -> str:
    """nvidia-smi -i argument naming the same physical GPU as the torch device."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index)


def kernel_sha(kernel: str) -> str:
    """Hash of everything that shapes a kernel's memory traffic: its source file, the shared
    device headers, the host launcher (tile schedule, tensor maps) and any other header of the
    package that the kernel's source includes."""
    csrc = os.path.join(ROOT, "tiled_attention_08_gb300", "csrc")
    shared = ("fa_internal.h", "fa_ptx.cuh", "fa_api.cu")
    with open(os.path.join(csrc, KERNEL_SOURCES[kernel]), "rb") as f:
        src = f.read()
    extra = sorted(n for n in set(re.findall(rb'#include "([A-Za-z0-9_.]+)"', src))
                   if n.decode() not in shared and os.path.exists(os.path.join(csrc, n.decode())))
    h = hashlib.sha256()
    h.update(src)
    for name in shared:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    for name in extra:
        with open(os.path.join(csrc, name.decode()), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel's source
    changed since the counters were taken (or no capture exists for it)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None, "no ncu traffic record"
    rec = d.get(kernel, {}).get(workload)
    if not rec:
        return None, "no ncu capture for this kernel/workload"
    if rec.get("source_sha") != kernel_sha(kernel):
        return None, "kernel changed since the ncu capture"
    return float(rec["dram_bytes_per_launch"]), rec.get("note", "")


# ---------------------------------------------------------------------------------------
# CPU oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------------------
def oracle_sample_seconds(w, inp, heads, prefix_len=None):
    """Times the fp64 oracle's forward + backward on the given heads (optionally only the
    first `prefix_len` queries and keys: a causal prefix is a complete sub-problem)."""
    import oracle
    oracle.build()
    L = w.L if prefix_len is None else min(w.L, prefix_len)
    t = 0.0
    for (b, h) in heads:
        f = [inp[n][b, h, :L].double().numpy() for n in ("q", "k", "v", "do")]
        t0 = time.perf_counter()
        oracle.forward(f[0], f[1], f[2], w.scale, w.causal)
        oracle.backward(f[0], f[1], f[2], f[3], w.scale, w.causal)
        t += time.perf_counter() - t0
    return t, L


def step_flops(w, L=None):
    from tiled_attention_08_gb300 import perfmodel as pm
    L = w.L if L is None else L
    return pm.flops_fwd(w.B, w.H, L, w.D, w.causal) + pm.flops_bwd(w.B, w.H, L, w.D, w.causal)


def cpu_baseline(w, inp, budget_s=12.0, max_heads=64):
    import oracle
    from tiled_attention_08_gb300 import perfmodel as pm
    heads_all = [(i % w.B, (i * 7) % w.H) for i in range(w.B * w.H)]
    done, secs = [], 0.0
    for hd in heads_all[:max_heads]:
        s, _ = oracle_sample_seconds(w, inp, [hd])
        done.append(hd)
        secs += s
        if secs >= budget_s:
            break
    per_head = pm.flops_fwd(1, 1, w.L, w.D, w.causal) + pm.flops_bwd(1, 1, w.L, w.D, w.causal)
    flops = per_head * len(done)
    return {"value": flops / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(secs, 3),
            "sample": f"fp64 oracle forward+backward of {len(done)} full head(s) of "
                      f"{w.name} (L={w.L}, D={w.D}, causal={w.causal}), about {budget_s:.0f} s "
                      f"of CPU work; heads are independent so per-head throughput stands for "
                      f"the whole batch"}


def run_reference(args, w):
    """The oracle as it stands, on the host cores: each step one bounded sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    import oracle
    import workloads
    oracle.build()
    inp = workloads.make_inputs(w, seed=0)
    # Size the per-step sample (a causal/plain prefix of one head) so the whole run stays
    # within about two minutes of CPU time.
    budget_per_step = 120.0 / max(1, args.steps + args.warmup)
    pref = min(w.L, 512)
    t, _ = oracle_sample_seconds(w, inp, [(0, 0)], pref)
    while pref < w.L and t * 3.5 < budget_per_step:
        pref = min(w.L, pref * 2)
        t, _ = oracle_sample_seconds(w, inp, [(0, 0)], pref)
    while pref > 64 and t > budget_per_step:
        pref //= 2
        t, _ = oracle_sample_seconds(w, inp, [(0, 0)], pref)
    heads = [(i % w.B, (i * 7) % w.H) for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        oracle_sample_seconds(w, inp, [heads[i]], pref)
    secs = 0.0
    for i in range(args.steps):
        s, _ = oracle_sample_seconds(w, inp, [heads[args.warmup + i]], pref)
        secs += s
    from tiled_attention_08_gb300 import perfmodel as pm
    per = pm.flops_fwd(1, 1, pref, w.D, w.causal) + pm.flops_bwd(1, 1, pref, w.D, w.causal)
    value = per * args.steps / secs / 1e12
    sample = (f"per step: fp64 oracle forward+backward of one head of {w.name}, first {pref} "
              f"of {w.L} queries and keys (a complete sub-problem of the same shape family)")
    cores = oracle.num_threads()
    return {"metric": METRIC, "impl": "reference", "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) tensors; no dataset or weights)",
            "config": dict(w.describe(), parallelism="host cores (OpenMP)"),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------------------
# The CUDA path
# ---------------------------------------------------------------------------------------
def run_ours(args, w):
    import torch
    import tiled_attention_08_gb300 as fa
    import workloads
    from tiled_attention_08_gb300 import build as fa_build
    from tiled_attention_08_gb300 import perfmodel as pm

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(world, "nccl")
    if rank == 0 or not os.path.exists(fa.library_path()):
        fa_build.build()
    barrier(dev)
    fa.load_library()
    if args.forward_pair and fa.fa_set_forward_pair(1) != fa.FA_OK:
        raise SystemExit("fa_set_forward_pair(1) failed")

    inp = workloads.make_inputs(w, seed=rank)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    B, H, L, D = w.B, w.H, w.L, w.D
    dt = fa.FA_BF16 if w.dtype == torch.bfloat16 else fa.FA_FP16
    o = torch.empty_like(q)
    lse = torch.empty((B, H, L), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, L, D)
    ws = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    causal = int(w.causal)

    def call_fwd(qq, kk, vv):
        st = fa.fa_fwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, H, L, D, w.scale, causal, dt, sh)
        if st != fa.FA_OK:
            raise fa.FaError("fa_fwd", st)

    def call_bwd(qq, kk, vv, dd):
        st = fa.fa_bwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(), dd.data_ptr(),
                       lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                       ws_bytes, B, H, L, D, w.scale, causal, dt, sh)
        if st != fa.FA_OK:
            raise fa.FaError("fa_bwd", st)

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)  # creates the underlying cudaEvent_t
        return evs

    # Warm-up.
    for _ in range(args.warmup):
        call_fwd(q, k, v)
        call_bwd(q, k, v, do)
    torch.cuda.synchronize(dev)
    st = fa.fa_get_device_status(sh)
    if st != fa.FA_OK:
        raise fa.FaError("warm-up", st)

    # Device-resident timed region: K steps, every kernel bracketed by events.
    K = args.steps
    kev = [new_events(8) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_selector(dev))
    sampler.start()
    time.sleep(0.3)
    launches0 = fa.fa_launch_count()
    barrier(dev)
    torch.cuda.synchronize(dev)
    t0.record(stream)
    for i in range(K):
        e = kev[i]
        fa.fa_trace_next_call([e[0].cuda_event, e[1].cuda_event], 1)
        call_fwd(q, k, v)
        fa.fa_trace_next_call([x.cuda_event for x in e[2:8]], 3)
        call_bwd(q, k, v, do)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    launches = fa.fa_launch_count() - launches0
    barrier(dev)
    clocks = sampler.stop()
    st = fa.fa_get_device_status(sh)
    if st != fa.FA_OK:
        raise fa.FaError("timed region", st)

    ms_local = t0.elapsed_time(t1)
    ms = reduce_max(ms_local, dev)
    flops_rank = step_flops(w) * K
    flops_all = reduce_sum(flops_rank, dev)
    value = flops_all / (ms * 1e-3) / 1e12

    kern_ms = {name: statistics.mean(kev[i][2 * j].elapsed_time(kev[i][2 * j + 1])
                                     for i in range(K))
               for j, name in enumerate(KERNELS)}
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    total_kms = sum(kern_ms.values())
    kernels = {}
    for name in KERNELS:
        f = pm.flops_kernel(name, B, H, L, D, w.causal)
        by = pm.bytes_kernel(name, B, H, L, D)
        t = kern_ms[name] * 1e-3
        kernels[name] = {"ms": round(kern_ms[name], 4), "launches": K,
                         "share": round(kern_ms[name] / total_kms, 4),
                         "tflops": round(f / t / 1e12, 2) if f else 0.0,
                         "gbps": round(by / t / 1e9, 1)}
    fwd_ms = kern_ms["fa_fwd"]
    bwd_ms = kern_ms["bwd_pre"] + kern_ms["bwd_dkdv"] + kern_ms["bwd_dq"]
    fwd_tf = pm.flops_fwd(B, H, L, D, w.causal) / (fwd_ms * 1e-3) / 1e12
    bwd_tf = pm.flops_bwd(B, H, L, D, w.causal) / (bwd_ms * 1e-3) / 1e12

    dom = max(("fa_fwd", "bwd_dkdv", "bwd_dq"), key=lambda n: kern_ms[n])
    dom_flops = pm.flops_kernel(dom, B, H, L, D, w.causal)
    achieved = dom_flops / (kern_ms[dom] * 1e-3) / 1e12
    traffic, traffic_note = profiled_traffic(dom, w.name)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2),
                "peak": peak_tf, "unit": "TFLOP/s", "frac": round(achieved / peak_tf, 4),
                "traffic": traffic, "traffic_note": traffic_note,
                "algorithmic_bytes": pm.bytes_kernel(dom, B, H, L, D),
                "peak_source": f"{peak_src} bf16_tflops (burst, cuBLAS bf16 GEMM)"
                               + (" of measured" if peak_src == "measured" else " of fallback")}

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms / K, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype_name,
        "data": "synthetic (seeded N(0,1) tensors; no dataset or weights)",
        "config": dict(w.describe(),
                       parallelism=("replicas: one independent copy per GPU"
                                    if world > 1 else "single GPU"),
                       step="fa_fwd + fa_bwd (4 kernels)",
                       forward=("CTA pairs (fa_set_forward_pair(1))" if args.forward_pair
                                else "single CTAs"),
                       l2=f"inputs larger than L2 ({q.numel() * 2 / 2**20:.0f} MiB per tensor); "
                          "no flush"),
        "fwd_tflops": round(fwd_tf, 2), "bwd_tflops": round(bwd_tf, 2),
        "fwd_frac_of_peak": round(fwd_tf / peak_tf, 4),
        "bwd_frac_of_peak": round(bwd_tf / peak_tf, 4),
        "peak_tflops": peak_tf, "peak_hbm_gbs": peak_bw,
        "kernels": kernels,
        "step_stats": _step_stats(kev, K),
        "roofline": roofline,
        "gpu_launches": int(reduce_sum(launches, dev)),
        "clocks": clocks,
    }
    if not args.no_e2e:
        del q, k, v, do, o, lse, dq, dk, dv, ws  # the e2e pass allocates its own buffer sets
        result["e2e"] = run_e2e(w, inp, dev, K)
    if world == 1 and not args.no_configs:
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        result["configs"] = run_configs(dev, skip=w.name)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, inp)
    return result if rank == 0 else None


L2_BYTES = 129 * 2**20  # GB300 L2


def _step_stats(kev, steps):
    """Mean and median over the timed steps of the forward (its call's events) and of the
    backward (the sum of its three kernels' events in the same step), in ms."""
    fwd = [kev[i][0].elapsed_time(kev[i][1]) for i in range(steps)]
    bwd = [sum(kev[i][2 * j].elapsed_time(kev[i][2 * j + 1]) for j in range(1, 4))
           for i in range(steps)]
    return {"fwd_ms_mean": round(statistics.mean(fwd), 4),
            "fwd_ms_median": round(statistics.median(fwd), 4),
            "bwd_ms_mean": round(statistics.mean(bwd), 4),
            "bwd_ms_median": round(statistics.median(bwd), 4)}


def _time_config(w, dev, peaks, dropout_p=0.0):
    """Times one workload's fa_fwd + fa_bwd through the C ABI with every kernel bracketed by
    CUDA events, sampling clocks meanwhile (with dropout on P: fa_fwd_ex + fa_bwd_ex on the
    same contiguous tensors; the FLOP count stays that of the attention itself).  Inputs that fit in L2 get an L2 flush before every
    step, outside the kernels' events: a write of a 256 MiB buffer, then a read of another one,
    so each step starts with none of its data in L2 and with no dirty lines left for its own
    kernels to write back.  The step count is chosen from the warm-up so the timed region lasts
    about half a second."""
    import torch
    import tiled_attention_08_gb300 as fa
    import workloads
    from tiled_attention_08_gb300 import perfmodel as pm
    inp = workloads.make_inputs(w, seed=0)
    q, k, v, do = (inp[n].to(dev) for n in ("q", "k", "v", "do"))
    B, H, L, D = w.B, w.H, w.L, w.D
    dt = fa.FA_BF16 if w.dtype == torch.bfloat16 else fa.FA_FP16
    o = torch.empty_like(q)
    lse = torch.empty((B, H, L), device=dev, dtype=torch.float32)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, L, D)
    ws = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream
    flush = None
    if q.numel() * q.element_size() < L2_BYTES:
        flush = (torch.empty(256 * 2**20, dtype=torch.uint8, device=dev),
                 torch.ones(64 * 2**20, dtype=torch.float32, device=dev))

    contig = (H * L * D, L * D, D)

    def step(ev=None):
        if flush is not None:
            flush[0].fill_(1)
            flush[1].sum()
        if ev is not None:
            fa.fa_trace_next_call([ev[0].cuda_event, ev[1].cuda_event], 1)
        if dropout_p > 0.0:
            st = fa.fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              lse.data_ptr(), [contig] * 4, B, H, L, L, D, w.scale,
                              int(w.causal), dropout_p, 1234, dt, sh)
        else:
            st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), B, H, L, D, w.scale, int(w.causal), dt, sh)
        if st != fa.FA_OK:
            raise fa.FaError("fa_fwd", st)
        if ev is not None:
            fa.fa_trace_next_call([x.cuda_event for x in ev[2:8]], 3)
        if dropout_p > 0.0:
            st = fa.fa_bwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                              do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                              dv.data_ptr(), ws.data_ptr(), ws_bytes, [contig] * 8, B, H, L, L,
                              D, w.scale, int(w.causal), dropout_p, 1234, 1, dt, sh)
        else:
            st = fa.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                           dv.data_ptr(), ws.data_ptr(), ws_bytes, B, H, L, D, w.scale,
                           int(w.causal), dt, sh)
        if st != fa.FA_OK:
            raise fa.FaError("fa_bwd", st)

    def events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)
        return evs

    warm = [events(8) for _ in range(3)]
    for ev in warm:
        step(ev)
    torch.cuda.synchronize(dev)
    t_step = min(sum(ev[2 * j].elapsed_time(ev[2 * j + 1]) for j in range(4)) for ev in warm)
    steps = int(max(10, min(400, math.ceil(500.0 / max(t_step, 1e-3)))))
    kev = [events(8) for _ in range(steps)]
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_selector(dev))
    sampler.start()
    time.sleep(0.3)
    for i in range(steps):
        step(kev[i])
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    st = fa.fa_get_device_status(sh)
    if st != fa.FA_OK:
        raise fa.FaError(w.name, st)
    kern_ms = {name: statistics.mean(kev[i][2 * j].elapsed_time(kev[i][2 * j + 1])
                                     for i in range(steps))
               for j, name in enumerate(KERNELS)}
    peak_tf = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    fwd_ms = kern_ms["fa_fwd"]
    bwd_ms = kern_ms["bwd_pre"] + kern_ms["bwd_dkdv"] + kern_ms["bwd_dq"]
    fwd_tf = pm.flops_fwd(B, H, L, D, w.causal) / (fwd_ms * 1e-3) / 1e12
    bwd_tf = pm.flops_bwd(B, H, L, D, w.causal) / (bwd_ms * 1e-3) / 1e12
    dom = max(("fa_fwd", "bwd_dkdv", "bwd_dq"), key=lambda n: kern_ms[n])
    dom_tf = pm.flops_kernel(dom, B, H, L, D, w.causal) / (kern_ms[dom] * 1e-3) / 1e12
    tot_flops = pm.flops_fwd(B, H, L, D, w.causal) + pm.flops_bwd(B, H, L, D, w.causal)
    return {
        "B": B, "H": H, "L": L, "D": D, "causal": w.causal, "dtype": w.dtype_name,
        "row_scaled": w.row_scaled, "dropout_p": dropout_p, "steps": steps,
        "l2": ("flushed before every step (256 MiB written, then 256 MiB read)"
               if flush is not None else "inputs larger than L2"),
        "fwd_ms": round(fwd_ms, 4), "bwd_ms": round(bwd_ms, 4),
        "fwd_tflops": round(fwd_tf, 2), "bwd_tflops": round(bwd_tf, 2),
        "fwd_bwd_tflops": round(tot_flops / ((fwd_ms + bwd_ms) * 1e-3) / 1e12, 2),
        "fwd_frac_of_peak": round(fwd_tf / peak_tf, 4),
        "bwd_frac_of_peak": round(bwd_tf / peak_tf, 4),
        "fwd_hbm_gbs": round(pm.bytes_fwd(B, H, L, D) / (fwd_ms * 1e-3) / 1e9, 1),
        "bwd_hbm_gbs": round(pm.bytes_bwd(B, H, L, D) / (bwd_ms * 1e-3) / 1e9, 1),
        "kernels_ms": {n: round(kern_ms[n], 4) for n in KERNELS},
        "step_stats": _step_stats(kev, steps),
        "dominant": {"kernel": dom, "tflops": round(dom_tf, 2),
                     "frac": round(dom_tf / peak_tf, 4)},
        "clocks": clocks,
    }


def _time_forward_latency(w, dev, launches=1000):
    """Latency of single forward launches (a one-tile problem is launch-bound): each of
    `launches` calls is bracketed by CUDA events on the launching stream, and the median and
    the mean over them are reported, with the mean of the same calls back to back."""
    import torch
    import tiled_attention_08_gb300 as fa
    import workloads
    inp = workloads.make_inputs(w, seed=0, with_do=False)
    q, k, v = (inp[n].to(dev) for n in ("q", "k", "v"))
    B, H, L, D = w.B, w.H, w.L, w.D
    dt = fa.FA_BF16 if w.dtype == torch.bfloat16 else fa.FA_FP16
    o = torch.empty_like(q)
    lse = torch.empty((B, H, L), device=dev, dtype=torch.float32)
    stream = torch.cuda.current_stream(dev)
    sh = stream.cuda_stream

    def call():
        st = fa.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                       B, H, L, D, w.scale, int(w.causal), dt, sh)
        if st != fa.FA_OK:
            raise fa.FaError("fa_fwd", st)

    for _ in range(20):
        call()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(launches)]
    for a, b in evs:
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_selector(dev))
    sampler.start()
    time.sleep(0.3)
    for a, b in evs:
        fa.fa_trace_next_call([a.cuda_event, b.cuda_event], 1)
        call()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(launches):
        call()
    t1.record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    st = fa.fa_get_device_status(sh)
    if st != fa.FA_OK:
        raise fa.FaError(w.name, st)
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in evs)
    return {"B": B, "H": H, "L": L, "D": D, "causal": w.causal, "dtype": w.dtype_name,
            "forward_only": True, "launches": launches,
            "fwd_latency_us_median": round(statistics.median(us), 3),
            "fwd_latency_us_mean": round(statistics.mean(us), 3),
            "fwd_latency_us_p90": round(us[int(0.9 * (len(us) - 1))], 3),
            "fwd_back_to_back_us": round(t0.elapsed_time(t1) * 1e3 / launches, 3),
            "l2": "warm (the 66 KB problem stays in L2)", "clocks": clocks}


def _time_decode(w, dev, peaks, steps=50):
    """One decode step over a paged cache (fa_decode_paged) timed with the library's per-kernel
    CUDA events.  The cache (several GB) is far larger than L2, so no flush is needed.  HBM
    bytes are algorithmic: every cached token's K and V row read once, plus q, O, LSE, the
    sequence lengths and the table entries in use."""
    import torch
    import tiled_attention_08_gb300 as fa
    import workloads
    inp = workloads.make_decode_inputs(w, seed=0, device=dev)
    stream = torch.cuda.current_stream(dev)
    o = torch.empty_like(inp["q"])
    lse = torch.empty((w.B, w.H), device=dev, dtype=torch.float32)

    def call(ev=None):
        if ev is not None:
            fa.fa_trace_next_call([e.cuda_event for e in ev], 2)
        fa.decode_paged(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                        inp["seq_lens"], w.scale, out=o, lse=lse)

    def events():
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        for e in evs:
            e.record(stream)
        return evs

    for _ in range(3):
        call()
    evs = [events() for _ in range(steps)]
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(gpu_selector(dev))
    sampler.start()
    time.sleep(0.3)
    t0 = time.perf_counter()
    for ev in evs:
        call(ev)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    st = fa.fa_get_device_status(stream.cuda_stream)
    if st != fa.FA_OK:
        raise fa.FaError(w.name, st)
    n_kern = 1 if fa.fa_decode_workspace_bytes(w.B, w.H, w.D, inp["block_tables"].shape[1]) == 0 \
        else 2
    ms = statistics.mean(sum(ev[2 * j].elapsed_time(ev[2 * j + 1]) for j in range(n_kern))
                         for ev in evs)
    lens = inp["seq_lens"].long()
    tokens = int(lens.sum())
    pages = int(((lens + workloads.PAGE_TOKENS - 1) // workloads.PAGE_TOKENS).sum())
    elt = 2
    by = (2 * tokens * w.H * w.D * elt + 2 * w.B * w.H * w.D * elt + w.B * w.H * 4 + w.B * 4 +
          pages * 4)
    peak_bw = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    gbs = by / (ms * 1e-3) / 1e9
    flops = 4.0 * tokens * w.H * w.D
    return dict(w.describe(), steps=steps, kernels=n_kern, tokens=tokens,
                us_per_step=round(ms * 1e3, 2), hbm_gbs=round(gbs, 1),
                hbm_frac_of_peak=round(gbs / peak_bw, 4),
                tflops=round(flops / (ms * 1e-3) / 1e12, 2),
                algorithmic_bytes=by, l2="cache larger than L2 (no flush)",
                roofline={"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_bw,
                          "unit": "GB/s", "frac": round(gbs / peak_bw, 4)},
                clocks=clocks)


DROPOUT_CONFIG = ("llama2_7b_L2048", 0.1)  # the Llama-2-7B layer with dropout on P


def run_configs(dev, skip):
    """Every other workload of the path, each timed on its own (see _time_config), the
    Llama-2-7B layer once more with dropout on P, and the decode step over a paged cache
    (_time_decode)."""
    import workloads
    peaks, _ = load_peaks()
    out = {}
    for name, w in workloads.WORKLOADS.items():
        if name == skip:
            continue
        out[name] = _time_config(w, dev, peaks) if w.backward else _time_forward_latency(w, dev)
    name, p = DROPOUT_CONFIG
    out[f"{name}_dropout{p}"] = _time_config(workloads.WORKLOADS[name], dev, peaks, dropout_p=p)
    for name, w in workloads.DECODE_WORKLOADS.items():
        out[name] = _time_decode(w, dev, peaks)
    return out


def run_e2e(w, inp, dev, K):
    """End to end through the same API.  Every step copies its inputs (q, k, v, dO) from pinned
    host memory to the device, runs fa_fwd + fa_bwd, and copies every output (o, lse, dq, dk,
    dv) back to pinned host memory, all inside the timed region.  Steps are pipelined the way
    a user streaming batches would run them: two device buffer sets and three streams, so the
    host-to-device copies of step i+1 and the device-to-host copies of step i-1 overlap the
    kernels of step i (the copy engines move both directions at once)."""
    import torch
    import tiled_attention_08_gb300 as fa
    B, H, L, D = w.B, w.H, w.L, w.D
    dt = fa.FA_BF16 if w.dtype == torch.bfloat16 else fa.FA_FP16
    causal = int(w.causal)
    pin = {n: inp[n].pin_memory() for n in ("q", "k", "v", "do")}
    like = pin["q"]
    host_out = {n: torch.empty(like.shape, dtype=like.dtype, pin_memory=True)
                for n in ("o", "dq", "dk", "dv")}
    host_out["lse"] = torch.empty((B, H, L), dtype=torch.float32, pin_memory=True)
    sets = []
    for _ in range(2):
        d = {n: torch.empty(like.shape, dtype=like.dtype, device=dev)
             for n in ("q", "k", "v", "do", "o", "dq", "dk", "dv")}
        d["lse"] = torch.empty((B, H, L), dtype=torch.float32, device=dev)
        sets.append(d)
    ws_bytes = fa.fa_bwd_workspace_bytes(B, H, L, D)
    ws = torch.empty(max(ws_bytes, 16), device=dev, dtype=torch.uint8)
    h2d = sum(t.numel() * t.element_size() for t in pin.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    in_ready = [torch.cuda.Event() for _ in range(2)]
    run_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i & 1
        d = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(run_done[b])  # step i-2's kernels have read set b's inputs
            for n in ("q", "k", "v", "do"):
                d[n].copy_(pin[n], non_blocking=True)
            in_ready[b].record(s_in)
        s_run.wait_event(in_ready[b])
        if i >= 2:
            s_run.wait_event(out_done[b])  # step i-2's outputs of set b are on the host
        sh = s_run.cuda_stream
        st = fa.fa_fwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["o"].data_ptr(),
                       d["lse"].data_ptr(), B, H, L, D, w.scale, causal, dt, sh)
        if st != fa.FA_OK:
            raise fa.FaError("fa_fwd (e2e)", st)
        st = fa.fa_bwd(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["o"].data_ptr(),
                       d["do"].data_ptr(), d["lse"].data_ptr(), d["dq"].data_ptr(),
                       d["dk"].data_ptr(), d["dv"].data_ptr(), ws.data_ptr(), ws_bytes,
                       B, H, L, D, w.scale, causal, dt, sh)
        if st != fa.FA_OK:
            raise fa.FaError("fa_bwd (e2e)", st)
        run_done[b].record(s_run)
        with torch.cuda.stream(s_out):
            s_out.wait_event(run_done[b])
            for n in ("o", "lse", "dq", "dk", "dv"):
                host_out[n].copy_(d[n], non_blocking=True)
            out_done[b].record(s_out)

    for i in range(2):  # warm the copy path and both buffer sets
        step(i)
    torch.cuda.synchronize(dev)
    barrier(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    e0.record(s_in)
    for i in range(K):
        step(i)
    s_out.synchronize()  # every step's outputs are on the host
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    e2e_ms = max(e0.elapsed_time(e1), wall * 1e3)
    e2e_ms = reduce_max(e2e_ms, dev)
    e2e_value = reduce_sum(step_flops(w) * K, dev) / (e2e_ms * 1e-3) / 1e12
    st = fa.fa_get_device_status(s_run.cuda_stream)
    if st != fa.FA_OK:
        raise fa.FaError("e2e region", st)
    return {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / K, 4),
            "pipeline": "2 device buffer sets; host-to-device copies, kernels and device-to-host "
                        "copies on 3 streams, so copies of neighbouring steps overlap a step's "
                        "kernels; every step's inputs and outputs cross the host link"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size B (smaller profiling cases)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end pass (profiling runs)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config measurements of the other workloads")
    ap.add_argument("--forward-pair", action="store_true",
                    help="run the forward on CTA pairs (D = 128; fa_set_forward_pair(1))")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    import workloads
    if args.workload not in workloads.WORKLOADS:
        ap.error(f"unknown workload; choose from {sorted(workloads.WORKLOADS)}")
    w = workloads.WORKLOADS[args.workload]
    if args.batch is not None:
        if args.batch < 1:
            ap.error("--batch must be positive")
        from dataclasses import replace
        w = replace(w, name=f"{w.name}_B{args.batch}", B=args.batch)
    if not w.backward:
        ap.error("the benchmark step is forward + backward; pick a workload with a backward")
    if args.impl == "reference":
        res = run_reference(args, w)
    else:
        res = run_ours(args, w)
    if res is not None:
        print(json.dumps(res), flush=True)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
