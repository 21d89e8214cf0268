"""Benchmark of the fused exact attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one forward pass (tile scheduling, Q/K/V tile loads, S = Q K^T,
masking + online softmax, correction, P V, epilogue) over one batch of
synthetic BF16 inputs, the workload being BF16 non-causal, head dim 128,
16 heads, 4 sequences of 4096 tokens (16384 tokens, hidden 2048), N(0,1).
The metric is attention TFLOP/s = 4*B*H*N^2*d / t (half for causal).

Prints one JSON line (rank 0). With several GPUs (torchrun) each rank runs an
independent replica of the workload (weak scaling, no collective on the data
path); the value is the total work of all ranks over the slowest rank's time.
``--impl reference`` times the fp64 CPU oracle on the host cores instead, on
a bounded sample of the same workload.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD = {"workload": "attn_fwd bf16 non-causal d128", "B": 4, "N": 4096, "H": 16, "Hkv": 16, "d": 128,
            "causal": False, "dtype": "bf16", "inputs": "N(0,1) seed 0"}
METRIC = "attention fwd TFLOP/s (4BHN^2d, 1/2 causal)"
L2_FLUSH_BYTES = 512 << 20
L2_NOTE = "flushed between timed iterations (512 MiB written, then read back so no dirty line is written back inside the timed region)"


def l2_flush(buf) -> None:
    """Evicts the L2 before a timed call: writes a buffer larger than the L2
    (129 MB) and reads it back, so the dirty lines the write leaves go to HBM
    here and not while the timed kernel streams its own inputs."""
    buf.zero_()
    buf.max()


def flops_of(w) -> float:
    f = 4.0 * w["B"] * w["H"] * w["N"] ** 2 * w["d"]
    return f / 2 if w["causal"] else f


FWD_BF16_KERNEL_SOURCES = ("attn_fwd2_kernel.cuh", "attn_fwd_pair_kernel.cuh", "attn_common.cuh", "ptx.cuh",
                           "fwd_launch.cuh", "attn_fwd_d128.cu", "launchers.h")
FWD_FP8_KERNEL_SOURCES = ("attn_fwd2_kernel.cuh", "attn_fwd_pair_kernel.cuh", "attn_common.cuh", "ptx.cuh",
                          "fwd_launch.cuh", "attn_fwd_fp8.cu", "fp8_launchers.h", "launchers.h")
PREPASS_KERNEL_SOURCES = ("attn_fp8_prepass.cu", "fp8_prepass.h", "ptx.cuh")
BWD_KERNEL_SOURCES = ("attn_bwd.cu", "api_internal.h", "attn_common.cuh", "bwd_launchers.h", "ptx.cuh")
DECODE_KT_KERNEL_SOURCES = ("attn_decode_kt.cuh", "attn_decode_kt.cu", "attn_fwd2_kernel.cuh", "attn_common.cuh",
                            "ptx.cuh", "fwd_launch.cuh", "launchers.h")


def kernel_digest(files) -> str:
    """sha256 over the named csrc files and the nvcc flags they are built with."""
    import hashlib

    from exact_attention_45_gb300 import build as _b
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(_b.CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    # flags without include paths (-I and its argument), so the digest is the
    # same wherever the checkout lives
    flags, skip = [], False
    for f in _b.ARCH + _b.NVCC_FLAGS:
        if skip or f == "-I":
            skip = f == "-I"
            continue
        flags.append(f)
    h.update(" ".join(flags).encode())
    return h.hexdigest()


def profiled_traffic(profile: str, files):
    """DRAM bytes per launch recorded by an ncu capture summarised under
    profiles/, if that capture ran the kernel sources built now (same digest
    of `files`); None once the kernel has changed since."""
    path = os.path.join(ROOT, "profiles", profile)
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and line.split(":")[0].strip() in ("kernel_source_digest", "traffic_bytes_per_launch"):
                key, val = line.split(":", 1)
                rec[key.strip()] = val.strip()
    if rec.get("kernel_source_digest") != kernel_digest(files) or "traffic_bytes_per_launch" not in rec:
        return None
    return int(rec["traffic_bytes_per_launch"])


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as fh:
            pk = json.load(fh)
        return {"bf16_tflops": pk["bf16_tflops"], "bf16_tflops_sustained": pk["bf16_tflops_sustained"],
                "hbm_gbs": pk["hbm_gbs"], "source": "measured"}
    return {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


# ------------------------------------------------------------------ distributed plumbing
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_seconds: float, local_flops: float, group=None):
    """(max seconds over ranks, total flops over ranks); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_seconds, local_flops
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    f = torch.tensor([local_flops], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    dist.all_reduce(f, op=dist.ReduceOp.SUM, group=group)
    return float(t.item()), float(f.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = os.path.join("/tmp", f"attn45_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.fh = open(self.out, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            # nvidia-smi takes a while to start: wait for its first samples so
            # that the timed region is covered
            t0 = time.time()
            while time.time() - t0 < 10.0:
                self.fh.flush()
                with open(self.out) as fh:
                    if sum(1 for _ in fh) >= 2:
                        break
                time.sleep(0.05)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.out):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.out):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        os.remove(self.out)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        loaded = [s for s, p in zip(sm, power) if p > 0.5 * max(power)] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(smax), "samples": len(sm),
                "power_w_max": max(power), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ oracle (CPU baseline)
def cpu_model() -> str:
    """The host CPU's model name (x86 /proc/cpuinfo, else lscpu, else the
    machine type)."""
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine() or "unknown"


def cpu_oracle_rate(w, budget_s: float = 12.0, seed: int = 0, threads: int | None = None):
    """Time the fp64 oracle on a seeded sample of rows of the workload; returns
    (TFLOP/s extrapolated to the metric's flop count, threads, sample text)."""
    import numpy as np

    import attn_inputs as gen
    import oracle as O
    q, k, v = gen.qkv_fixed(w["B"], w["N"], w["H"], w["Hkv"], w["d"], seed=seed)
    threads = threads or os.cpu_count() or 1
    per_row = 4.0 * w["N"] * w["d"] * (0.5 if w["causal"] else 1.0)
    rows = 256
    t_used = 0.0
    while True:
        rs, rh, ri = gen.sample_rows([w["N"]] * w["B"], w["H"], rows, seed=seed)
        t0 = time.perf_counter()
        O.attention(q, k, v, causal=w["causal"], rows=(rs, rh, ri), nthreads=threads)
        t_used = time.perf_counter() - t0
        if t_used >= budget_s * 0.5 or rows >= w["B"] * w["H"] * w["N"]:
            break
        rows = int(min(rows * max(2.0, budget_s / max(t_used, 1e-3) * 0.8), w["B"] * w["H"] * w["N"]))
    n = len(rs)
    rate = per_row * n / t_used / 1e12
    return rate, threads, f"{n} seeded (b,h,row) query rows of the workload, {t_used:.1f} s"


def cpu_baseline(w, budget_s: float):
    """The oracle timed on all host cores (the reported figure) and on one
    thread, with the CPU model named."""
    rate, threads, sample = cpu_oracle_rate(w, budget_s=budget_s)
    rate1, _, sample1 = cpu_oracle_rate(w, budget_s=max(2.0, budget_s / 3), threads=1)
    return {"value": round(rate, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample,
            "cpu_model": cpu_model(),
            "one_thread": {"value": round(rate1, 6), "unit": "TFLOP/s", "cores": 1, "sample": sample1}}


# ------------------------------------------------------------------ GPU arm
def run_ours(args):
    import torch
    import torch.distributed as dist

    import attn_inputs as gen
    import exact_attention_45_gb300 as A

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl")
    w = dict(WORKLOAD)
    B, N, H, Hkv, d = w["B"], w["N"], w["H"], w["Hkv"], w["d"]
    q_h, k_h, v_h = gen.qkv_fixed(B, N, H, Hkv, d, seed=rank)
    q, k, v = q_h.cuda(), k_h.cuda(), v_h.cuda()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    lib = A.capi()
    scale = 1.0 / math.sqrt(d)

    def launch():
        rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, Hkv, N, d,
                          int(w["causal"]), scale, 0, stream.cuda_stream)
        if rc != 0:
            raise A.AttnError(rc, lib.attn_last_error_message().decode())

    for _ in range(args.warmup):
        l2_flush(flush)
        launch()
    torch.cuda.synchronize()
    if A.attn_get_device_error() != 0:
        raise RuntimeError("device error during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        barrier()
        for i in range(args.steps):
            l2_flush(flush)                    # L2 flushed between timed iterations
            starts[i].record(stream)
            launch()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier()
    clocks = clk.summary()
    times_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    kernel_s = sum(times_ms) / 1e3
    local_flops = flops_of(w) * args.steps
    t_max, total_flops = aggregate(kernel_s, local_flops)
    value = total_flops / t_max / 1e12

    # end to end through the same C-ABI call with host buffers: every step
    # copies its q, k, v from pinned host memory and reads o and lse back, all
    # inside the timed region. The copies run on their own streams beside the
    # kernels (device tensors double-buffered; events order each reuse): the
    # inputs of step i+1 go up and the outputs of step i-1 come down while
    # step i computes.
    q_p, k_p, v_p = (t.pin_memory() for t in (q_h, k_h, v_h))
    o_p = torch.empty(o.shape, dtype=o.dtype).pin_memory()
    l_p = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    bufs = [(q, k, v, o, lse), tuple(torch.empty_like(t) for t in (q, k, v, o, lse))]
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    up_done, comp_done, down_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    for e_ in comp_done + down_done:
        e_.record(stream)

    def launch_buf(bq, bk, bv, bo, bl):
        rc = lib.attn_fwd(bq.data_ptr(), bk.data_ptr(), bv.data_ptr(), bo.data_ptr(), bl.data_ptr(), B, H, Hkv, N,
                          d, int(w["causal"]), scale, 0, stream.cuda_stream)
        if rc != 0:
            raise A.AttnError(rc, lib.attn_last_error_message().decode())

    def e2e_step(i):
        bq, bk, bv, bo, bl = bufs[i % 2]
        with torch.cuda.stream(s_up):
            s_up.wait_event(comp_done[i % 2])          # step i-2's kernel has read these inputs
            bq.copy_(q_p, non_blocking=True)
            bk.copy_(k_p, non_blocking=True)
            bv.copy_(v_p, non_blocking=True)
            up_done[i % 2].record(s_up)
        stream.wait_event(up_done[i % 2])
        stream.wait_event(down_done[i % 2])            # step i-2's outputs have been read back
        launch_buf(bq, bk, bv, bo, bl)
        comp_done[i % 2].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(comp_done[i % 2])
            o_p.copy_(bo, non_blocking=True)
            l_p.copy_(bl, non_blocking=True)
            down_done[i % 2].record(s_down)

    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e2e_steps = min(args.steps, 200)          # each moves ~270 MB over the host link
    e0.record(stream)
    s_up.wait_event(e0)
    s_down.wait_event(e0)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(down_done[(e2e_steps - 1) % 2])
    stream.wait_stream(s_up)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3
    e2e_max, e2e_flops = aggregate(e2e_s, flops_of(w) * e2e_steps)
    if A.attn_get_device_error() != 0:
        raise RuntimeError("device error during timing")

    pk = peaks()
    avg_launch_s = kernel_s / args.steps
    achieved = flops_of(w) / avg_launch_s / 1e12
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {**w, "global_batch": B * world, "seq_len": N, "parallelism": f"replicas{world}",
                   "l2": L2_NOTE},
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                     "traffic": profiled_traffic("attn_fwd2_bf16_d128_n4096_noncausal.md", FWD_BF16_KERNEL_SOURCES),
                     "source_digest": kernel_digest(FWD_BF16_KERNEL_SOURCES)[:16],
                     "peak_source": f"{pk['source']} bf16 burst (cuBLAS)", "kernel": "attn_fwd2_kernel<128,128,2,false,false,BF16>"},
        "e2e": {"value": round(e2e_flops / e2e_max / 1e12, 2), "unit": "TFLOP/s",
                "h2d_bytes_per_step": (q.numel() + k.numel() + v.numel()) * 2,
                "d2h_bytes_per_step": o.numel() * 2 + lse.numel() * 4,
                "copies": "pinned host buffers; H2D and D2H on their own streams beside the kernels, device tensors double-buffered"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    if rank == 0 and not args.no_fp8:
        line["fp8"] = fp8_measure(min(args.steps, 100), args.warmup)
    if rank == 0 and not args.no_decode:
        line["decode"] = decode_measure(min(args.steps, 100), args.warmup)
    if rank == 0 and not args.no_bwd:
        line["bwd"] = bwd_measure(min(args.steps, 50), args.warmup)
    if rank == 0 and not args.no_fp8:
        line["fp8_varlen"] = fp8_varlen_measure(min(args.steps, 20), args.warmup)
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1 and dist.is_initialized():
        dist.destroy_process_group()


def bwd_measure(steps: int, warmup: int, seed: int = 0):
    """Backward (dQ, dK, dV) on the forward's shape (B=4, N=4096, H=16, d=128,
    non-causal, bf16): row sums, the main kernel and the dQ conversion, timed
    with CUDA events, L2 flushed before each call. Work = 2.5 x the forward's
    (five N x N x d GEMMs instead of two): 10 B H N^2 d flops."""
    import torch

    import attn_inputs as gen
    import exact_attention_45_gb300 as A
    w = dict(WORKLOAD)
    B, N, H, d = w["B"], w["N"], w["H"], w["d"]
    q, k, v = (t.cuda() for t in gen.qkv_fixed(B, N, H, H, d, seed=seed))
    do = gen.qkv_fixed(B, N, H, H, d, seed=seed + 100)[0].cuda()
    o, lse = A.attn_fwd(q, k, v)
    ws = torch.empty(A.attn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    call = lambda: A.attn_bwd(q, k, v, o, lse, do, workspace=ws, dq=dq, dk=dk, dv=dv)
    for _ in range(warmup):
        l2_flush(flush)
        call()
    ev = []
    for _ in range(steps):
        l2_flush(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        ev.append((e0, e1))
    torch.cuda.synchronize()
    if A.attn_get_device_error() != 0:
        raise RuntimeError("device error in the backward")
    t = sum(a.elapsed_time(b) for a, b in ev) / steps / 1e3
    fl = 2.5 * flops_of(w)
    pk = peaks()
    return {
        "config": {"workload": "attn_bwd bf16 non-causal d128", "B": B, "N": N, "H": H, "d": d},
        "ms": round(t * 1e3, 4), "tflops": round(fl / t / 1e12, 2),
        "roofline": {"bound": "tensor", "achieved": round(fl / t / 1e12, 2), "peak": pk["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(fl / t / 1e12 / pk["bf16_tflops"], 4),
                     "flops": fl, "peak_source": f"{pk['source']} bf16 burst (cuBLAS)",
                     "traffic": profiled_traffic("attn_bwd_bf16_d128_n4096_noncausal.md", BWD_KERNEL_SOURCES),
                     "source_digest": kernel_digest(BWD_KERNEL_SOURCES)[:16]},
        "gpu_launches_per_step": 4,
    }


def fp8_varlen_measure(steps: int, warmup: int, seed: int = 0):
    """FP8 over packed sequences on the GQA varlen shape: 8 sequences with
    lengths uniform in [1k, 32k] (seed 0), H=32, Hkv=8, d=128, causal, outlier
    inputs, per-block scales + rotation. Work = sum over sequences of
    2 H n^2 d (causal half of 4 H n^2 d). Pre-pass and forward timed apart
    with CUDA events, L2 flushed before each call."""
    import numpy as np
    import torch

    import attn_inputs as gen
    import exact_attention_45_gb300 as A
    lengths = gen.varlen_lengths(8, 1024, 32768, seed=seed)
    q, k, v, cu = gen.qkv_varlen(lengths, 32, 8, 128, seed=seed, dist="outlier")
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    dcu = torch.as_tensor(cu, dtype=torch.int32).cuda()
    pre = A.attn_fp8_prepass_varlen(q, k, v, dcu)
    o = torch.empty((q.shape[0], 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((32, q.shape[0]), dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def timed(fn):
        for _ in range(warmup):
            l2_flush(flush)
            fn()
        ev = []
        for _ in range(steps):
            l2_flush(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / steps / 1e3

    t_fwd = timed(lambda: A.attn_fwd_fp8_varlen(pre, causal=True, out=o, lse=lse))
    t_pre = timed(lambda: A.attn_fp8_prepass_varlen(q, k, v, dcu))
    if A.attn_get_device_error() != 0:
        raise RuntimeError("device error in the FP8 varlen path")
    fl = float(sum(2.0 * 32 * float(n) ** 2 * 128 for n in lengths))
    pk = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"]
    return {
        "config": {"workload": "fp8 varlen GQA causal d128", "nseq": 8, "lengths": "uniform [1024, 32768], seed 0",
                   "H": 32, "Hkv": 8, "d": 128, "tokens": int(np.sum(lengths))},
        "fwd_tflops": round(fl / t_fwd / 1e12, 2), "fwd_ms": round(t_fwd * 1e3, 4),
        "fwd_roofline": {"bound": "tensor", "achieved": round(fl / t_fwd / 1e12, 2), "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": round(fl / t_fwd / 1e12 / fp8_peak, 4),
                         "peak_source": f"2 x {pk['source']} bf16 burst"},
        "prepass_ms": round(t_pre * 1e3, 4),
        "gpu_launches_per_step": 5,
    }


DECODE = {"workload": "split-KV decode bf16 d128", "B": 8, "H": 32, "Hkv": 8, "d": 128, "Nmax": 32768,
          "seqlens": "uniform integers in [1024, 32768], seed 0"}


def decode_measure(steps: int, warmup: int, seed: int = 0, splits: int = 0, group: int = 0):
    """Split-KV decode (one query token per sequence and head over a KV cache)
    on the GQA shape of the varlen configuration: 8 sequences with cached
    lengths uniform in [1k, 32k], H=32, Hkv=8, d=128, bf16. One launch per call
    (cached-key tiles divided evenly between persistent CTAs, partials merged
    in the kernel). HBM-bound: the algorithmic bytes are the cached K and V
    rows each sequence attends to, plus q, o and lse. Timed with CUDA events,
    L2 flushed before each call."""
    import torch

    import attn_inputs as gen
    import exact_attention_45_gb300 as A
    w = dict(DECODE)
    if group > 0:
        w["H"] = group * w["Hkv"]
    B, H, Hkv, d, nmax = w["B"], w["H"], w["Hkv"], w["d"], w["Nmax"]
    seqlens = gen.varlen_lengths(B, 1024, nmax, seed=seed)
    q, _, _ = gen.qkv_fixed(B, 1, H, Hkv, d, seed=seed)
    _, k, v = gen.qkv_fixed(B, nmax, Hkv, Hkv, d, seed=seed + 1)
    q, k, v = q[:, 0].contiguous().cuda(), k.cuda(), v.cuda()
    sl = torch.as_tensor(seqlens, dtype=torch.int32).cuda()
    splits = splits if splits > 0 else A.attn_decode_num_splits(B, Hkv, nmax)
    ws = torch.empty(A.attn_decode_workspace_size(B, H, d, splits), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H), dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    call = lambda: A.attn_decode(q, k, v, sl, num_splits=splits, workspace=ws, out=o, lse=lse)
    for _ in range(warmup):
        l2_flush(flush)
        call()
    ev = []
    for _ in range(steps):
        l2_flush(flush)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        ev.append((e0, e1))
    torch.cuda.synchronize()
    if A.attn_get_device_error() != 0:
        raise RuntimeError("device error in the decode path")
    t = sum(a.elapsed_time(b) for a, b in ev) / steps / 1e3
    kv_bytes = int(sum(seqlens)) * Hkv * d * 2 * 2
    io_bytes = q.numel() * 2 * 2 + lse.numel() * 4
    pk = peaks()
    gbs = (kv_bytes + io_bytes) / t / 1e9
    return {
        "config": {k2: v2 for k2, v2 in w.items()}, "num_splits": splits, "ms": round(t * 1e3, 4),
        "tokens_per_s": round(B * H / t, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                     "frac": round(gbs / pk["hbm_gbs"], 4), "algorithmic_bytes": kv_bytes + io_bytes,
                     "peak_source": f"{pk['source']} copy", "kernel": (f"decode_kt_kernel<{d},{H // Hkv},bf16>" if (H // Hkv <= 16 or H // Hkv in (24, 32))
                                else "attn_fwd2_kernel decode units + combine"),
                     "traffic": profiled_traffic("attn_decode_bf16_d128_gqa32x8_32k.md", DECODE_KT_KERNEL_SOURCES),
                     "source_digest": kernel_digest(DECODE_KT_KERNEL_SOURCES)[:16]},
        "gpu_launches_per_step": 1, "l2": L2_NOTE,
    }


def fp8_measure(steps: int, warmup: int, seed: int = 0):
    """The FP8 path on the same shape (B=4, N=4096, H=16, d=128, non-causal)
    with the outlier inputs: pre-pass (Hadamard rotation + block quantisation,
    HBM-bound) and the e4m3 forward (tensor-bound), each timed with CUDA events
    on its own with L2 flushed in between. Returns a dict for the JSON line."""
    import torch

    import attn_inputs as gen
    import exact_attention_45_gb300 as A
    w = dict(WORKLOAD)
    B, N, H, d = w["B"], w["N"], w["H"], w["d"]
    q, k, v = (t.cuda() for t in gen.qkv_fixed(B, N, H, H, d, seed=seed, dist="outlier"))
    ws = torch.empty(A.attn_fp8_workspace_size(B, H, H, N, d, "block"), dtype=torch.uint8, device="cuda")
    pre = A.attn_fp8_prepass(q, k, v, mode="block", rotate=True)
    o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")

    def timed(fn):
        for _ in range(warmup):
            l2_flush(flush)
            fn()
        ts = []
        for _ in range(steps):
            l2_flush(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ts) / steps / 1e3

    t_fwd = timed(lambda: A.attn_fwd_fp8(pre, out=o, lse=lse))
    t_pre = timed(lambda: A.attn_fp8_prepass(q, k, v, mode="block", rotate=True))
    t_all = timed(lambda: A.attn_fwd_fp8_auto(q, k, v, mode="block", rotate=True, workspace=ws, out=o, lse=lse))
    if A.attn_get_device_error() != 0:
        raise RuntimeError("device error in the FP8 path")
    fl = flops_of(w)
    pk = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"]     # e4m3 dense rate = 2x bf16 (nominal 4.5 vs 2.25 PFLOP/s)
    elems = B * N * H * d
    pre_bytes = 3 * elems * 2 + 3 * elems   # read Q, K, V once, write the three code tensors
    return {
        "inputs": "N(0,1) + N(0,100) w.p. 0.001, seed 0", "mode": "per-block scales + Hadamard rotation",
        "fwd_tflops": round(fl / t_fwd / 1e12, 2), "fwd_ms": round(t_fwd * 1e3, 4),
        "fwd_roofline": {"bound": "tensor", "achieved": round(fl / t_fwd / 1e12, 2), "peak": fp8_peak,
                         "unit": "TFLOP/s", "frac": round(fl / t_fwd / 1e12 / fp8_peak, 4),
                         "peak_source": f"2 x {pk['source']} bf16 burst",
                         "traffic": profiled_traffic("attn_fwd2_fp8_d128_n4096_noncausal.md", FWD_FP8_KERNEL_SOURCES),
                         "source_digest": kernel_digest(FWD_FP8_KERNEL_SOURCES)[:16]},
        "prepass_ms": round(t_pre * 1e3, 4),
        "prepass_roofline": {"bound": "hbm", "achieved": round(pre_bytes / t_pre / 1e9, 1), "peak": pk["hbm_gbs"],
                             "unit": "GB/s", "frac": round(pre_bytes / t_pre / 1e9 / pk["hbm_gbs"], 4),
                             "algorithmic_bytes": pre_bytes,
                             "traffic": profiled_traffic("attn_fp8_prepass_d128_n4096.md", PREPASS_KERNEL_SOURCES),
                             "source_digest": kernel_digest(PREPASS_KERNEL_SOURCES)[:16]},
        "prepass_plus_fwd_tflops": round(fl / t_all / 1e12, 2),
        "gpu_launches_per_step": 5,
    }


def run_sweep(args):
    """TFLOP/s of every BF16 configuration of the benchmark set (one GPU):
    the hidden-2048 sweep (d=64/H=32 and d=128/H=16, N = 512..16384,
    B*N = 16384), d=256/H=8 for N = 1024..16384, causal and not, and the GQA
    varlen causal batch. One JSON object per line on stdout."""
    import torch

    import attn_inputs as gen
    import exact_attention_45_gb300 as A
    torch.cuda.set_device(0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    pk = peaks()
    cases = [(d, H, N, c) for d, H in ((64, 32), (128, 16)) for N in (512, 1024, 2048, 4096, 8192, 16384)
             for c in (False, True)]
    cases += [(256, 8, N, c) for N in (1024, 2048, 4096, 8192, 16384) for c in (False, True)]
    if args.sweep_dims:
        keep = {int(x) for x in args.sweep_dims.split(",")}
        cases = [c for c in cases if c[0] in keep]

    def timeit(fn, reps):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            l2_flush(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ts) / 1e3

    for d, H, N, causal in cases:
        B = 16384 // N
        q, k, v = (t.cuda() for t in gen.qkv_fixed(B, N, H, H, d, seed=0))
        o = torch.empty_like(q)
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        t = timeit(lambda: A.attn_fwd(q, k, v, causal=causal, out=o, lse=lse), args.sweep_reps)
        fl = 4.0 * B * H * N * N * d / (2 if causal else 1)
        # algorithmic HBM bytes: read Q, K, V once, write O and the lse
        nbytes = B * N * (2 * H + 2 * H) * d * 2 + B * H * N * 4
        print(json.dumps({"d": d, "H": H, "N": N, "B": B, "causal": causal, "ms": round(t * 1e3, 4),
                          "tflops": round(fl / t / 1e12, 1), "frac": round(fl / t / 1e12 / pk["bf16_tflops"], 4),
                          "hbm_gbs": round(nbytes / t / 1e9, 1), "hbm_frac": round(nbytes / t / 1e9 / pk["hbm_gbs"], 4),
                          "bytes": nbytes}),
              flush=True)
    if args.sweep_dims and 128 not in keep:
        return
    lengths = gen.varlen_lengths(8, 1024, 32768, seed=0)
    q, k, v, cu = gen.qkv_varlen(lengths, 32, 8, 128, seed=0)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    dcu = torch.as_tensor(cu, dtype=torch.int32, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((32, q.shape[0]), dtype=torch.float32, device="cuda")
    t = timeit(lambda: A.attn_fwd_varlen(q, k, v, dcu, causal=True, out=o, lse=lse), args.sweep_reps)
    fl = sum(4.0 * 32 * int(n) ** 2 * 128 / 2 for n in lengths)
    print(json.dumps({"varlen_gqa": [int(n) for n in lengths], "H": 32, "Hkv": 8, "d": 128, "causal": True,
                      "ms": round(t * 1e3, 4), "tflops": round(fl / t / 1e12, 1),
                      "frac": round(fl / t / 1e12 / pk["bf16_tflops"], 4)}), flush=True)


def run_sweep_fp8(args):
    """FP8 forward over the FP8 benchmark set (one GPU): hidden size 2048
    (d=128 with H=16, d=256 with H=8; --sweep-dims keeps a subset),
    N = 1024..16384 with B*N = 16384, outlier inputs; at d=128 the four
    quantisation variants (per-block or per-tensor scales, with or without the
    Hadamard rotation) non-causal, and causal for per-block + rotation; at
    d=256 per-block + rotation, non-causal and causal. Pre-pass and forward
    timed separately (median of --sweep-reps, L2 flushed). One JSON object per
    line on stdout."""
    import torch

    import attn_inputs as gen
    import exact_attention_45_gb300 as A
    torch.cuda.set_device(0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    pk = peaks()
    fp8_peak = 2.0 * pk["bf16_tflops"]

    def timeit(fn, reps):
        for _ in range(3):
            fn()
        ts = []
        for _ in range(reps):
            l2_flush(flush)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in ts) / 1e3

    dims = [int(x) for x in args.sweep_dims.split(",") if x] or [128, 256]
    all_variants = [("block", True, False), ("block", False, False), ("tensor", True, False),
                    ("tensor", False, False), ("block", True, True)]
    for d, N in ((d, N) for d in dims for N in (1024, 2048, 4096, 8192, 16384)):
        H = 2048 // d
        variants = all_variants if d == 128 else [("block", True, False), ("block", True, True)]
        B = 16384 // N
        q, k, v = (t.cuda() for t in gen.qkv_fixed(B, N, H, H, d, seed=0, dist="outlier"))
        o = torch.empty((B, N, H, d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
        for mode, rot, causal in variants:
            pre = A.attn_fp8_prepass(q, k, v, mode=mode, rotate=rot)
            t_pre = timeit(lambda: A.attn_fp8_prepass(q, k, v, mode=mode, rotate=rot), args.sweep_reps)
            t_fwd = timeit(lambda: A.attn_fwd_fp8(pre, causal=causal, out=o, lse=lse), args.sweep_reps)
            fl = 4.0 * B * H * N * N * d / (2 if causal else 1)
            print(json.dumps({"d": d, "H": H, "N": N, "B": B, "mode": mode, "rotate": rot, "causal": causal,
                              "prepass_ms": round(t_pre * 1e3, 4), "fwd_ms": round(t_fwd * 1e3, 4),
                              "fwd_tflops": round(fl / t_fwd / 1e12, 1),
                              "frac_of_2x_bf16": round(fl / t_fwd / 1e12 / fp8_peak, 4)}), flush=True)
    if A.attn_get_device_error() != 0:
        raise RuntimeError("device error in the FP8 sweep")


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    w = dict(WORKLOAD)
    vals = []
    sample = ""
    threads = os.cpu_count() or 1
    for _ in range(args.warmup):
        cpu_oracle_rate(w, budget_s=2.0)
    for _ in range(args.steps):
        rate, threads, sample = cpu_oracle_rate(w, budget_s=args.cpu_budget / max(1, args.steps) * 2)
        vals.append(rate)
    value = statistics.mean(vals)
    per_step_s = flops_of(w) / (value * 1e12)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step_s * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**w, "global_batch": w["B"], "seq_len": w["N"], "parallelism": "cpu"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample + " per step (extrapolated to the full workload's flops)",
                         "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fp8", action="store_true", help="skip the FP8 sub-measurement")
    ap.add_argument("--no-decode", action="store_true", help="skip the split-KV decode sub-measurement")
    ap.add_argument("--no-bwd", action="store_true", help="skip the backward sub-measurement")
    ap.add_argument("--decode-splits", type=int, default=0, help="decode key-range splits (0 = automatic)")
    ap.add_argument("--decode-group", type=int, default=0,
                    help="--workload decode: query heads per KV head (default the workload's 4)")
    ap.add_argument("--workload", choices=("bf16", "fp8", "decode", "bwd"), default="bf16",
                    help="fp8 / decode: run only that path (e.g. for profiling)")
    ap.add_argument("--sweep", action="store_true", help="time every BF16 configuration instead")
    ap.add_argument("--sweep-fp8", action="store_true", help="time the FP8 configurations and quantisation variants")
    ap.add_argument("--sweep-reps", type=int, default=20)
    ap.add_argument("--sweep-dims", default="", help="comma-separated head dims the BF16 sweep keeps (default all)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)      # at least 3 untimed warm-up steps
    if args.workload == "fp8":
        import torch
        torch.cuda.set_device(0)
        print(json.dumps({"fp8": fp8_measure(args.steps, args.warmup)}), flush=True)
    elif args.workload == "bwd":
        import torch
        torch.cuda.set_device(0)
        print(json.dumps({"bwd": bwd_measure(args.steps, args.warmup)}), flush=True)
    elif args.workload == "decode":
        import torch
        torch.cuda.set_device(0)
        print(json.dumps({"decode": decode_measure(args.steps, args.warmup, splits=args.decode_splits,
                                                   group=args.decode_group)}), flush=True)
    elif args.sweep:
        run_sweep(args)
    elif args.sweep_fp8:
        run_sweep_fp8(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
