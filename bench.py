"""Benchmark of the KDA hot path (libkda) on GB300.

One step = one kda_chunk_fwd prefill over the packed variable-length
workload (64 sequences, lengths U{256..8192}, H=32, dk=dv=128, bf16 q/k/v,
fp32 z/beta/state, nonzero initial state, final state returned).  `value` is
prefill throughput in Mtokens/s (tokens, not head-tokens).  The decode step
(256 requests x 32 heads, 1000 steps, state updated in place) is measured in
the same run and reported under "decode" as state-update HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl kda|reference]

For N > 1 launch one rank per GPU with torch.distributed.run; each rank runs
its own workload (seed = rank), no data-path collective: weak scaling.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "KDA prefill Mtokens/s (H=32,d=128) & decode state-update HBM GB/s vs peak"
UNIT = "Mtokens/s"
PREFILL_BYTES_PER_HEAD_TOKEN = 3 * 256 + 512 + 4 + 256  # q,k,v bf16 + z fp32 + beta + o bf16
STATE_BYTES = 128 * 128 * 4
# Algorithmic GEMM FLOPs per head-token of the chunked form at chunk C, d = dk = dv:
# five C x C x d products (the two Gram matrices, T'K+, T'V, PU) and three C x d x d
# (WS, Q+S, Khat^T U) per C tokens = 10 C d + 6 d^2.
CHUNK = 64
FLOPS_PER_HEAD_TOKEN = 10 * CHUNK * 128 + 6 * 128 * 128
# Reverse mode (kda_recurrent_bwd), fp32 CUDA cores, per head-token: two
# forward passes over the state (the stored states, then the rebuild) at 5
# flops per state element (decay, the e reduction, the rank-1 write) and the
# reverse step at 16 (read-out, y, dq^, dk^, dalpha and the decayed dS).
BWD_FLOPS_PER_HEAD_TOKEN = (2 * 5 + 16) * 128 * 128
# Chunked reverse mode (kda_chunk_bwd), tf32 tensor-core products, per 16-token
# chunk (C = 16, d = 128): the forward chunk products that rebuild the states
# (C x C x d Gram, C x d x d for K+S, C x C x d for T'R, d x d x C state update)
# and the reverse step's products (the two C x C x d Grams and T'R again, then
# C x C x d + C x d x d for dU, C x C x d for dR, three C x d x d for dK~, dO S^T
# and dR S^T, two C x C x d for dT' and dP, d x d x 2C for dS, four C x C x d
# for the rest of dQ+, dK+, dK-, and two C^3 for the UT transform); 2 flops per
# multiply-add.
def _chunk_bwd_macs(C=16, d=128):
    fwd = C * C * d + C * d * d + C * C * d + d * d * C
    rev_common = 2 * C * C * d + C * d * d + C * C * d
    rev = (C * C * d + C * d * d) + C * C * d + 3 * C * d * d + 2 * C * C * d \
        + d * d * 2 * C + 4 * C * C * d + 2 * C ** 3
    return fwd + rev_common + rev


CBWD_FLOPS_PER_HEAD_TOKEN = 2 * _chunk_bwd_macs() // 16
# tf32 tensor-core peak: the measured bf16 peak times the nominal tf32 / bf16
# ratio (1.1 / 2.25 PFLOP/s dense).
TF32_PER_BF16 = 1.1 / 2.25
# Bytes a reverse pass cannot avoid per head-token: q, k, v, d out (bf16),
# z (fp32) and beta read; dq, dk, dv, dz (fp32) and dbeta written.
BWD_BYTES_PER_HEAD_TOKEN = 4 * 256 + 512 + 4 + 4 * 512 + 4
# fp32 CUDA-core peak: 152 SMs x 128 FP32 lanes x 2 flops per FMA x 2.07 GHz.
FP32_ALU_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except OSError:
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------- distributed --

def dist_info():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist, device):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(tokens_per_rank, world, seconds):
    """Whole-job throughput: tokens all ranks processed / max-over-ranks time."""
    return tokens_per_rank * world / seconds / 1e6


# ------------------------------------------------------- measured traffic --

# DRAM bytes of one prefill launch as counted by ncu (dram__bytes_read.sum +
# dram__bytes_write.sum), recorded under profiles/ together with a hash of
# the sources the kernel is compiled from.  The record is used only while
# those sources are unchanged, and only for the workload it was taken on.
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "kda_chunk_tc_dram_traffic_varlen.txt")
KERNEL_SOURCES = ["linear_attention_layer_gb300/csrc/kda_chunk_tc.cu",
                  "linear_attention_layer_gb300/csrc/tc_ptx.cuh",
                  "linear_attention_layer_gb300/csrc/kda_common.cuh",
                  "linear_attention_layer_gb300/csrc/kda_launch.h",
                  "include/kda.h"]


def kernel_sources_sha256():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def read_record(path):
    rec = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#") and ":" in line:
                k, v = line.split(":", 1)
                rec[k.strip()] = v.strip()
    return rec


TENSOR_RECORD = os.path.join(ROOT, "profiles", "kda_chunk_tc_tensor_pipe_prefill.txt")


def measured_tensor_pipe():
    """ncu tensor-pipe utilisation of the prefill kernel (busy SM), or None if stale."""
    try:
        rec = read_record(TENSOR_RECORD)
        if rec.get("sources_sha256") != kernel_sources_sha256():
            return None
        return float(rec["sm__pipe_tensor_cycles_active_pct"])
    except (OSError, KeyError, ValueError):
        return None


def measured_traffic(workload):
    """Bytes per launch from the record, or None if absent or stale."""
    try:
        rec = read_record(TRAFFIC_RECORD)
        if rec.get("workload") != workload or rec.get("sources_sha256") != kernel_sources_sha256():
            return None
        return int(rec["dram__bytes_read.sum"]) + int(rec["dram__bytes_write.sum"])
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- clocks --

class NvmlClockSampler:
    """SM clock, its maximum and the clock-event reasons, read through NVML
    (read-only queries, libnvidia-ml from the driver) every `period` seconds
    on a host thread while the timed region runs.  start() / stop() bracket
    the region; summary() has the same keys as ClockSampler's."""
    # nvmlClocksEventReason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown"}

    def __init__(self, gpu_uuid, period=0.005):
        import ctypes
        import threading
        self.ct, self.threading = ctypes, threading
        self.period = period
        self.samples = []
        self.thread = None
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.handle = ctypes.c_void_p()
        if not gpu_uuid or lib.nvmlDeviceGetHandleByUUID(gpu_uuid.encode(),
                                                          ctypes.byref(self.handle)) != 0:
            raise OSError("no NVML handle for this GPU")
        self.reason_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(
            self.handle, 1, ctypes.byref(mx)) == 0 else None

    def _read(self):
        ct = self.ct
        mhz, reasons = ct.c_uint(), ct.c_ulonglong()
        if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, ct.byref(mhz)) != 0:
            return None
        bits = int(reasons.value) if self.reason_fn(self.handle, ct.byref(reasons)) == 0 else 0
        return float(mhz.value), bits

    def _loop(self):
        import time
        while not self.stop_flag.is_set():
            v = self._read()
            if v is not None:
                self.samples.append(v)
            time.sleep(self.period)

    def start(self):
        self.stop_flag = self.threading.Event()
        self.thread = self.threading.Thread(target=self._loop, daemon=True)
        self.thread.start()

    def stop(self):
        if self.thread is not None:
            self.stop_flag.set()
            self.thread.join()
            self.thread = None

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml"}
        reasons = set()
        for _, bits in self.samples:
            for bit, name in self.REASONS.items():
                if bits & bit:
                    reasons.add(name)
        return {"sm_mhz": statistics.median(m for m, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": sorted(reasons),
                "samples": len(self.samples), "source": "nvml"}


def clock_sampler(gpu_uuid):
    """NVML sampler when the driver's library answers, else nvidia-smi."""
    try:
        return NvmlClockSampler(gpu_uuid)
    except (OSError, AttributeError):
        return ClockSampler(gpu_uuid)


class ClockSampler:
    """nvidia-smi sampled every 50 ms while the timed region runs (fallback)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id=None):
        self.proc = None
        self.lines = []
        self.gpu_id = gpu_id

    def start(self):
        self.__enter__()

    def stop(self):
        self.__exit__(None, None, None)

    def __enter__(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": "nvidia-smi"}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "source": "nvidia-smi"}


# ------------------------------------------------------------ CPU oracle --

def cpu_oracle_sample(budget_s=12.0, seed=0, max_seqs=64):
    """Time the fp64 oracle (as it stands) on whole sequences of the varlen
    workload, all 32 heads each, until `budget_s` of wall time is used.
    Returns (tokens/s, head_tokens, threads, description)."""
    import oracle
    import workloads
    lens = workloads.varlen_lengths(seed=seed)
    done_tok, elapsed, used = 0, 0.0, 1
    n = 0
    while elapsed < budget_s and n < min(max_seqs, len(lens)):
        p = workloads.random_problem([lens[n]], 32, 128, 128, init_std=0.1, seed=seed + n,
                                     name="varlen-sample")
        t0 = time.perf_counter()
        _, _, used = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host,
                                      p.initial_state)
        elapsed += time.perf_counter() - t0
        done_tok += lens[n]
        n += 1
    desc = (f"{n} whole sequence(s) of the varlen workload ({done_tok} tokens x 32 heads, "
            f"dk=dv=128), fp64 per-token recurrence, {elapsed:.1f} s")
    return done_tok / elapsed, done_tok * 32, used, desc


def cpu_oracle_one_core(seed=0, tokens=512):
    """The same oracle on one host thread: one sequence of `tokens` tokens x
    32 heads (about a second or two of CPU work).  Returns (tokens/s, description)."""
    import oracle
    import workloads
    p = workloads.random_problem([tokens], 32, 128, 128, init_std=0.1, seed=seed,
                                 name="varlen-sample")
    t0 = time.perf_counter()
    oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host, p.initial_state, threads=1)
    dt = time.perf_counter() - t0
    return tokens / dt, (f"one {tokens}-token sequence x 32 heads (dk=dv=128), one thread, "
                         f"{dt:.1f} s")


def reference_arm(args):
    """The oracle as it stands on the host cores: `--impl reference`."""
    rank, world, _ = dist_info()
    if rank != 0:
        return 0
    import oracle
    import workloads
    lens = workloads.varlen_lengths(seed=0)
    # one step = one whole sequence x 32 heads (about a second of CPU work)
    per_step = []
    used = 1
    for i in range(args.warmup + args.steps):
        L = lens[i % len(lens)]
        p = workloads.random_problem([L], 32, 128, 128, init_std=0.1, seed=i,
                                     name="varlen-sample")
        t0 = time.perf_counter()
        _, _, used = oracle.recurrent(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens_host,
                                      p.initial_state)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            per_step.append((L, dt))
    tok = sum(L for L, _ in per_step)
    sec = sum(dt for _, dt in per_step)
    value = tok / sec / 1e6
    sample = (f"each step one whole sequence of the varlen workload (lengths "
              f"{[L for L, _ in per_step]}), all 32 heads, dk=dv=128")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sec / len(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "varlen", "description": "64 seqs U{256..8192}, H=32, "
                   "dk=dv=128, bf16 inputs widened to fp64, initial state N(0,0.1)",
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ GPU ---

def event_time_ms(fn, stream):
    import torch
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    fn()
    b.record(stream)
    return a, b


def bench_prefill(kda, p, steps, warmup, dist, device, split=False, clk=None):
    import torch
    stream = torch.cuda.current_stream()
    out = torch.empty_like(p.v)
    fin = torch.empty((p.num_seqs, p.meta["num_heads"], p.meta["dk"], p.meta["dv"]),
                      dtype=torch.float32, device=p.v.device)
    ws = None
    if split:  # scratch that lets few long sequences split across SMs (allocated once)
        nbytes = kda.chunk_fwd_workspace_size(p.num_seqs, p.total_tokens, p.meta["num_heads"],
                                              p.meta["dk"], p.meta["dv"], p.q.dtype,
                                              p.cu_seqlens_host)
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def step():
        kda.chunk_fwd(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, out=out,
                      final_state=fin, cu_seqlens_host=p.cu_seqlens_host, workspace=ws)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    evs = []
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start()
    t_start.record(stream)
    for _ in range(steps):
        evs.append(event_time_ms(step, stream))
    t_end.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.stop()
    barrier(dist)
    torch.cuda.synchronize()
    total_ms = t_start.elapsed_time(t_end)
    per_launch = [a.elapsed_time(b) for a, b in evs]
    err = kda.get_device_error()
    if err != 0:
        raise RuntimeError(f"device error word {err} after the timed prefill")
    return total_ms, per_launch


def bench_backward(kda, p, steps, warmup, device, clk=None, chunked=False):
    """kda_recurrent_bwd (chunked: kda_chunk_bwd) over the prefill workload
    with random cotangents (d out bf16, d final state fp32).  Returns (total
    ms, per-launch ms)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(99)
    H = p.meta["num_heads"]
    d_out = torch.randn(p.v.shape, device=device, generator=g).to(p.q.dtype)
    d_fin = torch.randn((p.num_seqs, H, 128, 128), device=device, generator=g)
    size_fn = kda.chunk_bwd_workspace_size if chunked else kda.recurrent_bwd_workspace_size
    bwd_fn = kda.chunk_bwd if chunked else kda.recurrent_bwd
    nbytes = size_fn(H, p.q.dtype, p.cu_seqlens_host)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
    T = p.total_tokens
    f32 = dict(dtype=torch.float32, device=device)
    grads = (torch.empty((T, H, 128), **f32), torch.empty((T, H, 128), **f32),
             torch.empty((T, H, 128), **f32), torch.empty((T, H, 128), **f32),
             torch.empty((T, H), **f32), torch.empty((p.num_seqs, H, 128, 128), **f32))
    stream = torch.cuda.current_stream()

    def step():
        bwd_fn(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, d_out, d_fin,
               cu_seqlens_host=p.cu_seqlens_host, workspace=ws, grads=grads)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = []
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start()
    t0.record(stream)
    for _ in range(steps):
        evs.append(event_time_ms(step, stream))
    t1.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.stop()
    err = kda.get_device_error()
    if err != 0:
        raise RuntimeError(f"device error word {err} after the timed backward")
    del grads, ws, d_out, d_fin
    torch.cuda.empty_cache()
    return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in evs]


def bench_short_conv(kda, p, steps, warmup, device, width=4, clk=None):
    """kda_short_conv on q and on k of the prefill workload (width 4, with an
    incoming and an outgoing convolution state).  Returns (total ms, per-step ms)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(77)
    H, D, N = p.meta["num_heads"], p.meta["dk"], p.num_seqs
    wq = torch.randn((H, D, width), device=device, generator=g) * 0.5
    wk = torch.randn((H, D, width), device=device, generator=g) * 0.5
    sq = torch.randn((N, H, D, width - 1), device=device, generator=g)
    sk = torch.randn((N, H, D, width - 1), device=device, generator=g)
    yq, yk = torch.empty_like(p.q), torch.empty_like(p.k)
    fq, fk = torch.empty_like(sq), torch.empty_like(sk)
    stream = torch.cuda.current_stream()

    def step():
        kda.short_conv(p.q, wq, p.cu_seqlens, sq, out=yq, final_state=fq)
        kda.short_conv(p.k, wk, p.cu_seqlens, sk, out=yk, final_state=fk)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    evs = []
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start()
    t0.record(stream)
    for _ in range(steps):
        evs.append(event_time_ms(step, stream))
    t1.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.stop()
    err = kda.get_device_error()
    if err != 0:
        raise RuntimeError(f"device error word {err} after the timed convolution")
    return t0.elapsed_time(t1), [a.elapsed_time(b) for a, b in evs]


def bench_fused_prefill(kda, p, steps, warmup, device, width=4, clk=None):
    """kda_chunk_fwd_fused (the short convolution of raw q, k inside the
    prefill kernel) against the separate path (kda_short_conv of q and of k,
    then kda_chunk_fwd) on the same workload.  Returns (fused ms per step,
    separate ms per step)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(78)
    H, N = p.meta["num_heads"], p.num_seqs
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    wq = torch.randn((H, 128, width), **f32) * 0.5
    wk = torch.randn((H, 128, width), **f32) * 0.5
    sq = torch.randn((N, H, 128, width - 1), **f32)
    sk = torch.randn((N, H, 128, width - 1), **f32)
    out = torch.empty_like(p.v)
    fin = torch.empty((N, H, 128, 128), dtype=torch.float32, device=device)
    yq, yk = torch.empty_like(p.q), torch.empty_like(p.k)
    fq, fk = torch.empty_like(sq), torch.empty_like(sk)
    stream = torch.cuda.current_stream()

    def fused():
        kda.chunk_fwd_fused(p.q, p.k, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state,
                            conv_weight_q=wq, conv_weight_k=wk, conv_state_q=sq,
                            conv_state_k=sk, out=out, final_state=fin,
                            cu_seqlens_host=p.cu_seqlens_host)

    def separate():
        kda.short_conv(p.q, wq, p.cu_seqlens, sq, out=yq, final_state=fq)
        kda.short_conv(p.k, wk, p.cu_seqlens, sk, out=yk, final_state=fk)
        kda.chunk_fwd(yq, yk, p.v, p.z, p.beta, p.cu_seqlens, p.initial_state, out=out,
                      final_state=fin, cu_seqlens_host=p.cu_seqlens_host)

    res = []
    for fn, c in ((fused, clk), (separate, None)):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        if c is not None:
            c.start()
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        if c is not None:
            c.stop()
        res.append(a.elapsed_time(b) / steps)
    if kda.get_device_error() != 0:
        raise RuntimeError("device error word set after the fused prefill")
    return res[0], res[1]


def bench_spec_decode_fused(kda, B, H, W, steps, device, seed=0, clk=None, width=4):
    """The speculative-decoding step with the short convolution of raw q, k
    (width 4, states advanced by the replay) and the per-head RMS output norm
    fused in: one kda_decode_replay_window_fused call per step.
    Returns (ms per step, accepted tokens per step)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed + 1)
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    q = torch.randn((B, W, H, 128), **f32).to(torch.bfloat16)
    k = torch.randn((B, W, H, 128), **f32).to(torch.bfloat16)
    v = torch.randn((B, W, H, 128), **f32).to(torch.bfloat16)
    z = torch.randn((B, W, H, 128), **f32)
    beta = torch.sigmoid(torch.randn((B, W, H), **f32))
    state = torch.randn((B, H, 128, 128), **f32) * 0.1
    fz = dict(conv_weight_q=torch.randn((H, 128, width), **f32) * 0.5,
              conv_weight_k=torch.randn((H, 128, width), **f32) * 0.5,
              conv_state_q=torch.randn((B, H, 128, width - 1), **f32),
              conv_state_k=torch.randn((B, H, 128, width - 1), **f32),
              out_norm_weight=torch.ones((H, 128), dtype=torch.float32, device=device),
              out_norm_eps=1e-6)
    out = torch.empty((B, W, H, 128), dtype=torch.bfloat16, device=device)
    acc = torch.randint(0, W + 1, (steps + 3, B), generator=g, device=device, dtype=torch.int32)
    stream = torch.cuda.current_stream()
    win = (q, k, v, z, beta)

    def step(i):
        kda.decode_replay_window_fused(win, acc[i], win, state, out=out, **fz)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start()
    a.record(stream)
    for i in range(steps):
        step(3 + i)
    b.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.stop()
    if kda.get_device_error() != 0:
        raise RuntimeError("device error word set after the fused speculative-decoding steps")
    return a.elapsed_time(b) / steps, float(acc[3:].sum().item()) / steps


def bench_spec_decode(kda, B, H, W, steps, device, seed=0, clk=None):
    """Speculative decoding: per step one kda_decode_replay_window call -- the
    replay of the previous window's accepted prefix and the outputs of the
    next window of W drafts, one state read and one write.  Acceptance
    lengths are drawn U{0..W} (seeded).
    Returns (ms per step, accepted tokens per step)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    unit = lambda x: x / torch.linalg.vector_norm(x, dim=-1, keepdim=True)
    q = unit(torch.randn((B, W, H, 128), **f32)).to(torch.bfloat16)
    k = unit(torch.randn((B, W, H, 128), **f32)).to(torch.bfloat16)
    v = torch.randn((B, W, H, 128), **f32).to(torch.bfloat16)
    z = torch.randn((B, W, H, 128), **f32)
    beta = torch.sigmoid(torch.randn((B, W, H), **f32))
    state = torch.randn((B, H, 128, 128), **f32) * 0.1
    out = torch.empty((B, W, H, 128), dtype=torch.bfloat16, device=device)
    acc = torch.randint(0, W + 1, (steps + 3, B), generator=g, device=device, dtype=torch.int32)
    stream = torch.cuda.current_stream()

    prev = (q, k, v, z, beta)

    def step(i):  # replay the last window's accepted prefix, then the next window's outputs
        kda.decode_replay_window(prev, acc[i], q, k, v, z, beta, state, out=out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start()
    a.record(stream)
    for i in range(steps):
        step(3 + i)
    b.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.stop()
    if kda.get_device_error() != 0:
        raise RuntimeError("device error word set after the speculative-decoding steps")
    return a.elapsed_time(b) / steps, float(acc[3:].sum().item()) / steps


def bench_decode(kda, d, steps, device, clk=None):
    import torch
    stream = torch.cuda.current_stream()
    out = torch.empty_like(d.v[0])
    warm = 3
    for t in range(warm):
        kda.decode_step(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], d.state, out=out)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start()
    a.record(stream)
    for t in range(steps):
        kda.decode_step(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], d.state, out=out)
    b.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.stop()
    return a.elapsed_time(b)


def bench_decode_fused(kda, d, steps, device, width=4, clk=None):
    """kda_decode_step_fused over the decode workload: raw q, k through the
    short convolution (width 4, states advanced in place) and the outputs
    through the per-head RMS norm, one launch per step."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(79)
    N, H = d.meta["num_requests"], d.meta["num_heads"]
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    fz = dict(conv_weight_q=torch.randn((H, 128, width), **f32) * 0.5,
              conv_weight_k=torch.randn((H, 128, width), **f32) * 0.5,
              conv_state_q=torch.randn((N, H, 128, width - 1), **f32),
              conv_state_k=torch.randn((N, H, 128, width - 1), **f32),
              out_norm_weight=torch.ones((H, 128), dtype=torch.float32, device=device),
              out_norm_eps=1e-6)
    stream = torch.cuda.current_stream()
    out = torch.empty_like(d.v[0])
    for t in range(3):
        kda.decode_step_fused(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], d.state, out=out, **fz)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    if clk is not None:
        clk.start()
    a.record(stream)
    for t in range(steps):
        kda.decode_step_fused(d.q[t], d.k[t], d.v[t], d.z[t], d.beta[t], d.state, out=out, **fz)
    b.record(stream)
    torch.cuda.synchronize()
    if clk is not None:
        clk.stop()
    if kda.get_device_error() != 0:
        raise RuntimeError("device error word set after the fused decode steps")
    return a.elapsed_time(b)


def bench_e2e(kda, p, steps, device, groups=8, warmup=3):
    """End to end through kda_chunk_fwd_host: inputs and outputs in pinned host
    memory, every step copies the batch in, computes and copies out and the
    final state back (groups of sequences overlapped), all inside the timed
    region.  The device staging area is allocated once, outside it; `warmup`
    (at least 3) untimed steps first."""
    import torch
    stream = torch.cuda.current_stream()
    hq, hk, hv, hz, hb = (getattr(p, n).cpu().pin_memory() for n in ("q", "k", "v", "z", "beta"))
    hs0 = p.initial_state.cpu().pin_memory() if p.initial_state is not None else None
    H, dk, dv = p.meta["num_heads"], p.meta["dk"], p.meta["dv"]
    out_h = torch.empty(p.v.shape, dtype=p.v.dtype).pin_memory()
    fin_h = torch.empty((p.num_seqs, H, dk, dv), dtype=torch.float32).pin_memory()
    nbytes = kda.chunk_fwd_host_workspace_size(p.num_seqs, p.total_tokens, H, dk, dv, p.q.dtype)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=device)
    ins = [hq, hk, hv, hz, hb] + ([hs0] if hs0 is not None else [])
    h2d = sum(t.numel() * t.element_size() for t in ins) + 4 * (p.num_seqs + 1)
    d2h = out_h.numel() * out_h.element_size() + fin_h.numel() * 4

    def step():
        kda.chunk_fwd_host(hq, hk, hv, hz, hb, p.cu_seqlens_host, hs0, out=out_h,
                           final_state=fin_h, workspace=ws, groups=groups)

    for _ in range(max(3, warmup)):
        step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    per = []
    a.record(stream)
    for _ in range(steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        per.append((e0, e1))
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    bench_e2e.min_ms = min(x.elapsed_time(y) for x, y in per)
    # the link itself: one 1 GiB pinned copy each way, timed alone
    link = {}
    big_h = torch.empty(1 << 30, dtype=torch.uint8).pin_memory()
    big_d = torch.empty(1 << 30, dtype=torch.uint8, device=device)
    for name, dst, src in (("h2d", big_d, big_h), ("d2h", big_h, big_d)):
        dst.copy_(src, non_blocking=True)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        dst.copy_(src, non_blocking=True)
        e1.record(stream)
        torch.cuda.synchronize()
        link[name] = (1 << 30) / (e0.elapsed_time(e1) * 1e-3) / 1e9
    del big_h, big_d
    return ms, h2d, d2h, link


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--skip", default="",
                    help="comma list of: decode,e2e,cpu,long,spec,bwd,cbwd,conv,prefill,tiny,fused")
    ap.add_argument("--bwd-steps", type=int, default=3)
    ap.add_argument("--workload", default="varlen", choices=["varlen", "long", "prefill"])
    ap.add_argument("--split", action="store_true",
                    help="pass scratch so that few long sequences are split across SMs")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import linear_attention_layer_gb300 as kda
    import workloads

    rank, world, local = dist_info()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (libkda has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    kda.load()
    skip = set(filter(None, args.skip.split(",")))
    peaks, peak_src = load_peaks()

    # ---- prefill (the step) ----
    p = workloads.prefill_workload(args.workload, device=device, seed=rank)
    torch.cuda.synchronize()
    H = p.meta["num_heads"]
    T = p.total_tokens
    N = p.num_seqs
    gpu_uuid = None
    try:
        gpu_uuid = str(torch.cuda.get_device_properties(device).uuid)
        if gpu_uuid and not gpu_uuid.startswith("GPU-"):
            gpu_uuid = "GPU-" + gpu_uuid
    except Exception:
        gpu_uuid = None
    clk = clock_sampler(gpu_uuid)
    total_ms, per_launch = bench_prefill(kda, p, args.steps, args.warmup, dist, device,
                                         split=args.split, clk=clk)
    total_ms = max_over_ranks(total_ms, dist, device)
    ms_per_step = total_ms / args.steps
    value = weak_scaling_value(T, world, total_ms / 1e3 / args.steps)
    launch_ms = statistics.mean(per_launch)
    state_io = (2 if p.initial_state is not None else 1) * N * H * STATE_BYTES
    alg_bytes = T * H * PREFILL_BYTES_PER_HEAD_TOKEN + 4 * (N + 1) + state_io
    achieved = alg_bytes / (launch_ms * 1e-3) / 1e9
    hbm_peak = peaks["hbm_gbs"]
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                "traffic": None if args.split else measured_traffic(args.workload),
                "kernel": "kda_chunk_fwd", "algorithmic_bytes_per_launch": alg_bytes,
                "peak_source": f"{peak_src} hbm_gbs"}
    flops = T * H * FLOPS_PER_HEAD_TOKEN
    tflops = flops / (launch_ms * 1e-3) / 1e12
    tc_burst, tc_sust = peaks.get("bf16_tflops"), peaks.get("bf16_tflops_sustained")
    tensor = {"algorithmic_tflops": round(tflops, 2), "flops_per_head_token": FLOPS_PER_HEAD_TOKEN,
              "chunk": CHUNK,
              "frac_of_bf16_burst": round(tflops / tc_burst, 4) if tc_burst else None,
              "frac_of_bf16_sustained": round(tflops / tc_sust, 4) if tc_sust else None,
              "ncu_tensor_pipe_util_pct": measured_tensor_pipe()}
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "description": workloads.DESCRIPTIONS[args.workload],
                   "num_seqs": N, "total_tokens": T, "num_heads": H, "dk": 128, "dv": 128,
                   "l2": "inputs larger than L2 (no flush)", "parallelism": f"replicas x{world}",
                   "split_long_sequences": bool(args.split)},
        "roofline": roofline,
        "head_tokens_per_s_M": round(weak_scaling_value(T * H, world, total_ms / 1e3 / args.steps), 2),
        "tensor": tensor,
        "roofline_fraction_max": round(max(achieved / hbm_peak,
                                           tflops / tc_burst if tc_burst else 0.0), 4),
        "clocks": clk.summary(),
        "gpu_launches": args.steps,
    }

    # ---- the short convolution fused into the prefill, against the separate calls ----
    if "fused" not in skip:
        fpclk = clock_sampler(gpu_uuid)
        fu_ms, sep_ms = bench_fused_prefill(kda, p, args.steps, args.warmup, device, clk=fpclk)
        fu_bytes = alg_bytes + 2 * 2 * N * H * 128 * 3 * 4  # + q, k convolution states in and out
        fu_gbs = fu_bytes / (fu_ms * 1e-3) / 1e9
        line["prefill_conv_fused"] = {
            "value": round(weak_scaling_value(T, world, fu_ms / 1e3), 3), "unit": UNIT,
            "ms_per_step": round(fu_ms, 4), "kernel": "kda_chunk_fwd_fused",
            "separate_ms_per_step": round(sep_ms, 4),
            "separate": "kda_short_conv (q), kda_short_conv (k), kda_chunk_fwd",
            "workload": workloads.DESCRIPTIONS[args.workload] + "; raw q, k, convolution width 4",
            "roofline": {"bound": "hbm", "achieved": round(fu_gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(fu_gbs / hbm_peak, 4),
                         "algorithmic_bytes_per_launch": fu_bytes},
            "clocks": fpclk.summary(), "gpu_launches": 3 * args.steps}

    # ---- the 4 x 4096-token, 16-head prefill (workspace offered: the planner
    # decides whether splitting sequences across SMs pays) ----
    if "prefill" not in skip and args.workload != "prefill":
        p2 = workloads.prefill_workload("prefill", device=device, seed=rank)
        torch.cuda.synchronize()
        pclk = clock_sampler(gpu_uuid)
        p2_ms, p2_launch = bench_prefill(kda, p2, args.steps, args.warmup, dist, device,
                                         split=True, clk=pclk)
        p2_ms = max_over_ranks(p2_ms, dist, device)
        T2, H2, N2 = p2.total_tokens, p2.meta["num_heads"], p2.num_seqs
        p2_bytes = T2 * H2 * PREFILL_BYTES_PER_HEAD_TOKEN + 4 * (N2 + 1) + N2 * H2 * STATE_BYTES
        p2_launch_ms = statistics.mean(p2_launch)
        p2_gbs = p2_bytes / (p2_launch_ms * 1e-3) / 1e9
        p2_ws = kda.chunk_fwd_workspace_size(N2, T2, H2, 128, 128, p2.q.dtype, p2.cu_seqlens_host)
        line["prefill"] = {
            "value": round(weak_scaling_value(T2, world, p2_ms / 1e3 / args.steps), 3),
            "unit": UNIT, "ms_per_step": round(p2_ms / args.steps, 4),
            "workload": workloads.DESCRIPTIONS["prefill"],
            "units": N2 * H2, "split_planned": bool(p2_ws),
            "roofline": {"bound": "hbm", "achieved": round(p2_gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(p2_gbs / hbm_peak, 4),
                         "algorithmic_bytes_per_launch": p2_bytes},
            "clocks": pclk.summary(), "gpu_launches": args.steps * (3 if p2_ws else 1)}
        del p2
        torch.cuda.empty_cache()

    # ---- the tiny fp32 call (B=1, H=1, T=64, d=32): launch-latency bound ----
    if "tiny" not in skip:
        pt = workloads.prefill_workload("tiny", device=device, seed=rank)
        t_out = torch.empty_like(pt.v)
        t_fin = torch.empty((1, 1, 32, 32), dtype=torch.float32, device=device)

        def tiny_call():
            kda.chunk_fwd(pt.q, pt.k, pt.v, pt.z, pt.beta, pt.cu_seqlens, None, out=t_out,
                          final_state=t_fin, cu_seqlens_host=pt.cu_seqlens_host)

        for _ in range(max(args.warmup, 10)):
            tiny_call()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream()
        single = []
        for _ in range(50):  # one call between a synchronize and the next
            a, b = event_time_ms(tiny_call, stream)
            torch.cuda.synchronize()
            single.append(a.elapsed_time(b))
        n_b = 500
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        a.record(stream)
        for _ in range(n_b):
            tiny_call()
        b.record(stream)
        torch.cuda.synchronize()
        host_us = (time.perf_counter() - t0) / n_b * 1e6
        # the device's own time per call: a spin kernel holds the GPU while the
        # host enqueues every call, so the calls then run back to back
        torch.cuda._sleep(int(2.0e9 * (n_b * (host_us + 20.0) * 1e-6)))
        a.record(stream)
        for _ in range(n_b):
            tiny_call()
        b.record(stream)
        torch.cuda.synchronize()
        dev_us = a.elapsed_time(b) / n_b * 1e3
        if kda.get_device_error() != 0:
            raise RuntimeError("device error word set after the tiny calls")
        line["tiny"] = {
            "value": round(dev_us, 2), "unit": "us per call",
            "value_is": "device time per call with the calls queued ahead of the GPU",
            "higher_is_better": False, "workload": workloads.DESCRIPTIONS["tiny"],
            "bound": "launch latency (41 KB of data)",
            "single_call_us_synchronised": round(statistics.median(single) * 1e3, 2),
            "host_us_per_call": round(host_us, 2),
            "calls": 50 + 2 * n_b, "gpu_launches": 50 + 2 * n_b}
        del pt

    # ---- reverse mode over the same workload ----
    if "bwd" not in skip:
        bclk = clock_sampler(gpu_uuid)
        b_ms, b_launch = bench_backward(kda, p, args.bwd_steps, args.warmup, device, clk=bclk)
        b_launch_ms = statistics.mean(b_launch)
        b_flops = T * H * BWD_FLOPS_PER_HEAD_TOKEN
        b_tf = b_flops / (b_launch_ms * 1e-3) / 1e12
        b_bytes = T * H * BWD_BYTES_PER_HEAD_TOKEN + 3 * N * H * STATE_BYTES
        b_gbs = b_bytes / (b_launch_ms * 1e-3) / 1e9
        line["backward"] = {
            "value": round(weak_scaling_value(T, world, b_ms / 1e3 / args.bwd_steps), 3),
            "unit": UNIT, "ms_per_step": round(b_ms / args.bwd_steps, 3),
            "steps": args.bwd_steps, "kernel": "kda_recurrent_bwd",
            "workload": workloads.DESCRIPTIONS[args.workload] + "; random d out and d final state",
            "roofline": {"bound": "alu", "achieved": round(b_tf, 2),
                         "peak": round(FP32_ALU_TFLOPS, 1), "unit": "TFLOP/s",
                         "frac": round(b_tf / FP32_ALU_TFLOPS, 4), "traffic": None,
                         "flops_per_head_token": BWD_FLOPS_PER_HEAD_TOKEN,
                         "peak_source": "fp32 CUDA-core peak from unit counts and the 2.07 GHz "
                                        "maximum SM clock"},
            "hbm": {"achieved": round(b_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(b_gbs / hbm_peak, 4), "algorithmic_bytes_per_launch": b_bytes},
            "clocks": bclk.summary(), "gpu_launches": args.bwd_steps}

    # ---- the chunked tensor-core reverse mode over the same workload ----
    if "cbwd" not in skip:
        cbclk = clock_sampler(gpu_uuid)
        c_ms, c_launch = bench_backward(kda, p, args.bwd_steps, args.warmup, device, clk=cbclk,
                                        chunked=True)
        c_launch_ms = statistics.mean(c_launch)
        c_flops = T * H * CBWD_FLOPS_PER_HEAD_TOKEN
        c_tf = c_flops / (c_launch_ms * 1e-3) / 1e12
        tf32_peak = peaks["bf16_tflops_sustained"] * TF32_PER_BF16
        c_bytes = T * H * BWD_BYTES_PER_HEAD_TOKEN + 3 * N * H * STATE_BYTES
        c_gbs = c_bytes / (c_launch_ms * 1e-3) / 1e9
        line["backward_chunked"] = {
            "value": round(weak_scaling_value(T, world, c_ms / 1e3 / args.bwd_steps), 3),
            "unit": UNIT, "ms_per_step": round(c_ms / args.bwd_steps, 3),
            "steps": args.bwd_steps, "kernel": "kda_chunk_bwd",
            "workload": workloads.DESCRIPTIONS[args.workload] + "; random d out and d final state",
            "roofline": {"bound": "tensor", "achieved": round(c_tf, 2),
                         "peak": round(tf32_peak, 1), "unit": "TFLOP/s",
                         "frac": round(c_tf / tf32_peak, 4), "traffic": None,
                         "flops_per_head_token": CBWD_FLOPS_PER_HEAD_TOKEN,
                         "peak_source": f"{peak_src} bf16_tflops_sustained x nominal "
                                        "tf32/bf16 ratio 1.1/2.25"},
            "hbm": {"achieved": round(c_gbs, 1), "peak": hbm_peak, "unit": "GB/s",
                    "frac": round(c_gbs / hbm_peak, 4), "algorithmic_bytes_per_launch": c_bytes},
            "clocks": cbclk.summary(), "gpu_launches": args.bwd_steps}

    # ---- the Q/K short convolution + Swish over the same workload ----
    if "conv" not in skip:
        cclk = clock_sampler(gpu_uuid)
        c_ms, c_steps = bench_short_conv(kda, p, args.steps, args.warmup, device, clk=cclk)
        c_step_ms = statistics.mean(c_steps)
        # per head-token: q and k read and their outputs written (bf16); per
        # (sequence, head): both states read and written, 3 x 128 fp32 each
        c_bytes = T * H * 4 * 256 + 4 * N * H * 128 * 3 * 4 + 2 * H * 128 * 4 * 4
        c_gbs = c_bytes / (c_step_ms * 1e-3) / 1e9
        line["short_conv"] = {
            "value": round(c_gbs, 1), "unit": "GB/s", "ms_per_step": round(c_ms / args.steps, 4),
            "steps": args.steps, "kernel": "kda_short_conv", "width": 4,
            "workload": workloads.DESCRIPTIONS[args.workload] + "; q and k, width 4, with states",
            "roofline": {"bound": "hbm", "achieved": round(c_gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(c_gbs / hbm_peak, 4), "traffic": None,
                         "algorithmic_bytes_per_step": c_bytes},
            "clocks": cclk.summary(), "gpu_launches": 4 * args.steps}

    # ---- the long single-sequence workload, split across SMs ----
    if "long" not in skip and args.workload != "long":
        del p
        torch.cuda.empty_cache()
        pl = workloads.prefill_workload("long", device=device, seed=rank)
        torch.cuda.synchronize()
        lclk = clock_sampler(gpu_uuid)
        l_ms, l_launch = bench_prefill(kda, pl, args.steps, args.warmup, dist, device, split=True,
                                       clk=lclk)
        l_ms = max_over_ranks(l_ms, dist, device)
        Tl, Hl = pl.total_tokens, pl.meta["num_heads"]
        l_bytes = Tl * Hl * PREFILL_BYTES_PER_HEAD_TOKEN + 4 * (pl.num_seqs + 1) + \
            pl.num_seqs * Hl * STATE_BYTES
        l_launch_ms = statistics.mean(l_launch)
        l_gbs = l_bytes / (l_launch_ms * 1e-3) / 1e9
        line["long"] = {
            "value": round(weak_scaling_value(Tl, world, l_ms / 1e3 / args.steps), 3), "unit": UNIT,
            "ms_per_step": round(l_ms / args.steps, 4), "workload": workloads.DESCRIPTIONS["long"],
            "split_long_sequences": True,
            "roofline": {"bound": "hbm", "achieved": round(l_gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(l_gbs / hbm_peak, 4),
                         "algorithmic_bytes_per_launch": l_bytes},
            "clocks": lclk.summary(),
            "gpu_launches": 3 * args.steps}  # per step: segment pass, state scan, final pass
        del pl
        torch.cuda.empty_cache()
        p = None

    # ---- decode ----
    if "decode" not in skip:
        del p
        torch.cuda.empty_cache()
        p = None
        d = workloads.decode_workload(device=device, seed=rank, steps=args.decode_steps + 3)
        torch.cuda.synchronize()
        dclk = clock_sampler(gpu_uuid)
        dec_ms = bench_decode(kda, d, args.decode_steps, device, clk=dclk)
        per_step_ms = dec_ms / args.decode_steps
        Nq, Hq = d.meta["num_requests"], d.meta["num_heads"]
        dec_bytes = Nq * Hq * (2 * STATE_BYTES + 3 * 256 + 512 + 4 + 256)
        gbs = dec_bytes / (per_step_ms * 1e-3) / 1e9
        line["decode"] = {
            "value": round(gbs, 1), "unit": "GB/s", "ms_per_step": round(per_step_ms, 5),
            "steps": args.decode_steps, "workload": workloads.DESCRIPTIONS["decode"],
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(gbs / hbm_peak, 4), "traffic": None,
                         "kernel": "kda_decode_step", "algorithmic_bytes_per_launch": dec_bytes,
                         "peak_source": f"{peak_src} hbm_gbs"},
            "clocks": dclk.summary(), "gpu_launches": args.decode_steps}
        # the same steps with the convolution of raw q, k and the output norm fused in
        fdclk = clock_sampler(gpu_uuid)
        fdec_ms = bench_decode_fused(kda, d, args.decode_steps, device, clk=fdclk)
        f_step_ms = fdec_ms / args.decode_steps
        f_bytes = dec_bytes + Nq * Hq * 2 * 2 * 128 * 3 * 4  # + q, k convolution states in and out
        f_gbs = f_bytes / (f_step_ms * 1e-3) / 1e9
        line["decode_fused"] = {
            "value": round(f_gbs, 1), "unit": "GB/s", "ms_per_step": round(f_step_ms, 5),
            "steps": args.decode_steps, "kernel": "kda_decode_step_fused",
            "fused": "short convolution (width 4) of raw q, k + per-head RMS output norm",
            "workload": workloads.DESCRIPTIONS["decode"],
            "roofline": {"bound": "hbm", "achieved": round(f_gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(f_gbs / hbm_peak, 4),
                         "algorithmic_bytes_per_launch": f_bytes},
            "clocks": fdclk.summary(), "gpu_launches": args.decode_steps}
        del d
        torch.cuda.empty_cache()

    # ---- speculative decoding: window of drafts + replay of the accepted prefix ----
    if "spec" not in skip:
        Bs, Hs, Ws, ns = 256, 32, 4, 200
        sclk = clock_sampler(gpu_uuid)
        s_ms, s_acc = bench_spec_decode(kda, Bs, Hs, Ws, ns, device, seed=rank, clk=sclk)
        # per (request, head): the state read and written once; the W new drafts'
        # inputs (q, k, v bf16, z fp32, beta) and outputs; the accepted drafts' inputs
        tok_in = 3 * 256 + 512 + 4
        s_bytes = int(Bs * Hs * (2 * STATE_BYTES + Ws * (tok_in + 256)) + s_acc * Hs * tok_in)
        s_gbs = s_bytes / (s_ms * 1e-3) / 1e9
        line["spec_decode"] = {
            "value": round(s_acc * Hs / (s_ms * 1e-3) / 1e6, 3), "unit": "M accepted head-tokens/s",
            "ms_per_step": round(s_ms, 5), "window": Ws, "accepted_tokens_per_step": s_acc,
            "workload": f"{Bs} requests x H={Hs}, dk=dv=128, window {Ws}, acceptance U{{0..{Ws}}}",
            "roofline": {"bound": "hbm", "achieved": round(s_gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(s_gbs / hbm_peak, 4),
                         "algorithmic_bytes_per_step": s_bytes},
            "clocks": sclk.summary(), "gpu_launches": ns}

    # ---- the same step with the short convolution and the output norm fused in ----
    if "spec" not in skip:
        Bs, Hs, Ws, ns = 256, 32, 4, 200
        fclk = clock_sampler(gpu_uuid)
        f_ms, f_acc = bench_spec_decode_fused(kda, Bs, Hs, Ws, ns, device, seed=rank, clk=fclk)
        tok_in = 3 * 256 + 512 + 4
        conv_state = 2 * 128 * 3 * 4  # q and k convolution states of one (request, head)
        f_bytes = int(Bs * Hs * (2 * STATE_BYTES + 2 * conv_state + Ws * (tok_in + 256)) +
                      f_acc * Hs * tok_in)
        f_gbs = f_bytes / (f_ms * 1e-3) / 1e9
        line["spec_decode_fused"] = {
            "value": round(f_acc * Hs / (f_ms * 1e-3) / 1e6, 3),
            "unit": "M accepted head-tokens/s", "ms_per_step": round(f_ms, 5), "window": Ws,
            "accepted_tokens_per_step": f_acc, "kernel": "kda_decode_replay_window_fused",
            "fused": "short convolution (width 4) of raw q, k + per-head RMS output norm",
            "workload": f"{Bs} requests x H={Hs}, dk=dv=128, window {Ws}, acceptance U{{0..{Ws}}}",
            "roofline": {"bound": "hbm", "achieved": round(f_gbs, 1), "peak": hbm_peak,
                         "unit": "GB/s", "frac": round(f_gbs / hbm_peak, 4),
                         "algorithmic_bytes_per_step": f_bytes},
            "clocks": fclk.summary(), "gpu_launches": ns}

    # ---- end to end through host buffers ----
    if "e2e" not in skip:
        if p is None:
            p = workloads.prefill_workload(args.workload, device=device, seed=rank)
        groups = 16
        ms, h2d, d2h, link = bench_e2e(kda, p, args.e2e_steps, device, groups=groups,
                                       warmup=args.warmup)
        ms = max_over_ranks(ms, dist, device)
        line["e2e"] = {"value": round(weak_scaling_value(T, world, ms / 1e3), 3), "unit": UNIT,
                       "ms_per_step": round(ms, 3), "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
                       "warmup": max(3, args.warmup),
                       "copy_gbs_effective": round((h2d + d2h) / (ms * 1e-3) / 1e9, 1),
                       "min_ms_per_step": round(bench_e2e.min_ms, 3),
                       "link_gbs_1gib_pinned_copy": {k: round(v, 1) for k, v in link.items()},
                       "api": "kda_chunk_fwd_host (pinned host buffers, copies overlapped with "
                              f"the kernels over {groups} groups of sequences)",
                       "gpu_launches": groups * args.e2e_steps}

    # ---- CPU oracle baseline (rank 0, N = 1 only) ----
    if "cpu" not in skip and rank == 0 and world == 1:
        tps, htok, used, desc = cpu_oracle_sample(args.cpu_budget)
        tps1, desc1 = cpu_oracle_one_core()
        line["cpu_baseline"] = {"value": round(tps / 1e6, 6), "unit": UNIT, "cores": used,
                                "kind": "oracle", "sample": desc,
                                "one_core": {"value": round(tps1 / 1e6, 6), "unit": UNIT,
                                             "cores": 1, "sample": desc1}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
