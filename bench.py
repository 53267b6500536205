"""Throughput of the bf16 attention forward on one GB300, one JSON line.

A step is one call of fa_fwd over the whole workload (default: B=1, H=32,
N=16384, D=128, causal, the long-context throughput configuration), with the
inputs already resident in device memory.  FLOPs per step = 4*D*P where P is
the exact number of (query, key) pairs the mask allows (causal counts the
lower triangle including the diagonal).  The inputs (Q, K, V: 384 MiB) are
larger than the 126 MiB L2, so no flush is needed between timed steps.

Also reported on the same line:
  roofline      dominant kernel (the tcgen05 forward) against the measured
                dense bf16 tensor peak; its duration is timed with CUDA events
                on the launching stream;
  e2e           the same metric through the C ABI with host buffers: every
                step copies Q, K, V from pinned host memory and O and LSE
                back, all inside the timed region, through fa_fwd_from_host
                (the copies of one group of heads overlap the computation of
                the next);
  cpu_baseline  the fp64 CPU oracle timed on a bounded sample of the same
                workload on this host's cores (rank 0, N=1 only);
  clocks        SM clocks, power and throttle reasons sampled (NVML, read
                only) every 2 ms during the timed region, and SM cycles per
                step at the median clock.

--impl reference times the CPU oracle alone (the reference arm).
Multi-GPU: one process per GPU under torchrun; the path shards by
(batch, head) with no exchange, so every rank runs its own full workload
(weak scaling) and rank 0 reports the units of all ranks over the slowest
rank's time.
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
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "attention fwd TFLOP/s on 1 GB300 and % of dense bf16 tensor peak"
L2_BYTES = 126 << 20
# MUFU ex2.approx.ftz.f32 results per clock per SM, measured on a GB300 with
# independent exponentials on every SM sub-partition (about 8 lanes per clock
# each).  Every visible score takes at least one exponential, so this rate
# bounds the attention FLOP rate at D=64 and below, beside the tensor roofline.
EX2_PER_CLK_PER_SM = 31.0
UNIT = "TFLOP/s"
FALLBACK_PEAK_TFLOPS = 1900.0   # used only when MEASURED_PEAKS.json is absent
HOST_LEAD_CYCLES = 400_000      # about 0.2 ms of SM clock: the host's lead on the device


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"bf16_tflops": FALLBACK_PEAK_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


# The sources each timed kernel is built from; a DRAM-traffic figure taken
# by ncu stays valid only while these files are unchanged.
KERNEL_SOURCES = {
    "fwd_bf16_kernel": ("fa_fwd_bf16.cu", "fa_fwd_softmax.cuh", "fa_tc_common.cuh", "sm103_ptx.cuh",
                        "fa_internal.h", "fa_api.cu"),
    "bwd_kernel": ("fa_bwd_bf16.cu", "fa_tc_common.cuh", "sm103_ptx.cuh", "fa_internal.h", "fa_api.cu"),
    "fwd_fp32_kernel": ("fa_fwd_fp32.cu", "fa_internal.h", "fa_api.cu"),
    "fwd_onetile_kernel": ("fa_fwd_onetile.cu", "fa_fwd_softmax.cuh", "fa_tc_common.cuh", "sm103_ptx.cuh",
                           "fa_internal.h", "fa_api.cu"),
    "fwd_halves_kernel": ("fa_fwd_halves.cu", "fa_fwd_softmax.cuh", "fa_tc_common.cuh", "sm103_ptx.cuh",
                          "fa_internal.h", "fa_api.cu"),
}


_COMMENT = re.compile(r"//[^\n]*|/\*.*?\*/", re.S)


def kernel_source_hash(kernel: str) -> str:
    """Hash of the kernel's sources with comments and blank space removed, so
    that editing a comment keeps profiled counters valid."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "exact_tiled_attention_23_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            code = _COMMENT.sub("", f.read())
        h.update(name.encode())
        h.update(" ".join(code.split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, if it
    was taken on the kernel's current sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)
    ent = rec.get(workload)
    if not ent or ent.get("kernel") != kernel or ent.get("source_hash") != kernel_source_hash(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


class _Nvml:
    """Read-only NVML queries through ctypes (clocks, power, clock-event
    reasons).  Nothing here changes a GPU setting."""

    # clock-event reason bits of nvml.h
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.dev = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.max_mhz = self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn):
        v = self.ct.c_uint()
        if fn(self.dev, self.ct.c_int(1), self.ct.byref(v)) != 0:    # NVML_CLOCK_SM
            raise OSError("clock query failed")
        return float(v.value)

    def sample(self):
        sm = self._clock(self.lib.nvmlDeviceGetClockInfo)
        bits = self.ct.c_ulonglong()
        self.reasons_fn(self.dev, self.ct.byref(bits))
        mw = self.ct.c_uint()
        self.lib.nvmlDeviceGetPowerUsage(self.dev, self.ct.byref(mw))
        reasons = [n for b, n in self.REASONS.items() if bits.value & b]
        return sm, self.max_mhz, mw.value / 1e3, reasons


class ClockSampler:
    """SM clock, power and clock-event reasons sampled every few milliseconds
    while the timed loop runs: NVML through ctypes in a thread (every 2 ms),
    else nvidia-smi (every 10 ms).  Entering waits for the first sample, so
    even a region of a few tens of milliseconds carries several."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.002

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.thread = None
        self.samples = []            # (sm_mhz, max_mhz, watts, [reasons])
        self.source = "none"
        self._stop = threading.Event()
        self._first = threading.Event()

    def __enter__(self):
        try:
            nv = _Nvml(self.gpu)
            nv.sample()
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll_nvml, args=(nv,), daemon=True)
        except (OSError, AttributeError):
            try:
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                     "--format=csv,noheader,nounits", "-lms", "10"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                self.thread = threading.Thread(target=self._read_smi, daemon=True)
            except OSError:
                self.proc = None
        if self.thread is not None:
            self.thread.start()
            self._first.wait(timeout=5.0)
        return self

    def _poll_nvml(self, nv):
        while not self._stop.is_set():
            try:
                self.samples.append(nv.sample())
            except OSError:
                pass
            self._first.set()
            time.sleep(self.PERIOD_S)

    def _read_smi(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.proc.stdout:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, mx = float(parts[1]), float(parts[2])
                watts = float(parts[3]) if parts[3] not in ("", "[N/A]") else float("nan")
            except ValueError:
                continue
            self.samples.append((sm, mx, watts, [n for n, v in zip(names, parts[5:9]) if v.lower() == "active"]))
            self._first.set()

    def __exit__(self, *exc):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": self.source}
        sm = [x[0] for x in self.samples]
        watts = [x[2] for x in self.samples if x[2] == x[2]]
        reasons = sorted({r for x in self.samples for r in x[3]})
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max(x[1] for x in self.samples),
                "power_w_max": max(watts) if watts else None, "reasons": reasons,
                "samples": len(sm), "source": self.source}


# ------------------------------------------------------------ multi-rank
def slowest_rank_ms(local_ms: float, world: int, device=None) -> float:
    """Max over ranks of the timed region (each rank runs its own replica)."""
    if world <= 1:
        return float(local_ms)
    t = torch.tensor([float(local_ms)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, slowest_ms: float, world: int) -> float:
    """Whole-job TFLOP/s: every rank does `steps` steps of `flops_per_step`
    (weak scaling), all within the slowest rank's time."""
    return world * flops_per_step * steps / (slowest_ms * 1e-3) / 1e12


# --------------------------------------------------------------------- oracle
_F32_CACHE = {}


def oracle_sample(inp, budget_s: float, seed: int = 0):
    """Time the fp64 oracle on randomly chosen query rows of the workload for
    about `budget_s` seconds; returns (flops, seconds, rows, threads)."""
    import oracle

    w = inp.workload
    lib = oracle.library()
    threads = lib.max_threads()
    if w.name not in _F32_CACHE:
        _F32_CACHE[w.name] = tuple(np.ascontiguousarray(x.float().numpy()) for x in (inp.q, inp.k, inp.v))
    qf, kf, vf = _F32_CACHE[w.name]
    kv = None if inp.kv_len is None else inp.kv_len.numpy()
    rng = np.random.default_rng(seed)
    total_rows = w.B * w.H * w.N

    def flops_of(rows):
        i = rows % w.N
        b = rows // (w.N * w.H)
        L = np.full(rows.shape, w.N) if kv is None else np.clip(kv[b], 0, w.N)
        nk = np.minimum(L, i + 1) if w.causal else L
        return float(4 * w.D * nk.sum())

    # calibrate on growing batches (>= 0.2 s), then run one batch sized to the budget
    n = max(threads, 16)
    while True:
        rows = rng.integers(0, total_rows, n)
        t0 = time.perf_counter()
        lib.attention_rows(qf, kf, vf, rows, causal=w.causal, scale=w.scale, kv_len=kv)
        dt = time.perf_counter() - t0
        if dt >= min(0.2, budget_s / 4) or n >= total_rows:
            break
        n = min(total_rows, n * 4)
    n = int(min(total_rows, max(n, n * budget_s / max(dt, 1e-6))))
    rows = rng.integers(0, total_rows, n)
    t0 = time.perf_counter()
    lib.attention_rows(qf, kf, vf, rows, causal=w.causal, scale=w.scale, kv_len=kv)
    dt = time.perf_counter() - t0
    return flops_of(rows), dt, n, threads


def run_reference(args, rank, world):
    if rank != 0:
        return
    inp = workloads.make(args.workload)
    w = inp.workload
    vals = []
    for _ in range(args.warmup):
        oracle_sample(inp, budget_s=min(1.0, args.ref_step_seconds), seed=1)
    t_all = 0.0
    flops_all = 0.0
    rows_all = 0
    threads = 1
    for s in range(args.steps):
        f, dt, n, threads = oracle_sample(inp, budget_s=args.ref_step_seconds, seed=100 + s)
        vals.append(f / dt / 1e12)
        t_all += dt
        flops_all += f
        rows_all += n
    value = flops_all / t_all / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_all / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{rows_all} random query rows of {w.name} over {args.steps} steps "
                                   f"({t_all:.1f} s in all), fp64 two-pass naive attention"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import exact_tiled_attention_23_gb300 as fa

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    fa.build()
    fa.load()
    inp = workloads.make(args.workload, heads=args.heads, dtype=args.dtype, seq=args.seq, dim=args.dim)
    w = inp.workload
    B, H, N, D = w.B, w.H, w.N, w.D
    pairs = workloads.unmasked_pairs(N, w.causal, None if inp.kv_len is None else inp.kv_len.tolist(), B, H)
    flops = 4.0 * D * pairs

    q, k, v = inp.q.to(dev), inp.k.to(dev), inp.v.to(dev)
    kv = inp.kv_len.to(dev) if inp.kv_len is not None else None
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sp = stream.cuda_stream
    kv_ptr = kv.data_ptr() if kv is not None else None
    fwd = {"bf16": fa.fa_fwd, "fp16": fa.fa_fwd_f16, "fp32": fa.fa_fwd_fp32}[w.dtype]
    splits = None
    if args.splits is not None:
        if w.dtype != "bf16":
            raise SystemExit("--splits needs a bf16 workload")
        splits = args.splits if args.splits > 0 else fa.fa_fwd_splitkv_auto_splits(B, H, N, D)
        ws_bytes = fa.fa_fwd_splitkv_workspace_bytes(B, H, N, D, splits)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)   # outside the timed region

    if args.pass_ == "bwd":
        if w.dtype not in ("bf16", "fp16"):
            raise SystemExit("--pass bwd needs a bf16 or fp16 workload")
        bwd = fa.fa_bwd_f16 if w.dtype == "fp16" else fa.fa_bwd
        # the forward's outputs and an upstream gradient, made outside the timed region
        fa.forward(q, k, v, causal=w.causal, kv_len=kv, out=o, lse=lse)
        gen = torch.Generator("cpu").manual_seed(w.seed + 99)
        d_o = torch.randn(q.shape, generator=gen).to(q.dtype).to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
        bwd_ws_bytes = fa.fa_bwd_workspace_bytes(B, H, N, D)
        bwd_ws = torch.empty(bwd_ws_bytes, dtype=torch.uint8, device=dev)
        flops = 10.0 * D * pairs          # five products of 2*D flops per visible pair

    def step():
        if args.pass_ == "bwd":
            st = bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), d_o.data_ptr(),
                     lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D,
                     w.causal, float("nan"), kv_ptr, bwd_ws.data_ptr(), bwd_ws_bytes, sp)
        elif splits is not None:
            st = fa.fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   B, H, N, D, w.causal, float("nan"), kv_ptr, splits,
                                   workspace.data_ptr(), ws_bytes, sp)
        else:
            st = fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                     B, H, N, D, w.causal, float("nan"), kv_ptr, sp)
        if st != fa.FA_OK:
            raise fa.FAError(st, "fa_fwd")

    torch.cuda.synchronize(dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fa_device_status(sp) != fa.FA_OK:
        raise RuntimeError("device status not OK after warm-up")

    # ---- timed region: K steps, events on the launching stream -------------
    input_bytes = sum(x.numel() * x.element_size() for x in (q, k, v))
    flush = args.flush_l2 == "on" or (args.flush_l2 == "auto" and input_bytes < 2 * L2_BYTES)
    scratch = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if flush else None
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            t_begin = torch.cuda.Event(enable_timing=True)
            t_end = torch.cuda.Event(enable_timing=True)
            # A bounded device-side wait ahead of the loop (and after every
            # flush) lets the host queue the next step before the GPU reaches
            # it, so a step interval holds device time only, not the host's
            # call overhead.  Neither wait lies inside a timed interval.
            torch.cuda._sleep(HOST_LEAD_CYCLES * 4)
            t_begin.record(stream)
            for s in range(args.steps):
                if flush:
                    scratch.fill_(s & 0xFF)     # evict the inputs from L2 (not timed)
                    torch.cuda._sleep(HOST_LEAD_CYCLES)
                starts[s].record(stream)
                step()
                ends[s].record(stream)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    kernel_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    # with a flush, the timed work is the sum of the step intervals (flushes excluded)
    total_ms = sum(kernel_ms) if flush else t_begin.elapsed_time(t_end)
    if fa.fa_device_status(sp) != fa.FA_OK:
        raise RuntimeError("device status not OK after the timed loop")
    t_max = slowest_rank_ms(total_ms, world, dev)
    value = job_throughput(flops, args.steps, t_max, world)
    avg_kernel_ms = sum(kernel_ms) / len(kernel_ms)

    peaks, peak_kind = measured_peaks()
    achieved = flops / (avg_kernel_ms * 1e-3) / 1e12
    if w.dtype in ("bf16", "fp16"):
        # fp16 and bf16 have the same dense tensor rate (kind::f16)
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAK_TFLOPS))
        # the kernel the library runs for these sizes (FA_FWD_TILES forces one)
        choice = fa.fa_fwd_kernel_choice(B, H, N, D)
        kname = ("bwd_kernel" if args.pass_ == "bwd" else
                 "fwd_bf16_kernel" if splits is not None else
                 {1: "fwd_onetile_kernel", 3: "fwd_halves_kernel"}.get(choice, "fwd_bf16_kernel"))
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": profiled_traffic(w.name, kname),
                    "peak_kind": f"{peak_kind} dense bf16 (burst)",
                    "kernel": kname, "flops_per_launch": flops}
    else:
        # fp32 FMA on the CUDA cores: 152 SMs x 128 lanes x 2 flops x max SM clock
        peak = 152 * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
        roofline = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                    "frac": achieved / peak, "traffic": profiled_traffic(w.name, "fwd_fp32_kernel"),
                    "peak_kind": "fp32 FMA, derived from unit counts and max clock",
                    "kernel": "fwd_fp32_kernel", "flops_per_launch": flops}
    hbm_bytes = input_bytes + o.numel() * o.element_size() + lse.numel() * 4
    roofline["hbm_gbs"] = hbm_bytes / (avg_kernel_ms * 1e-3) / 1e9
    roofline["hbm_frac"] = roofline["hbm_gbs"] / float(peaks.get("hbm_gbs", 6800.0))
    roofline["algorithmic_bytes_per_launch"] = hbm_bytes

    # ---- e2e through the C ABI with host buffers ---------------------------
    e2e = None
    if not args.no_e2e and args.pass_ == "fwd":
        hq, hk, hv = (x.pin_memory() for x in (inp.q, inp.k, inp.v))
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hl = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        e2e_steps = max(3, min(args.steps, 20))
        # 16-bit single-pass forward: the library's host entry point, which
        # overlaps the copies of one group of heads with the computation of
        # the next; otherwise copy in, compute, copy out
        from_host = w.dtype in ("bf16", "fp16") and splits is None
        groups = fa.fa_fwd_from_host_auto_groups(B, H, N, D) if from_host else 0

        def e2e_step():
            if from_host:
                st = fa.fa_fwd_from_host(hq.data_ptr(), hk.data_ptr(), hv.data_ptr(), ho.data_ptr(),
                                         hl.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), B, H, N, D, w.causal, float("nan"), kv_ptr,
                                         w.dtype == "fp16", groups, sp)
                if st != fa.FA_OK:
                    raise fa.FAError(st, "fa_fwd_from_host")
                return
            with torch.cuda.stream(stream):
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
                step()
                ho.copy_(o, non_blocking=True)
                hl.copy_(lse, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e_ms = e0.elapsed_time(e1) / e2e_steps
        h2d = sum(x.numel() * x.element_size() for x in (hq, hk, hv))
        d2h = ho.numel() * ho.element_size() + hl.numel() * hl.element_size()
        e2e = {"value": world * flops / (e_ms * 1e-3) / 1e12, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e_ms,
               "steps": e2e_steps,
               "path": (f"fa_fwd_from_host ({groups} head groups, copies overlapped with compute)"
                        if from_host else "copy in, compute, copy out")}

    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return

    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        f, dt, n, threads = oracle_sample(inp, budget_s=args.cpu_seconds)
        cpu = {"value": f / dt / 1e12, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": f"{n} random query rows of {w.name} ({dt:.1f} s), fp64 two-pass naive attention"}

    line = {
        "metric": METRIC if args.pass_ == "fwd" else METRIC.replace("attention fwd", "attention bwd"),
        "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "B": B, "H": H, "N": N, "D": D, "causal": w.causal,
                   "padded": w.padded, "flops_per_step": flops, "unmasked_pairs": pairs,
                   "l2": ("256 MiB write before every step (flush not timed)" if flush else
                          "inputs (Q,K,V) larger than L2; no flush between steps" if input_bytes >= L2_BYTES else
                          f"no flush: inputs (Q,K,V, {input_bytes >> 20} MiB) stay in L2 between steps (warm)"),
                   "parallelism": f"replicas x{world} (no exchange)",
                   "path": (("fa_bwd_f16" if w.dtype == "fp16" else "fa_bwd") if args.pass_ == "bwd" else
                            "fa_fwd" if splits is None else f"fa_fwd_splitkv (splits={splits})")},
        "pct_of_peak": 100.0 * value / world / peak,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": args.steps * (3 if args.pass_ == "bwd" else 2 if splits is not None else 1),
        "clocks": clk.summary(),
    }
    if line["clocks"]["sm_mhz"]:
        # SM cycles per step at the sampled median clock: comparable across
        # boxes whose clocks differ
        line["clocks"]["kcycles_per_step"] = t_max / args.steps * 1e-3 * line["clocks"]["sm_mhz"] * 1e3
    if roofline["bound"] == "tensor":
        # the exp2 ceiling: exponentials per second x FLOPs of the metric per
        # visible score (4D forward, 10D backward), at the sampled SM clock
        mhz = line["clocks"]["sm_mhz"] or float(peaks.get("sm_max_mhz", 2070.0))
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        per_score = (10 if args.pass_ == "bwd" else 4) * D
        ceiling = EX2_PER_CLK_PER_SM * sms * mhz * 1e6 * per_score / 1e12
        roofline["exp2_ceiling"] = ceiling
        roofline["exp2_frac"] = roofline["achieved"] / ceiling
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=list(workloads.WORKLOADS))
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=8.0)
    ap.add_argument("--heads", type=int, default=None,
                    help="override the workload's head count (smaller profiling captures)")
    ap.add_argument("--flush-l2", choices=["auto", "on", "off"], default="auto",
                    help="write a 256 MiB buffer before every timed step (auto: when Q,K,V fit in 2x L2)")
    ap.add_argument("--seq", type=int, default=None,
                    help="override the workload's sequence length N (IO probe, profiler captures)")
    ap.add_argument("--dim", type=int, default=None,
                    help="override the workload's head dimension D")
    ap.add_argument("--dtype", choices=["bf16", "fp16"], default=None,
                    help="override the element type of a 16-bit workload")
    ap.add_argument("--splits", type=int, default=None,
                    help="time the split-KV path with this many key ranges (0 = automatic)")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward pass (fa_bwd)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)          # at least 3 untimed warm-up steps
    rank, world, local = dist_env()
    if args.impl == "reference":
        # the whole reference run (warm-up + timed samples) stays within ~4 minutes
        args.ref_step_seconds = min(args.ref_step_seconds, 200.0 / (args.steps + args.warmup))
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
