"""Benchmark of the fused attention forward (no KV cache) on GB300.

One step = one forward pass of the whole hot path (one kernel launch) over
one batch of the workload's synthetic inputs, resident in HBM. L2 is flushed
before every timed step (a 256 MiB buffer is rewritten, then another 256 MiB
buffer is read so that no dirty line is left to be written back inside the
timed step) and each step's kernel is timed with CUDA events on the
launching stream.

Prints ONE JSON line (rank 0). Metric: attention forward TFLOP/s counting
only unmasked (query, key) pairs, FLOPs = 4 * B * H * D * pairs.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

--impl reference times the fp64 CPU oracle on the host cores over a bounded
sample of the same workload (the reference arm of this benchmark).
Under torchrun (N > 1) every rank runs an independent replica of the
workload (no data-path collective; the workload's (batch, head) units are
independent), timings are max-reduced over ranks, scaling is weak.
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
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "gqa_s4096_d128"
METRIC = "attention fwd TFLOP/s (unmasked FLOPs) and % of GB300 BF16 tensor peak"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20  # GB300 L2 (about 129 MB)
# GPU spin (clock cycles, ~100 us) enqueued before each timed step's start
# event: the GPU stays busy while the host enqueues the step, so the event pair
# brackets the step's kernels and not host launch latency (which the e2e
# number includes).
SPIN_CYCLES = 200_000
KERNEL_NAME = "fa_fwd_bf16_tc_kernel"
# Workloads whose oracle figure is also taken on one host thread.
SINGLE_THREAD_WORKLOADS = ("tiny_f32", "mha_s1024_d64", "gqa_s4096_d128")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ----------------------------------------------------------------- FLOP accounting
def visible_pairs(S: int, causal: bool, window: int) -> int:
    """Number of (query, key) pairs the mask leaves visible in one (b, h)."""
    if not causal:
        if window is None or window <= 0 or window >= S:
            return S * S
        W = window  # keys within W - 1 on either side, clipped at both ends
        return S * (2 * W - 1) - W * (W - 1)
    if window is None or window <= 0 or window >= S:
        return S * (S + 1) // 2
    W = window
    return W * (W + 1) // 2 + (S - W) * W


def visible_keys_of_row(i: int, S: int, causal: bool, window: int) -> int:
    windowed = window is not None and window > 0
    hi = i if causal else (min(S - 1, i + window - 1) if windowed else S - 1)
    lo = max(0, i - window + 1) if windowed else 0
    return hi - lo + 1


def workload_flops(w) -> float:
    return 4.0 * w.B * w.H * w.D * visible_pairs(w.S, w.causal, w.window)


def algorithmic_bytes(w) -> int:
    """Minimum HBM traffic of one launch: read Q, K, V once, write O and LSE."""
    e = 2 if w.dtype == "bf16" else 4
    return (2 * w.B * w.S * w.H * w.D * e + 2 * w.B * w.S * w.Hkv * w.D * e
            + 4 * w.B * w.H * w.S)


# ----------------------------------------------------------------- KV-cache accounting
KV_METRIC = "KV-cache attention HBM GB/s (algorithmic bytes: visible cache rows, Q, O, LSE)"
KV_KERNEL_NAME = "fa_decode_bf16_tc_kernel"


def kv_row_range(L: int, Sq: int, s: int, causal: bool, window: int):
    """Visible keys [lo, hi] of query row s of a batch holding L keys."""
    pos = L - Sq + s
    windowed = window is not None and window > 0
    lo = max(0, pos - window + 1) if windowed else 0
    hi = min(pos, L - 1) if causal else (min(pos + window - 1, L - 1) if windowed else L - 1)
    return lo, hi


def kv_flops(w, lens) -> float:
    pairs = 0
    for L in lens:
        for s in range(w.Sq):
            lo, hi = kv_row_range(int(L), w.Sq, s, w.causal, w.window)
            pairs += max(0, hi - lo + 1)
    return 4.0 * w.H * w.D * pairs


def kv_algorithmic_bytes(w, lens) -> int:
    """Cache rows some query of the batch sees (K and V, once), Q read, O and
    LSE written."""
    rows = 0
    for L in lens:
        lo, _ = kv_row_range(int(L), w.Sq, 0, w.causal, w.window)
        _, hi = kv_row_range(int(L), w.Sq, w.Sq - 1, w.causal, w.window)
        rows += max(0, hi - lo + 1)
    return (2 * rows * w.Hkv * w.D * 2 + 2 * w.B * w.Sq * w.H * w.D * 2
            + 4 * w.B * w.H * w.Sq)


# ----------------------------------------------------------------- peaks / traffic
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_digest(kernel_file: str = "fa_fwd_tc.cu") -> str:
    """Digest of a kernel's source file and every local header it includes
    (transitively): a profile taken on other source no longer applies."""
    csrc = os.path.join(ROOT, "attention_fa2_forward_gb300", "csrc")
    inc_dirs = [csrc, os.path.join(ROOT, "include")]
    seen, todo = set(), [kernel_file]
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        for d in inc_dirs:
            path = os.path.join(d, name)
            if os.path.exists(path):
                seen.add(name)
                with open(path) as f:
                    todo += re.findall(r'^#include "([^"]+)"', f.read(), flags=re.M)
                break
    h = hashlib.sha256()
    for name in sorted(seen):
        path = next(os.path.join(d, name) for d in inc_dirs
                    if os.path.exists(os.path.join(d, name)))
        with open(path, "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = KERNEL_NAME,
                     kernel_file: str = "fa_fwd_tc.cu"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel source (matching digest); else None."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)\s*\(kernel source digest ([0-9a-f]+)\)",
                  text)
    if not m or m.group(2) != kernel_source_digest(kernel_file):
        return None
    return int(m.group(1))


# ----------------------------------------------------------------- end to end
def prefill_traffic(w):
    """Profiled DRAM bytes per launch of the kernel that serves workload w:
    the bf16 tensor-core kernel up to D = 128, the one-Q-tile kernel above, the
    fp32 tensor-core kernel for fp32 D 64/128 (none for the CUDA-core path)."""
    if w.dtype == "bf16":
        if w.D > 128:
            return profiled_traffic(w.name, KV_KERNEL_NAME, "fa_decode_tc.cu")
        return profiled_traffic(w.name)
    if w.D in (64, 128):
        return profiled_traffic(w.name, "fa_fwd_f32x3_kernel", "fa_fwd_f32x3.cu")
    return None


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (ctypes) while the
    timed region runs. Reads settings only."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x2: "applications_clocks_setting", 0x10: "sync_boost"}

    def __init__(self, index: int, period_s: float = 0.002):
        self.index, self.period = index, period_s
        self.samples, self.reasons = [], set()
        self.max_mhz = None
        self._stop = threading.Event()
        self._thread = None
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            if self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.handle, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.ok = True
        except OSError:
            self.ok = False

    def _sample(self):
        mhz = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
            self.samples.append(mhz.value)
        fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(self.nvml, "nvmlDeviceGetCurrentClocksThrottleReasons")
        if fn(self.handle, ctypes.byref(rs)) == 0:
            for bit, name in self.REASONS.items():
                if rs.value & bit:
                    self.reasons.add(name)

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(self.period)

    def start(self):
        """Start sampling and return once the first sample is in, so that the
        thread's start-up (NVML's first calls) falls before the timed region
        rather than inside its first step."""
        if self.ok:
            self._thread = threading.Thread(target=self._run, daemon=True)
            self._thread.start()
            t0 = time.perf_counter()
            while not self.samples and time.perf_counter() - t0 < 0.2:
                time.sleep(0.001)

    def stop(self):
        if self.ok and self._thread is not None:
            self._stop.set()
            self._thread.join()
            if not self.samples:
                self._sample()

    def summary(self):
        if not self.ok:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        return {"sm_mhz": statistics.median(self.samples) if self.samples else None,
                "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                "samples": len(self.samples)}


# ----------------------------------------------------------------- L2 flush
class L2Flush:
    """Between timed steps: write a buffer larger than L2 (evicting the
    inputs), then read a second one, so the write's dirty lines are written
    back before the step instead of during it. Outside the timed region."""

    NOTE = ("flushed before every step: 256 MiB written, then another 256 MiB read (L2 holds "
            "no input and no dirty line when the step starts)")

    def __init__(self, device, enabled: bool = True):
        import torch
        n = L2_FLUSH_BYTES // 4 if enabled else 0
        self.w = torch.empty(n, dtype=torch.float32, device=device)
        self.r = torch.ones(n, dtype=torch.float32, device=device)
        self.enabled = enabled

    def __call__(self):
        if self.enabled:
            self.w.zero_()
            self.sink = self.r.sum()


def step_stats(kernel_ms):
    """Mean and median of per-step times (ms)."""
    return statistics.fmean(kernel_ms), statistics.median(kernel_ms)


def host_cost_us(call, n: int = 200):
    """Host microseconds per call of `call` (which enqueues GPU work and does
    not synchronise), averaged over n calls after a warm-up."""
    import torch
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        call()
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    return dt / n * 1e6


# ----------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        os.environ.setdefault("MASTER_PORT", "29511")
        dist.init_process_group(backend)
    return dist if world > 1 else None


def max_over_ranks(value: float, dist) -> float:
    if dist is None:
        return value
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------- oracle sample
def oracle_sample_rows(w, target_flops: float):
    """Evenly spread query rows whose oracle work is about target_flops."""
    total = workload_flops(w)
    frac = min(1.0, target_flops / total)
    n = max(2, int(round(w.S * frac)))
    if n >= w.S:
        return list(range(w.S))
    step = w.S / n
    return sorted({min(w.S - 1, int(i * step + step / 2)) for i in range(n)})


def sampled_flops(w, rows) -> float:
    keys = sum(visible_keys_of_row(i, w.S, w.causal, w.window) for i in rows)
    return 4.0 * w.B * w.H * w.D * keys


def run_oracle_sample(w, q, k, v, rows, nthreads):
    import oracle
    t0 = time.perf_counter()
    oracle.mha_forward(q[:, rows], k, v, w.scale, w.causal, w.window, rows=rows,
                       nthreads=nthreads)
    return time.perf_counter() - t0


# ----------------------------------------------------------------- arms
def bench_reference(args, w, world, rank):
    """The fp64 oracle on the host cores: each step evaluates a bounded,
    evenly spread sample of the workload's query rows (all batches, heads)."""
    if rank != 0:
        return None
    import oracle
    from attention_fa2_forward_gb300.inputs import workload_inputs
    oracle.build()
    q, k, v = workload_inputs(w)
    nthreads = oracle.default_threads()
    # Size the per-step sample from a short calibration run.
    probe_rows = oracle_sample_rows(w, 2e9)
    t = run_oracle_sample(w, q, k, v, probe_rows, nthreads)
    rate = sampled_flops(w, probe_rows) / max(t, 1e-6)
    per_step_s = max(0.2, min(8.0, 120.0 / max(1, args.steps + args.warmup)))
    rows = oracle_sample_rows(w, rate * per_step_s)
    for _ in range(args.warmup):
        run_oracle_sample(w, q, k, v, rows, nthreads)
    times = [run_oracle_sample(w, q, k, v, rows, nthreads) for _ in range(args.steps)]
    fl = sampled_flops(w, rows)
    total_s = sum(times)
    value = fl * args.steps / total_s / 1e12
    sample = (f"{len(rows)} of {w.S} query rows (evenly spread), all {w.B} batches x {w.H} heads, "
              f"{fl / 1e9:.2f} GFLOP per step")
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def bench_ours(args, w, world, rank, local, dist):
    import torch

    import attention_fa2_forward_gb300 as fa
    from attention_fa2_forward_gb300.inputs import workload_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    lib = fa.load_library()
    q_h, k_h, v_h = workload_inputs(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    mask = "causal" if w.causal else "none"
    f32_tc = w.dtype == "f32" and w.D in (64, 128)
    launches_per_step = 3 if f32_tc else 1  # fp32 on the tensor cores: two split kernels + main
    ws = None
    if f32_tc:
        ws = torch.empty(int(lib.fa_mha_no_cache_f32_tc_workspace(w.B, w.S, w.Hkv, w.D)),
                         dtype=torch.uint8, device=dev)

    def step():
        fa.mha_no_cache(q, k, v, w.scale, mask, w.window, out=out, lse=lse, workspace=ws)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("kernel reported a timed-out wait during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    t_wall = time.perf_counter()
    for s in range(args.steps):
        flush()
        torch.cuda._sleep(SPIN_CYCLES)
        starts[s].record(stream)
        step()
        ends[s].record(stream)
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t_wall
    clocks.stop()
    barrier(dist)
    kernel_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    local_ms = sum(kernel_ms)
    mean_ms, median_ms = step_stats(kernel_ms)
    total_ms = max_over_ranks(local_ms, dist)
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("kernel reported a timed-out wait in the timed region")

    # ---- host cost of one call through the C ABI (argument checks, cached
    # tensor maps, launch; no synchronisation), and of ctypes itself
    dt = fa.DTYPE_BF16 if w.dtype == "bf16" else fa.DTYPE_F32
    mcode = fa.MASK_CAUSAL if w.causal else fa.MASK_NONE
    cargs = (out.data_ptr(), lse.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), w.B, w.S,
             w.H, w.Hkv, w.D, w.scale, mcode, w.window)
    if f32_tc:
        def c_call():
            lib.fa_mha_no_cache_f32_tc(*cargs, ws.data_ptr(), ws.numel(), stream.cuda_stream)
    else:
        def c_call():
            lib.fa_mha_no_cache(*cargs, dt, stream.cuda_stream)
    host_us = host_cost_us(c_call)
    ctypes_us = host_cost_us(lambda: lib.fa_version())
    py_us = host_cost_us(step)

    # ---- end to end through the C ABI's host-buffer entry point: pinned host
    # q, k, v in, pinned out and lse back, copies inside the timed region
    e2e = None
    if not args.no_e2e:
        qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        e2e_steps = max(2, min(args.steps, 20))
        st2 = [stream, torch.cuda.Stream(dev)]
        ws_bytes = fa.host_workspace_bytes(w.B, w.S, w.H, w.Hkv, w.D, q_h.dtype)
        wss = [torch.empty(ws_bytes, dtype=torch.uint8, device=dev) for _ in st2]
        outps = [torch.empty(q_h.shape, dtype=q_h.dtype, pin_memory=True) for _ in st2]
        lseps = [torch.empty((w.B, w.H, w.S), dtype=torch.float32, pin_memory=True)
                 for _ in st2]

        def run_e2e(n):
            # step i on stream i % 2 with its own workspace: step i+1's copy in
            # overlaps step i's kernel, step i's copy out overlaps step i+1's
            # kernel (separate copy engines for each direction)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            ev0.record(st2[0])
            st2[1].wait_event(ev0)
            done = [None, None]
            for i in range(n):
                sl = i % 2
                if done[sl] is not None:
                    st2[sl].wait_event(done[sl])
                fa.mha_no_cache_host(qp, kp, vp, outps[sl], wss[sl], w.scale, mask, w.window,
                                     lse=lseps[sl], stream=st2[sl])
                done[sl] = torch.cuda.Event()
                done[sl].record(st2[sl])
            for sl in range(2):
                if done[sl] is not None:
                    st2[0].wait_event(done[sl])
            ev1.record(st2[0])
            torch.cuda.synchronize()
            return ev0.elapsed_time(ev1) / n

        run_e2e(2)  # warm-up
        barrier(dist)
        e2e_ms = max_over_ranks(run_e2e(e2e_steps) * e2e_steps, dist) / e2e_steps
        if fa.device_status() != fa.FA_OK:
            raise RuntimeError("kernel reported a timed-out wait in the end-to-end run")
        h2d = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
        d2h = outps[0].numel() * outps[0].element_size() + lseps[0].numel() * 4
        e2e = {"value": world * workload_flops(w) / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
               "api": "fa_mha_no_cache_host (C ABI, pinned host buffers)",
               "pipeline": "steps alternate over two streams and workspaces: step i+1's copy "
                           "in overlaps step i's kernel and copy out"}

    # ---- CPU baseline: the oracle on a bounded sample, rank 0 at N=1 only
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        nthreads = oracle.default_threads()
        rows = oracle_sample_rows(w, 2e9)
        t = run_oracle_sample(w, q_h, k_h, v_h, rows, nthreads)
        rate = sampled_flops(w, rows) / max(t, 1e-6)
        rows = oracle_sample_rows(w, rate * args.cpu_seconds)
        t = run_oracle_sample(w, q_h, k_h, v_h, rows, nthreads)
        fl = sampled_flops(w, rows)
        cpu = {"value": fl / t / 1e12, "unit": "TFLOP/s", "cores": nthreads, "kind": "oracle",
               "sample": f"{len(rows)} of {w.S} query rows (evenly spread), all {w.B} batches "
                         f"x {w.H} heads: {fl / 1e9:.1f} GFLOP in {t:.1f} s"}
        if w.name in SINGLE_THREAD_WORKLOADS:
            rows1 = oracle_sample_rows(w, rate / nthreads * args.cpu_seconds / 3)
            t1 = run_oracle_sample(w, q_h, k_h, v_h, rows1, 1)
            fl1 = sampled_flops(w, rows1)
            cpu["single_thread"] = {
                "value": fl1 / t1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                "sample": f"{len(rows1)} of {w.S} query rows: {fl1 / 1e9:.2f} GFLOP in "
                          f"{t1:.1f} s"}

    flops = workload_flops(w)
    ms_per_step = total_ms / args.steps
    value = world * flops / (ms_per_step * 1e-3) / 1e12
    peaks, peak_src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_note = "bf16 burst, MEASURED_PEAKS.json"
    if w.dtype == "f32":
        # fp32 runs as six bf16 part products per contraction: its ceiling in
        # useful fp32 FLOPs is the bf16 peak / 6.
        peak /= 6.0
        peak_note = "bf16 burst / 6 part products, MEASURED_PEAKS.json"
    achieved = flops / (mean_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "achieved_median": flops / (median_ms * 1e-3) / 1e12,
                "traffic": prefill_traffic(w),
                "peak_source": f"{peak_src} ({peak_note})"
                if peak_src == "measured" else "fallback",
                "algorithmic_bytes": algorithmic_bytes(w),
                "hbm_gbs": algorithmic_bytes(w) / (mean_ms * 1e-3) / 1e9}
    return {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": median_ms,
        "value_median": world * flops / (median_ms * 1e-3) / 1e12,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if w.dtype == "bf16" else "f32 (three bf16 parts per value, fp32 accumulation)",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "B": w.B, "S": w.S, "H": w.H,
                   "Hkv": w.Hkv, "D": w.D, "mask": mask, "window": w.window,
                   "flops_per_step": flops, "l2": L2Flush.NOTE,
                   "timing": "CUDA events around each step; a GPU spin before the start event "
                             "hides host launch latency (e2e includes it)",
                   "host_us_per_call": host_us,
                   "host_us_note": "CPU time of one C-ABI call (checks, cached tensor maps, "
                                   "launch; no sync) through ctypes, whose own cost is "
                                   "ctypes_us_per_call; python_us_per_call is the Python "
                                   "binding's call",
                   "ctypes_us_per_call": ctypes_us, "python_us_per_call": py_us,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "pct_of_peak": 100.0 * value / (peak * world),
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clocks.summary(), "gpu_launches": args.steps * launches_per_step,
        "wall_s_timed_region": wall_s,
    }


def bench_kv_reference(args, w, world, rank):
    """The fp64 oracle's KV-cache form on the host cores, on the first batches
    of the workload (bounded to a few seconds per step)."""
    if rank != 0:
        return None
    import oracle
    from attention_fa2_forward_gb300.inputs import kv_workload_inputs
    oracle.build()
    q, k, v, lens = kv_workload_inputs(w)
    nthreads = oracle.default_threads()
    nb = max(1, min(w.B, 2))

    def one():
        t0 = time.perf_counter()
        oracle.mha_forward_kvcache(q[:nb], k[:nb], v[:nb], w.scale, lens[:nb].numpy(), w.causal,
                                   w.window, nthreads=nthreads)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one()
    times = [one() for _ in range(args.steps)]
    sub = lens[:nb].tolist()
    byts = kv_algorithmic_bytes(type(w)(**{**w.__dict__, "B": nb}), sub)
    value = byts * args.steps / sum(times) / 1e9
    sample = f"batches 0..{nb - 1} of {w.B} (all heads, all query rows): {byts / 1e6:.1f} MB"
    return {
        "impl": "reference", "metric": KV_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sum(times) / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": nthreads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def bench_kv_ours(args, w, world, rank, local, dist):
    """One attention step over resident KV caches per timed step (the caches
    live in HBM, as in decoding; e2e copies the step's queries and lengths in
    and its output out)."""
    import torch

    import attention_fa2_forward_gb300 as fa
    from attention_fa2_forward_gb300.inputs import kv_workload_inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load_library()
    q_h, k_h, v_h, lens_h = kv_workload_inputs(w)
    q, k, v, lens = q_h.to(dev), k_h.to(dev), v_h.to(dev), lens_h.to(dev)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    mask = "causal" if w.causal else "none"
    splits, ws_bytes = fa.kv_cache_plan(w.B, w.Sq, w.S_cache, w.H, w.Hkv, w.D, mask, w.window,
                                        args.splits)
    ws = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)

    def step():
        fa.mha_kv_cache(q, k, v, lens, w.scale, mask, w.window, num_splits=args.splits, out=out,
                        lse=lse, workspace=ws)

    # Inputs larger than L2 need no flush between steps (a 256 MiB write would
    # leave dirty lines whose write-back competes with the kernel's reads).
    cache_bytes = 2 * k.numel() * k.element_size()
    big_inputs = cache_bytes > 2 * L2_BYTES
    flush = L2Flush(dev, enabled=not big_inputs)
    l2_note = (f"no flush: the step reads {cache_bytes / 1e6:.0f} MB of KV cache, more than "
               f"the {L2_BYTES / 1e6:.0f} MB L2" if big_inputs else L2Flush.NOTE)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("kernel reported a timed-out wait during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    for s in range(args.steps):
        flush()
        torch.cuda._sleep(SPIN_CYCLES)
        starts[s].record(stream)
        step()
        ends[s].record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    barrier(dist)
    kernel_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    local_ms = sum(kernel_ms)
    _, median_ms = step_stats(kernel_ms)
    total_ms = max_over_ranks(local_ms, dist)
    if fa.device_status() != fa.FA_OK:
        raise RuntimeError("kernel reported a timed-out wait in the timed region")

    lens_list = lens_h.tolist()
    byts = kv_algorithmic_bytes(w, lens_list)
    flops = kv_flops(w, lens_list)
    ms_per_step = total_ms / args.steps
    value = world * byts / (ms_per_step * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        qp, lp = q_h.pin_memory(), lens_h.pin_memory()
        outp = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        e2e_steps = max(1, min(args.steps, 20))

        def e2e_step():
            q.copy_(qp, non_blocking=True)
            lens.copy_(lp, non_blocking=True)
            step()
            outp.copy_(out, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist) / e2e_steps
        e2e = {"value": world * byts / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": qp.numel() * qp.element_size() + lp.numel() * 4,
               "d2h_bytes_per_step": outp.numel() * outp.element_size(),
               "ms_per_step": e2e_ms, "note": "KV caches resident on the device"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res = bench_kv_reference(argparse.Namespace(steps=1, warmup=0), w, 1, 0)
        cpu = res["cpu_baseline"]

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = byts / (local_ms / args.steps * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": profiled_traffic(w.name, KV_KERNEL_NAME, "fa_decode_tc.cu"),
                "peak_source": f"{peak_src} (HBM copy, MEASURED_PEAKS.json)"
                if peak_src == "measured" else "fallback",
                "algorithmic_bytes": byts,
                "tflops": flops / (local_ms / args.steps * 1e-3) / 1e12}
    return {
        "metric": KV_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": median_ms, "value_median": world * byts / (median_ms * 1e-3) / 1e9,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "B": w.B, "Sq": w.Sq,
                   "S_cache": w.S_cache, "H": w.H, "Hkv": w.Hkv, "D": w.D, "mask": mask,
                   "window": w.window, "lens": "ragged" if w.ragged else "full",
                   "splits": splits, "bytes_per_step": byts, "flops_per_step": flops,
                   "l2": l2_note,
                   "timing": "CUDA events around each step; a GPU spin before the start event "
                             "hides host launch latency (e2e includes it)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        "clocks": clocks.summary(), "gpu_launches": args.steps * (2 if splits > 1 else 1),
    }


TOPK_METRIC = "top-K selection HBM GB/s (algorithmic bytes: scores read once, values and indices written)"


def topk_bytes(w) -> int:
    return w.B * w.V * 4 + w.B * w.K * 8


def bench_topk_reference(args, w, world, rank):
    """The numpy top-K oracle on the host cores, on the first rows of the
    workload."""
    if rank != 0:
        return None
    from attention_fa2_forward_gb300.inputs import make_scores
    from oracle import topk as topk_oracle
    scores = make_scores(w.B, w.V, w.seed).numpy()
    rows = max(1, min(w.B, 16))

    def one():
        t0 = time.perf_counter()
        topk_oracle.topk(scores[:rows], w.K)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        one()
    times = [one() for _ in range(args.steps)]
    byts = rows * w.V * 4 + rows * w.K * 8
    value = byts * args.steps / sum(times) / 1e9
    sample = f"rows 0..{rows - 1} of {w.B}: {byts / 1e6:.1f} MB per step"
    return {
        "impl": "reference", "metric": TOPK_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sum(times) / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def bench_topk_ours(args, w, world, rank, local, dist):
    import torch

    import attention_fa2_forward_gb300 as fa
    from attention_fa2_forward_gb300.inputs import make_scores

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load_library()
    scores_h = make_scores(w.B, w.V, w.seed)
    scores = scores_h.to(dev)
    values = torch.empty((w.B, w.K), dtype=torch.float32, device=dev)
    indices = torch.empty((w.B, w.K), dtype=torch.int32, device=dev)
    chunks, ws_bytes = fa.topk_plan(w.B, w.V, w.K)
    ws = torch.empty(max(ws_bytes, 8), dtype=torch.uint8, device=dev)
    # Scores larger than L2 need no flush between steps: a launch reads each
    # score once, and steady-state ncu counters (cache control off) show every
    # launch reading all of them from DRAM; a flush would instead leave L2
    # full of dirty lines that the kernel pays to write back.
    big = scores.numel() * 4 > L2_BYTES
    flush = L2Flush(dev, enabled=not big)
    stream = torch.cuda.current_stream(dev)

    def step():
        fa.topk(scores, w.K, values=values, indices=indices, workspace=ws)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(torch.cuda.current_device())
    barrier(dist)
    torch.cuda.synchronize()
    clocks.start()
    for s in range(args.steps):
        flush()
        torch.cuda._sleep(SPIN_CYCLES)
        starts[s].record(stream)
        step()
        ends[s].record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    barrier(dist)
    kernel_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    local_ms = sum(kernel_ms)
    _, median_ms = step_stats(kernel_ms)
    total_ms = max_over_ranks(local_ms, dist)
    byts = topk_bytes(w)
    ms_per_step = total_ms / args.steps
    value = world * byts / (ms_per_step * 1e-3) / 1e9

    e2e = None
    if not args.no_e2e:
        sp = scores_h.pin_memory()
        vp = torch.empty(values.shape, dtype=values.dtype, pin_memory=True)
        ip = torch.empty(indices.shape, dtype=indices.dtype, pin_memory=True)
        e2e_steps = max(1, min(args.steps, 20))

        def e2e_step():
            scores.copy_(sp, non_blocking=True)
            step()
            vp.copy_(values, non_blocking=True)
            ip.copy_(indices, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist) / e2e_steps
        e2e = {"value": world * byts / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": sp.numel() * 4,
               "d2h_bytes_per_step": vp.numel() * 4 + ip.numel() * 4, "ms_per_step": e2e_ms}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = bench_topk_reference(argparse.Namespace(steps=1, warmup=0), w, 1, 0)["cpu_baseline"]

    peaks, peak_src = load_peaks()
    peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    achieved = byts / (local_ms / args.steps * 1e-3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak,
                "traffic": profiled_traffic(w.name, "topk_chunk_kernel", "topk.cu"),
                "peak_source": f"{peak_src} (HBM copy, MEASURED_PEAKS.json)"
                if peak_src == "measured" else "fallback",
                "algorithmic_bytes": byts}
    return {
        "metric": TOPK_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "ms_per_step_median": median_ms, "value_median": world * byts / (median_ms * 1e-3) / 1e9,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "shape": w.describe(), "B": w.B, "V": w.V, "K": w.K,
                   "chunks_per_row": chunks, "bytes_per_step": byts,
                   "l2": (f"no flush: the step reads {scores.numel() * 4 / 1e6:.0f} MB, more "
                          f"than the {L2_BYTES / 1e6:.0f} MB L2") if big
                   else L2Flush.NOTE,
                   "timing": "CUDA events around each step; a GPU spin before the start event "
                             "hides host launch latency (e2e includes it)",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
        # rows of 1, 2, 4 or 8 chunks are finished by the chunk kernel (no workspace);
        # other plans add a merge kernel
        "clocks": clocks.summary(), "gpu_launches": args.steps * (1 if ws_bytes == 0 else 2),
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--splits", type=int, default=0,
                    help="KV-cache workloads: key-range splits (0: the library's choice)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    from attention_fa2_forward_gb300.inputs import KV_WORKLOADS, TOPK_WORKLOADS, WORKLOADS
    arms = {}
    for table, ref, ours in ((WORKLOADS, bench_reference, bench_ours),
                             (KV_WORKLOADS, bench_kv_reference, bench_kv_ours),
                             (TOPK_WORKLOADS, bench_topk_reference, bench_topk_ours)):
        for name, wl in table.items():
            arms[name] = (wl, ref, ours)
    if args.workload not in arms:
        ap.error(f"unknown workload {args.workload!r} (choose from {sorted(arms)})")
    w, ref_arm, our_arm = arms[args.workload]
    world, rank, local = dist_env()
    if args.impl == "reference":
        res = ref_arm(args, w, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return 0
    dist = init_dist(world, "nccl")
    res = our_arm(args, w, world, rank, local, dist)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
