#!/usr/bin/env python3
"""Benchmark of the fused attention forward on one or more B300s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl ours|reference]

A step is one attention forward (one ``attn_fwd`` call through the C ABI)
over the whole workload, inputs resident in device memory. The default
workload is the long-context prefill shape B=2, H=32, S=8192, d=128, bf16,
causal. Workloads named ``bwd_*`` time the backward pass instead (one
``attn_bwd`` call: dQ, dK, dV from q, k, v, O, LSE and dO), counted as 2.5
times the forward's FLOPs. Prints ONE JSON line on rank 0.

With N > 1 (one process per GPU, launched by torch.distributed.run; given
--gpus N outside such a launch, the script starts the N ranks itself) every
rank runs the same workload on its own GPU (independent replicas: the heads
of the batch are independent, nothing is exchanged), timing is bracketed by
barriers, the time is the max over ranks and ``value`` counts all ranks' work.

``--impl reference`` times the CPU oracle (fp64, the host's cores) on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("attention fwd TFLOP/s (4·B·H·Sq·Sk·d, causal halved) "
          "and % of B300 tensor peak")
METRIC_BWD = ("attention bwd TFLOP/s (2.5 x 4·B·H·Sq·Sk·d, causal halved) "
              "and % of B300 tensor peak")


def metric_of(w) -> str:
    return METRIC_BWD if w.backward else METRIC
DEFAULT_WORKLOAD = "b2h32s8192d128_causal"
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL_SOURCES = ["exact_attention_forward_14_b300/csrc/attn_fwd_kernel.cuh",
                  "exact_attention_forward_14_b300/csrc/ptx.cuh"]
# the backward's traffic also depends on how the host launches its kernels
# (dK/dV and dQ side by side on split SMs), so the host file is part of it
KERNEL_SOURCES_BWD = ["exact_attention_forward_14_b300/csrc/attn_bwd_kernel.cuh",
                      "exact_attention_forward_14_b300/csrc/ptx.cuh",
                      "exact_attention_forward_14_b300/csrc/attn_api.cu"]
KERNEL_SOURCES_D256 = ["exact_attention_forward_14_b300/csrc/attn_fwd_d256.cuh",
                       "exact_attention_forward_14_b300/csrc/attn_fwd_kernel.cuh",
                       "exact_attention_forward_14_b300/csrc/ptx.cuh"]
PROFILES = os.path.join(ROOT, "profiles")


def kernel_source_hash(sources=KERNEL_SOURCES) -> str:
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def ncu_traffic(workload: str, sources=KERNEL_SOURCES):
    """DRAM bytes per launch (per call, for the backward's three kernels) from
    the JSON block of a committed ncu summary (profiles/*.md), only while the
    kernel sources still match the capture."""
    import glob
    import re
    want = kernel_source_hash(sources)
    for path in sorted(glob.glob(os.path.join(PROFILES, "*.md"))):
        with open(path) as f:
            text = f.read()
        for block in re.findall(r"```json\n(.*?)```", text, flags=re.S):
            try:
                entry = json.loads(block)
            except ValueError:
                continue
            if entry.get("workload") == workload and entry.get("kernel_hash") == want:
                return entry.get("dram_bytes_per_launch")
    return None


class ClockSampler:
    """Samples SM clock, power and throttle reasons with ``nvidia-smi -lms``
    in a background reader while the timed region runs. Only samples that
    arrive between enter() and exit() are kept."""

    QUERY = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    FLAGS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int, period_ms: int = 20):
        self.period_ms = period_ms
        self.rows = []
        self.error = None
        self._proc = None
        self._thread = None
        self._active = False
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.index = device_index
        if vis and vis.split(",")[device_index].strip().isdigit():
            self.index = int(vis.split(",")[device_index])

    def _reader(self):
        for line in self._proc.stdout:
            if self._active:
                self.rows.append(line.strip())

    def start(self):
        """Starts nvidia-smi and returns once its first line has arrived."""
        import subprocess
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 f"-lms={self.period_ms}", f"-i={self.index}"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self._proc.stdout.readline()
            if not first:
                raise RuntimeError("nvidia-smi printed nothing")
        except Exception as e:
            self.error = f"{type(e).__name__}: {e}"
            self._proc = None
            return self
        self._thread = threading.Thread(target=self._reader, daemon=True)
        self._thread.start()
        return self

    def __enter__(self):
        self._active = True
        return self

    def __exit__(self, *exc):
        self._active = False
        if self._proc is not None:
            self._proc.terminate()
            self._proc.wait()
            self._thread.join(timeout=2)

    def summary(self):
        mhz, maxes, watts, reasons = [], [], [], set()
        for r in self.rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 8:
                continue
            try:
                mhz.append(float(f[0]))
                maxes.append(float(f[1]))
                watts.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(self.FLAGS, f[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(mhz) if mhz else None,
               "sm_max_mhz": max(maxes) if maxes else None,
               "power_w_max": max(watts) if watts else None,
               "reasons": sorted(reasons), "samples": len(mhz),
               "source": f"nvidia-smi -lms {self.period_ms}"}
        if self.error:
            out["error"] = self.error
        if getattr(self, "nvml_error", None):
            out["nvml_error"] = self.nvml_error
        return out


class NvmlClockSampler:
    """Samples the SM clock, power and clock-event reasons through NVML (the
    driver's libnvidia-ml, called with ctypes) from a background thread every
    ~1 ms while the timed region runs, so even a region of a few milliseconds
    gets samples (nvidia-smi's loop cannot go much below 20 ms). Same
    interface as ClockSampler, which is the fallback when NVML cannot be
    loaded."""

    NVML_CLOCK_SM = 1
    # clock-event reason bits (nvml.h)
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device_index: int, period_s: float = 0.001):
        self.period_s = period_s
        self.index = ClockSampler(device_index).index
        self.rows = []  # (sm_mhz, max_mhz, watts, reasons bitmask)
        self.error = None
        self.ok = False
        self._thread = None
        self._stop = threading.Event()
        self._active = False

    def start(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)):
                raise RuntimeError("nvmlDeviceGetHandleByIndex_v2 failed")
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)):
                raise RuntimeError("nvmlDeviceGetMaxClockInfo failed")
            self._lib, self._h, self._max = lib, h, float(mx.value)
            self._reasons = (getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                             or lib.nvmlDeviceGetCurrentClocksThrottleReasons)
        except Exception as e:  # no NVML: the caller falls back to nvidia-smi
            self.error = f"{type(e).__name__}: {e}"
            return self
        self.ok = True
        self._thread = threading.Thread(target=self._loop, daemon=True)
        self._thread.start()
        return self

    def _loop(self):
        import ctypes
        clk, mw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self._active:
                if (self._lib.nvmlDeviceGetClockInfo(self._h, self.NVML_CLOCK_SM, ctypes.byref(clk))
                        == 0 and self._lib.nvmlDeviceGetPowerUsage(self._h, ctypes.byref(mw)) == 0
                        and self._reasons(self._h, ctypes.byref(rs)) == 0):
                    self.rows.append((float(clk.value), self._max, mw.value / 1000.0, rs.value))
            time.sleep(self.period_s)

    def __enter__(self):
        self._active = True
        return self

    def __exit__(self, *exc):
        self._active = False
        self._stop.set()
        if self._thread is not None:
            self._thread.join(timeout=2)

    def summary(self):
        reasons = sorted({name for *_, r in self.rows for name, b in self.REASONS.items()
                          if r & b})
        mhz = [r[0] for r in self.rows]
        out = {"sm_mhz": statistics.median(mhz) if mhz else None,
               "sm_max_mhz": max(r[1] for r in self.rows) if mhz else None,
               "power_w_max": max(r[2] for r in self.rows) if mhz else None,
               "reasons": reasons, "samples": len(mhz),
               "source": f"NVML (libnvidia-ml), every {self.period_s * 1e3:g} ms"}
        if self.error:
            out["error"] = self.error
        return out


def clock_sampler(device_index: int):
    """NVML sampler when NVML answers, else the nvidia-smi one (whose summary
    then names NVML's error)."""
    s = NvmlClockSampler(device_index).start()
    if s.ok:
        return s
    fallback = ClockSampler(device_index).start()
    fallback.nvml_error = s.error
    return fallback


# ------------------------------------------------------------ CPU oracle --

def _oracle_inputs(w):
    """The workload's inputs in the oracle's form (drawn once): bf16 bits, or
    for the FP8 workload E4M3 codes and block scales from the oracle's own
    quantiser."""
    os.environ.setdefault("OMP_NUM_THREADS", str(len(os.sched_getaffinity(0))))
    import oracle
    from exact_attention_forward_14_b300 import inputs
    if w.dtype == "e4m3":
        qc, kc, vc = (oracle.quantize_fp8_e4m3(t.numpy()) for t in inputs.draw_workload_f32(w))
        return {"dtype": "e4m3", "q": qc[0], "k": kc[0], "v": vc[0],
                "q_scale": qc[1], "k_scale": kc[1], "v_scale": vc[1]}
    q, k, v = inputs.draw_workload_16(w)
    bits = {"dtype": w.dtype, "q": inputs.bits16(q), "k": inputs.bits16(k),
            "v": inputs.bits16(v)}
    if w.backward:
        bits["do"] = inputs.bits16(inputs.draw_grad_out(w.B, w.Sq, w.Hq, w.d, w.seed, w.dtype))
    return bits


def _oracle_sample(w, bits, target_s: float, seed: int, n_fixed: int | None = None):
    """Times the oracle on a row sample of workload w: n_fixed random rows, or
    a sample grown until it takes ~target_s of CPU work.
    Returns (flops_of_sample, seconds, n_rows, threads)."""
    import numpy as np
    import oracle

    def rows_flops(rows):
        i = rows % w.Sq
        if w.causal:
            vis = np.clip(i + (w.Sk - w.Sq) + 1, 0, w.Sk)
        else:
            vis = np.full(rows.shape, w.Sk)
        return float(4.0 * w.d * vis.sum()) * (2.5 if w.backward else 1.0)

    rng = np.random.default_rng(seed)
    total = w.B * w.Hq * w.Sq
    n = n_fixed or 64
    while True:
        rows = np.sort(rng.choice(total, size=min(n, total), replace=False)).astype(np.int64)
        t0 = time.perf_counter()
        if w.backward:  # dQ of the sampled rows (each recomputes its O and LSE)
            oracle.attn_bwd_sampled(bits["q"], bits["k"], bits["v"], bits["do"], w.causal,
                                    w.scale, rows, np.zeros(0, np.int64), dtype=bits["dtype"])
        else:
            oracle.attn_fwd(bits["q"], bits["k"], bits["v"], w.causal, w.scale,
                            dtype=bits["dtype"], q_scale=bits.get("q_scale"),
                            k_scale=bits.get("k_scale"), v_scale=bits.get("v_scale"), rows=rows)
        dt = time.perf_counter() - t0
        if n_fixed or dt >= target_s or n >= total:
            return rows_flops(rows), dt, rows.size, int(os.environ["OMP_NUM_THREADS"])
        n = int(min(total, max(2 * n, n * target_s / max(dt, 1e-3) * 1.05)))


def cpu_model() -> str:
    """The host CPU's model name (Linux), or the platform's processor string."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.processor() or "unknown"


def cpu_baseline(w, target_s: float = 12.0):
    flops, dt, n, threads = _oracle_sample(w, _oracle_inputs(w), target_s, seed=1)
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "cpu": cpu_model(),
            "sample": f"{n} random query rows of all (b, h) of the workload "
                      f"({flops / 1e9:.1f} GFLOP by the metric's count) in {dt:.1f} s, "
                      + ("fp64 oracle dQ rows (O, LSE recomputed per row), OpenMP"
                         if w.backward else "fp64 two-pass oracle, OpenMP")}


def count_ranks(backend: str = "gloo") -> int:
    """Number of ranks that joined this job (1 without torch.distributed):
    every rank adds 1 in an all-reduce. Leaves no process group behind."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world == 1:
        return 1
    import torch
    import torch.distributed as dist
    dist.init_process_group(backend)
    t = torch.ones(1, dtype=torch.int64)
    dist.all_reduce(t)
    dist.destroy_process_group()
    return int(t.item())


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    ranks = count_ranks()  # every rank joins, so n_gpus counts the ranks that ran
    if rank != 0:
        return 0
    per_step = max(0.05, args.ref_seconds / (args.steps + args.warmup))
    bits = _oracle_inputs(w)
    _, _, n_step, _ = _oracle_sample(w, bits, per_step, seed=99)  # calibrate the step size
    flops_t = []
    for s in range(args.warmup + args.steps):
        flops, dt, n, threads = _oracle_sample(w, bits, per_step, seed=100 + s, n_fixed=n_step)
        if s >= args.warmup:
            flops_t.append((flops, dt, n))
    tot_f = sum(f for f, _, _ in flops_t)
    tot_t = sum(t for _, t, _ in flops_t)
    value = tot_f / tot_t / 1e12
    line = {
        "impl": "reference", "metric": metric_of(w), "value": value, "unit": "TFLOP/s",
        "n_gpus": ranks, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot_t / len(flops_t), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "cpu": cpu_model(),
                         "sample": f"each step: ~{flops_t[0][2]} random query rows of the "
                                   "workload through the fp64 oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------ L2 residency --

L2_BYTES = 126 * 2 ** 20  # B300 L2 (nominal); the device's own figure is used when larger


def step_bytes(w):
    """(input, output) bytes of one step as the path reads and writes them
    once: Q, K, V (and the FP8 block scales; for the backward also O, LSE and
    dO; for the RMSNorm prologue its weights) in, O and LSE (dQ, dK, dV for the
    backward) out."""
    esz = 1 if w.dtype == "e4m3" else 2
    nq, nkv = w.B * w.Sq * w.Hq * w.d, w.B * w.Sk * w.Hkv * w.d
    lse = 4 * w.B * w.Hq * w.Sq
    inb = esz * (nq + 2 * nkv)
    if w.dtype == "e4m3":
        inb += 4 * (w.B * w.Hq * -(-w.Sq // 64) + 2 * w.B * w.Hkv * -(-w.Sk // 64))
    if w.qknorm:
        inb += 2 * (w.Hq + w.Hkv) * w.d
    if w.backward:
        return inb + 2 * 2 * nq + lse, 2 * (nq + 2 * nkv)
    return inb, 2 * nq + lse


def l2_flush_bytes(w, l2_bytes: int = L2_BYTES) -> int:
    """Bytes to write between timed steps: none when one step's inputs alone
    are larger than the L2 (every step then streams them from HBM), else a
    buffer of twice the L2, which leaves none of them resident."""
    return 0 if step_bytes(w)[0] > l2_bytes else 2 * l2_bytes


def l2_label(w) -> str:
    if not l2_flush_bytes(w):
        return "inputs larger than L2 (no flush)"
    return (f"inputs ({step_bytes(w)[0] / 1e6:.3f} MB) fit in L2: a buffer of twice the L2 is "
            "written before every timed step, outside its CUDA events; value and ms_per_step "
            "are the sum of the per-step events (L2-cold); l2_warm gives back-to-back steps")


def workload_config(w, nsplit=None):
    c = {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Sq": w.Sq, "Sk": w.Sk,
         "d": w.d, "causal": w.causal, "dtype": w.dtype, "l2": l2_label(w)}
    if nsplit:
        c["splitkv_ranges"] = nsplit
    return c


# ------------------------------------------------------ rank arithmetic --

def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The slowest rank's figure (every rank gets it); x itself with one rank."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(flops_per_step: float, steps: int, world: int, total_ms: float) -> float:
    """Whole-job throughput: every rank ran `steps` steps of `flops_per_step`
    in (at most) total_ms."""
    return world * flops_per_step * steps / (total_ms * 1e-3) / 1e12


# ------------------------------------------------------ MUFU microbench --

def mufu_ex2_rate(w, num_sms: int, sm_mhz: float):
    """ex2.approx throughput per SM per clock from the self-test library's
    microbenchmark (one CTA per SM), and the TFLOP/s ceiling it would set on
    its own: every score element needs one exp2 and 4 d tensor FLOPs."""
    import ctypes
    import statistics as st
    import torch
    path = os.path.join(ROOT, "exact_attention_forward_14_b300", "libattn_selftest.so")
    lib = ctypes.CDLL(path)
    lib.attn_selftest_ex2_rate.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                           ctypes.c_void_p, ctypes.c_void_p]
    lib.attn_selftest_ex2_rate.restype = ctypes.c_int
    iters = 2048
    cyc = torch.zeros(num_sms, dtype=torch.int64, device="cuda")
    sink = torch.zeros(1024, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream or None
    for _ in range(2):  # the first launch warms the clocks and the instruction cache
        rc = lib.attn_selftest_ex2_rate(iters, num_sms, cyc.data_ptr(), sink.data_ptr(), stream)
        if rc != 0:
            return None
    rates = [1024 * 8 * iters / c for c in cyc.cpu().tolist() if c > 0]
    rate = st.median(rates)
    ceiling = None if not sm_mhz else rate * num_sms * sm_mhz * 1e6 * 4 * w.d / 1e12
    return {"ex2_per_clk_per_sm": rate, "implied_ceiling_tflops": ceiling,
            "at_sm_mhz": sm_mhz,
            "note": "one exp2 per score element against 4 d tensor FLOPs, at the SM clock "
                    "sampled in the timed region (null when no sample arrived); "
                    "microbenchmark in csrc/mufu_rate.cu"}


# ------------------------------------------------------------- GPU path --

def e2e_pipelined(args, host_in, bufs, step, dev, dist, world, flops):
    """The step end to end through the public call: each step's inputs are
    copied from pinned host memory to the device and its outputs back, as a
    caller streaming many problems would do it. Three streams and two buffer
    sets overlap step k's compute with the copies of steps k-1 and k+1, and
    the two copy directions with each other; every step still moves all of
    its own bytes. The timed region starts on an idle device (pipeline fill
    included) and ends when the last result has reached the host."""
    import torch
    sets = [bufs, {"in": tuple(torch.empty_like(t) for t in bufs["in"]),
                   "out": tuple(torch.empty_like(t) for t in bufs["out"])}]
    host_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in bufs["out"]]
                for _ in range(2)]
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    e_steps = max(3, min(args.steps, 20))
    n = e_steps + 2
    ev_in = [torch.cuda.Event() for _ in range(n)]
    ev_cmp = [torch.cuda.Event() for _ in range(n)]
    ev_out = [torch.cuda.Event() for _ in range(n)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(n):
        b = k % 2
        if k == 2:  # two untimed steps, then start from an idle device
            torch.cuda.synchronize(dev)
            if dist is not None:
                dist.barrier()
            e0.record(s_in)
        if k >= 2:
            s_in.wait_event(ev_cmp[k - 2])  # step k-2 has finished reading set b
        with torch.cuda.stream(s_in):
            for dst, src in zip(sets[b]["in"], host_in):
                dst.copy_(src, non_blocking=True)
        ev_in[k].record(s_in)
        s_cmp.wait_event(ev_in[k])
        if k >= 2:
            s_cmp.wait_event(ev_out[k - 2])  # set b's outputs of step k-2 are on the host
        step(sets[b], s_cmp.cuda_stream)
        ev_cmp[k].record(s_cmp)
        s_out.wait_event(ev_cmp[k])
        with torch.cuda.stream(s_out):
            for dst, src in zip(host_out[b], sets[b]["out"]):
                dst.copy_(src, non_blocking=True)
        ev_out[k].record(s_out)
    e1.record(s_out)
    torch.cuda.synchronize(dev)
    e_ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    return {"value": job_tflops(flops, e_steps, world, e_ms), "unit": "TFLOP/s",
            "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in host_in),
            "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in bufs["out"]),
            "ms_per_step": e_ms / e_steps,
            "pipelined": "3 streams, 2 buffer sets: copies overlap neighbouring steps' compute"}


def quant_rate(reps: int = 20):
    """Rate of the FP8 block quantiser (attn_quantize_fp8_e4m3, outside the
    attention's timed region) on one operand of the FP8 workload: fp32
    [4, 4096, 16, 128] -> E4M3 codes + per-block scales. Each call is timed
    alone with CUDA events after a write of twice the L2 (L2-cold); prints one
    JSON line with the median and the HBM rate its bytes imply, against the
    measured copy bandwidth."""
    import torch
    import exact_attention_forward_14_b300 as ea
    from exact_attention_forward_14_b300 import inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = inputs.WORKLOADS["fp8_b4h16s4096d128"]
    x = inputs.draw_workload_f32(w)[0].to(dev)
    for _ in range(5):
        ea.quantize_fp8(x)
    torch.cuda.synchronize(dev)
    flush = torch.empty(2 * 126 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    times = []
    clocks = clock_sampler(0)
    with clocks:
        for r in range(reps):
            flush.fill_(float(r))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            codes, scales = ea.quantize_fp8(x)
            e1.record()
            torch.cuda.synchronize(dev)
            times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    nbytes = x.numel() * 4 + codes.numel() + scales.numel() * 4
    peaks, src = load_peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9
    print(json.dumps({"kernel": "quantize_fp8_kernel", "shape": list(x.shape), "us_median": ms * 1e3,
                      "bytes": nbytes, "hbm_gbs": gbs, "peak_gbs": peaks["hbm_gbs"], "peak_source": src,
                      "frac": gbs / peaks["hbm_gbs"], "l2": "a buffer of twice the L2 written before each call",
                      "clocks": clocks.summary()}), flush=True)
    return 0


def gemm_peaks(n: int = 8192, reps: int = 40):
    """Library GEMM rates on this GPU at n x n x n, as context for the FP8
    roofline: cuBLASLt E4M3 x E4M3 -> bf16 (torch._scaled_mm, unit tensor
    scales, with and without fast accumulation) beside a cuBLAS bf16 matmul.
    Inputs are N(0,1) draws; each figure is the mean of `reps` back-to-back
    calls after 5 warm-ups, timed with CUDA events. Prints one JSON line."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(7)
    a16 = torch.randn(n, n, device=dev, generator=g).to(torch.bfloat16)
    b16 = torch.randn(n, n, device=dev, generator=g).to(torch.bfloat16)
    a8 = a16.to(torch.float8_e4m3fn)
    b8 = b16.to(torch.float8_e4m3fn).t()  # column-major second operand
    one = torch.ones((), device=dev, dtype=torch.float32)
    calls = {
        "bf16": lambda: torch.matmul(a16, b16),
        "fp8": lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one,
                                        out_dtype=torch.bfloat16),
        "fp8_fast_accum": lambda: torch._scaled_mm(a8, b8, scale_a=one, scale_b=one,
                                                   out_dtype=torch.bfloat16,
                                                   use_fast_accum=True),
    }
    out = {"n": n, "reps": reps}
    clocks = clock_sampler(0)
    with clocks:
        for name, f in calls.items():
            for _ in range(5):
                f()
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(reps):
                f()
            e1.record()
            torch.cuda.synchronize(dev)
            out[f"{name}_tflops"] = 2.0 * n ** 3 / (e0.elapsed_time(e1) / reps * 1e-3) / 1e12
    out["fp8_over_bf16"] = max(out["fp8_tflops"], out["fp8_fast_accum_tflops"]) / out["bf16_tflops"]
    out["clocks"] = clocks.summary()
    print(json.dumps(out), flush=True)
    return 0


def run_ours(args, w):
    import torch
    import exact_attention_forward_14_b300 as ea
    from exact_attention_forward_14_b300 import inputs

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but {world} rank(s) were launched")
    if local >= torch.cuda.device_count():
        raise SystemExit(f"rank {rank}: local rank {local} but only "
                         f"{torch.cuda.device_count()} visible GPU(s)")
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    # inputs: seeded CPU draw, then resident on the device
    if w.dtype == "e4m3":
        qf, kf, vf = inputs.draw_workload_f32(w)
        q8, qs = ea.quantize_fp8(qf.to(dev))
        k8, ks = ea.quantize_fp8(kf.to(dev))
        v8, vs = ea.quantize_fp8(vf.to(dev))
        dev_in = (q8, k8, v8, qs, ks, vs)
        del qf, kf, vf
        # what a caller of the FP8 entry point holds: codes and block scales
        host = tuple(t.cpu().pin_memory() for t in dev_in)
    else:
        hq, hk, hv = inputs.draw_workload_16(w)
        host = tuple(t.pin_memory() for t in (hq, hk, hv))
        dev_in = tuple(t.to(dev) for t in host)
    o = torch.empty((w.B, w.Sq, w.Hq, w.d),
                    dtype=torch.float16 if w.dtype == "f16" else torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Hq, w.Sq), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    ws, nsplit = None, 0
    if w.splits:
        nsplit = w.splits
        rc, planned, wbytes = ea.attn_splitkv_plan(w.B, w.Hq, w.Sq, w.Sk, w.d, w.causal)
        if rc != ea.ATTN_OK:
            raise ea.AttnError(rc, "attn_splitkv_plan")
        if nsplit < 0:
            nsplit = planned
        wbytes = nsplit * w.B * w.Hq * w.Sq * (w.d + 1) * 4
        ws = torch.empty(wbytes // 4, dtype=torch.float32, device=dev)

    bwd = None
    if w.backward:
        # the backward pass's inputs: q, k, v, the forward's O and LSE on
        # them, and dO (all resident); outputs dQ, dK, dV
        code = ea.ATTN_F16 if w.dtype == "f16" else ea.ATTN_BF16
        h_do = inputs.draw_grad_out(w.B, w.Sq, w.Hq, w.d, w.seed, w.dtype).pin_memory()
        d_o = h_do.to(dev)
        q, k, v = dev_in
        rc = ea.attn_fwd(q, k, v, o, lse, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.causal, w.scale,
                         code, stream)
        if rc != ea.ATTN_OK:
            raise ea.AttnError(rc, "attn_fwd")
        rc, wbytes = ea.attn_bwd_workspace_size(w.B, w.Hq, w.Sq)
        if rc != ea.ATTN_OK:
            raise ea.AttnError(rc, "attn_bwd_workspace_size")
        bwd = {"code": code, "do": d_o, "h_do": h_do,
               "grads": (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)),
               "ws": torch.empty(wbytes // 4, dtype=torch.float32, device=dev)}

    norm = None
    if w.qknorm:
        wq = inputs.draw_norm_weights(w.Hq * w.d, w.seed + 50, w.dtype).to(dev)
        wk = inputs.draw_norm_weights(w.Hkv * w.d, w.seed + 51, w.dtype).to(dev)
        norm = (wq, wk, torch.empty_like(dev_in[0]), torch.empty_like(dev_in[1]))

    code16 = ea.ATTN_F16 if w.dtype == "f16" else ea.ATTN_BF16
    # one step's device buffers: its inputs (copied in by the e2e leg) and its outputs
    if bwd is not None:
        default_bufs = {"in": tuple(dev_in) + (o, lse, bwd["do"]), "out": bwd["grads"]}
    else:
        default_bufs = {"in": tuple(dev_in), "out": (o, lse)}

    def prologue(bufs=default_bufs, st=None):
        q, k = bufs["in"][0], bufs["in"][1]
        wq, wk, qn, kn = norm
        rc = ea.attn_qk_rmsnorm(q, k, wq, wk, qn, kn, w.B, w.Sq, w.Sk, w.Hq, w.Hkv, w.d, 1e-6,
                                code16, st if st is not None else stream)
        if rc != ea.ATTN_OK:
            raise ea.AttnError(rc, "attn_qk_rmsnorm")
        return qn, kn

    def step(bufs=default_bufs, st=None):
        st = st if st is not None else stream
        if bwd is not None:
            q, k, v, o_, lse_, d_o = bufs["in"]
            dq, dk, dv = bufs["out"]
            rc = ea.attn_bwd(q, k, v, o_, lse_, d_o, dq, dk, dv, w.B, w.Hq, w.Hkv, w.Sq,
                             w.Sk, w.d, w.causal, w.scale, bwd["code"], bwd["ws"],
                             bwd["ws"].numel() * 4, st)
            if rc != ea.ATTN_OK:
                raise ea.AttnError(rc, "attn_bwd")
            return
        o_, lse_ = bufs["out"]
        if norm is not None:
            qn, kn = prologue(bufs, st)
            rc = ea.attn_fwd(qn, kn, bufs["in"][2], o_, lse_, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d,
                             w.causal, w.scale, code16, st)
        elif ws is not None:
            q, k, v = bufs["in"]
            rc = ea.attn_fwd_splitkv(q, k, v, o_, lse_, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d,
                                     w.causal, w.scale, code16, nsplit, ws, ws.numel() * 4, st)
        elif w.dtype == "e4m3":
            q8, k8, v8, qs, ks, vs = bufs["in"]
            rc = ea.attn_fwd_fp8(q8, k8, v8, qs, ks, vs, o_, lse_, w.B, w.Hq, w.Hkv, w.Sq, w.Sk,
                                 w.d, w.causal, w.scale, st)
        else:
            q, k, v = bufs["in"]
            rc = ea.attn_fwd(q, k, v, o_, lse_, w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.d, w.causal,
                             w.scale, code16, st)
        if rc != ea.ATTN_OK:
            raise ea.AttnError(rc, "attn_fwd")

    # small workloads: evict the inputs from L2 before every timed step
    flush = None
    if l2_flush_bytes(w):
        l2_dev = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 0)
        flush = torch.empty(l2_flush_bytes(w, max(L2_BYTES, l2_dev)), dtype=torch.uint8,
                            device=dev)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    st = ea.attn_device_status(stream)
    if st != ea.ATTN_OK:
        raise ea.AttnError(st, "warm-up")

    # timed region: K back-to-back launches, an event pair around each
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    clocks = clock_sampler(local)
    with clocks:
        if args.profiler_range:
            torch.cuda.profiler.start()
        t0.record(stream)
        for i, (a, b) in enumerate(ev):
            if flush is not None:
                flush.fill_(i & 0xFF)
            a.record(stream)
            step()
            b.record(stream)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        if args.profiler_range:
            torch.cuda.profiler.stop()
    if dist is not None:
        dist.barrier()
    st = ea.attn_device_status(stream)
    if st != ea.ATTN_OK:
        raise ea.AttnError(st, "timed region")
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    # with the flush, the steps' own events; without it, the whole region
    total_ms = sum(launch_ms) if flush is not None else t0.elapsed_time(t1)
    total_ms = max_over_ranks(total_ms, dist, dev)
    ms_per_step = total_ms / args.steps
    flops = w.flops()
    value = job_tflops(flops, args.steps, world, total_ms)

    # the same steps back to back with the inputs left in L2
    l2_warm = None
    if flush is not None:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0.record(stream)
        for _ in range(args.steps):
            step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        st = ea.attn_device_status(stream)
        if st != ea.ATTN_OK:
            raise ea.AttnError(st, "L2-warm steps")
        warm_ms = max_over_ranks(t0.elapsed_time(t1), dist, dev)
        l2_warm = {"value": job_tflops(flops, args.steps, world, warm_ms), "unit": "TFLOP/s",
                   "ms_per_step": warm_ms / args.steps}
        del flush

    # end to end through the public API: every step copies its inputs from
    # pinned host memory and reads its results back (see e2e_pipelined)
    e2e = None
    if host is not None:
        host_in = list(host)
        if bwd is not None:
            host_in += [o.cpu().pin_memory(), lse.cpu().pin_memory(), bwd["h_do"]]
        e2e = e2e_pipelined(args, host_in, default_bufs, step, dev, dist, world, flops)

    prologue_line = None
    if norm is not None:
        # the RMSNorm kernel on its own (HBM-bound): algorithmic bytes = Q and K
        # read and written once, plus the weights
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 50
        prologue()
        torch.cuda.synchronize(dev)
        p0.record(stream)
        for _ in range(reps):
            prologue()
        p1.record(stream)
        torch.cuda.synchronize(dev)
        pms = p0.elapsed_time(p1) / reps
        nbytes = 2 * 2 * (w.B * w.Sq * w.Hq * w.d + w.B * w.Sk * w.Hkv * w.d) + \
            2 * (w.Hq + w.Hkv) * w.d
        peaks_p, src_p = load_peaks()
        gbs = nbytes / (pms * 1e-3) / 1e9
        prologue_line = {"kernel": "qk_rmsnorm_kernel", "ms": pms, "bound": "hbm",
                         "achieved": gbs, "peak": peaks_p["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks_p["hbm_gbs"], "bytes": nbytes,
                         "peak_source": f"{src_p} hbm copy"}

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peaks, peaks_src = load_peaks()
    mean_launch_ms = statistics.mean(launch_ms)
    # the backward pass runs 7 matrix products per visible (query, key) pair
    # (dK/dV kernel 4, dQ kernel 3) against the metric's 5
    executed = flops * (7.0 / 5.0 if bwd is not None else 1.0)
    achieved = executed / (mean_launch_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"] * (2.0 if w.dtype == "e4m3" else 1.0)
    roofline = {
        "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
        "frac": achieved / peak,
        "traffic": ncu_traffic(w.name, KERNEL_SOURCES_BWD if bwd is not None else
                               KERNEL_SOURCES_D256 if w.d == 256 else KERNEL_SOURCES),
        "kernel": (f"attn_bwd (bwd_prep_kernel + bwd_dkdv_kernel + bwd_dq_kernel)<{w.d},"
                   f"{str(w.dtype == 'f16').lower()}>, executed FLOPs (7 products per pair)"
                   if bwd is not None else
                   f"attn_fwd_d256_kernel<{str(w.dtype == 'f16').lower()}>" if w.d == 256 else
                   f"attn_fwd_kernel<{w.d},{str(w.dtype == 'e4m3').lower()},"
                   f"{str(w.dtype == 'f16').lower()}>"),
        "peak_source": (f"{peaks_src} bf16 burst" if w.dtype != "e4m3"
                        else f"{peaks_src} bf16 burst x 2 (nominal fp8/bf16 ratio)"),
        "frac_of_sustained": achieved / (peaks.get("bf16_tflops_sustained", peak) *
                                         (2.0 if w.dtype == "e4m3" else 1.0)),
        "launch_ms_median": statistics.median(launch_ms),
    }
    line = {
        "metric": metric_of(w), "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": workload_config(w, nsplit), "clocks": clocks.summary(), "e2e": e2e,
        "gpu_launches": args.steps * (3 if bwd is not None else
                                      2 if (ws is not None or norm is not None) else 1),
        "roofline": roofline,
    }
    if prologue_line is not None:
        line["prologue"] = prologue_line
    if l2_warm is not None:
        # small problems are latency-bound: the call's time and the HBM rate
        # its compulsory bytes imply
        in_b, out_b = step_bytes(w)
        med = statistics.median(launch_ms)
        line["l2_warm"] = l2_warm
        line["per_call"] = {"us_median": med * 1e3, "bytes": in_b + out_b,
                            "hbm_gbs": (in_b + out_b) / (med * 1e-3) / 1e9}
    if not w.backward:
        props = torch.cuda.get_device_properties(dev)
        # the ceiling uses the clock sampled in the timed region; none without samples
        line["mufu"] = mufu_ex2_rate(w, props.multi_processor_count, line["clocks"].get("sm_mhz"))
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def launch_ranks(n: int, argv) -> int:
    """Re-runs this script as n ranks on this node (one per GPU) through
    torch.distributed.run, rendezvous on 127.0.0.1; returns their exit code.
    Used when --gpus N > 1 is given outside a torchrun launch."""
    import socket
    import subprocess
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={n}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the CPU oracle timing (e.g. under a profiler)")
    ap.add_argument("--gemm-peaks", action="store_true",
                    help="only time library bf16 and FP8 GEMMs (8192^3) and exit")
    ap.add_argument("--quant-rate", action="store_true",
                    help="only time the FP8 block quantiser on one FP8-workload operand and exit")
    ap.add_argument("--profiler-range", action="store_true",
                    help="bracket the timed region with cudaProfilerStart/Stop, so that ncu "
                         "--replay-mode app-range measures it as a whole (kernels that run "
                         "side by side included); never for a bench value")
    ap.add_argument("--ref-seconds", type=float, default=150.0,
                    help="--impl reference: seconds of oracle work over all steps (bounded sample)")
    args = ap.parse_args(argv)
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # N replicas need N processes: start them here rather than run one
        return launch_ranks(args.gpus, sys.argv[1:] if argv is None else list(argv))
    if args.gemm_peaks:
        return gemm_peaks()
    if args.quant_rate:
        return quant_rate()
    from exact_attention_forward_14_b300 import inputs
    w = inputs.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
