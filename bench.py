"""Benchmark of the Mixtral sparse-MoE feed-forward layer on B300.

One "step" = one MoE layer call (router + top-2 gate, dispatch, W1/W3 grouped
GEMM with fused SwiGLU, W2 grouped GEMM with gate scaling, combine) on one
batch of synthetic Mixtral-shaped input (d=4096, d_ff=14336, 8 experts, top-2,
seeded random weights; no checkpoint).  The headline workload is prefill with
T=4096 tokens; the decode regime (T=32) is measured in the same run and
reported as microseconds per layer.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 launch under torch.distributed.run: every rank runs an independent
replica on its own GPU with its own batch (the layer is per-token independent:
data parallel over tokens, no collective on the data path); the barrier and
the max over ranks are for timing only.

--impl reference times the fp64 CPU oracle (the only other implementation of
the layer there is) on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (T=4096 prefill) & µs/layer decode T=32; % of BF16/HBM roofline"


# DRAM traffic of the dominant kernel (W1/W3 grouped GEMM) per launch at the
# prefill workload, from one ncu capture, kept with a hash of the sources that
# define the kernel: the figure is reported only while they are unchanged.
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_w13_prefill_t4096.json")
W13_SOURCES = [os.path.join(ROOT, "sparse_mixture_experts_54_b300", "csrc", f)
               for f in ("gemm_tc2.cu", "common.cuh", "combine_epi.cuh")]


def w13_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    for f in W13_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def w13_traffic():
    """(bytes per launch, note) from the committed capture, or (None, why)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no capture committed"
    with open(TRAFFIC_FILE) as f:
        t = json.load(f)
    if t.get("source_sha256") != w13_source_hash():
        return None, "kernel changed since the capture"
    return int(t["dram_bytes_per_launch"]), t.get("command", "")


# Headline windows up to this long are timed against the burst GEMM peak.
BURST_WINDOW_MS = 250.0


def peaks():
    p = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            m = json.load(f)
        p.update({k: float(m[k]) for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained") if k in m})
        p["source"] = "measured"
    return p


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus: int):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws > 1:
        import torch.distributed as dist
        rank = int(os.environ["RANK"])
        local = int(os.environ.get("LOCAL_RANK", rank))
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
        return rank, ws, dist
    if torch.cuda.is_available():
        torch.cuda.set_device(0)
    return 0, 1, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(v: float, dist) -> float:
    if dist is None:
        return v
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """Samples of SM clock, power and clock-event reasons while the bench runs.

    A thread reads them through the driver's NVML library every 5 ms (read-only
    queries, by ctypes), so that even a 20-call headline window of ~40 ms holds
    several; without it the sampler falls back to nvidia-smi every 200 ms.  Samples are timestamped when taken; summary()
    keeps those inside the timed windows marked with window()."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    PERIOD_S = 0.005

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.samples = []   # (time, sm MHz, max sm MHz, power W, set of reasons)
        self.windows = []
        self._stop = threading.Event()
        self._t = None

    @staticmethod
    def _nvml():
        """Read-only NVML queries through the driver's library (ctypes): a function
        returning (sm MHz, power W, clock-event reason bits) and the max SM MHz."""
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit")
        return lib

    def _nvml_handle(self, lib):
        h = ctypes.c_void_p()
        try:   # the device torch calls `index`, found by its PCI address
            prop = torch.cuda.get_device_properties(self.index)
            bus = f"{prop.pci_domain_id:08x}:{prop.pci_bus_id:02x}:{prop.pci_device_id:02x}.0".encode()
            if lib.nvmlDeviceGetHandleByPciBusId_v2(ctypes.c_char_p(bus), ctypes.byref(h)) == 0:
                return h
        except Exception:
            pass
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByIndex")
        return h

    def __enter__(self):
        try:
            lib = self._nvml()
            h = self._nvml_handle(lib)
            try:
                get_reasons = lib.nvmlDeviceGetCurrentClocksEventReasons
            except AttributeError:
                get_reasons = lib.nvmlDeviceGetCurrentClocksThrottleReasons
            # nvml.h clock-event reason bits
            bits = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                    "hw_thermal_slowdown": 0x40}
            NVML_CLOCK_SM = 1
            mx = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, NVML_CLOCK_SM, ctypes.byref(mx)) != 0:
                raise RuntimeError("nvmlDeviceGetMaxClockInfo")
            smax = float(mx.value)
            clk, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()

            def poll():
                while not self._stop.is_set():
                    if (lib.nvmlDeviceGetClockInfo(h, NVML_CLOCK_SM, ctypes.byref(clk)) == 0 and
                            lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 and
                            get_reasons(h, ctypes.byref(rs)) == 0):
                        r = rs.value
                        self.samples.append((time.monotonic(), float(clk.value), smax, pw.value / 1000.0,
                                             {k for k, b in bits.items() if r & b}))
                    self._stop.wait(self.PERIOD_S)

            self._t = threading.Thread(target=poll, daemon=True)
            self._t.start()
            return self
        except Exception:
            pass
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                reasons = {k for k, f in zip(self.REASONS, parts[4:8]) if f.lower() == "active"}
                self.samples.append((time.monotonic(), float(parts[0]), float(parts[1]), float(parts[2]), reasons))
            except ValueError:
                continue

    def wait_first(self, timeout_s: float = 5.0):
        t0 = time.monotonic()
        while self._t is not None and not self.samples and time.monotonic() - t0 < timeout_s:
            time.sleep(0.01)

    def window(self, t0: float, t1: float, name: str = "headline"):
        self.windows.append((name, t0, t1))

    def __exit__(self, *a):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self._t is not None and self.proc is None:
            self._t.join(timeout=1.0)

    def summary(self, which=("headline",)):
        """Clock record of the samples inside the named timed windows."""
        wins = [(a, b) for (n, a, b) in self.windows if n in which]
        inside = [smp for smp in list(self.samples) if any(a <= smp[0] <= b for a, b in wins)]
        timed_s = sum(b - a for a, b in wins)
        source = "nvml, every 5 ms" if self.proc is None else "nvidia-smi, every 200 ms"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "source": source,
                    "timed_seconds": round(timed_s, 3), "note": "no sample inside the timed region"}
        reasons = set().union(*(smp[4] for smp in inside))
        return {"sm_mhz": statistics.median(smp[1] for smp in inside), "sm_max_mhz": inside[-1][2],
                "reasons": sorted(reasons), "samples": len(inside),
                "power_w_median": statistics.median(smp[3] for smp in inside), "source": source,
                "timed_seconds": round(timed_s, 3)}


# ----------------------------------------------------------------------------- workloads
def algorithmic(T: int, counts, d=4096, F=14336, n=8, k=2):
    """FLOPs and bytes of one layer call that the method itself requires."""
    flops_router = 2.0 * T * d * n
    flops_w13 = 4.0 * k * T * d * F
    flops_w2 = 2.0 * k * T * d * F
    touched = sum(1 for c in counts if c > 0)
    w_bytes = touched * 3.0 * d * F * 2
    act_bytes = 2.0 * T * d * 2 + n * d * 4
    return dict(flops=flops_router + flops_w13 + flops_w2, flops_w13=flops_w13, flops_w2=flops_w2,
                bytes=w_bytes + act_bytes, weight_bytes=w_bytes, touched=touched)


class L2Flush:
    """Writes a buffer twice the size of L2 (126 MB) so that the next call reads its
    weights from HBM, then reads a second one of the same size: the written lines
    are dirty, and without the read their write-back to HBM would fall inside the
    next timed call (up to 126 MB, ~20 us of the copy bandwidth)."""

    def __init__(self, nbytes: int = 256 << 20):
        self.buf = torch.empty(nbytes // 4, dtype=torch.int32, device="cuda")
        self.clean = torch.ones(nbytes // 4, dtype=torch.int32, device="cuda")
        self.sink = torch.empty((), dtype=torch.int64, device="cuda")

    def __call__(self):
        self.buf.fill_(1)
        torch.sum(self.clean, dim=0, dtype=torch.int64, out=self.sink)


def timed_per_call(fn, steps: int, stream, flush=None):
    """Mean ms of fn() over `steps` calls, each bracketed by its own CUDA events on
    the stream; with `flush`, L2 is overwritten before each call (outside the
    events)."""
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        if flush is not None:
            flush()
        e0.record(stream)
        fn()
        e1.record(stream)
    torch.cuda.synchronize()
    return statistics.fmean(e0.elapsed_time(e1) for e0, e1 in ev)


def run_ours(args, rank, world, dist):
    from sparse_mixture_experts_54_b300 import _lib, inputs
    from sparse_mixture_experts_54_b300.layer import MoELayer

    pk = peaks()
    wp = inputs.workload("prefill_t4096")
    wd = inputs.workload("decode_t32")
    # every rank draws its own batch (data parallel over tokens); experts are the same model
    W1, W3, W2 = inputs.make_experts(wp, "cuda")
    xp = inputs.make_x(wp, "cuda", seed=rank)
    xd = inputs.make_x(wd, "cuda", seed=rank)
    Wg, _ = inputs.make_router(wp, "cuda")
    m = MoELayer(wp.d, wp.d_ff, wp.n_experts, wp.k)
    m.reserve(wp.T)
    stream = torch.cuda.current_stream()
    flush = L2Flush()
    yp = torch.empty((wp.T, wp.d), dtype=torch.bfloat16, device="cuda")
    yd = torch.empty((wd.T, wd.d), dtype=torch.bfloat16, device="cuda")

    def timed(x, y, steps, warmup, stage_timing, clk=None, window=None):
        """Mean ms per call over `steps` back-to-back calls (CUDA events on the stream).

        With stage_timing the library also records events around each kernel;
        those calls give the per-kernel breakdown."""
        for _ in range(warmup):
            m.forward(x, Wg, W1, W3, W2, y=y)
        torch.cuda.synchronize()
        m.set_option(_lib.MOE_OPT_STAGE_TIMING, 1 if stage_timing else 0)
        m.stage_times()   # drop warm-up records
        barrier(dist)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.monotonic()
        e0.record(stream)
        for _ in range(steps):
            m.forward(x, Wg, W1, W3, W2, y=y)
        e1.record(stream)
        torch.cuda.synchronize()
        if clk is not None:
            clk.window(t0, time.monotonic(), window)
        barrier(dist)
        ms = e0.elapsed_time(e1) / steps
        stages, calls = m.stage_times()
        m.set_option(_lib.MOE_OPT_STAGE_TIMING, 0)
        assert m.status() == 0, _lib.moe_error_string(m.status())
        return max_over_ranks(ms, dist), stages

    def timed_decode(steps, stage_timing, clk=None, window=None):
        """Decode calls, L2 flushed before each one, CUDA events around each call."""
        for _ in range(args.warmup):
            m.forward(xd, Wg, W1, W3, W2, y=yd)
        torch.cuda.synchronize()
        m.set_option(_lib.MOE_OPT_STAGE_TIMING, 1 if stage_timing else 0)
        m.stage_times()
        barrier(dist)
        t0 = time.monotonic()
        ms = timed_per_call(lambda: m.forward(xd, Wg, W1, W3, W2, y=yd), steps, stream, flush)
        if clk is not None:
            clk.window(t0, time.monotonic(), window)
        barrier(dist)
        stages, _ = m.stage_times()
        m.set_option(_lib.MOE_OPT_STAGE_TIMING, 0)
        assert m.status() == 0, _lib.moe_error_string(m.status())
        return max_over_ranks(ms, dist), stages

    # routing statistics of the batches (for the algorithmic byte count)
    r = m.route(xp, Wg)
    counts_p = r["counts"].cpu().tolist()
    idx_p = r["topk_idx"].cpu()
    r = m.route(xd, Wg)
    counts_d = r["counts"].cpu().tolist()

    with ClockSampler(torch.cuda.current_device()) as clk:
        clk.wait_first()
        # headline: K uninstrumented back-to-back calls after W warm-ups
        ms_p, _ = timed(xp, yp, args.steps, args.warmup, False, clk, "headline")
        # the same K calls again with per-kernel events: the kernels' shares of a call
        ms_pi, stages_p = timed(xp, yp, args.steps, 0, True, clk, "prefill_stages")
        ms_d, _ = timed_decode(args.decode_steps, False, clk, "decode")
        ms_di, stages_d = timed_decode(max(args.decode_steps // 4, 3), True, clk, "decode_stages")
        # sustained: a pre-roll into the power-capped steady state, then >= 2 s timed
        sus = None
        if args.sustained_s > 0:
            n_sus = max(int(args.sustained_s / (ms_p * 1e-3)), args.steps)
            n_pre = max(int(1.0 / (ms_p * 1e-3)), 1)
            ms_s, _ = timed(xp, yp, n_sus, n_pre, False, clk, "sustained")
            ms_si, stages_s = timed(xp, yp, max(n_sus // 3, args.steps), 0, True, clk, "sustained_stages")
            sus = dict(ms=ms_s, calls=n_sus, ms_i=ms_si, stages=stages_s)
    clocks = clk.summary(("headline",))

    # skewed, locally correlated routing at 32k context (router bias, repeated rows)
    skew = run_skewed(args, W1, W3, W2, pk, dist) if not args.no_skewed else None

    # end to end: pinned host x in, host y out, through the host-buffer entry point
    xh = xp.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    for _ in range(args.warmup):
        m.forward_host(xh, Wg, W1, W3, W2, yh)
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        m.forward_host(xh, Wg, W1, W3, W2, yh)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist)

    # decode with fp8 (e4m3) expert weights, power-of-two row scales
    fp8 = run_fp8_decode(args, m, W1, W3, W2, Wg, pk, dist, flush) if not args.no_fp8 else None

    alg_p = algorithmic(wp.T, counts_p)
    alg_d = algorithmic(wd.T, counts_d)
    tok_s = world * wp.T / (ms_p * 1e-3)
    # dominant kernel: the W1/W3 grouped GEMM (2/3 of the FLOPs).  Its duration in
    # the headline run = the headline's ms per call x its share of a call in the
    # per-kernel events of the same calls repeated right after.
    k13 = "expert_w1w3_swiglu"
    share = stages_p[k13] / sum(stages_p.values())
    k13_ms = ms_p * share
    achieved = alg_p["flops_w13"] / (k13_ms * 1e-3) / 1e12
    traffic, traffic_note = w13_traffic()
    # The peak that fits the window: the burst GEMM rate for a window of a few tens
    # of calls (clocks near their maximum), the sustained one for a window long
    # enough to reach the power-capped steady state.
    window_ms = ms_p * args.steps
    kind = "burst" if window_ms <= BURST_WINDOW_MS else "sustained"
    peak = pk["bf16_tflops"] if kind == "burst" else pk["bf16_tflops_sustained"]
    roofline = {"kernel": "expert_w1w3_swiglu (tcgen05 grouped GEMM + SwiGLU on CTA pairs)", "bound": "tensor",
                "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                "frac": round(achieved / peak, 4),
                "peak_kind": f"bf16 {kind} ({pk['source']}): the headline window is {args.steps} calls, "
                             f"{window_ms:.0f} ms ({'at most' if kind == 'burst' else 'over'} "
                             f"{BURST_WINDOW_MS:.0f} ms)",
                "frac_of_burst": round(achieved / pk["bf16_tflops"], 4),
                "frac_of_sustained": round(achieved / pk["bf16_tflops_sustained"], 4),
                "frac_of_nominal_2250": round(achieved / 2250.0, 4),
                "flops_per_launch": alg_p["flops_w13"],
                "duration_us": round(k13_ms * 1e3, 1),
                "duration_source": "headline ms_per_step x the kernel's share of the per-kernel CUDA-event times "
                                   "of the same calls repeated right after",
                "share": round(share, 4), "instrumented_us": round(stages_p[k13] * 1e3, 1),
                "traffic": traffic, "traffic_unit": "bytes per launch (dram read + write)",
                "traffic_source": traffic_note}
    layer_tflops = alg_p["flops"] / (ms_p * 1e-3) / 1e12
    dec_gbs = alg_d["bytes"] / (ms_d * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(tok_s, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_p, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0, 1/sqrt(fan_in)) weights, unit-RMS x)",
        "config": {"workload": "prefill_t4096", "T": wp.T, "d": wp.d, "d_ff": wp.d_ff, "n_experts": wp.n_experts,
                   "k": wp.k, "parallelism": f"replicas x{world} (data parallel over tokens)",
                   "l2": "prefill: inputs larger than L2 (2.82 GB of expert weights streamed per step); "
                         "decode: L2 overwritten (256 MB written, then 256 MB read so no dirty line is left) before each timed call"},
        "layer": {"us_per_layer": round(ms_p * 1e3, 1), "tflops": round(layer_tflops, 1),
                  "frac_of_bf16_burst": round(layer_tflops / pk["bf16_tflops"], 4),
                  "frac_of_bf16_nominal_2250": round(layer_tflops / 2250.0, 4), "expert_loads": counts_p},
        "decode_t32": {"us_per_layer": round(ms_d * 1e3, 1), "weight_gbytes": round(alg_d["weight_bytes"] / 1e9, 3),
                       "experts_touched": alg_d["touched"], "achieved_gbs": round(dec_gbs, 1),
                       "frac_of_hbm": round(dec_gbs / pk["hbm_gbs"], 4),
                       "frac_of_hbm_nominal_8000": round(dec_gbs / 8000.0, 4),
                       "timing": "L2 overwritten before each call; CUDA events around each call",
                       "stages_us": {k: round(v * 1e3, 1) for k, v in stages_d.items()},
                       "roofline": {"bound": "hbm", "achieved": round(dec_gbs, 1), "peak": pk["hbm_gbs"],
                                    "unit": "GB/s", "frac": round(dec_gbs / pk["hbm_gbs"], 4),
                                    "bytes_per_step": int(alg_d["bytes"])}},
        "stages_us": {k: round(v * 1e3, 1) for k, v in stages_p.items()},
        "instrumented_ms_per_step": {"prefill": round(ms_pi, 4), "decode": round(ms_di, 4)},
        "roofline": roofline,
        "sustained": None,
        "skewed_t32768": skew,
        "decode_fp8": fp8,
        "e2e": {"value": round(world * wp.T / (ms_e2e * 1e-3), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": int(xh.numel() * xh.element_size()),
                "d2h_bytes_per_step": int(yh.numel() * yh.element_size()),
                "ms_per_step": round(ms_e2e, 4), "entry_point": "moe_forward_host"},
        "gpu_launches": 3 * args.steps,   # route, W1/W3 GEMM, W2 GEMM (combine in its epilogue) per call
        "timing": {"prefill_steps": args.steps, "decode_steps": args.decode_steps,
                   "per_kernel": "CUDA events recorded by the library around each kernel on the call's stream"},
        "clocks": clocks,
    }
    if sus is not None:
        share_s = sus["stages"][k13] / sum(sus["stages"].values())
        k13_s = sus["ms"] * share_s
        ach_s = alg_p["flops_w13"] / (k13_s * 1e-3) / 1e12
        lt = alg_p["flops"] / (sus["ms"] * 1e-3) / 1e12
        line["sustained"] = {
            "tokens_s": round(world * wp.T / (sus["ms"] * 1e-3), 1), "us_per_layer": round(sus["ms"] * 1e3, 1),
            "calls": sus["calls"], "timed_seconds": round(sus["ms"] * sus["calls"] / 1e3, 2),
            "layer_tflops": round(lt, 1), "layer_frac_of_nominal_2250": round(lt / 2250.0, 4),
            "roofline": {"kernel": k13, "bound": "tensor", "achieved": round(ach_s, 1),
                         "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                         "frac": round(ach_s / pk["bf16_tflops_sustained"], 4),
                         "peak_kind": f"bf16 sustained ({pk['source']})", "duration_us": round(k13_s * 1e3, 1),
                         "share": round(share_s, 4)},
            "stages_us": {k: round(v * 1e3, 1) for k, v in sus["stages"].items()},
            "clocks": clk.summary(("sustained",)),
            "note": "after a 1 s pre-roll of the same calls; per-kernel shares from the instrumented calls that follow"}
    m.close()
    host = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        host = dict(x=xp.cpu(), Wg=Wg.cpu(), W=(W1.cpu(), W3.cpu(), W2.cpu()), gpu_idx=idx_p)
    del xp, xd, W1, W3, W2, Wg
    torch.cuda.empty_cache()
    if not args.no_stack:
        line["stack32"] = run_stack(args, dist)
    return line, host


def run_fp8_decode(args, m, W1, W3, W2, Wg, pk, dist, flush):
    """Decode batches through moe_forward_fp8: the same experts quantised to e4m3
    with one power-of-two scale per weight row (1.41 GB of weight bytes instead
    of 2.82 GB), the same router.  L2 overwritten before each call, CUDA events
    around each call."""
    from sparse_mixture_experts_54_b300 import _lib, inputs

    q, s = {}, {}
    for name, t in (("W1", W1), ("W3", W3), ("W2", W2)):
        q[name], s[name] = inputs.quantize_e4m3_rows(t)
    args8 = (q["W1"], s["W1"], q["W3"], s["W3"], q["W2"], s["W2"])
    stream = torch.cuda.current_stream()
    w = inputs.workload("decode_t32")
    out = {"weights": "e4m3, one fp32 power-of-two scale per weight row", "us_per_layer": {},
           "timing": "L2 overwritten before each call; CUDA events around each call"}

    def timed(T, steps, stage_timing):
        x = inputs.make_x(w, "cuda", seed=17, T=T)
        y = torch.empty((T, w.d), dtype=torch.bfloat16, device="cuda")
        for _ in range(args.warmup):
            m.forward_fp8(x, Wg, *args8, y=y)
        torch.cuda.synchronize()
        m.set_option(_lib.MOE_OPT_STAGE_TIMING, 1 if stage_timing else 0)
        m.stage_times()
        barrier(dist)
        ms = timed_per_call(lambda: m.forward_fp8(x, Wg, *args8, y=y), steps, stream, flush)
        barrier(dist)
        stages, _ = m.stage_times()
        m.set_option(_lib.MOE_OPT_STAGE_TIMING, 0)
        assert m.status() == 0, _lib.moe_error_string(m.status())
        counts = m.route(x, Wg)["counts"].cpu().tolist()
        return max_over_ranks(ms, dist), stages, counts

    ms, _, counts = timed(32, args.decode_steps, False)
    _, stages, _ = timed(32, max(args.decode_steps // 4, 3), True)
    touched = sum(1 for c in counts if c > 0)
    wbytes = touched * (3 * w.d * w.d_ff + (2 * w.d_ff + w.d) * 4)   # e4m3 bytes + row scales
    nbytes = wbytes + 2 * 32 * w.d * 2 + w.n_experts * w.d * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    out["decode_t32"] = {"us_per_layer": round(ms * 1e3, 1), "weight_gbytes": round(wbytes / 1e9, 3),
                         "experts_touched": touched, "achieved_gbs": round(gbs, 1),
                         "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                         "stages_us": {k: round(v * 1e3, 1) for k, v in stages.items()},
                         "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": pk["hbm_gbs"],
                                      "unit": "GB/s", "frac": round(gbs / pk["hbm_gbs"], 4),
                                      "bytes_per_step": int(nbytes)}}
    for T in (1, 8, 128, 256):
        ms_t, _, _ = timed(T, max(args.decode_steps // 4, 20), False)
        out["us_per_layer"][str(T)] = round(ms_t * 1e3, 1)
    out["us_per_layer"]["32"] = round(ms * 1e3, 1)
    out["kernel"] = "e4m3 weights into the 8-bit MMA against hi/lo e4m3 token rows (MOE_OPT_FP8_WIDEN 0)"
    # the exact widening kernel beside it (bitwise equal to the bf16 path on the dequantised weights)
    m.set_option(_lib.MOE_OPT_FP8_WIDEN, 1)
    ms_w, stages_w, _ = timed(32, max(args.decode_steps // 4, 20), False)
    m.set_option(_lib.MOE_OPT_FP8_WIDEN, 0)
    out["widened_t32_us_per_layer"] = round(ms_w * 1e3, 1)
    del q, s, args8
    torch.cuda.empty_cache()
    return out


def run_skewed(args, W1, W3, W2, pk, dist):
    """One layer call at T=32768 with the skewed router bias and consecutive-token
    locality (same expert weights as the headline workload)."""
    from sparse_mixture_experts_54_b300 import _lib, inputs
    from sparse_mixture_experts_54_b300.layer import MoELayer

    w = inputs.workload("skewed_t32768")
    rank = int(os.environ.get("RANK", "0"))
    x = inputs.make_x(w, "cuda", seed=rank)
    Wg, b = inputs.make_router(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, bias=b)
    m.reserve(w.T)
    r = m.route(x, Wg)
    counts = r["counts"].cpu().tolist()
    first = r["topk_idx"][:, 0]
    repeat = float((first[1:] == first[:-1]).float().mean().item())
    y = torch.empty_like(x)
    for _ in range(2):
        m.forward(x, Wg, W1, W3, W2, y=y)
    steps = max(args.steps // 50, 5)
    m.set_option(_lib.MOE_OPT_STAGE_TIMING, 1)
    m.stage_times()
    torch.cuda.synchronize()
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        m.forward(x, Wg, W1, W3, W2, y=y)
    e1.record()
    torch.cuda.synchronize()
    barrier(dist)
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, dist)
    stages, _ = m.stage_times()
    assert m.status() == 0, _lib.moe_error_string(m.status())
    m.close()
    alg = algorithmic(w.T, counts)
    tf = alg["flops"] / (ms * 1e-3) / 1e12
    return {"us_per_layer": round(ms * 1e3, 1), "tokens_s": round(w.T / (ms * 1e-3), 1), "tflops": round(tf, 1),
            "frac_of_bf16_sustained": round(tf / pk["bf16_tflops_sustained"], 4),
            "expert_loads": counts, "hot_expert_share": round(max(counts) / sum(counts), 4),
            "first_choice_repeat_rate": round(repeat, 4), "steps": steps,
            "stages_us": {k: round(v * 1e3, 1) for k, v in stages.items()},
            "note": "timed with per-stage events on; router bias [1.5,0.5,0,0,0,0,-0.5,-1], row repeat p=0.5"}


def run_stack(args, dist):
    """The 32-layer stack (h <- h + MoE_l(RMSNorm(h)) per layer, layer l seeded
    1000 + l; ~90 GB of expert weights resident): microseconds per layer through
    moe_stack_forward for the decode sweep and one prefill pass."""
    from sparse_mixture_experts_54_b300 import _lib, inputs
    from sparse_mixture_experts_54_b300.layer import MoELayer

    w = inputs.workload("decode_t32")
    layers = []
    for l in range(inputs.STACK_LAYERS):
        Wg, _ = inputs.make_router(w, "cuda", seed=1000 + l)
        layers.append((Wg,) + inputs.make_experts(w, "cuda", seed=1000 + l))
    torch.cuda.synchronize()
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k)
    m.reserve(inputs.STACK_PREFILL_T)
    L = len(layers)

    def per_layer_us(T, passes, force_path=0):
        m.set_option(_lib.MOE_OPT_FORCE_PATH, force_path)
        h0 = inputs.make_x(w, "cuda", seed=2000 + T, T=T)
        h = h0.clone()
        m.stack_forward(h, layers, 1e-5)   # warm-up pass
        torch.cuda.synchronize()
        barrier(dist)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(passes):
            m.stack_forward(h, layers, 1e-5)
        e1.record()
        torch.cuda.synchronize()
        barrier(dist)
        assert m.status() == 0, _lib.moe_error_string(m.status())
        return max_over_ranks(e0.elapsed_time(e1) * 1e3 / (passes * L), dist)

    out = {"layers": L, "expert_weight_gbytes": round(L * 3 * w.n_experts * w.d * w.d_ff * 2 / 1e9, 2),
           "timing": "CUDA events around whole stack passes (h updated in place; weights streamed from HBM)",
           "decode_us_per_layer": {}, "decode_path_us_per_layer": {}}
    for T in inputs.STACK_DECODE_T:
        out["decode_us_per_layer"][str(T)] = round(per_layer_us(T, args.stack_passes), 1)
        if T > 64:
            out["decode_path_us_per_layer"][str(T)] = round(per_layer_us(T, args.stack_passes, force_path=2), 1)
    Tp = inputs.STACK_PREFILL_T
    us = per_layer_us(Tp, max(args.stack_passes // 4, 2))
    out["prefill_t8192_us_per_layer"] = round(us, 1)
    out["prefill_t8192_tokens_s_per_layer"] = round(Tp / (us * 1e-6), 1)
    out["prefill_t8192_stack_ms"] = round(us * L / 1e3, 2)
    m.close()
    del layers
    torch.cuda.empty_cache()
    return out


# ----------------------------------------------------------------------------- oracle timing
def time_oracle(x, Wg, W, budget_s: float, min_tokens: int, seed: int = 0):
    """Time the fp64 oracle on a bounded, seeded sample of the batch's tokens."""
    import numpy as np

    import oracle
    from sparse_mixture_experts_54_b300 import inputs

    # already host arrays when the caller converted them once (the reference arm)
    xo = x if isinstance(x, np.ndarray) else inputs.to_oracle(x)
    Wgo = Wg if isinstance(Wg, np.ndarray) else inputs.to_oracle(Wg)
    W1, W3, W2 = (t if isinstance(t, np.ndarray) else inputs.to_oracle(t) for t in W)
    threads = oracle.max_threads()
    T = xo.shape[0]
    order = inputs.sample_tokens(T, T, seed).numpy()
    rng = np.random.default_rng(seed)
    rng.shuffle(order)
    done, t_total = 0, 0.0
    batch = max(threads, 1)
    while done < T:
        toks = np.sort(order[done:done + batch])
        t0 = time.perf_counter()
        oracle.moe_forward(xo[toks], Wgo, W1, W3, W2, 2, nthreads=threads)
        t_total += time.perf_counter() - t0
        done += len(toks)
        if t_total >= budget_s and done >= min_tokens:
            break
    return dict(tokens=done, seconds=t_total, threads=threads, tok_s=done / t_total)


def routing_near_ties(host, K: int = 2, eps: float = 1e-6):
    """The cpu_baseline leg's fp64 routing of every prefill token against the GPU's
    top-K indices: near ties (fp64 logits of ranks 1..K+1 closer than eps, where
    fp32 on the GPU may order them either way) and index mismatches outside them."""
    import numpy as np

    import oracle
    from sparse_mixture_experts_54_b300 import inputs

    logits = oracle.router_logits(inputs.to_oracle(host["x"]), inputs.to_oracle(host["Wg"]))
    idx, _ = oracle.select_topk(logits, K)
    srt = -np.sort(-logits, axis=1)
    gaps = srt[:, :K] - srt[:, 1:K + 1]
    near = np.any(gaps < eps, axis=1)
    gpu = host["gpu_idx"].numpy()
    mism = int(np.sum(np.any(gpu != idx, axis=1) & ~near))
    return {"tokens": int(logits.shape[0]), "near_ties": int(near.sum()), "index_mismatches_outside_near_ties": mism,
            "rule": f"fp64 router logits of ranks 1..{K + 1} closer than {eps:g}",
            "source": "cpu_baseline leg: the oracle's fp64 routing of every token vs the GPU's top-k"}


def cpu_baseline_block(res, T):
    return {"value": round(res["tok_s"], 3), "unit": "tokens/s", "cores": res["threads"], "kind": "oracle",
            "sample": f"{res['tokens']} of the {T} prefill tokens (seeded sample), full routing + 2 SwiGLU experts "
                      f"each in fp64, {res['seconds']:.1f} s on {res['threads']} host threads"}


def run_reference(args, rank, world):
    from sparse_mixture_experts_54_b300 import inputs

    if rank != 0:
        return None
    w = inputs.workload("prefill_t4096")
    # the oracle runs on the host: draw the inputs on the GPU when there is one (fast), then copy
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    W = tuple(inputs.to_oracle(t) for t in inputs.make_experts(w, dev))
    x = inputs.to_oracle(inputs.make_x(w, dev))
    Wg = inputs.to_oracle(inputs.make_router(w, dev)[0])
    per_step = []
    res = None
    # each step is a bounded sample, sized so that the whole run stays within a few minutes
    budget = args.ref_budget_s if args.ref_budget_s is not None else \
        min(6.0, 150.0 / max(args.warmup + args.steps, 1))
    for i in range(args.warmup + args.steps):
        res = time_oracle(x, Wg, W, budget_s=budget, min_tokens=1, seed=i)
        if i >= args.warmup:
            per_step.append(res)
    tok_s = sum(r["tokens"] for r in per_step) / sum(r["seconds"] for r in per_step)
    ms_per_step = w.T / tok_s * 1e3
    cb = cpu_baseline_block(dict(res, tok_s=tok_s, tokens=sum(r["tokens"] for r in per_step),
                                 seconds=sum(r["seconds"] for r in per_step)), w.T)
    return {"impl": "reference", "metric": METRIC, "value": round(tok_s, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 1),
            "ms_per_step_kind": "extrapolated: T=4096 tokens divided by the oracle's rate on the timed samples "
                                "(each step times a bounded sample, not the whole batch)",
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0, 1/sqrt(fan_in)) weights, unit-RMS x)",
            "config": {"workload": "prefill_t4096", "T": w.T, "d": w.d, "d_ff": w.d_ff, "n_experts": w.n_experts,
                       "k": w.k, "parallelism": "host cores (OpenMP over tokens)",
                       "sample": "each step: a bounded seeded sample of the T=4096 tokens"},
            "cpu_baseline": cb,
            "e2e": {"value": round(tok_s, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def profile_step(args):
    """A few untimed forward calls of one workload, for ncu captures (no timing, no oracle)."""
    from sparse_mixture_experts_54_b300 import _lib, inputs
    from sparse_mixture_experts_54_b300.layer import MoELayer

    torch.cuda.set_device(0)
    w = inputs.workload(args.profile_step, **({"T": args.profile_T} if args.profile_T else {}))
    W1, W3, W2 = inputs.make_experts(w, "cuda")
    x = inputs.make_x(w, "cuda")
    Wg, b = inputs.make_router(w, "cuda")
    m = MoELayer(w.d, w.d_ff, w.n_experts, w.k, bias=b)
    if args.force_path:
        m.set_option(_lib.MOE_OPT_FORCE_PATH, args.force_path)
    if args.gemm_pair:
        m.set_option(_lib.MOE_OPT_GEMM_PAIR, args.gemm_pair)
    if args.fp8:
        q = [inputs.quantize_e4m3_rows(t) for t in (W1, W3, W2)]
        del W1, W3, W2
        for _ in range(args.warmup + 1):
            m.forward_fp8(x, Wg, q[0][0], q[0][1], q[1][0], q[1][1], q[2][0], q[2][1])
    else:
        for _ in range(args.warmup + 1):
            m.forward(x, Wg, W1, W3, W2)
    torch.cuda.synchronize()
    assert m.status() == 0
    print(f"profile_step {w.name} (T={w.T}): {args.warmup + 1} forward calls done", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--decode-steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-stack", action="store_true", help="skip the 32-layer stack measurement")
    ap.add_argument("--no-skewed", action="store_true", help="skip the skewed T=32768 measurement")
    ap.add_argument("--no-fp8", action="store_true", help="skip the fp8-weight decode measurements")
    ap.add_argument("--fp8", action="store_true", help="with --profile-step: fp8 expert weights (moe_forward_fp8)")
    ap.add_argument("--stack-passes", type=int, default=8)
    ap.add_argument("--sustained-s", type=float, default=2.5,
                    help="seconds of back-to-back prefill calls for the sustained leg (0: skip it)")
    ap.add_argument("--cpu-budget-s", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=None,
                    help="oracle seconds per reference step (default: min(6, 150 / (warmup + steps)))")
    ap.add_argument("--profile-step", default=None, help="workload name: run warmup+1 untimed calls (for ncu)")
    ap.add_argument("--force-path", type=int, default=0)
    ap.add_argument("--profile-T", type=int, default=0, help="with --profile-step: batch size other than the workload's")
    ap.add_argument("--gemm-pair", type=int, default=0,
                    help="with --profile-step: grouped-GEMM tiling (1 single CTA, 2 CTA pairs; 0 the default)")
    args = ap.parse_args()
    if args.profile_step:
        profile_step(args)
        return
    if args.warmup < 3:
        args.warmup = 3

    rank, world, dist = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if rank == 0:
            print(json.dumps(line), flush=True)
        return
    line, host = run_ours(args, rank, world, dist)
    if rank == 0:
        if host is not None:
            res = time_oracle(host["x"], host["Wg"], host["W"], budget_s=args.cpu_budget_s, min_tokens=8)
            line["cpu_baseline"] = cpu_baseline_block(res, 4096)
            line["near_ties"] = routing_near_ties(host)
        else:
            line["cpu_baseline"] = None
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
