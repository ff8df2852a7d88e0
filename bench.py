#!/usr/bin/env python
"""MoE layer forward throughput on B300 (one JSON line on rank 0).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                [--per-config A,B,...] [--impl ours|reference]

A step is one full moe_layer_forward (router, gating/top-k, capacity/dispatch,
gather, grouped gate/up + SwiGLU, grouped down, combine) over one batch of
synthetic inputs that are already resident in HBM.  ``value`` is tokens/s over
all ranks; with N > 1 every rank runs an independent replica (the layer shards
by tokens with no exchange), so scaling is weak.

The headline is the DeepSeek-V3-shaped prefill layer, the largest layer that
fits one GPU (its GEMMs are the tensor-bound half of the metric).  The line's
``per_config`` object carries the same measurement for the Mixtral-shaped
layer, the DeepSeek-V3-shaped decode layer (the HBM-bound half) and the
Switch-shaped capacity layer.  Every configuration reports the K-step figure
(burst clocks) and, under ``sustained``, a seconds-long loop of the same step
that runs into the power cap, against the sustained tensor peak.

--impl reference times the float64 CPU oracle (the only reference
implementation: the pages print no code) on the host cores, on a bounded
sample of the headline workload.
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
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("MoE-layer tokens/s on 1 B300; % of bf16 tensor peak (prefill) / "
          "HBM BW (decode)")

WORKLOAD_TEXT = {
    "mixtral": "Mixtral-8x7B-shaped MoE layer (T=4096, d=4096, E=8, top-2, SwiGLU d_ff=14336, "
               "softmax + renorm, bf16, fp32 accumulate)",
    "dsv3_prefill": "DeepSeek-V3-shaped MoE prefill layer (T=8192, d=7168, E=256 top-8, "
                    "d_ff=2048, 1 shared expert d_ff=2048, sigmoid, renorm x2.5, bf16)",
    "switch": "Switch-style capacity layer (T=16384, d=2048, E=64 top-1, d_ff=8192, softmax, "
              "C=ceil(T/E*1.25)=320, Zipf(1.2) router bias, bf16)",
    "dsv3_prefill_noaux": "DeepSeek-V3-shaped MoE prefill layer with DeepSeek-V3's router "
                          "(T=8192, d=7168, E=256 top-8 ranked by sigmoid + selection bias, "
                          "8 groups / 4 kept, d_ff=2048, 1 shared expert, renorm x2.5, bf16)",
    "switch_expert_choice": "Switch-shaped layer routed by expert choice (T=16384, d=2048, "
                            "E=64, each expert takes C=T/E=256 tokens, d_ff=8192, softmax "
                            "scores, bf16)",
    "dsv3_decode_fp8": "DeepSeek-V3-shaped decode layer with E4M3 expert weights (T=64, "
                       "d=7168, E=256 top-8, d_ff=2048, 1 shared expert, sigmoid, renorm x2.5, "
                       "bf16 activations, one fp32 scale per weight row)",
    "dsv3_prefill_fp8": "DeepSeek-V3-shaped MoE prefill layer with E4M3 expert weights (T=8192, "
                        "d=7168, E=256 top-8, d_ff=2048, 1 shared expert, sigmoid, renorm x2.5, "
                        "bf16 activations, one fp32 scale per weight row)",
    "dsv3_decode": "DeepSeek-V3-shaped decode layer (T=64, d=7168, E=256 top-8, d_ff=2048, "
                   "1 shared expert, sigmoid, renorm x2.5, bf16)",
    "tiny": "tiny fp32 layer (T=64, d=128, E=4 top-2, d_ff=256)",
}

FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


HEADLINE = "dsv3_prefill"
PER_CONFIG = ("mixtral", "dsv3_decode", "switch", "dsv3_decode_fp8")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--per-config", default=",".join(PER_CONFIG),
                    help="comma-separated workloads measured after the headline one and "
                         "reported under per_config ('' for none)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample-tokens", type=int, default=16)
    ap.add_argument("--cpu-steps", type=int, default=3)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--sustain-ms", type=float, default=2000.0,
                    help="length of the sustained (power-capped) loop per workload; 0 skips it")
    ap.add_argument("--experts", type=int, default=None,
                    help="profiling aid: keep the workload's per-expert GEMM shapes but use "
                         "this many experts (tokens scaled to keep rows per expert)")
    return ap.parse_args(argv)


# ---------------------------------------------------------------------------
# environment helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# Sources of the grouped GEMM kernels whose DRAM counters profiles/traffic.json
# stores: each record names the files its kernel is built from (default: the
# bf16 tokens-in-M kernel) and the digest of those files when it was captured.
GEMM_SOURCES = ("experts_tc.cu", "tc_common.cuh")
E2E_PIPELINE = 2   # batches in flight in the end-to-end leg


def source_digest(names=GEMM_SOURCES) -> str:
    """Digest of grouped-GEMM CUDA sources, to tell whether stored ncu
    counters still describe the current kernels."""
    h = hashlib.sha256()
    files = [os.path.join(ROOT, "top_routing_expert_gate_b300", "csrc", n) for n in names]
    for f in files:
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def stored_traffic(workload: str, stage: str):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        t = json.load(f)
    rec = t.get(workload, {}).get(stage)
    if not rec or rec.get("source_digest") != source_digest(tuple(rec.get("sources",
                                                                           GEMM_SOURCES))):
        return None
    return rec.get("dram_bytes_per_launch")


# Polls one GPU through NVML, the driver's management library, called with
# ctypes (read-only queries: SM clock, its maximum, the active clock-event
# reasons), and prints "host_time sm_mhz max_mhz reason_mask" per sample until
# it is terminated.  A process of its own, so that the bench's Python thread
# holding the interpreter lock cannot delay the samples.
_NVML_POLL_SRC = r"""
import ctypes, sys, time
nv = ctypes.CDLL("libnvidia-ml.so.1")
if nv.nvmlInit_v2() != 0:
    sys.exit(1)
h = ctypes.c_void_p()
if nv.nvmlDeviceGetHandleByPciBusId_v2(sys.argv[1].encode(), ctypes.byref(h)) != 0:
    sys.exit(1)
period = float(sys.argv[2])
try:
    reasons = nv.nvmlDeviceGetCurrentClocksEventReasons
except AttributeError:
    reasons = nv.nvmlDeviceGetCurrentClocksThrottleReasons
SM = 1   # NVML_CLOCK_SM
clk, mx, mask = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
if nv.nvmlDeviceGetMaxClockInfo(h, SM, ctypes.byref(mx)) != 0:
    sys.exit(1)
out = sys.stdout
while True:
    t = time.time()
    if nv.nvmlDeviceGetClockInfo(h, SM, ctypes.byref(clk)) != 0 or \
            reasons(h, ctypes.byref(mask)) != 0:
        sys.exit(1)
    out.write("%.6f %d %d %d\n" % (t, clk.value, mx.value, mask.value))
    out.flush()
    time.sleep(period)
"""


class ClockSampler:
    """SM clock and clock-event reasons sampled during the timed window.

    A child process polls NVML every 5 ms (read-only queries), so that even a
    20 ms window holds a few samples; `nvidia-smi -lms 50` stands in when
    the NVML library cannot be loaded.  Only the samples taken inside the timed window
    (mark_begin .. mark_end, host wall clock) enter the summary.  Nothing
    here changes a GPU setting."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    # NVML clock-event reason bits of the four reasons above
    REASON_BITS = (0x8, 0x40, 0x20, 0x4)
    PERIOD_S = 0.005

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        self.nvml_lines = []
        self.dev = device_index
        self.t0 = self.t1 = None
        self.source = None

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def _smi_id(self):
        import torch
        try:
            p = torch.cuda.get_device_properties(self.dev)
            return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            return vis.split(",")[self.dev] if vis else str(self.dev)

    def start(self):
        # the NVML poller, once it has taken its first sample; else nvidia-smi
        try:
            self.proc = subprocess.Popen(
                [sys.executable, "-c", _NVML_POLL_SRC, self._smi_id(), str(self.PERIOD_S)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            first = self.proc.stdout.readline()
            if first.strip():
                self.nvml_lines = [first]
                self.source = "nvml"
                return
            self.proc.wait(timeout=5)
        except (OSError, subprocess.TimeoutExpired):
            pass
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", self._smi_id()],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        lines = [ln for ln in out.splitlines() if ln.strip()]
        if self.source == "nvml":
            self.nvml_lines += lines
        else:
            self.lines = lines

    @staticmethod
    def _stamp(text):
        import datetime
        try:
            return datetime.datetime.strptime(text.strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
        except ValueError:
            return None

    def _in_window(self, ts):
        return ts is None or self.t0 is None or self.t1 is None or self.t0 <= ts <= self.t1

    def summary(self):
        sm, mx, reasons = [], None, set()
        for ln in self.nvml_lines:
            parts = ln.split()
            try:
                ts, mhz, top, mask = float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3])
            except (ValueError, IndexError):
                continue
            if not self._in_window(ts):
                continue
            sm.append(mhz)
            mx = top
            reasons |= {n for n, b in zip(self.REASONS, self.REASON_BITS) if mask & b}
        names = list(self.REASONS)
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 10:
                continue
            if not self._in_window(self._stamp(parts[0])):
                continue
            try:
                sm.append(float(parts[2]))
                mx = float(parts[3])
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# algorithmic work
# ---------------------------------------------------------------------------

def algorithmic_work(shape, counts):
    """FLOPs and bytes of one forward: router + kept assignments + shared."""
    T, d, E, F, Fs = shape.T, shape.d, shape.E, shape.F, shape.F_s
    kept = int(sum(counts))
    touched = int(sum(1 for c in counts if c > 0))
    eb = 2 if shape.dtype == "bf16" else 4
    fp8 = getattr(shape, "weight_format", "act") == "fp8"
    wb = 1 if fp8 else eb          # bytes per expert weight (E4M3 codes: 1)
    sb = 4 if fp8 else 0           # bytes of the fp32 scale of one weight row
    fl_router = 2.0 * T * E * d
    fl_gate_up = 2.0 * kept * 2 * F * d + 2.0 * T * 2 * Fs * d
    fl_down = 2.0 * kept * F * d + 2.0 * T * Fs * d
    b_gate_up = touched * 2 * F * (d * wb + sb) + 2 * Fs * (d * wb + sb)
    b_down = touched * d * (F * wb + sb) + d * (Fs * wb + sb)
    return {"kept": kept, "touched": touched, "flops_router": fl_router,
            "flops_gate_up": fl_gate_up, "flops_down": fl_down,
            "flops": fl_router + fl_gate_up + fl_down,
            "bytes_gate_up": b_gate_up, "bytes_down": b_down,
            "weight_bytes": b_gate_up + b_down + E * d * eb}


# ---------------------------------------------------------------------------
# float64 oracle timing (reference arm and cpu_baseline)
# ---------------------------------------------------------------------------

def oracle_samples(shape, sample_tokens: int, n: int, seed: int = 0):
    """The token sample of each oracle step (sorted token ids)."""
    import numpy as np
    rng = np.random.default_rng(seed)
    m = min(sample_tokens, shape.T)
    return [np.sort(rng.choice(shape.T, size=m, replace=False)) for _ in range(n)]


def _oracle_inputs(shape, inputs):
    from workloads.generate import to_f64
    return (to_f64(inputs["x"]), to_f64(inputs["w_router"]), to_f64(inputs["router_bias"]),
            to_f64(inputs.get("score_bias")), to_f64(inputs.get("shared_gate")))


def experts_reached(shape, inputs, samples):
    """Routed experts whose weights the sampled tokens' outputs use (one
    untimed routing pass of the oracle over the whole batch)."""
    import numpy as np
    from oracle import moe_oracle as O
    x, wr, bias, sbias, _ = _oracle_inputs(shape, inputs)
    toks = np.unique(np.concatenate(samples))
    z = O.router_logits(x, wr, bias)
    if getattr(shape, "routing", "token") == "expert":
        C = O.expert_choice_capacity(shape.T, shape.E, shape.k)
        ec = O.expert_choice(O.gate_scores(z, shape.gate), C)
        return [e for e in range(shape.E) if np.isin(ec["tokens"][e], toks).any()]
    r = O.route(z, shape.k, shape.gate, shape.renormalize, shape.rsf,
                O.expert_capacity(shape.T, shape.E, shape.capacity_factor), score_bias=sbias,
                n_group=max(shape.n_group, 1), topk_group=shape.topk_group)
    kept = r["drop_mask"].reshape(shape.T, shape.k)[toks] == 0
    return sorted(set(r["topk_idx"][toks][kept].tolist()))


class WidenedExperts:
    """Float64 expert weights for the oracle, widened once before timing and
    kept resident on the host (as the GPU's weights are resident in HBM).
    Only experts some sampled token reaches are widened; a workload with the
    same weight tensors (same shapes and seed) reuses what is already here."""

    def __init__(self):
        self.key = None
        self.experts = {}
        self.shared = None

    def prepare(self, shape, inputs, needed):
        import torch
        from oracle import moe_oracle as O
        from workloads.generate import to_f64
        key = (shape.d, shape.E, shape.F, shape.F_s, shape.dtype,
               getattr(shape, "weight_format", "act"))
        if key != self.key:
            self.key, self.experts, self.shared = key, {}, None

        def widen(name, e=None):
            t = inputs[name] if e is None else inputs[name][e]
            if inputs.get(name + "_scale") is None:
                return to_f64(t)
            sc = inputs[name + "_scale"] if e is None else inputs[name + "_scale"][e]
            codes = t.detach().contiguous().view(torch.uint8).cpu().numpy()
            return O.dequantize_rows(codes, to_f64(sc))

        for e in needed:
            if e not in self.experts:
                self.experts[e] = (widen("w_gate", e), widen("w_up", e), widen("w_down", e))
        if inputs.get("ws_gate") is not None and self.shared is None:
            self.shared = (widen("ws_gate"), widen("ws_up"), widen("ws_down"))
        return self.experts, (self.shared if inputs.get("ws_gate") is not None else None)


def time_oracle(shape, inputs, samples, warmup: int = 0, cache: Optional[WidenedExperts] = None):
    """Oracle forward on the host, one step per token sample: routing of all
    T tokens and the layer output of the sampled tokens.  Returns the times of
    the steps after ``warmup``."""
    from oracle import moe_oracle as O
    cache = cache or WidenedExperts()
    experts, shared = cache.prepare(shape, inputs, experts_reached(shape, inputs, samples))
    x, wr, bias, sbias, sgate = _oracle_inputs(shape, inputs)
    cap = O.expert_capacity(shape.T, shape.E, shape.capacity_factor)
    times = []
    for i, toks in enumerate(samples):
        t0 = time.perf_counter()
        if getattr(shape, "routing", "token") == "expert":
            O.moe_layer_expert_choice(x, wr, experts,
                                      O.expert_choice_capacity(shape.T, shape.E, shape.k),
                                      shape.gate, shared=shared, tokens=toks)
        else:
            O.moe_layer_forward(x, wr, experts, k=shape.k, gate=shape.gate,
                                renormalize=shape.renormalize, routed_scaling_factor=shape.rsf,
                                capacity=cap, router_bias=bias, shared=shared, tokens=toks,
                                score_bias=sbias, n_group=max(shape.n_group, 1),
                                topk_group=shape.topk_group, shared_gate=sgate)
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    return times


def max_over_ranks(value: float, device) -> float:
    """The largest ``value`` over all ranks (the slowest replica sets the time);
    ``value`` itself when not running distributed."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def tensor_bound(work, stage: str, peaks, tensor_key: str) -> bool:
    """True when a GEMM stage's algorithmic FLOPs take longer at the tensor
    peak than its algorithmic weight bytes at the copy bandwidth."""
    if stage not in ("gate_up", "down"):
        return False
    f = work["flops_gate_up"] if stage == "gate_up" else work["flops_down"]
    b = work["bytes_gate_up"] if stage == "gate_up" else work["bytes_down"]
    return f / (peaks[tensor_key] * 1e12) >= b / (peaks["hbm_gbs"] * 1e9)


def tokens_per_second(tokens_per_rank: int, world: int, ms_per_step: float) -> float:
    """Whole-job throughput: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / (ms_per_step * 1e-3)


def cores_available():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def timed_oracle(shape, inputs, samples, warmup: int = 0, threads: Optional[int] = None,
                 cache: Optional[WidenedExperts] = None):
    """Oracle timing with the BLAS pools limited to `threads` (default: every
    core of this process's affinity); returns the step times and the BLAS
    threads in effect while they ran.  Without threadpoolctl the BLAS
    default (one thread per core) stays and the affinity count is reported."""
    n = threads or cores_available()
    try:
        from threadpoolctl import threadpool_info, threadpool_limits
    except ImportError:
        return time_oracle(shape, inputs, samples, warmup, cache), n
    with threadpool_limits(limits=n, user_api="blas"):
        used = max([p["num_threads"] for p in threadpool_info() if p["user_api"] == "blas"]
                   or [1])
        times = time_oracle(shape, inputs, samples, warmup, cache)
    return times, used


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def workload_shape(name: str, experts: Optional[int] = None):
    from workloads import SHAPES
    shape = SHAPES[name]
    if experts is not None and experts != shape.E:
        from dataclasses import replace
        T = max(1, shape.T * experts // shape.E)
        shape = replace(shape, name=f"{shape.name}_E{experts}", E=experts,
                        k=min(shape.k, experts), T=T)
    return shape


def roofline(work, stage_ms, peaks, peak_src, tensor_key, peak_note):
    """Roofline record of the dominant (longest) stage: its bound is the roof
    its algorithmic work reaches first (FLOPs at the tensor peak vs bytes at
    the copy bandwidth): tensor for the prefill GEMMs, HBM for decode and for
    the Switch layer's few kept tokens over many touched experts."""
    dom = max(stage_ms, key=stage_ms.get)
    if tensor_bound(work, dom, peaks, tensor_key):
        flops = work["flops_gate_up"] if dom == "gate_up" else work["flops_down"]
        achieved = flops / (stage_ms[dom] * 1e-3) / 1e12
        peak = peaks[tensor_key]
        return {"bound": "tensor", "kernel": f"grouped_{dom}", "stage": dom,
                "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": f"{tensor_key} ({peak_src}; {peak_note})"}
    nbytes = work["bytes_gate_up"] if dom == "gate_up" else (
        work["bytes_down"] if dom == "down" else work["weight_bytes"])
    achieved = nbytes / (stage_ms[dom] * 1e-3) / 1e9
    peak = peaks["hbm_gbs"]
    return {"bound": "hbm", "kernel": f"grouped_{dom}" if dom in ("gate_up", "down") else dom,
            "stage": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"hbm_gbs ({peak_src})"}


def layer_rates(work, ms_per_step, peaks, tensor_key):
    sec = ms_per_step * 1e-3
    return {"tflops": work["flops"] / sec / 1e12,
            # whole layer against the same tensor peak as the roofline
            "tensor_peak_frac": work["flops"] / sec / 1e12 / peaks[tensor_key],
            "weight_gbs": work["weight_bytes"] / sec / 1e9,
            # whole layer's weight stream against the measured copy bandwidth
            "hbm_frac": work["weight_bytes"] / sec / 1e9 / peaks["hbm_gbs"]}


def measure_workload(name, args, dev, world, rank, peaks, peak_src, oracle_cache):
    """One workload on this rank: warm-up, K timed steps, the sustained loop
    and the end-to-end leg.  Returns the record rank 0 reports (None on other
    ranks) and, on rank 0 of a one-GPU run, a function that times the oracle
    baseline on the host and adds it to the record: main calls those after
    every GPU measurement, so that the GPU does not sit idle (and clock down)
    between one workload's timed steps and the next one's."""
    import torch
    import torch.distributed as dist

    import top_routing_expert_gate_b300 as moe
    from top_routing_expert_gate_b300 import _binding as B
    from workloads import make_inputs

    shape = workload_shape(name, args.experts)
    inputs = make_inputs(shape, device=dev, seed=0)
    cfg = moe.config_from_shape(shape, out_dtype="fp32")
    ws = moe.Workspace(cfg, dev)
    w = moe.LayerWeights.from_inputs(inputs)
    T, d, E, k = shape.T, shape.d, shape.E, shape.k
    x = inputs["x"]
    y = torch.empty((T, d), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    drops = torch.empty(E, dtype=torch.int32, device=dev)
    mean_prob = torch.empty(E, dtype=torch.float32, device=dev)
    token_choice = getattr(shape, "routing", "token") == "token"   # expert choice: no top-k
    topk_idx = torch.empty((T, k), dtype=torch.int32, device=dev) if token_choice else None
    topk_w = torch.empty((T, k), dtype=torch.float32, device=dev) if token_choice else None
    stream = torch.cuda.current_stream(dev)
    NS = B.MOE_NUM_STAGES

    def new_events(n):
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for e in evs:
            e.record(stream)      # creates the underlying cudaEvent
        return evs

    def step(evs):
        return moe.moe_layer_forward_profiled(cfg, x, w.w_router, w.router_bias, w.score_bias,
                                              w.w_gate, w.w_up, w.w_down, w.ws_gate, w.ws_up,
                                              w.ws_down, w.shared_gate, w.scales, y, topk_idx,
                                              topk_w, counts, drops, mean_prob, ws, evs, stream)

    warm_events = new_events(NS + 1)
    for _ in range(args.warmup):
        step(warm_events)
    torch.cuda.synchronize(dev)
    if moe.moe_get_error(ws) != 0:
        raise RuntimeError(f"{name}: device status after warm-up")
    work = algorithmic_work(shape, counts.cpu().tolist())

    def timed_loop(n_steps):
        """n_steps layer calls between a barrier + synchronize on both sides;
        returns (ms per step over the slowest rank, per-stage ms, launches,
        clock summary)."""
        evs = [new_events(NS + 1) for _ in range(n_steps)]
        clocks = ClockSampler(dev.index if dev.index is not None else 0)
        clocks.start()
        time.sleep(0.3)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        launches = 0
        clocks.mark_begin()
        t0.record(stream)
        for i in range(n_steps):
            launches += step(evs[i])
        t1.record(stream)
        torch.cuda.synchronize(dev)
        clocks.mark_end()
        if world > 1:
            dist.barrier()
        clocks.stop()
        ms = max_over_ranks(t0.elapsed_time(t1), dev) / n_steps
        if moe.moe_get_error(ws) != 0:
            raise RuntimeError(f"{name}: device status after the timed steps")
        stage = {}
        for si, sname in enumerate(B.STAGE_NAMES):
            vals = [ev[si].elapsed_time(ev[si + 1]) for ev in evs]
            stage[sname] = sum(vals) / len(vals)
        return ms, stage, launches, clocks.summary()

    ms_per_step, stage_ms, launches, clk = timed_loop(args.steps)

    # a seconds-long loop of the same step, long enough to reach the power cap
    sustained = None
    if args.sustain_ms > 0:
        n_sus = max(args.steps, int(math.ceil(args.sustain_ms / ms_per_step)))
        s_ms, s_stage, _, s_clk = timed_loop(n_sus)
        s_key = "bf16_tflops_sustained" if "bf16_tflops_sustained" in peaks else "bf16_tflops"
        sustained = {"value": tokens_per_second(T, world, s_ms), "unit": "tokens/s",
                     "ms_per_step": s_ms, "steps": n_sus, "stage_ms": s_stage,
                     "roofline": roofline(work, s_stage, peaks, peak_src, s_key,
                                          "seconds-long loop"),
                     **layer_rates(work, s_ms, peaks, s_key), "clocks": s_clk}

    # end to end through the C ABI's host-buffer call: every step copies its
    # x from pinned host memory, runs the layer and copies y back.  Two
    # batches are in flight on two streams (each with its own staging buffers
    # and workspace), so that one batch's copies overlap the other's kernels.
    n_pipe = E2E_PIPELINE
    pipes = []
    for j in range(n_pipe):
        pipes.append({"stream": torch.cuda.Stream(dev), "x_host": x.cpu().pin_memory(),
                      "y_host": torch.empty((T, d), dtype=y.dtype).pin_memory(),
                      "x": torch.empty_like(x), "y": torch.empty_like(y),
                      "ws": ws if j == 0 else moe.Workspace(cfg, dev)})

    def e2e_step(i):
        p = pipes[i % n_pipe]
        moe.layer_forward_host(cfg, p["x_host"], w, p["ws"], p["x"], p["y"], p["y_host"],
                               stream=p["stream"])

    e2e_start = torch.cuda.Event(enable_timing=True)
    e2e_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    for i in range(2 * n_pipe):
        e2e_step(i)
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e2e_start.record(stream)
    for p in pipes:
        p["stream"].wait_event(e2e_start)
    for i in range(args.e2e_steps):
        e2e_step(i)
    for p in pipes:
        stream.wait_stream(p["stream"])
    e2e_end.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e2e_start.elapsed_time(e2e_end) / args.e2e_steps, dev)
    for p in pipes[1:]:
        if moe.moe_get_error(p["ws"]) != 0:
            raise RuntimeError(f"{name}: device status after the end-to-end steps")

    record = None
    if rank == 0:
        # The K-step loop (well under a second) is compared with the burst
        # tensor peak even when the power cap showed in its clock samples;
        # the seconds-long loop above uses the sustained one.
        capped = "sw_power_cap" in clk.get("reasons", [])
        tensor_key = "bf16_tflops"
        roof = roofline(work, stage_ms, peaks, peak_src, tensor_key,
                        "short timed loop" + ("; power cap seen" if capped else ""))
        # counters of a reduced-expert run do not describe the full workload
        roof["traffic"] = None if args.experts else stored_traffic(name, roof["stage"])
        record = {
            "workload": WORKLOAD_TEXT[name], "name": shape.name,
            "value": tokens_per_second(T, world, ms_per_step), "unit": "tokens/s",
            "ms_per_step": ms_per_step, "steps": args.steps, "dtype": shape.dtype,
            **layer_rates(work, ms_per_step, peaks, tensor_key),
            "stage_ms": stage_ms, "roofline": roof, "gpu_launches": launches, "clocks": clk,
            "e2e": {"value": tokens_per_second(T, world, e2e_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": x.numel() * x.element_size(),
                    "d2h_bytes_per_step": y.numel() * y.element_size(),
                    "api": "moe_layer_forward_host", "batches_in_flight": E2E_PIPELINE},
            "sustained": sustained,
            "config": {"workload": WORKLOAD_TEXT[name], "name": shape.name,
                       "global_batch_tokens": world * T, "parallelism": f"replicas x{world}",
                       "l2": "inputs larger than L2: every step streams "
                             f"{work['weight_bytes'] / 1e9:.2f} GB of expert weights "
                             "(L2 126 MB)",
                       "kept_assignments": work["kept"], "touched_experts": work["touched"]},
        }
    cpu_job = None
    if record is not None and world == 1 and not args.no_cpu_baseline:
        def cpu_job(rec=record, shape=shape, inputs=inputs):
            samples = oracle_samples(shape, args.cpu_sample_tokens, args.cpu_steps)
            times, used = timed_oracle(shape, inputs, samples, cache=oracle_cache)
            t = statistics.mean(times)
            rec["cpu_baseline"] = {
                "value": len(samples[0]) / t, "unit": "tokens/s", "cores": used,
                "kind": "oracle",
                "sample": f"{args.cpu_steps} oracle steps, each: routing of all {T} tokens + "
                          f"layer output of {len(samples[0])} sampled tokens (float64; the "
                          "experts they reach widened to float64 before timing)"}
            if name == "tiny":
                # the small layer's single-thread figure beside the all-core one
                times1, _ = timed_oracle(shape, inputs, samples, threads=1, cache=oracle_cache)
                rec["cpu_baseline"]["single_thread_value"] = (len(samples[0]) /
                                                              statistics.mean(times1))
    del pipes, w, ws, x, y
    if cpu_job is None:
        del inputs
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    return record, cpu_job


def reference_main(args, rank, local_rank):
    """The reference arm: the float64 oracle as it stands, timed on the host
    cores on a bounded sample of the headline workload."""
    import torch
    from workloads import make_inputs
    if rank != 0:
        return 0
    if torch.cuda.is_available():
        torch.cuda.set_device(local_rank)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    shape = workload_shape(args.workload, args.experts)
    inputs = make_inputs(shape, device=dev, seed=0)
    samples = oracle_samples(shape, args.cpu_sample_tokens, args.warmup + args.steps)
    times, used = timed_oracle(shape, inputs, samples, args.warmup)
    t = statistics.mean(times)
    m = len(samples[0])
    val = m / t
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * t, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD_TEXT[args.workload], "name": shape.name},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": used, "kind": "oracle",
                             "sample": f"per step: routing of all {shape.T} tokens + layer "
                                       f"output of {m} sampled tokens"},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return reference_main(args, rank, local_rank)

    import torch
    import torch.distributed as dist

    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peaks, peak_src = load_peaks()
    cache = WidenedExperts()

    names = [args.workload] + [n for n in args.per_config.split(",")
                               if n and n != args.workload]
    for n in names:
        if n not in WORKLOAD_TEXT:
            raise SystemExit(f"unknown workload {n!r}")
    records, cpu_jobs = {}, []
    for n in names:
        records[n], job = measure_workload(n, args, dev, world, rank, peaks, peak_src, cache)
        if job is not None:
            cpu_jobs.append(job)
    # the host-side oracle baselines, once the GPU measurements are done
    for job in cpu_jobs:
        job()
    del cpu_jobs

    if rank == 0:
        head = records[args.workload]
        line = {
            "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": head["dtype"],
            "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights)",
            "config": head["config"],
            **{k: head[k] for k in ("tflops", "tensor_peak_frac", "weight_gbs", "hbm_frac",
                                    "stage_ms", "roofline", "gpu_launches", "clocks", "e2e",
                                    "sustained")},
        }
        if "cpu_baseline" in head:
            line["cpu_baseline"] = head["cpu_baseline"]
        line["per_config"] = {n: records[n] for n in names[1:]}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
