#!/usr/bin/env python
"""Benchmark of the recalibrated MoE expert backward on GB300.

One step = one pass of the whole path over one synthetic MoE layer with its
inputs resident in HBM: dispatch permutation, LRM score, quota rule and
per-expert top-q selection, compaction, the four grouped expert-backward
products and the dx scatter (9 kernel launches up to 2^17 routed pairs). The metric is
retained rows per second, M / step time, with M = sum_e q_e the retained
token-expert pairs. The L2 is flushed (a 256 MiB write) before every timed
step, outside the step's CUDA events.

The default layer is the largest single-GPU workload, shaped like
GLM4.5-106B-A12B (T = 16384, D = 4096, H = 1408, E = 128, top-8, BF16); the
headline is its rho = 1/2 point, and the same line carries the whole
retention sweep (rho = 1/4, 1/2, 3/4, 1 at fixed routed pairs N) with a
least-squares fit of step time against the retained rows M, plus one timed
pass of each other workload (``configs``).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
    python bench.py --impl reference ...   # the CPU oracle on a bounded sample

Under torchrun (N > 1) every rank runs an independent replica of the layer
(no collective on the data path); value = rows of all ranks / max time.
Rank 0 prints one JSON line.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "retained-pair expert-backward rows/s; grouped-GEMM % BF16 peak; select GB/s"
DEFAULT_CONFIG = "glm45-106b-a12b-t16k"
# the other workloads timed once each into the line's "configs" table
OTHER_WORKLOADS = ["qwen3-30b-a3b-t4k", "qwen3-30b-a3b-t32k", "stress-e256"]
FLUSH_BYTES = 256 << 20
SEGMENTS = ["dispatch", "score", "select", "compact", "fc2_dgrad", "fc2_wgrad",
            "fc1_wgrad", "fc1_dgrad", "scatter_dx"]
# kernels whose names the launch list shows for each segment
KERNEL_NAMES = {
    "dispatch": "dispatch_fused_kernel",
    "score": "score_kernel", "select": "select_kernel", "compact": "compact_kernel",
    "fc2_dgrad": "grouped_gemm_kernel<0, 1, 0>", "fc2_wgrad": "grouped_gemm_kernel<1, 0, 0>",
    "fc1_wgrad": "grouped_gemm_kernel<2, 0, 0>", "fc1_dgrad": "grouped_gemm_kernel<3, 1, 0>",
    "scatter_dx": "dx_gather_kernel",
}
FUSED_DISPATCH_MAX_PAIRS = 1 << 17  # above it dispatch takes three launches
# the forward expert pass that produces the saved state, timed on its own
FWD_SEGMENTS = ["dispatch", "gather", "fc1_fwd", "fc2_fwd", "combine"]
FWD_KERNEL_NAMES = {
    "dispatch": "dispatch_fused_kernel", "gather": "gather_tokens_kernel",
    "fc1_fwd": "grouped_gemm_kernel<4, 1, 0>", "fc2_fwd": "grouped_gemm_kernel<5, 1, 0>",
    "combine": "combine_kernel",
}


# FC1 dgrad runs on 256 x 512 tiles (third template argument 1) when 2H spans
# at least this many 64-deep K blocks
WIDE_FC1_DGRAD_MIN_KBLOCKS = 32


def segment_kernels(seg: str, cfg, fwd: bool = False) -> str:
    """Kernel name(s) of a segment as the launch list shows them."""
    if seg == "dispatch" and cfg.N > FUSED_DISPATCH_MAX_PAIRS:
        return "dispatch_hist_kernel + dispatch_scan_kernel + dispatch_scatter_kernel"
    if seg == "fc1_dgrad" and not fwd and 2 * cfg.H // 64 >= WIDE_FC1_DGRAD_MIN_KBLOCKS:
        return "grouped_gemm_kernel<3, 1, 1>"
    if seg == "score" and cfg.dtype == "bf16" and cfg.K <= 8:
        # BF16 layers: the instantiation with the fewest 16-byte chunks per lane
        # (GV for a g row, HV for a phi row) that covers the row lengths
        gl, hl = -(-cfg.D // 256), -(-cfg.H // 256)
        for gv in (8, 16):
            for hv in (1, 2, 3, 4, 6):
                if gl <= gv and hl <= hv:
                    return f"score_upfront_kernel<{gv}, {hv}>"
    return (FWD_KERNEL_NAMES if fwd else KERNEL_NAMES)[seg]


def kernels_per_step(N: int) -> int:
    """Launches of one step: dispatch (1 or 3), score, select (with the quota
    rule), compact, four grouped GEMMs, dx scatter."""
    return (1 if N <= FUSED_DISPATCH_MAX_PAIRS else 3) + 8
# source file of each segment's kernel (for the traffic record's freshness check)
KERNEL_SOURCE = {
    "dispatch": "dispatch.cu", "score": "score.cu",
    "select": "select.cu", "compact": "compact.cu", "fc2_dgrad": "gemm_tc.cu",
    "fc2_wgrad": "gemm_tc.cu", "fc1_wgrad": "gemm_tc.cu", "fc1_dgrad": "gemm_tc.cu",
    "scatter_dx": "compact.cu",
}


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--rate", default=None, help="retention rate num/den (default: the "
                    "workload's first rate)")
    ap.add_argument("--override", default="",
                    help="comma-separated shape overrides of the workload, e.g. T=2048,E=16 "
                    "(a scaled variant; the workload name records them)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-forward", action="store_true",
                    help="skip the separate timing of the forward expert pass")
    ap.add_argument("--backward", choices=["compacted", "gathered"], default="gathered",
                    help="compacted: the products read compacted copies of x, [a | b] and "
                    "phi; gathered: compaction writes only the gradient rows and the "
                    "products read the others in place")
    ap.add_argument("--no-other-backward", action="store_true",
                    help="skip timing the step with the other --backward variant")
    ap.add_argument("--index-sweep", action="store_true",
                    help="supplementary: time the dispatch permutation and the selection "
                         "(with the quota rule) alone over routed-pair counts 2^15..2^22 "
                         "and print one JSON line; the headline run is not made")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the retention sweep of a workload that has several rates")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other workloads into the line's configs table")
    ap.add_argument("--no-recompute", action="store_true",
                    help="skip the timing of the backward step that recomputes [a | b]")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic bytes and flops per launch
# ---------------------------------------------------------------------------
def algorithmic(cfg, M: int, gathered: bool = False) -> dict:
    """Bytes (and flops) each segment must move at minimum, per launch
    (gathered: compaction writes only the gradient rows)."""
    T, D, H, E, K = cfg.T, cfg.D, cfg.H, cfg.E, cfg.K
    N = T * K
    s = 2 if cfg.dtype == "bf16" else 4
    W = E * D * H * s  # one expert weight tensor, all experts
    return {
        "dispatch": {"bytes": 4 * N + 8 * N + 8 * E},
        "score": {"bytes": T * D * s + N * H * s + 4 * N + 4 * N + 4 * N},
        "select": {"bytes": 4 * N + N + 4 * M + 24 * E},
        "compact": {"bytes": (2 * M * D * s if gathered else 2 * M * (2 * D + 3 * H) * s)
                    + 4 * M * 4 + 5 * N},
        "fc2_dgrad": {"bytes": M * D * s + W + 2 * (M * 2 * H * s), "flops": 2 * M * D * H},
        "fc2_wgrad": {"bytes": M * H * s + M * D * s + E * H * D * 4, "flops": 2 * M * D * H},
        "fc1_wgrad": {"bytes": M * D * s + M * 2 * H * s + 2 * E * D * H * 4,
                      "flops": 4 * M * D * H},
        "fc1_dgrad": {"bytes": M * 2 * H * s + 2 * W + M * D * 4, "flops": 4 * M * D * H},
        "scatter_dx": {"bytes": M * D * 4 + T * D * 4 + 8 * N},
    }


def algorithmic_fwd(cfg) -> dict:
    """Bytes (and flops) each forward segment must move at minimum, per launch."""
    T, D, H, E, K = cfg.T, cfg.D, cfg.H, cfg.E, cfg.K
    N = T * K
    s = 2 if cfg.dtype == "bf16" else 4
    W = E * D * H * s
    return {
        "dispatch": {"bytes": 4 * N + 8 * N + 8 * E},
        "gather": {"bytes": T * D * s + N * D * s + 4 * N},
        "fc1_fwd": {"bytes": N * D * s + 2 * W + N * 3 * H * s, "flops": 4 * N * D * H},
        "fc2_fwd": {"bytes": N * H * s + W + N * D * s, "flops": 2 * N * D * H},
        "combine": {"bytes": N * D * s + 8 * N + T * D * 4},
    }


def roofline_of(a: dict, ms: float, peaks: dict) -> dict:
    """Bound, achieved and fraction of one kernel from its algorithmic work."""
    t_hbm = a["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = a.get("flops", 0) / (peaks["bf16_tflops"] * 1e12)
    if t_tc > t_hbm:
        achieved = a["flops"] / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1),
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    else:
        achieved = a["bytes"] / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
    roof["frac"] = round(achieved / roof["peak"], 4)
    return roof


def roofline_time_ms(a: dict, peaks: dict) -> float:
    """The least time a segment could take: its algorithmic bytes at the
    measured copy bandwidth or its flops at the measured BF16 peak, whichever
    is longer."""
    t_hbm = a["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = a.get("flops", 0) / (peaks["bf16_tflops"] * 1e12)
    return max(t_hbm, t_tc) * 1e3


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": float(pk["hbm_gbs"]), "bf16_tflops": float(pk["bf16_tflops"]),
                "bf16_tflops_sustained": float(pk.get("bf16_tflops_sustained",
                                                      pk["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def source_sha(fname: str) -> str:
    p = os.path.join(ROOT, "demand_side_expert_gb300", "csrc", fname)
    with open(p, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:12]


def load_traffic(workload: str) -> dict:
    """DRAM bytes per launch recorded from ncu, keyed by segment, fresh only."""
    out = {}
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return out
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            seg, wl, sha, nbytes = line.split()[:4]
            if wl == workload and seg in KERNEL_SOURCE and sha == source_sha(KERNEL_SOURCE[seg]):
                out[seg] = int(nbytes)
    return out


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# our path
# ---------------------------------------------------------------------------
def aggregate_ranks(time_s: float, rows: int, device, dist=None):
    """(max time over ranks, rows summed over ranks); replicas, weak scaling."""
    if dist is None:
        return time_s, float(rows)
    import torch

    t = torch.tensor([time_s, float(rows)], dtype=torch.float64, device=device)
    tmax = t.clone()
    dist.all_reduce(tmax, op=dist.ReduceOp.MAX)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(tmax[0]), float(t[1])


def workload_of(args):
    from workloads import get_config

    over = {}
    for item in filter(None, args.override.split(",")):
        k, v = item.split("=")
        over[k.strip()] = int(v)
    cfg = get_config(args.config, **over)
    if over:
        tag = ",".join(f"{k}={v}" for k, v in sorted(over.items()))
        cfg = type(cfg)(**{**cfg.__dict__, "name": f"{cfg.name}[{tag}]"})
    return cfg


def headline_rate(cfg, args):
    """The retention rate of the headline line: --rate, else the middle of a
    retention sweep (rho = 1/2 on the GLM-shaped layer), else the workload's rate."""
    if args.rate:
        return tuple(int(v) for v in args.rate.split("/"))
    if (1, 2) in cfg.rates:
        return (1, 2)
    return cfg.rates[0]


def make_step(pipe, inp, ab, phi, rate, cfg, stream, gathered):
    """One step of the whole path as a function of a list of events: with
    seg=False only its first and last events are recorded, so consecutive
    kernels overlap as they do without timing."""
    from demand_side_expert_gb300 import lrm

    def step(ev, seg=True):
        def mark(j):
            if seg or j == 0 or j == len(SEGMENTS):
                ev[j].record(stream)

        mark(0)
        pipe.dispatch(inp["topk_idx"])
        mark(1)
        pipe.score_pairs(inp["alpha"], inp["g"], phi)
        mark(2)
        pipe.select_rate(rate[0], rate[1], cfg.cap)
        mark(3)
        pipe.compact(inp["alpha"], inp["x"], inp["g"], ab, phi, gathered=gathered)
        mark(4)
        if gathered:  # the products read x, ab and phi rows in place
            for j, part in enumerate((lrm.LRM_BWD_FC2_DGRAD, lrm.LRM_BWD_FC2_WGRAD,
                                      lrm.LRM_BWD_FC1_WGRAD, lrm.LRM_BWD_FC1_DGRAD,
                                      lrm.LRM_BWD_SCATTER_DX)):
                pipe.expert_bwd_gathered(inp["x"], ab, phi, inp["w_gate"], inp["w_up"],
                                         inp["w_down"], parts=part)
                mark(5 + j)
            return
        pipe.fc2_dgrad(inp["w_down"])
        mark(5)
        pipe.fc2_wgrad()
        mark(6)
        pipe.fc1_wgrad()
        mark(7)
        pipe.fc1_dgrad(inp["w_gate"], inp["w_up"])
        mark(8)
        pipe.scatter_dx()
        mark(9)

    return step


def time_layer(pipe, inp, ab, phi, rate, cfg, flush, stream, steps, warmup, gathered,
               dist=None):
    """Warm-up, then `steps` headline steps (events at their two ends only,
    the L2 flushed before each, outside the events), then a second pass of
    `steps` steps with an event between every call for the per-segment
    times. Returns the retained rows and the times in ms."""
    import torch

    step = make_step(pipe, inp, ab, phi, rate, cfg, stream, gathered)
    dev = pipe.device

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(len(SEGMENTS) + 1)]

    for _ in range(max(warmup, 0)):
        flush.fill_(1)
        step(new_events())
    torch.cuda.synchronize(dev)
    if pipe.device_error() != 0:
        raise RuntimeError(f"device error word {pipe.device_error()} after warm-up")
    M = pipe.retained_rows
    events = [new_events() for _ in range(steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(steps):
        flush.fill_(1)  # L2 flush outside the step's events
        step(events[i], seg=False)
    torch.cuda.synchronize(dev)
    if dist:
        dist.barrier()
    wall = time.perf_counter() - wall0
    seg_events = [new_events() for _ in range(steps)]
    for i in range(steps):
        flush.fill_(1)
        step(seg_events[i], seg=True)
    torch.cuda.synchronize(dev)
    if pipe.device_error() != 0:
        raise RuntimeError(f"device error word {pipe.device_error()} after timing")
    seg_ms = {s: [ev[j].elapsed_time(ev[j + 1]) for ev in seg_events]
              for j, s in enumerate(SEGMENTS)}
    return {"M": M, "step_ms": [ev[0].elapsed_time(ev[-1]) for ev in events],
            "seg_ms": seg_ms,
            "seg_step_ms": statistics.mean(ev[0].elapsed_time(ev[-1]) for ev in seg_events),
            "wall": wall}


# HBM-bound segments that also get a size-matched copy: the same bytes moved by
# a plain device-to-device copy (half read, half written), timed the same way
COPY_MATCHED = ("score", "compact", "scatter_dx")


def size_matched_copies(cfg, M: int, gathered: bool, flush, stream, reps: int = 10) -> dict:
    """For each segment in COPY_MATCHED: the mean time of a device-to-device
    copy that moves that segment's algorithmic bytes, with the L2 flushed
    before each copy and CUDA events around the copy alone. The measured copy
    peak is taken on gigabytes; a launch that moves tens of megabytes spends a
    visible share of its time in launch, ramp-up and drain, which this copy
    shows at the segment's own size."""
    import torch

    alg = algorithmic(cfg, M, gathered)
    out = {}
    for seg in COPY_MATCHED:
        nbytes = alg[seg]["bytes"]
        half = max(16, (nbytes // 2) // 16 * 16)
        src = torch.ones(half, dtype=torch.uint8, device=flush.device)
        dst = torch.empty_like(src)
        times = []
        with torch.cuda.stream(stream):
            for i in range(reps + 3):
                flush.fill_(1)
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dst.copy_(src)
                e1.record(stream)
                e1.synchronize()
                if i >= 3:
                    times.append(e0.elapsed_time(e1))
        ms = statistics.mean(times)
        out[seg] = {"bytes": 2 * half, "ms": round(ms, 4),
                    "gbs": round(2 * half / (ms * 1e-3) / 1e9, 1)}
        del src, dst
    return out


def attach_copies(summary: dict, copies: dict) -> None:
    for seg, c in copies.items():
        k = summary["kernels"][seg]
        k["size_matched_copy"] = c
        k["frac_size_matched_copy"] = round(k["gbs"] / c["gbs"], 4) if c["gbs"] else None


def largest_segment(pipe) -> int:
    return int(pipe.counts.max().item()) if pipe.E else 0


def layer_summary(cfg, rate, t: dict, peaks: dict, gathered: bool, n_max: int) -> dict:
    """Per-kernel times, GB/s and TFLOP/s, the dominant kernel's roofline and
    the grouped products' totals of one timed layer."""
    M = t["M"]
    seg_ms = t["seg_ms"]
    alg = algorithmic(cfg, M, gathered)
    traffic = load_traffic(cfg.name)
    kernels = {}
    for s in SEGMENTS:
        ms = statistics.mean(seg_ms[s])
        k = {"ms": round(ms, 4), "kernels": segment_kernels(s, cfg),
             "gbs": round(alg[s]["bytes"] / (ms * 1e-3) / 1e9, 1),
             "frac_hbm": round(alg[s]["bytes"] / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4)}
        if "flops" in alg[s]:
            k["tflops"] = round(alg[s]["flops"] / (ms * 1e-3) / 1e12, 1)
            k["frac_bf16"] = round(alg[s]["flops"] / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"],
                                   4)
        if s in traffic:  # DRAM bytes of one launch from an ncu capture of this build
            k["dram_bytes"] = traffic[s]
            k["dram_gbs"] = round(traffic[s] / (ms * 1e-3) / 1e9, 1)
        kernels[s] = k
    # the selection is one CTA per expert: its time is set by the largest
    # segment, not by bytes (latency-bound)
    kernels["select"]["us"] = round(1e3 * kernels["select"]["ms"], 2)
    kernels["select"]["bound"] = "latency (one CTA per expert; the largest segment sets it)"
    kernels["select"]["largest_segment"] = n_max
    if "dram_bytes" not in kernels["compact"]:
        kernels["compact"]["dram_bytes"] = None
    kernels["compact"]["note"] = (
        "gbs counts the algorithmic bytes (a token's g row once per retained pair); "
        "dram_gbs counts the DRAM bytes ncu measured for one launch (g rows re-read from L2)")
    dominant = max(SEGMENTS, key=lambda s: statistics.mean(seg_ms[s]))
    a = alg[dominant]
    roof = roofline_of(a, statistics.mean(seg_ms[dominant]), peaks)
    roof["traffic"] = traffic.get(dominant)
    roof["kernel"] = segment_kernels(dominant, cfg)
    roof["algorithmic_bytes"] = a["bytes"]
    if "flops" in a:
        roof["algorithmic_flops"] = a["flops"]
    roof["peak_source"] = f"{peaks['source']} (MEASURED_PEAKS.json burst)" \
        if peaks["source"] == "measured" else "fallback"
    gemm = ["fc2_dgrad", "fc2_wgrad", "fc1_wgrad", "fc1_dgrad"]
    gemm_ms = sum(statistics.mean(seg_ms[s]) for s in gemm)
    gemm_flops = sum(alg[s]["flops"] for s in gemm)
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12
    ms = statistics.mean(t["step_ms"])
    return {
        "rho": f"{rate[0]}/{rate[1]}", "retained_rows": M, "ms_per_step": round(ms, 4),
        "rows_per_s": round(M / (ms * 1e-3), 1),
        "ms_per_step_with_segment_events": round(t["seg_step_ms"], 4),
        "grouped_gemm_tflops": round(gemm_tflops, 1),
        "grouped_gemm_pct_bf16_peak": round(100 * gemm_tflops / peaks["bf16_tflops"], 2),
        # the four products' summed roofline times over their summed measured times
        # (each product bound by HBM or the tensor pipe, whichever is slower)
        "grouped_gemm_roofline_frac": round(
            sum(roofline_time_ms(alg[s], peaks) for s in gemm) / gemm_ms, 4),
        "select_gbs": round(alg["select"]["bytes"] / (kernels["select"]["ms"] * 1e-3) / 1e9, 1),
        "kernels": kernels, "roofline": roof,
    }


def linear_fit(xs, ys) -> dict:
    """Least-squares line y = a + b x with R^2 and the largest residual."""
    n = len(xs)
    mx, my = sum(xs) / n, sum(ys) / n
    sxx = sum((x - mx) ** 2 for x in xs)
    b = sum((x - mx) * (y - my) for x, y in zip(xs, ys)) / sxx if sxx else 0.0
    a = my - b * mx
    res = [y - (a + b * x) for x, y in zip(xs, ys)]
    sst = sum((y - my) ** 2 for y in ys)
    r2 = 1.0 - sum(r * r for r in res) / sst if sst else 1.0
    return {"a": a, "b": b, "r2": r2, "max_abs_residual": max(abs(r) for r in res)}


def sweep_summary(cfg, points: list, peaks: dict) -> dict:
    """Step time against retained rows M over a retention sweep at fixed N."""
    fit = linear_fit([p["retained_rows"] for p in points], [p["ms_per_step"] for p in points])
    s = 2 if cfg.dtype == "bf16" else 4
    fixed_bytes = 3 * cfg.E * cfg.D * cfg.H * (s + 4)  # weights in, FP32 weight gradients out
    return {
        "routed_pairs": cfg.N,
        "points": points,
        "fit": {"model": "ms_per_step = intercept_ms + ns_per_retained_row * M / 1e6",
                "intercept_ms": round(fit["a"], 4),
                "ns_per_retained_row": round(fit["b"] * 1e6, 3),
                "r2": round(fit["r2"], 5),
                "max_abs_residual_us": round(fit["max_abs_residual"] * 1e3, 1)},
        "intercept_reading": {
            "weights_in_and_fp32_weight_gradients_out_bytes": fixed_bytes,
            "their_time_at_measured_hbm_ms": round(fixed_bytes / (peaks["hbm_gbs"] * 1e9) * 1e3,
                                                   4)},
    }


def prepare_layer(cfg, dev, seed):
    """Generate one layer, allocate its buffers and lay out the saved state in
    dispatch order (the forward side, done once, not timed)."""
    from demand_side_expert_gb300 import RecalibratedExpertBackward
    from workloads import generate

    inp = generate(cfg, device=dev, seed=seed)
    pipe = RecalibratedExpertBackward(cfg.T, cfg.D, cfg.H, cfg.E, cfg.K, cfg.dtype, dev)
    pipe.dispatch(inp["topk_idx"])
    ab = pipe.to_dispatch_order(inp["ab_pair"])
    phi = pipe.to_dispatch_order(inp["phi_pair"])
    del inp["ab_pair"], inp["phi_pair"]
    return inp, pipe, ab, phi


def run_ours(args, rank: int, world: int, local_rank: int):
    import torch

    from workloads import get_config

    gathered = args.backward == "gathered"
    dist = None
    if world > 1:
        import torch.distributed as dist

    cfg = workload_of(args)
    rate = headline_rate(cfg, args)
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    inp, pipe, ab, phi = prepare_layer(cfg, dev, cfg.seed + rank)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    clocks = ClockSampler(local_rank)
    clocks.start()
    t = time_layer(pipe, inp, ab, phi, rate, cfg, flush, stream, args.steps, args.warmup,
                   gathered, dist)
    n_max = largest_segment(pipe)
    M = t["M"]
    copies = size_matched_copies(cfg, M, gathered, flush, stream)
    total_s = sum(t["step_ms"]) / 1e3
    total_max, rows_sum = aggregate_ranks(total_s, M * args.steps, dev, dist)
    peaks = load_peaks()

    # the retention sweep of a layer that has one: same N, growing M
    sweep = None
    if len(cfg.rates) > 1 and not args.no_sweep and not args.rate:
        points = []
        for r in cfg.rates:
            tr = t if r == rate else time_layer(pipe, inp, ab, phi, r, cfg, flush, stream,
                                                args.steps, args.warmup, gathered)
            sm = layer_summary(cfg, r, tr, peaks, gathered, n_max)
            points.append({k: sm[k] for k in (
                "rho", "retained_rows", "ms_per_step", "rows_per_s",
                "grouped_gemm_tflops", "grouped_gemm_pct_bf16_peak",
                "grouped_gemm_roofline_frac", "select_gbs")}
                | {"segments_ms": {s: sm["kernels"][s]["ms"] for s in SEGMENTS},
                   "score_frac_hbm": sm["kernels"]["score"]["frac_hbm"],
                   "compact_frac_hbm": sm["kernels"]["compact"]["frac_hbm"]})
        sweep = sweep_summary(cfg, points, peaks)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(pipe, inp, ab, phi, rate, cfg, flush, stream, args)
    fwd = None
    if not args.no_forward:
        fwd = run_forward(pipe, inp, cfg, flush, stream, args)
    rec = None
    if not args.no_recompute:
        rec = run_recompute(pipe, inp, phi, rate, cfg, flush, stream, args)
    other = None
    if not args.no_other_backward:
        other = run_other_backward(pipe, inp, ab, phi, rate, cfg, flush, stream, args)

    # the other workloads, one pass each with the same timing and L2 flush
    others = None
    if not args.no_configs and not args.override:
        del pipe, inp, ab, phi
        torch.cuda.empty_cache()
        others = {}
        for name in OTHER_WORKLOADS:
            if name == cfg.name:
                continue
            ocfg = get_config(name)
            orate = ocfg.rates[0]
            oinp, opipe, oab, ophi = prepare_layer(ocfg, dev, ocfg.seed + rank)
            ot = time_layer(opipe, oinp, oab, ophi, orate, ocfg, flush, stream, args.steps,
                            args.warmup, gathered)
            sm = layer_summary(ocfg, orate, ot, peaks, gathered, largest_segment(opipe))
            attach_copies(sm, size_matched_copies(ocfg, ot["M"], gathered, flush, stream))
            sm["workload"] = ocfg.name
            sm["T"], sm["D"], sm["H"], sm["E"], sm["K"] = ocfg.T, ocfg.D, ocfg.H, ocfg.E, ocfg.K
            sm["quota_cap"] = ocfg.cap
            sm["gpu_launches"] = kernels_per_step(ocfg.N) * 2 * args.steps
            others[name] = sm
            del oinp, opipe, oab, ophi
            torch.cuda.empty_cache()
    clk = clocks.stop()

    if rank != 0:
        return None

    head = layer_summary(cfg, rate, t, peaks, gathered, n_max)
    attach_copies(head, copies)
    line = {
        "metric": METRIC,
        "value": round(rows_sum / total_max, 1),
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_max * 1e3 / args.steps, 4),
        "ms_per_step_with_segment_events": head["ms_per_step_with_segment_events"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": cfg.dtype,
        "data": "synthetic (seeded router, SwiGLU forward state and cotangents)",
        "config": {
            "workload": f"{cfg.name} rho={rate[0]}/{rate[1]}", "layer": cfg.name,
            "T": cfg.T, "D": cfg.D, "H": cfg.H, "E": cfg.E, "K": cfg.K,
            "rho": f"{rate[0]}/{rate[1]}", "quota_cap": cfg.cap, "routed_pairs": cfg.N,
            "retained_rows": M, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
            "l2": "flushed by a 256 MiB write before every timed step (outside the events)",
            "inputs": "resident in HBM",
            "backward": args.backward,
        },
        "grouped_gemm_pct_bf16_peak": head["grouped_gemm_pct_bf16_peak"],
        "grouped_gemm_tflops": head["grouped_gemm_tflops"],
        "grouped_gemm_roofline_frac": head["grouped_gemm_roofline_frac"],
        "select_gbs": head["select_gbs"],
        "kernels": head["kernels"],
        "roofline": head["roofline"],
        # headline steps and the segmented pass over them
        "gpu_launches": kernels_per_step(cfg.N) * 2 * args.steps,
        "clocks": clk,
        "wall_s": round(t["wall"], 4),
    }
    if sweep is not None:
        line["rho_sweep"] = sweep
    if e2e is not None:
        line["e2e"] = e2e
    if fwd is not None:
        line["forward"] = fwd
    if rec is not None:
        line["recompute"] = rec
    if other is not None:
        line["other_backward"] = other
    if others:
        line["configs"] = others
    return line, cfg, rate


def run_other_backward(pipe, inp, ab, phi, rate, cfg, flush, stream, args):
    """The whole step again with the other backward variant (compacted copies
    vs in-place gathers), timed the same way, so both stand side by side."""
    import torch

    gathered = args.backward != "gathered"

    def step():
        pipe.step(inp["topk_idx"], inp["alpha"], inp["x"], inp["g"], ab, phi, inp["w_gate"],
                  inp["w_up"], inp["w_down"], rate=rate, cap=cfg.cap, gathered=gathered)

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for a, b in evs:
        flush.fill_(1)
        a.record(stream)
        step()
        b.record(stream)
    torch.cuda.synchronize()
    if pipe.device_error() != 0:
        raise RuntimeError(f"device error word {pipe.device_error()} in the other backward")
    ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    return {"backward": "gathered" if gathered else "compacted",
            "value": round(pipe.retained_rows / (ms * 1e-3), 1), "unit": "rows/s",
            "ms_per_step": round(ms, 4), "steps": args.steps}


def run_recompute(pipe, inp, phi, rate, cfg, flush, stream, args):
    """The same backward step without saved [a | b]: compaction copies no
    [a | b] rows and the gate/up product rebuilds them for the retained rows
    only (lrm_expert_fc1_recompute), then the four products and the scatter.
    Timed like the headline step; reported beside it."""
    import torch

    def step(ev):
        ev[0].record(stream)
        pipe.dispatch(inp["topk_idx"])
        pipe.score_pairs(inp["alpha"], inp["g"], phi)
        pipe.select_rate(rate[0], rate[1], cfg.cap)
        pipe.compact(inp["alpha"], inp["x"], inp["g"], None, phi)
        ev[1].record(stream)
        pipe.fc1_recompute(inp["w_gate"], inp["w_up"])
        ev[2].record(stream)
        pipe.expert_bwd(inp["w_gate"], inp["w_up"], inp["w_down"])
        ev[3].record(stream)

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(4)]

    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step(new_events())
    torch.cuda.synchronize()
    events = [new_events() for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(1)
        step(events[i])
    torch.cuda.synchronize()
    if pipe.device_error() != 0:
        raise RuntimeError(f"device error word {pipe.device_error()} in the recompute step")
    M = pipe.retained_rows
    ms = statistics.mean(ev[0].elapsed_time(ev[-1]) for ev in events)
    rec_ms = statistics.mean(ev[1].elapsed_time(ev[2]) for ev in events)
    s = 2 if cfg.dtype == "bf16" else 4
    a = {"bytes": M * cfg.D * s + 2 * cfg.E * cfg.D * cfg.H * s + M * 2 * cfg.H * s,
         "flops": 4 * M * cfg.D * cfg.H}
    roof = roofline_of(a, rec_ms, load_peaks())
    roof["kernel"] = FWD_KERNEL_NAMES["fc1_fwd"]
    return {"metric": "retained rows through the backward step per second, [a | b] recomputed",
            "value": round(M / (ms * 1e-3), 1), "unit": "rows/s", "ms_per_step": round(ms, 4),
            "steps": args.steps, "saved_state_bytes_avoided": cfg.N * 2 * cfg.H * s,
            "recompute_ms": round(rec_ms, 4), "recompute_roofline": roof,
            "gpu_launches": (kernels_per_step(cfg.N) + 1) * args.steps}


def run_forward(pipe, inp, cfg, flush, stream, args):
    """The forward expert pass that produces the saved state (dispatch, token
    gather, gate/up products with the SwiGLU epilogue, down products, combine)
    timed on its own with the same L2 flush and CUDA events. Reported beside
    the backward line; it is not part of the step the headline times."""
    import torch

    def step(ev):
        ev[0].record(stream)
        pipe.dispatch(inp["topk_idx"])
        ev[1].record(stream)
        pipe.gather_tokens(inp["x"])
        ev[2].record(stream)
        pipe.fc1_fwd(inp["w_gate"], inp["w_up"])
        ev[3].record(stream)
        pipe.fc2_fwd(inp["w_down"])
        ev[4].record(stream)
        pipe.combine(inp["alpha"])
        ev[5].record(stream)

    def new_events():
        return [torch.cuda.Event(enable_timing=True) for _ in range(len(FWD_SEGMENTS) + 1)]

    pipe.gather_tokens(inp["x"])  # allocates the forward buffers
    for _ in range(max(args.warmup, 3)):
        flush.fill_(1)
        step(new_events())
    torch.cuda.synchronize()
    events = [new_events() for _ in range(args.steps)]
    for i in range(args.steps):
        flush.fill_(1)
        step(events[i])
    torch.cuda.synchronize()
    if pipe.device_error() != 0:
        raise RuntimeError(f"device error word {pipe.device_error()} in the forward")
    seg = {s: statistics.mean(ev[j].elapsed_time(ev[j + 1]) for ev in events)
           for j, s in enumerate(FWD_SEGMENTS)}
    ms = statistics.mean(ev[0].elapsed_time(ev[-1]) for ev in events)
    alg = algorithmic_fwd(cfg)
    peaks = load_peaks()
    kernels = {}
    for s in FWD_SEGMENTS:
        k = {"ms": round(seg[s], 4), "kernels": segment_kernels(s, cfg, fwd=True),
             "gbs": round(alg[s]["bytes"] / (seg[s] * 1e-3) / 1e9, 1)}
        if "flops" in alg[s]:
            k["tflops"] = round(alg[s]["flops"] / (seg[s] * 1e-3) / 1e12, 1)
        kernels[s] = k
    dominant = max(FWD_SEGMENTS, key=lambda s: seg[s])
    roof = roofline_of(alg[dominant], seg[dominant], peaks)
    roof["kernel"] = FWD_KERNEL_NAMES[dominant]
    roof["traffic"] = None
    return {"metric": "routed rows through the forward expert pass per second",
            "value": round(cfg.N / (ms * 1e-3), 1), "unit": "rows/s",
            "ms_per_step": round(ms, 4), "steps": args.steps,
            "gpu_launches": (len(FWD_SEGMENTS) - 1 + (1 if cfg.N <= FUSED_DISPATCH_MAX_PAIRS
                                                      else 3)) * args.steps,
            "kernels": kernels, "roofline": roof}


def run_e2e(pipe, inp, ab, phi, rate, cfg, flush, stream, args):
    """Same metric through the public calls with host buffers: every step
    copies its inputs (routing, activations, cotangents, saved state) in from
    pinned host memory, runs the C-ABI calls, and copies its result -- dx, the
    input gradient handed to the layer below -- back to pinned host memory,
    all inside the timed region. Steps are pipelined the way a training loop
    would run them: two device input slots and two dx buffers, the host->device
    copies of step i+1 on one copy stream and the dx copy of step i on another,
    both overlapping step i's kernels on the compute stream (events order each
    slot's reuse). The weight gradients stay in HBM for the optimizer (the
    pages' CPU offload queue is not part of this path). Each step's inputs
    (185 MB on the default layer) are larger than the 129 MB L2, and its
    working set (weights and gradients) is several GB, so no flush is added."""
    import torch

    gathered = args.backward == "gathered"
    names = ("topk_idx", "alpha", "x", "g")
    host_in = {k: inp[k].cpu().pin_memory() for k in names}
    host_in["ab"] = ab.cpu().pin_memory()
    host_in["phi"] = phi.cpu().pin_memory()
    slot0 = {k: inp[k] for k in names}
    slot0["ab"], slot0["phi"] = ab, phi
    slots = [slot0, {k: torch.empty_like(v) for k, v in slot0.items()}]
    dx_bufs = [pipe.dx, torch.empty_like(pipe.dx)]
    host_dx = torch.empty(pipe.dx.shape, dtype=torch.float32, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_dx.numel() * host_dx.element_size()
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # slot s filled
    ev_done = [torch.cuda.Event() for _ in range(2)]   # step on slot s finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # dx buffer s copied out

    def issue(i):
        s = i % 2
        with torch.cuda.stream(h2d_stream):
            if i >= 2:
                h2d_stream.wait_event(ev_done[s])  # the step that read slot s is done
            for k, h in host_in.items():
                slots[s][k].copy_(h, non_blocking=True)
            ev_in[s].record(h2d_stream)
        stream.wait_event(ev_in[s])
        if i >= 2:
            stream.wait_event(ev_out[s])  # dx buffer s copied out two steps ago
        pipe.dx = dx_bufs[s]
        d = slots[s]
        pipe.step(d["topk_idx"], d["alpha"], d["x"], d["g"], d["ab"], d["phi"], inp["w_gate"],
                  inp["w_up"], inp["w_down"], rate=rate, cap=cfg.cap, gathered=gathered)
        ev_done[s].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(ev_done[s])
            host_dx.copy_(dx_bufs[s], non_blocking=True)
            ev_out[s].record(d2h_stream)

    steps = max(2, min(args.steps, 20))
    for i in range(4):  # warm-up, both slots
        issue(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        issue(i)
    stream.wait_event(ev_out[(steps - 1) % 2])
    e1.record(stream)
    e1.synchronize()
    tot = e0.elapsed_time(e1) / 1e3
    # the pipelined steps returned what a plain step on resident inputs gives
    pipe.dx = dx_bufs[0]
    d = slots[0]
    pipe.step(d["topk_idx"], d["alpha"], d["x"], d["g"], d["ab"], d["phi"], inp["w_gate"],
              inp["w_up"], inp["w_down"], rate=rate, cap=cfg.cap, gathered=gathered)
    torch.cuda.synchronize()
    if not torch.equal(host_dx, pipe.dx.cpu()):
        raise RuntimeError("pipelined end-to-end steps returned a different dx")
    M = pipe.retained_rows
    return {"value": round(M * steps / tot, 1), "unit": "rows/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(tot * 1e3 / steps, 3),
            "path": "pinned host -> HBM copies of each step's inputs (copy stream), the C-ABI "
                    "calls (compute stream), HBM -> pinned host copy of dx (second copy "
                    "stream); consecutive steps overlap through two input slots"}


# ---------------------------------------------------------------------------
# the CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_sample(cfg, rate, T_s: int, seed: int):
    """The first T_s tokens of the workload, as float64/int64 host arrays."""
    import numpy as np
    import torch

    from workloads import generate, with_tokens

    small = with_tokens(cfg, T_s) if T_s < cfg.T else cfg
    inp = generate(small, device="cuda" if torch.cuda.is_available() else "cpu", seed=seed)

    def f64(t):
        t = t.detach().cpu()
        return (t.float() if t.dtype == torch.bfloat16 else t).numpy().astype(np.float64)

    arrs = {k: f64(inp[k]) for k in ("alpha", "x", "g", "w_gate", "w_up", "w_down",
                                      "ab_pair", "phi_pair")}
    arrs["topk_idx"] = inp["topk_idx"].cpu().numpy().astype(np.int64)
    return small, arrs


def oracle_step(small, rate, a):
    import oracle

    out = oracle.recalibrated_backward(
        a["topk_idx"], a["alpha"], a["x"], a["g"], a["ab_pair"], a["phi_pair"], a["w_gate"],
        a["w_up"], a["w_down"], E=small.E, num=rate[0], den=rate[1], cap=small.cap)
    return int(out["sel_off"][-1])


def cpu_baseline(cfg, rate, T_s: int):
    small, a = oracle_sample(cfg, rate, T_s, cfg.seed)
    warm, aw = oracle_sample(cfg, rate, 16, cfg.seed + 1)
    oracle_step(warm, rate, aw)  # BLAS thread pool start-up, outside the timing
    t0 = time.perf_counter()
    M = oracle_step(small, rate, a)
    dt = time.perf_counter() - t0
    whole = "the whole workload" if small.T == cfg.T else \
        f"a {small.T}-token layer of {cfg.name}'s recipe (same D, H, E, K, rho)"
    return {"value": round(M / dt, 2), "unit": "rows/s", "cores": os.cpu_count(),
            "kind": "oracle",
            "sample": f"{whole}: whole path once, {M} retained rows in {dt:.1f} s; "
                      f"float64 NumPy (BLAS threads on all host cores)"}


def oracle_tokens(cfg, rate, seconds: float) -> int:
    """Tokens whose oracle pass takes about ``seconds`` on the host: a fixed
    part (first touch of the float64 weight-gradient buffers, 3*E*D*H*8
    bytes, at about 16 GB/s) plus 12*D*H float64 flops per retained row at
    about 250 GFLOP/s (NumPy's BLAS on 16 Arm cores, as measured)."""
    fixed = 3.0 * cfg.E * cfg.D * cfg.H * 8 / 1.6e10
    rows = max(seconds - fixed, 0.5) * 2.5e11 / (12.0 * cfg.D * cfg.H)
    tokens = int(rows / (cfg.K * rate[0] / rate[1] if rate[0] else cfg.K))
    return max(16, min(cfg.T, tokens))


def run_reference(args, rank: int):
    if rank != 0:
        return None
    cfg = workload_of(args)
    rate = headline_rate(cfg, args)
    per_step = 150.0 / max(1, args.steps + args.warmup)  # whole run within a few minutes
    small, a = oracle_sample(cfg, rate, oracle_tokens(cfg, rate, per_step), cfg.seed)
    for _ in range(max(args.warmup, 0)):
        oracle_step(small, rate, a)
    t0 = time.perf_counter()
    M = 0
    for _ in range(args.steps):
        M += oracle_step(small, rate, a)
    dt = time.perf_counter() - t0
    value = round(M / dt, 2)
    return {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3 / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name} rho={rate[0]}/{rate[1]}", "layer": cfg.name,
                   "T": cfg.T, "D": cfg.D, "H": cfg.H, "E": cfg.E, "K": cfg.K,
                   "rho": f"{rate[0]}/{rate[1]}", "sampled_tokens": small.T},
        "cpu_baseline": {"value": value, "unit": "rows/s", "cores": os.cpu_count(),
                         "kind": "oracle",
                         "sample": f"a {small.T}-token layer of {cfg.name}'s recipe per "
                                   f"step (same D, H, E, K, rho)"},
        "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_index_sweep(args):
    """The latency-bound index steps at growing N = T*K (K = 8, E = 128, zipf-skewed
    routing, rho = 1/2, random scores), each timed alone with CUDA events (L2 flushed
    before every launch): dispatch, selection with the quota rule, and the standalone
    quota rule. GB/s counts the algorithmic bytes: dispatch 4N + 16N + 8E, selection
    4N + N + 4M + 16E."""
    import torch
    from demand_side_expert_gb300 import lrm

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    E, K, num, den = 128, 8, 1, 2
    gen = torch.Generator(device=dev).manual_seed(0)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    probs = 1.0 / torch.arange(1, E + 1, device=dev, dtype=torch.float64) ** 1.2
    points = []
    for log_n in range(15, 23):
        N = 1 << log_n
        T = N // K
        shape = lrm.make_shape(T, 64, 64, E, K, lrm.LRM_BF16)
        ws_bytes = lrm.lrm_workspace_bytes(shape)
        ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
        topk = torch.multinomial(probs.float().expand(T, E), K, replacement=False,
                                 generator=gen).to(torch.int32)
        i32 = dict(dtype=torch.int32, device=dev)
        perm, inv = torch.empty(N, **i32), torch.empty(N, **i32)
        counts, off, quota = torch.empty(E, **i32), torch.empty(E + 1, **i32), torch.empty(E, **i32)
        score = torch.rand(N, generator=gen, device=dev)
        keep = torch.empty(N, dtype=torch.uint8, device=dev)
        sel_off, sel_pos = torch.empty(E + 1, **i32), torch.empty(N, **i32)
        calls = {
            "dispatch": lambda: lrm.lrm_dispatch_permute(shape, topk, perm, inv, counts, off,
                                                         ws, ws_bytes, None),
            "select": lambda: lrm.lrm_select_rate(shape, score, off, num, den, 0, quota, keep,
                                                  sel_off, sel_pos, ws, ws_bytes, None),
            # the standalone quota rule (the step folds it into the selection)
            "quota": lambda: lrm.lrm_quota_from_rate(counts, E, num, den, 0, quota, None),
        }
        point = {"N": N}
        for name, fn in calls.items():
            for _ in range(max(args.warmup, 3)):
                fn()
            times = []
            for _ in range(20):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            point[name + "_us"] = round(statistics.median(times) * 1e3, 2)
        M = int(sel_off[-1].item())
        point["M"] = M
        point["dispatch_gbs"] = round((20 * N + 8 * E) / (point["dispatch_us"] * 1e3), 1)
        point["select_gbs"] = round((5 * N + 4 * M + 16 * E) / (point["select_us"] * 1e3), 1)
        code = lrm.lrm_get_device_error(ws, ws_bytes)
        if code:
            raise RuntimeError(f"device error word {code} at N = {N}")
        points.append(point)
    return {"metric": "index steps alone over routed pairs N (supplementary sweep)",
            "unit": "GB/s", "data": "synthetic (zipf 1.2 routing over 128 experts, K = 8, "
            "rho = 1/2, uniform random scores)", "points": points}


def main():
    args = parse_args()
    if args.index_sweep:
        print(json.dumps(run_index_sweep(args)), flush=True)
        return
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    out = run_ours(args, rank, world, local_rank)
    if out is not None:
        line, cfg, rate = out
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(cfg, rate, oracle_tokens(cfg, rate, 15.0))
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
