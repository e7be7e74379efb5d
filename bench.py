#!/usr/bin/env python
"""Throughput of the W8A8 MoE layer on GB300, one JSON line on stdout.

    python bench.py [--gpus N --steps K --warmup W] [--config prefill|decode|wide|tiny|linear]
    python bench.py --impl reference ...      # the CPU oracle on the host cores

A step is one forward of the whole layer (router, top-k, permutation,
per-token quantisation, GEMM1 + SiLU epilogue, requantisation, GEMM2,
combine) over one batch of seeded synthetic input already resident in HBM.
The default workload is the prefill-shaped layer (T=8192 tokens, H=4096,
I=1536, 64 experts, top-2, Zipf(1.2) expert popularity).  Between timed
steps the L2 cache is flushed by writing a 256 MB buffer (untimed).

N > 1 (torchrun): every rank runs its own replica of the layer on its own GPU
(the layer is not sharded: replicas only); the value is the tokens of all
ranks divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "W8A8 MoE layer tokens/s at 1 GB300; % of INT8-tensor / HBM roofline"
L2_FLUSH_BYTES = 256 << 20
STAGES = ["router_topk", "scan", "permute_quant", "gemm1_gateup", "requant", "gemm2_down", "combine"]
LIN_STAGES = ["quant", "gemm"]
FUSED_STAGES = ["fused_layer"]


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--config", default="prefill", choices=["prefill", "decode", "wide", "tiny", "linear"])
    p.add_argument("--format", default="int8", choices=["int8", "fp8", "int8-smooth"],
                   help="int8: the W8A8 INT8 layer; fp8: its E4M3 variant; int8-smooth: the INT8 layer with "
                        "SmoothQuant-folded activations, per-expert factors (MoE configs only)")
    p.add_argument("--fused", action="store_true",
                   help="the INT8 MoE layer as one persistent kernel (moe_w8a8_forward_fused; T <= 128)")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args(argv)


# ----------------------------------------------------------------- ranks

class Ranks:
    """Rank bookkeeping; with WORLD_SIZE > 1 a torch.distributed group
    (NCCL on GPUs, gloo on CPU) provides the barrier and the max-reduction."""

    def __init__(self, backend=None):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", str(self.rank)))
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            if backend is None:
                import torch
                backend = "nccl" if torch.cuda.is_available() else "gloo"
            if not dist.is_initialized():
                dist.init_process_group(backend=backend)
            self.dist = dist
            self.backend = backend

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, value: float) -> float:
        if self.dist is None:
            return value
        import torch
        dev = "cuda" if self.backend == "nccl" else "cpu"
        t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def aggregate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * world / max_seconds if max_seconds > 0 else float("nan")


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.cmd = ["nvidia-smi", f"--id={gpu_index}", "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", f"-lms={period_ms}"]
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, flag in zip(names, parts[4:]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- workload

def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


# fp8 tensor peak = the measured bf16 peak x the nominal fp8 : bf16 ratio (4.5 : 2.25 PFLOP/s dense)
FP8_TO_BF16 = 2.0


def tensor_peak(peaks, fmt):
    """Dense tensor peak (TFLOP/s) of the format's contraction: the exact int8
    path runs on f16 tensor cores (the bf16 rate), E4M3 on the fp8 rate."""
    return peaks["bf16_tflops"] * (FP8_TO_BF16 if fmt == "fp8" else 1.0)


def describe(cfg, fmt="int8") -> str:
    from w8a8_quantised_moe_gb300 import workloads as wl
    if isinstance(cfg, wl.LinearConfig):
        return f"w8a8_linear M={cfg.M} K={cfg.K} N={cfg.N}"
    route = {"none": "uniform routing", "zipf": f"Zipf({cfg.zipf_s}) expert popularity",
             "normal": f"router bias N(0,{cfg.bias_std}^2)"}[cfg.bias]
    tail = {"fp8": ", E4M3 weights and activations",
            "int8-smooth": ", SmoothQuant-folded activations (per-expert factors)"}.get(fmt, "")
    return (f"moe_{cfg.name} T={cfg.T} H={cfg.H} I={cfg.I} E={cfg.E} top-{cfg.k}, {route}{tail}")


def get_config(name):
    from w8a8_quantised_moe_gb300 import workloads as wl
    return wl.LINEAR if name == "linear" else wl.CONFIGS[name]


def device_weights(cfg, seed, dev, fmt="int8"):
    """Expert weights drawn in fp32 on the device, quantised by the library."""
    import torch
    import w8a8_quantised_moe_gb300 as moe
    from w8a8_quantised_moe_gb300 import workloads as wl
    if isinstance(cfg, wl.LinearConfig):
        w = wl.expert_weight_fp32(cfg, "linear", 0, seed, device=dev)
        return moe.quantize_weights(w)
    quant = moe.fp8_quantize_weights if fmt == "fp8" else moe.quantize_weights
    code = torch.uint8 if fmt == "fp8" else torch.int8
    smooth = torch.from_numpy(wl.smoothing_factors(cfg, seed)).to(dev) if fmt == "int8-smooth" else None
    w13_q = torch.empty((cfg.E, 2 * cfg.I, cfg.H), dtype=code, device=dev)
    w13_s = torch.empty((cfg.E, 2 * cfg.I), dtype=torch.float32, device=dev)
    w2_q = torch.empty((cfg.E, cfg.H, cfg.I), dtype=code, device=dev)
    w2_s = torch.empty((cfg.E, cfg.H), dtype=torch.float32, device=dev)
    for e in range(cfg.E):
        w13 = wl.expert_weight_fp32(cfg, "w13", e, seed, device=dev)
        q, s = quant(w13) if smooth is None else moe.quantize_weights_smoothed(w13, smooth[e])
        w13_q[e].copy_(q)
        w13_s[e].copy_(s)
        q, s = quant(wl.expert_weight_fp32(cfg, "w2", e, seed, device=dev))
        w2_q[e].copy_(q)
        w2_s[e].copy_(s)
    return w13_q, w13_s, w2_q, w2_s


def oracle_weights(cfg, seed, dev, fmt="int8"):
    """The same fp32 draws, quantised by the CPU oracle (for the oracle's timing)."""
    import oracle
    from w8a8_quantised_moe_gb300 import workloads as wl
    if isinstance(cfg, wl.LinearConfig):
        return oracle.quantize_rows(wl.expert_weight_fp32(cfg, "linear", 0, seed, device=dev).cpu().numpy())
    quant = oracle.quantize_rows_fp8 if fmt == "fp8" else oracle.quantize_rows
    code = np.uint8 if fmt == "fp8" else np.int8
    smooth = wl.smoothing_factors(cfg, seed) if fmt == "int8-smooth" else None
    w13_q = np.empty((cfg.E, 2 * cfg.I, cfg.H), code)
    w13_s = np.empty((cfg.E, 2 * cfg.I), np.float32)
    w2_q = np.empty((cfg.E, cfg.H, cfg.I), code)
    w2_s = np.empty((cfg.E, cfg.H), np.float32)
    for e in range(cfg.E):
        w13 = wl.expert_weight_fp32(cfg, "w13", e, seed, device=dev).cpu().numpy()
        w13_q[e], w13_s[e] = quant(w13) if smooth is None else oracle.quantize_rows_smoothed(w13, smooth[e])
        w2_q[e], w2_s[e] = quant(wl.expert_weight_fp32(cfg, "w2", e, seed, device=dev).cpu().numpy())
    return w13_q, w13_s, w2_q, w2_s


def host_inputs(cfg, seed):
    from w8a8_quantised_moe_gb300 import workloads as wl
    if isinstance(cfg, wl.LinearConfig):
        return {"x": wl.linear_activations(cfg, seed)}
    inp = wl.make_moe_inputs(cfg, seed)
    return {"x": inp.x, "Wr": inp.Wr, "bias": inp.bias, "redrawn": inp.redrawn_rows, "seed": seed}


def tokens_of(cfg):
    from w8a8_quantised_moe_gb300 import workloads as wl
    return cfg.M if isinstance(cfg, wl.LinearConfig) else cfg.T


# ------------------------------------------------------------ CPU oracle

def oracle_sample_rate(cfg, inputs, oweights, target_s, max_tokens=None, fmt="int8"):
    """Tokens/s of the oracle forward on a sample of the workload's first
    tokens, sized to take about ``target_s`` seconds.  -> (rate, tokens, seconds)."""
    import oracle
    from w8a8_quantised_moe_gb300 import workloads as wl
    T = tokens_of(cfg)
    lim = T if max_tokens is None else min(T, max_tokens)

    def run(n):
        x = inputs["x"][:n]
        t0 = time.perf_counter()
        if isinstance(cfg, wl.LinearConfig):
            oracle.linear(x, *oweights)
        else:
            if fmt == "int8-smooth":
                oracle.moe_forward_smooth(x, inputs["Wr"], inputs["bias"], wl.smoothing_factors(cfg, inputs["seed"]),
                                          *oweights, cfg.k)
            else:
                fwd = oracle.moe_forward_fp8 if fmt == "fp8" else oracle.moe_forward
                fwd(x, inputs["Wr"], inputs["bias"], *oweights, cfg.k)
        return time.perf_counter() - t0

    n = min(lim, 8)
    dt = run(n)
    while dt < 0.5 * target_s and n < lim:
        n = min(lim, max(n * 2, int(n * target_s / max(dt, 1e-3))))
        dt = run(n)
    return n / dt, n, dt


# ------------------------------------------------------------- GPU timing

def algorithmic_work(cfg, offsets, peaks):
    """Algorithmic bytes and flops per launch of the two GEMMs.

    GEMM1: flops 2*S*(2I)*H over routed rows; bytes = int8 weights + fp32
    scales of the experts that received tokens + S*H int8 activation codes +
    S*I fp32 h.  GEMM2: flops 2*S*H*I; bytes = touched w2 + scales + S*I int8
    codes + S*H fp32 o.  Linear: flops 2*M*N*K; bytes = N*K + 4N + M*K + 2*M*N.
    """
    from w8a8_quantised_moe_gb300 import workloads as wl
    if isinstance(cfg, wl.LinearConfig):
        M, N, K = cfg.M, cfg.N, cfg.K
        return {"gemm": {"flops": 2.0 * M * N * K, "bytes": N * K + 4 * N + M * K + 2 * M * N}}
    S, H, I = cfg.T * cfg.k, cfg.H, cfg.I
    touched = int((np.diff(offsets) > 0).sum())
    return {
        "gemm1_gateup": {"flops": 2.0 * S * 2 * I * H,
                         "bytes": touched * (2 * I * H + 8 * I) + S * H + 4 * S * I, "touched": touched},
        "gemm2_down": {"flops": 2.0 * S * H * I,
                       "bytes": touched * (H * I + 4 * H) + S * I + 4 * S * H, "touched": touched},
    }


def layer_roofline_us(cfg, offsets, peaks, fmt="int8"):
    """Roofline time of the whole layer: max(weight+activation bytes at HBM
    peak, routed int8 MACs at the tensor peak)."""
    from w8a8_quantised_moe_gb300 import workloads as wl
    if isinstance(cfg, wl.LinearConfig):
        b = cfg.N * cfg.K + 4 * cfg.N + 2 * cfg.M * cfg.K + 2 * cfg.M * cfg.N
        f = 2.0 * cfg.M * cfg.N * cfg.K
    else:
        touched = int((np.diff(offsets) > 0).sum())
        b = (touched * (3 * cfg.H * cfg.I + 4 * (2 * cfg.I + cfg.H)) + 2 * cfg.T * cfg.H * 2
             + 4 * cfg.H * cfg.E)
        f = 2.0 * cfg.T * cfg.k * 3 * cfg.H * cfg.I
    t_b = b / (peaks["hbm_gbs"] * 1e9)
    t_f = f / (tensor_peak(peaks, fmt) * 1e12)
    return max(t_b, t_f) * 1e6, ("hbm" if t_b >= t_f else "tensor"), b, f


GEMM_SOURCES = {
    "int8": ("gemm.cu", "gemm_pair.cu", "gemm_skinny.cu", "gemm_skinny.cuh", "gemm_common.cuh", "ptx.cuh",
             "internal.h", "fused.cu", "router_small.cuh"),
    "fp8": ("fp8.cu", "gemm_fp8_pair.cu", "gemm_common.cuh", "ptx.cuh", "internal.h"),
}


def gemm_source_sha(fmt="int8"):
    """sha256 prefix of the format's GEMM kernel sources (keys the committed traffic)."""
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES[fmt]:
        with open(os.path.join(ROOT, "w8a8_quantised_moe_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_from_profiles(config_name, kernel, fmt="int8"):
    """dram bytes per launch of ``kernel`` from the committed ncu summary, if
    it was taken on the current source of the format's GEMM kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    ent = table.get(config_name, {}).get(kernel)
    if not ent or ent.get("gemm_src_sha256_16") != gemm_source_sha(fmt):
        return None
    return ent.get("dram_bytes_per_launch")


def tensor_rate_from_profiles(fmt="int8"):
    """The measured tcgen05 rate (TOPS) of the format's MMA kind, from the
    committed summary of the contraction-rate program, or None."""
    path = os.path.join(ROOT, "profiles", "tensor_rates.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        table = json.load(f)
    ent = table.get("e4m3" if fmt == "fp8" else "f16_int8_values")
    return None if not ent else ent.get("tops")


def run_ours(args, ranks: Ranks):
    import torch
    import w8a8_quantised_moe_gb300 as moe
    from w8a8_quantised_moe_gb300 import workloads as wl

    torch.cuda.set_device(ranks.local_rank)
    dev = torch.device("cuda", ranks.local_rank)
    stream = torch.cuda.current_stream()
    cfg = get_config(args.config)
    linear = isinstance(cfg, wl.LinearConfig)
    fmt = args.format
    if linear and fmt != "int8":
        raise SystemExit(f"--format {fmt} applies to the MoE configs")
    if args.fused and (linear or fmt != "int8" or not moe.fused_supported(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k)):
        raise SystemExit("--fused takes an INT8 MoE config that moe_w8a8_fused_supported accepts (T <= 128)")
    if fmt == "int8-smooth":
        smooth_dev = torch.from_numpy(wl.smoothing_factors(cfg, args.seed + ranks.rank)).to(dev)

        def fwd(*a, **kw):
            return moe.forward_smooth(*a[:3], smooth_dev, *a[3:], **kw)

        def fwd_debug(*a, fields=None, **kw):
            return moe.forward_smooth(*a[:3], smooth_dev, *a[3:], fields=fields, **kw)
    elif args.fused:
        fwd = moe.forward_fused

        def fwd_debug(*a, fields=None, **kw):
            return moe.forward_fused(*a, fields=fields, **kw)
    else:
        fwd = moe.fp8_forward if fmt == "fp8" else moe.forward
        fwd_debug = moe.fp8_forward_debug if fmt == "fp8" else moe.forward_debug
    peaks = measured_peaks()
    seed = args.seed + ranks.rank
    inputs = host_inputs(cfg, seed)
    weights = device_weights(cfg, seed, dev, fmt)
    x_host = torch.from_numpy(inputs["x"].view(np.int16)).view(torch.bfloat16)
    x = x_host.to(dev)
    T = tokens_of(cfg)
    if linear:
        w_q, w_s = weights
        ws = moe.new_workspace(moe.linear_workspace_size(cfg.M, cfg.N, cfg.K), dev)
        y = torch.empty((cfg.M, cfg.N), dtype=torch.bfloat16, device=dev)

        def step(xin, out):
            return moe.linear(xin, w_q, w_s, workspace=ws, out=out)
        stage_names = LIN_STAGES
    else:
        Wr = torch.from_numpy(inputs["Wr"]).to(dev)
        bias = None if inputs["bias"] is None else torch.from_numpy(inputs["bias"]).to(dev)
        w13_q, w13_s, w2_q, w2_s = weights
        ws = moe.new_workspace(moe.workspace_size(cfg.T, cfg.H, cfg.I, cfg.E, cfg.k), dev)
        y = torch.empty((cfg.T, cfg.H), dtype=torch.bfloat16, device=dev)

        def step(xin, out):
            return fwd(xin, Wr, bias, w13_q, w13_s, w2_q, w2_s, cfg.k, workspace=ws, out=out)
        stage_names = FUSED_STAGES if args.fused else STAGES
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    lib = moe._lib.load()

    # routing of this workload (for the algorithmic byte counts)
    if linear:
        offsets = None
    else:
        _, d = fwd_debug(x, Wr, bias, w13_q, w13_s, w2_q, w2_s, cfg.k, fields=("offsets", "topk_ids"))
        offsets = d["offsets"].cpu().numpy()
        shares = wl.realised_shares(d["topk_ids"].cpu().numpy(), cfg.E)

    for _ in range(args.warmup):
        flush.zero_()
        step(x, y)
    torch.cuda.synchronize()
    if moe.device_error(ws) != 0:
        raise RuntimeError("device error during warm-up")

    n_ev = 8
    K = args.steps
    # timed steps: one event pair around each whole step (the layer's kernels
    # overlap their set-up with the previous kernel's tail); the per-kernel
    # breakdown comes from a second pass with an event between every two
    # launches, which serialises them
    step_events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(K)]
    for row in [*step_events, *events]:  # materialise the driver events
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    handles = [ctypes_array(row) for row in events]  # (pointer, keep-alive array)

    ranks.barrier()
    torch.cuda.synchronize()
    with ClockSampler(ranks.local_rank) as clocks:
        launches0 = lib.moe_w8a8_launch_count()
        t_wall0 = time.perf_counter()
        for i in range(K):
            flush.zero_()  # untimed: outside the step's events
            step_events[i][0].record(stream)
            step(x, y)
            step_events[i][1].record(stream)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
        launches = lib.moe_w8a8_launch_count() - launches0
        # per-kernel breakdown (untimed for the value)
        for i in range(K):
            flush.zero_()
            moe._lib.check(lib.moe_w8a8_set_profile_events(handles[i][0], n_ev), "set_profile_events")
            step(x, y)
        lib.moe_w8a8_set_profile_events(None, 0)
        torch.cuda.synchronize()
        # keep the GPU busy long enough for the clock sampler (untimed)
        t_extra = time.perf_counter()
        while time.perf_counter() - t_extra < max(0.0, 1.0 - t_wall):
            flush.zero_()
            step(x, y)
            torch.cuda.synchronize()
    ranks.barrier()
    torch.cuda.synchronize()
    status = moe.device_error(ws)
    if status != 0:
        raise RuntimeError(f"device error in the timed region: {moe.STATUS.get(status)}")

    last = len(stage_names)
    step_ms = [a.elapsed_time(b) for a, b in step_events]
    stage_ms = {name: statistics.mean(events[i][j].elapsed_time(events[i][j + 1]) for i in range(K))
                for j, name in enumerate(stage_names)}
    serial_step_ms = statistics.mean(events[i][0].elapsed_time(events[i][last]) for i in range(K))
    gpu_s = sum(step_ms) / 1e3
    max_gpu_s = ranks.max(gpu_s)
    value = aggregate(T * K, ranks.world, max_gpu_s)

    # dominant kernel and its roofline
    work = algorithmic_work(cfg, offsets, peaks)
    if args.fused:  # one kernel: the whole layer's bytes and flops
        _, _, lb, lf = layer_roofline_us(cfg, offsets, peaks, fmt)
        work = {"fused_layer": {"flops": lf, "bytes": lb}}
    dom = max(work, key=lambda k: stage_ms[k])
    dom_ms = stage_ms[dom]
    w = work[dom]
    peak_t = tensor_peak(peaks, fmt)
    t_f = w["flops"] / (peak_t * 1e12)
    t_b = w["bytes"] / (peaks["hbm_gbs"] * 1e9)
    if t_f >= t_b:
        achieved = w["flops"] / (dom_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s"}
    else:
        achieved = w["bytes"] / (dom_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    probe = tensor_rate_from_profiles(fmt)
    if roof["bound"] == "tensor" and probe:  # the MMA kind's own measured rate, beside the cuBLAS peak
        roof["probe"] = {"peak": probe, "frac": achieved / probe, "unit": "TFLOP/s",
                         "source": "profiles/tcgen05_rates.md"}
    gemm_fmt = "fp8" if fmt == "fp8" else "int8"  # the smoothed layer runs the INT8 GEMM kernels
    roof["traffic"] = traffic_from_profiles(args.config + ("_fp8" if fmt == "fp8" else ""), dom, gemm_fmt)
    roof["kernel"] = dom
    roof["kernel_ms"] = dom_ms
    roof["algorithmic"] = {"flops": w["flops"], "bytes": w["bytes"]}
    roof["peak_source"] = peaks["source"] + (
        " (bf16 burst x 2, the nominal fp8 : bf16 ratio)" if fmt == "fp8"
        else " (bf16 burst; f16 tensor rate carries the exact int8 products)")
    layer_us, layer_bound, layer_bytes, layer_flops = layer_roofline_us(cfg, offsets, peaks, fmt)

    # end to end through the public API with host buffers: the MoE layers
    # through the host entry point (x copied in and y out inside the call,
    # token chunks overlapping the copies with compute on a second stream);
    # the linear layer with its copies around the device entry point
    x_pin = x_host.pin_memory()
    y_pin = torch.empty(y.shape, dtype=torch.bfloat16).pin_memory()
    x_dev2 = torch.empty_like(x)
    copy_stream = torch.cuda.Stream(device=dev)
    if linear or fmt == "int8-smooth":  # no host-resident entry point: copies around the device one
        def step_host():
            x_dev2.copy_(x_pin, non_blocking=True)
            step(x_dev2, y)
            y_pin.copy_(y, non_blocking=True)
        host_chunks = 1
    else:
        fwd_host = moe.fp8_forward_host if fmt == "fp8" else moe.forward_host

        def step_host():
            fwd_host(x_pin, Wr, bias, w13_q, w13_s, w2_q, w2_s, cfg.k, y_host=y_pin, x_dev=x_dev2, y_dev=y,
                     workspace=ws, stream=stream, copy_stream=copy_stream)
        host_chunks = moe.host_chunks(cfg.T, cfg.H, cfg.I, cfg.E)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(2):
        step_host()
    torch.cuda.synchronize()
    ranks.barrier()
    e2e_ms = 0.0
    for _ in range(K):
        flush.zero_()
        e0.record(stream)
        step_host()
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_value = aggregate(T * K, ranks.world, ranks.max(e2e_ms / 1e3))
    h2d = x.numel() * 2
    d2h = y.numel() * 2

    out = {
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": ranks.world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": max_gpu_s * 1e3 / K,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if fmt == "fp8" else "int8",
        "data": "synthetic (seeded; random-init expert weights quantised per channel)",
        "config": {
            "workload": describe(cfg, fmt),
            "parallelism": f"replicas x{ranks.world}" if ranks.world > 1 else "single GPU",
            "l2": "flushed between timed steps (256 MB write, untimed)",
            "arithmetic": ("E4M3 x E4M3 -> fp32 on the fp8 tensor cores (tcgen05 kind::f8f6f4), fp32 epilogues"
                           if fmt == "fp8" else
                           "int8 x int8 -> exact int32 on f16 tensor cores (tcgen05 kind::f16), fp32 epilogues"),
            "stage_ms": stage_ms,
            "stage_ms_note": "per-kernel pass with an event between launches (serialised), "
                             f"{serial_step_ms:.4f} ms per step there",
            "pdl": os.environ.get("MOE_W8A8_NO_PDL", "0") in ("", "0"),
            "layer_roofline_us": layer_us,
            "layer_bound": layer_bound,
            "layer_frac": layer_us / (max_gpu_s * 1e6 / K),
            "wall_s_timed_region": t_wall,
        },
        "roofline": roof,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "host_chunks": host_chunks},
        "gpu_launches": int(launches),
        "clocks": clocks.summary(),
    }
    if args.fused:
        out["config"]["layer_kernel"] = "one persistent cooperative kernel (moe_w8a8_forward_fused)"
        out["e2e"]["note"] = "through moe_w8a8_forward_host (the multi-kernel layer; no host entry for the fused one)"
    if not linear:
        out["config"]["touched_experts"] = int((np.diff(offsets) > 0).sum())
        out["config"]["top12_share"] = float(np.sort(shares)[::-1][:12].sum())
        out["config"]["redrawn_rows"] = int(inputs["redrawn"])

    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        import oracle
        oweights = oracle_weights(cfg, seed, dev, fmt)
        rate, n, dt = oracle_sample_rate(cfg, inputs, oweights, args.cpu_seconds, fmt=fmt)
        out["cpu_baseline"] = {"value": rate, "unit": "tokens/s", "cores": oracle.num_threads(),
                               "kind": "oracle",
                               "sample": f"first {n} tokens of the same workload, one oracle forward "
                                         f"({dt:.1f} s; OpenMP over tokens/slots)"}
    return out


def ctypes_array(events):
    import ctypes
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    return ctypes.cast(arr, ctypes.c_void_p), arr


def run_reference(args):
    """The CPU oracle as the reference arm: each step is one oracle forward on
    a bounded sample of the workload's tokens."""
    import torch
    import oracle
    cfg = get_config(args.config)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    fmt = args.format
    inputs = host_inputs(cfg, args.seed)
    oweights = oracle_weights(cfg, args.seed, dev, fmt)
    total = args.steps + args.warmup
    per_step_s = min(8.0, 150.0 / max(total, 1))
    _, n, _ = oracle_sample_rate(cfg, inputs, oweights, per_step_s, fmt=fmt)
    import w8a8_quantised_moe_gb300.workloads as wl
    x = inputs["x"][:n]

    def step():
        if isinstance(cfg, wl.LinearConfig):
            oracle.linear(x, *oweights)
        elif fmt == "int8-smooth":
            oracle.moe_forward_smooth(x, inputs["Wr"], inputs["bias"], wl.smoothing_factors(cfg, inputs["seed"]),
                                      *oweights, cfg.k)
        else:
            (oracle.moe_forward_fp8 if fmt == "fp8" else oracle.moe_forward)(
                x, inputs["Wr"], inputs["bias"], *oweights, cfg.k)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "tokens/s",
        "n_gpus": 1,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if fmt == "fp8" else "int8",
        "data": "synthetic (seeded)",
        "config": {"workload": describe(cfg, fmt), "parallelism": "host cores (OpenMP)",
                   "sample_tokens_per_step": n},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"first {n} of {tokens_of(cfg)} tokens per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        if int(os.environ.get("RANK", "0")) != 0:
            return 0
        print(json.dumps(run_reference(args)), flush=True)
        return 0
    ranks = Ranks()
    try:
        out = run_ours(args, ranks)
        if ranks.rank == 0:
            print(json.dumps(out), flush=True)
    finally:
        ranks.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
