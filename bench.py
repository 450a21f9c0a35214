"""Benchmark of the LatentMoE layer forward + backward on GB300 (libmoe).

Workload: T=16384 tokens, d=4096, latent l=1024, E=896 routed experts top-16,
2 shared experts (SwiGLU f=512), loss = sum(out * g): one step is the full
forward and backward (all expert, shared, projection and router gradients).
Inputs and weights are seeded synthetic bf16 (inputs.py), resident in HBM.

Prints one JSON line. `value` is whole-job tokens/s (device-timed with CUDA
events over exactly --steps steps after --warmup steps); `e2e` repeats the
measurement with the step's inputs copied from pinned host memory and the
input gradient copied back inside the timed region. Under torchrun each rank
runs an independent replica (the layer has no cross-GPU exchange here).

--impl reference times the fp64 CPU oracle instead (bounded token sample per
step, host cores), on the same metric.
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
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s fwd+bwd (896 experts, top-16); grouped GEMM % of BF16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
EXPERT_GEMMS = ("expert_gemm1_swiglu", "expert_gemm2_rowscale", "expert_dgrad2_swiglu_bwd",
                "expert_wgrad2", "expert_dgrad1", "expert_wgrad1")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--wgrad", default="f32", choices=["f32", "bf16"])
    ap.add_argument("--cpu-sample-tokens", type=int, default=128)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--fused-gather", action="store_true",
                    help="the grouped GEMMs gather their permuted rows themselves")
    ap.add_argument("--no-graph", action="store_true",
                    help="time eager launches instead of CUDA-graph replays of the step")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary workloads (T=4096 forward uniform / Zipf, EP rank)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="profiling case: override T (the JSON line then names that case)")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling case: override E (the JSON line then names that case)")
    ap.add_argument("--case", default="", choices=["", "topk", "permute", "gather", "combine"],
                    help="time one entry point alone on the workload's sizes (for ncu): "
                         "topk = moe_topk_from_logits on fp32 logits [T][E]; permute = "
                         "moe_permute; gather = moe_unpermute_combine_bwd; combine = "
                         "moe_unpermute_combine")
    return ap.parse_args()


def workload(args):
    import dataclasses

    from sparse_moe_layer_topk_gb300 import inputs as I
    cfg = I.CONFIGS[args.config]
    if args.tokens or args.experts:
        T = args.tokens or cfg.T
        E = args.experts or cfg.E
        cfg = dataclasses.replace(cfg, T=T, E=E, name=f"profile_case_T{T}_E{E}_top{cfg.k}")
    return cfg


def max_over_ranks(ms, world, device):
    """The slowest rank's time (ms): every rank's timed region covers the same
    number of steps, so the job finishes with the slowest one."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, T, steps, ms):
    """Whole-job throughput: every rank processes T tokens per step (replicas,
    weak scaling) in the slowest rank's time."""
    return world * T * steps / (ms / 1000.0)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------- algorithmic work

def kernel_work(cfg, T, wgrad_bytes=4):
    """Algorithmic (flops, bytes) per launch of each kernel label at token count T;
    weight gradients are written as fp32 (wgrad_bytes=4) or bf16 (2)."""
    d, l, E, k, S, f = cfg.d, cfg.l, cfg.E, cfg.k, cfg.S, cfg.f
    R = T * k
    nch = (T + 255) // 256  # token chunks of the routing-map kernels
    w13 = E * l * 2 * f * 2
    w2 = E * f * l * 2
    b = 2  # bf16 bytes
    g = wgrad_bytes
    return {
        "router_logits_gemm": (2 * T * d * E, T * d * b + d * E * b + T * E * 4),
        # the router and the down-projection as one GEMM over [Wr | W_dn] (x read once)
        "router_latent_gemm": (2 * T * d * (E + l),
                               T * d * b + d * (E + l) * b + T * E * 4 + T * l * b),
        "topk_sigmoid": (0, T * E * 4 + T * k * 12),
        "latent_proj_gemm": (2 * T * d * l, T * d * b + d * l * b + T * l * b),
        "permute_gather": (0, T * l * b + R * l * b + R * 4),
        "expert_gemm1_swiglu": (2 * R * l * 2 * f, R * l * b + w13 + R * f * b + R * 2 * f * b),
        "expert_gemm2_rowscale": (2 * R * f * l, R * f * b + w2 + R * l * b + R * 4),
        "shared_gemm1_swiglu": (2 * T * l * 2 * f * S, T * l * b + S * l * 2 * f * b + T * S * 3 * f * b),
        "shared_gemm2": (2 * T * S * f * l, T * S * f * b + S * f * l * b + T * l * b),
        "combine": (0, R * l * b + 2 * T * l * b + R * 4),
        "latent_proj_dgrad": (2 * T * d * l, T * d * b + d * l * b + T * l * b),
        "latent_proj_wgrad": (2 * T * d * l, T * d * b + T * l * b + d * l * g),
        "combine_bwd_gather": (0, T * l * b + R * l * b + R * 4),
        # dy and W2 in; the epilogue reads g, u, h and writes dg, du, w*h (6 f per
        # row) and the routing-weight gradient (its per-n-tile partials are the
        # engine's, not the algorithm's)
        "expert_dgrad2_swiglu_bwd": (2 * R * l * f, R * l * b + w2 + R * 6 * f * b + R * 4),
        "expert_wgrad2": (2 * R * f * l, R * f * b + R * l * b + E * f * l * g),
        "expert_dgrad1": (2 * R * 2 * f * l, R * 2 * f * b + w13 + R * l * b),
        "expert_wgrad1": (2 * R * l * 2 * f, R * l * b + R * 2 * f * b + E * l * 2 * f * g),
        "shared_dgrad2_swiglu_bwd": (2 * T * l * S * f, T * l * b + S * f * l * b + T * S * 5 * f * b),
        "shared_wgrad2": (2 * T * S * f * l, T * S * f * b + T * l * b + S * f * l * g),
        "shared_dgrad1": (2 * T * S * 2 * f * l, T * S * 2 * f * b + S * l * 2 * f * b + T * l * b),
        "shared_wgrad1": (2 * T * l * S * 2 * f, T * l * b + T * S * 2 * f * b + S * l * 2 * f * g),
        "permute_bwd_sum": (0, R * l * b + 2 * T * l * b + R * 4),
        # two epilogue warps per lane quadrant x one partial per 256-wide n tile
        "routing_weight_grad_reduce": (0, R * 4 * 2 * ((f + 255) // 256) + R * 4),
        "router_bwd_dlogits": (0, T * k * 16 + T * E * b),
        # The router backward's logit gradient dL has k nonzeros per token: its
        # algorithmic cost is 2 T k d per product, reading the k (value, id)
        # pairs per token (6 bytes each); the dense GEMMs that run it execute
        # the flops of DENSE_EXECUTED (the difference is counted as waste)
        "router_dgrad": (2 * T * k * d, T * k * 6 + d * E * b + 2 * T * d * b),
        "down_proj_router_dgrad": (2 * T * d * l + 2 * T * k * d,
                                   T * l * b + d * l * b + T * k * 6 + d * E * b + T * d * b),
        "router_wgrad": (2 * T * k * d, T * d * b + T * k * 6 + d * E * g),
        # routing maps: the per-chunk expert histogram (chunks of 256 tokens) is
        # this design's intermediate; hist reads the ids, scan turns the
        # histogram into per-chunk prefixes plus counts / offsets / schedule, maps
        # reads ids, weights and prefixes and writes slot_of, token_of and row_w
        "permute_hist": (0, R * 4 + nch * E * 4),
        "permute_scan": (0, 2 * nch * E * 4 + 3 * (E + 1) * 4),
        "permute_maps": (0, 2 * R * 4 + nch * E * 4 + E * 4 + 3 * R * 4),
        # the shared experts' K-split weight gradients: each launch reads its
        # slices' fp32 partials and writes the gradient (mean of the two launches)
        "splitk_reduce": (0, sum(m * n * (4 * s + g) for m, n, s in splitk_shapes(cfg, T)) // 2),
    }


def pick_bn(n):
    """Tile width of the GEMM engine for an N-wide output: 256 unless N is narrow or
    a 256-wide tail would waste more than a quarter."""
    return 256 if (n % 256 == 0 or (n > 512 and n % 256 >= 128)) else 128


def wgrad_splitk(m, n, kdim):
    """K slices of a dense weight gradient with few output tiles, as the library
    chooses them: enough for ~128 tiles, at most 4, each slice >= 1024 rows of K."""
    tiles = ((m + 127) // 128) * ((n + pick_bn(n) - 1) // pick_bn(n))
    s = 1
    while s < 4 and tiles * s * 2 <= 128 and kdim // (s * 2) >= 1024:
        s *= 2
    return s


def splitk_shapes(cfg, T):
    """(M, N, slices) of the shared experts' two weight gradients: dW2_sh [S f][l]
    and dW13_sh [l][S 2f], K = T."""
    sf, l = cfg.S * cfg.f, cfg.l
    return [(sf, l, wgrad_splitk(sf, l, T)), (l, 2 * sf, wgrad_splitk(l, 2 * sf, T))]


def dense_executed_flops(cfg, T):
    """Flops the dense router-backward GEMMs execute per launch (their
    algorithmic cost, in kernel_work, is the sparse 2 T k d per product)."""
    d, l, E = cfg.d, cfg.l, cfg.E
    return {"router_dgrad": 2 * T * E * d, "down_proj_router_dgrad": 2 * T * d * (l + E),
            "router_wgrad": 2 * T * d * E}


def load_peaks(path=None):
    """The measured peaks file as a dict ({} when it is absent or unreadable)."""
    p = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as fh:
                m = json.load(fh)
            return m if isinstance(m, dict) else {}
        except Exception:
            pass
    return {}


_NOT_A_PEAK = ("util", "pct", "percent", "frac", "ratio", "mhz", "clock", "time", "_ms", "bytes",
               "size", "watt", "power", "temp", "date", "count", "iters")


def _number(v, inner=True):
    """A positive number, or a record holding one directly under a value-like key."""
    if isinstance(v, bool):
        return None
    if isinstance(v, (int, float)) and v > 0:
        return float(v)
    if inner and isinstance(v, dict):
        for kk in ("value", "median", "gbs", "tflops", "mean"):
            x = _number(v.get(kk), inner=False)
            if x:
                return x
    return None


def _leaves(d, path=()):
    for key, v in d.items():
        kp = path + (str(key).lower(),)
        if isinstance(v, dict) and _number(v) is None:
            yield from _leaves(v, kp)
        else:
            yield kp, v


def _peak_val(peaks, names, words=(), avoid=()):
    """A peak from the measured file: one of the exact top-level `names` first,
    else the first numeric entry (nested or not) whose key path holds every one of
    `words` and none of `avoid` or of the words that mark a non-peak figure."""
    for n in names:
        x = _number(peaks.get(n))
        if x:
            return x
    if not words:
        return None
    for kp, v in _leaves(peaks):
        path = ".".join(kp)
        if all(w in path for w in words) and not any(w in path for w in avoid + _NOT_A_PEAK):
            x = _number(v)
            if x:
                return x
    return None


def burst_tc_peak(peaks):
    """(bf16 TFLOP/s, label) for a kernel timed on its own: the burst figure of
    the measured file, else the fallback burst number."""
    tc = _peak_val(peaks, ("bf16_tflops",), ("bf16",), avoid=("sustained",))
    if tc:
        return tc, "measured (burst)"
    return FALLBACK_PEAKS["bf16_tflops"], "fallback (burst)"


def roofline_peaks(peaks):
    """(HBM GB/s, its label, bf16 TFLOP/s for a kernel timed inside a step, its label).

    Each figure is labelled by where it came from: the measured file, or the
    fallback numbers when the file lacks it. A kernel timed inside a long step
    takes the sustained bf16 figure; only when the file has no sustained figure
    does the burst one stand in, and the label says so."""
    hbm = _peak_val(peaks, ("hbm_gbs", "hbm_GBs", "hbm"), ("hbm",))
    hbm_src = "measured (copy)"
    if not hbm:
        hbm, hbm_src = FALLBACK_PEAKS["hbm_gbs"], "fallback (copy)"
    tc = _peak_val(peaks, ("bf16_tflops_sustained",), ("bf16", "sustained"))
    tc_src = "measured (sustained)"
    if not tc:
        tc = _peak_val(peaks, ("bf16_tflops",), ("bf16",), avoid=("sustained",))
        tc_src = "measured (burst; the file has no sustained figure)"
    if not tc:
        tc, tc_src = FALLBACK_PEAKS["bf16_tflops_sustained"], "fallback (sustained)"
    return hbm, hbm_src, tc, tc_src


# the GEMM engine's sources: the DRAM traffic on record is for its kernels
GEMM_SOURCES = ("common.cuh", "gemm.h", "gemm_tc.cu")


def source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_moe_layer_topk_gb300", "csrc")
    for name in GEMM_SOURCES:
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def dram_traffic(label, workload):
    """Per-launch DRAM bytes of `label` from the committed ncu summary, or None
    when none was taken for this workload on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as fh:
            tab = json.load(fh)
    except Exception:
        return None
    ent = tab.get(workload, {}).get(label)
    if not ent or ent.get("source_hash") != source_hash():
        return None
    return ent.get("bytes_per_launch")


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        return parse_clock_samples(out)


def parse_clock_samples(out):
    """The `clocks` record from nvidia-smi's CSV lines (the ClockSampler fields,
    no header, no units): median SM clock, maximum SM clock, and every throttle
    reason seen active in any sample."""
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in out.strip().splitlines():
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            mx.append(float(parts[1]))
        except ValueError:
            continue
        for n, v in zip(names, parts[4:8]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
            "samples": len(sm)}


# ---------------------------------------------------------------- oracle timing

def oracle_sample_time(inp_cpu, n_tokens):
    """Time the fp64 oracle's forward + backward on the first n_tokens tokens."""
    import oracle as O
    sub = dict(inp_cpu)
    sub["x"] = inp_cpu["x"][:n_tokens]
    sub["g"] = inp_cpu["g"][:n_tokens]
    t0 = time.perf_counter()
    fwd = O.layer_forward(sub)
    O.layer_backward(sub, fwd)
    return time.perf_counter() - t0


def host_threads() -> int:
    """Threads the oracle's numpy BLAS calls may use: the BLAS/OpenMP thread limit
    when one is set, else the cores this process may run on."""
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var, "")
        if v.isdigit() and int(v) > 0:
            return int(v)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    world, rank, _ = dist_env()
    from sparse_moe_layer_topk_gb300 import inputs as I
    cfg = workload(args)
    line = {"impl": "reference", "metric": METRIC, "unit": "tokens/s", "higher_is_better": True}
    if rank != 0:
        return
    # bounded sample: at most ~1024 oracle tokens over the whole run (a few minutes
    # of fp64 host work), at least 4 per step
    n = max(4, min(args.cpu_sample_tokens, 1024 // max(1, args.steps + args.warmup)))
    inp = I.make_layer_inputs(cfg, T=n)
    for _ in range(args.warmup):
        oracle_sample_time(inp, n)
    times = [oracle_sample_time(inp, n) for _ in range(args.steps)]
    total = sum(times)
    value = n * args.steps / total
    cores = host_threads()
    line.update({
        "value": value, "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * total / args.steps, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "l": cfg.l, "E": cfg.E,
                   "k": cfg.k, "S": cfg.S, "f": cfg.f,
                   "sample": f"first {n} tokens of the workload per step, full weights"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} tokens fwd+bwd per step, {args.steps} steps"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    })
    print(json.dumps(line), flush=True)


def roofline_report(per_kernel, work, peaks, traffic_of, executed=None):
    """(roofline of the dominant kernel, per-kernel breakdown, grouped-GEMM % of bf16 peak).

    per_kernel: label -> (launches, total ms) over the timed steps; work: label ->
    algorithmic (flops, bytes) per launch; peaks: the tuple of roofline_peaks;
    traffic_of(label): ncu DRAM bytes per launch on record for that kernel, or None.
    A kernel's floor is the larger of its compute time and its memory time at the
    peaks; the dominant kernel (largest total time) is reported against whichever
    of the two bounds it. executed: label -> flops a launch executes where that
    exceeds its algorithmic flops (dense GEMMs over sparse operands); such kernels
    also report the executed rate and the executed flops' share that is waste."""
    hbm, hbm_src, tc, tc_src = peaks
    total = sum(v[1] for v in per_kernel.values())
    breakdown = {}
    for name, (cnt, tot) in sorted(per_kernel.items(), key=lambda kv: -kv[1][1]):
        fl, by = work.get(name, (0, 0))
        avg_s = tot / cnt / 1000.0
        floor_s = max(fl / (tc * 1e12), by / (hbm * 1e9))
        breakdown[name] = {"launches": cnt, "avg_us": round(avg_s * 1e6, 2),
                           "share": round(tot / total, 4),
                           "tflops": round(fl / avg_s / 1e12, 1) if fl else None,
                           "gbs": round(by / avg_s / 1e9, 1),
                           "roofline_frac": round(floor_s / avg_s, 3) if floor_s else None}
        if executed and name in executed:
            ex = executed[name]
            breakdown[name]["executed_tflops"] = round(ex / avg_s / 1e12, 1)
            breakdown[name]["executed_waste_frac"] = round(1.0 - fl / ex, 4) if ex else None
    roof = None
    if per_kernel:
        name, (cnt, tot) = max(per_kernel.items(), key=lambda kv: kv[1][1])
        fl, by = work.get(name, (0, 0))
        avg_s = tot / cnt / 1000.0
        if fl and fl / (tc * 1e12) >= by / (hbm * 1e9):
            roof = {"kernel": name, "bound": "tensor", "achieved": fl / avg_s / 1e12,
                    "peak": tc, "unit": "TFLOP/s", "frac": fl / avg_s / 1e12 / tc}
        else:
            roof = {"kernel": name, "bound": "hbm", "achieved": by / avg_s / 1e9, "peak": hbm,
                    "unit": "GB/s", "frac": by / avg_s / 1e9 / hbm}
        roof["traffic"] = traffic_of(name)
        roof["avg_launch_us"] = avg_s * 1e6
        roof["peak_source"] = tc_src if roof["bound"] == "tensor" else hbm_src
    g_fl = sum(work[n][0] * per_kernel[n][0] for n in EXPERT_GEMMS if n in per_kernel)
    g_ms = sum(per_kernel[n][1] for n in EXPERT_GEMMS if n in per_kernel)
    grouped_pct = 100.0 * (g_fl / (g_ms / 1000.0) / 1e12) / tc if g_ms else None
    return roof, breakdown, grouped_pct


# ---------------------------------------------------------------- GPU arm

def _event_time(fn, steps, warmup, stream):
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def secondary_workloads(steps, warmup, tc_peak):
    """Forward-only tokens/s at T=4096 (uniform and Zipf-skewed routing), the
    bench step with bf16 weight gradients and with the FP8 cache of g|u, and the
    expert-parallel rank workload (grouped SwiGLU GEMMs + return to arrival
    order, 14 experts x 65536 rows), each timed with CUDA events after warm-up.
    Returns a dict for the JSON line."""
    import numpy as np
    import torch

    from sparse_moe_layer_topk_gb300 import _lib as M
    from sparse_moe_layer_topk_gb300 import inputs as I
    from sparse_moe_layer_topk_gb300.layer import LatentMoELayer, weights_to_device
    out = {}
    stream = torch.cuda.current_stream()
    for cid in (1, 2):
        cfg = I.CONFIGS[cid]
        inp = I.make_layer_inputs(cfg)
        layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32)
        x = inp["x"].cuda()
        ms = _event_time(lambda: layer.forward(x), steps, warmup, stream)
        counts = layer.counts.cpu().numpy()
        out[cfg.name] = {"forward_ms": round(ms, 4), "tokens_per_s": cfg.T / (ms / 1000.0),
                         "experts_with_0_to_2_rows": int((counts <= 2).sum())}
        # grouped experts alone: natural expert order vs bucketed order (big experts first)
        w_ = layer.w
        E, R, l, f = cfg.E, layer.R, cfg.l, cfg.f
        order = torch.empty(E, dtype=torch.int32, device="cuda")
        sched_o = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        M.moe_expert_buckets(layer.counts, E, order, sched_o)

        def natural():
            M.moe_grouped_swiglu(layer.z_perm, w_["W13"], w_["W2"], layer.offsets,
                                 layer.tile_sched, layer.row_w, E, R, l, f, layer.gu, layer.h,
                                 layer.y_perm)

        def bucketed():
            M.moe_grouped_swiglu_ordered(layer.z_perm, w_["W13"], w_["W2"], layer.offsets, sched_o,
                                         order, layer.row_w, E, R, l, f, layer.gu, layer.h,
                                         layer.y_perm)
        out[cfg.name]["grouped_swiglu_ms"] = round(_event_time(natural, steps, warmup, stream), 4)
        out[cfg.name]["grouped_swiglu_bucketed_ms"] = round(
            _event_time(bucketed, steps, warmup, stream), 4)
        del layer, inp, x
        torch.cuda.empty_cache()
    # the bench step with bf16 weight gradients (halves the expert gradient writes)
    cfg = I.CONFIGS[4]
    inp = I.make_layer_inputs(cfg)
    layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_BF16)
    x, g = inp["x"].cuda(), inp["g"].cuda()
    layer.step(x, g)
    graph = layer.capture_step(x, g)
    ms = _event_time(graph.replay, steps, warmup, stream)
    out[cfg.name + "_bf16_wgrad"] = {"ms_per_step": round(ms, 4),
                                      "tokens_per_s": cfg.T / (ms / 1000.0)}
    del graph, layer
    torch.cuda.empty_cache()
    # the bench step with the routed experts' g|u cached in FP8 for the backward
    layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32, fp8_cache=True)
    layer.step(x, g)
    graph = layer.capture_step(x, g)
    ms = _event_time(graph.replay, steps, warmup, stream)
    M.moe_timing_report()
    M.moe_timing_enable(True)
    _event_time(lambda: layer.step(x, g), steps, 0, stream)
    M.moe_timing_enable(False)
    per = M.moe_timing_report()
    R, f = cfg.T * cfg.k, cfg.f
    out[cfg.name + "_fp8_cache"] = {
        "ms_per_step": round(ms, 4), "tokens_per_s": cfg.T / (ms / 1000.0),
        "gu_cache_bytes": R * 2 * f + R * (2 * f // 64) * 4, "gu_bf16_bytes": R * 2 * f * 2,
        "kernels_us": {n: round(per[n][1] / per[n][0] * 1000.0, 2)
                       for n in ("expert_gemm1_swiglu", "expert_dgrad2_swiglu_bwd") if n in per}}
    del graph, layer, inp, x, g
    torch.cuda.empty_cache()
    ep = I.make_ep_rank_inputs()
    c = ep["cfg"]
    counts = ep["counts"].numpy().astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    sched = np.concatenate([[0], np.cumsum((counts + 127) // 128)]).astype(np.int32)
    z, W13, W2, w = (ep["z_perm"].cuda(), ep["W13"].cuda(), ep["W2"].cuda(), ep["w"].cuda())
    off, sch = torch.from_numpy(offsets).cuda(), torch.from_numpy(sched).cuda()
    perm = ep["perm"].numpy()
    inv = np.empty(c.R, dtype=np.int32)
    inv[perm] = np.arange(c.R, dtype=np.int32)
    slot = torch.from_numpy(inv).reshape(c.R, 1).cuda()
    h = torch.empty(c.R, c.f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(c.R, c.l, dtype=torch.bfloat16, device="cuda")
    o = torch.empty(c.R, c.l, dtype=torch.bfloat16, device="cuda")

    def ep_step():
        M.moe_grouped_swiglu(z, W13, W2, off, sch, w, c.E, c.R, c.l, c.f, None, h, y)
        M.moe_unpermute_combine(y, slot, None, c.R, 1, c.l, o)

    M.moe_timing_report()
    M.moe_timing_enable(True)
    ms = _event_time(ep_step, steps, warmup, stream)
    M.moe_timing_enable(False)
    per = M.moe_timing_report()
    g_ms = sum(per[n][1] for n in ("expert_gemm1_swiglu", "expert_gemm2_rowscale") if n in per)
    g_n = per.get("expert_gemm1_swiglu", (1, 0))[0]
    flops = 2 * c.R * c.l * 2 * c.f + 2 * c.R * c.f * c.l
    g_avg = g_ms / max(g_n, 1) / 1000.0
    out[c.name] = {"ms": round(ms, 4), "rows_per_s": c.R / (ms / 1000.0),
                   "grouped_gemm_tflops": flops / g_avg / 1e12,
                   "grouped_gemm_pct_bf16_peak": 100.0 * flops / g_avg / 1e12 / tc_peak}
    return out


def run_ours(args):
    import torch
    import torch.distributed as dist

    from sparse_moe_layer_topk_gb300 import _lib as M
    from sparse_moe_layer_topk_gb300 import build as B
    from sparse_moe_layer_topk_gb300 import inputs as I
    from sparse_moe_layer_topk_gb300.layer import LatentMoELayer, weights_to_device

    world, rank, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        B.build_library()
    if world > 1:
        dist.barrier()
    M.load()
    cfg = workload(args)
    T = cfg.T
    inp = I.make_layer_inputs(cfg)
    wdt = M.MOE_DTYPE_F32 if args.wgrad == "f32" else M.MOE_DTYPE_BF16
    layer = LatentMoELayer(weights_to_device(inp), T, cfg.k, wdt, fused_gather=args.fused_gather)
    x = inp["x"].cuda()
    g = inp["g"].cuda()
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()

    for _ in range(args.warmup):
        layer.step(x, g)
    torch.cuda.synchronize()
    if int(layer.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(layer.err.item())}")

    # ---- device-timed region
    dev_uuid = None
    try:
        dev_uuid = "GPU-" + str(torch.cuda.get_device_properties(local).uuid)
    except Exception:
        dev_uuid = str(local)
    clocks = ClockSampler(dev_uuid)
    graph = None
    if not args.no_graph:
        # the step as one CUDA graph (no host launch gaps), replayed K times
        graph = layer.capture_step(x, g)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()

    def timed(fn, per_kernel_events):
        M.moe_timing_report()  # drop anything recorded so far
        M.moe_timing_enable(per_kernel_events)
        barrier()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record(stream)
        for _ in range(args.steps):
            fn()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier()
        M.moe_timing_enable(False)
        rep = M.moe_timing_report()
        t_ms = max_over_ranks(ev0.elapsed_time(ev1), world, "cuda")
        return t_ms, rep

    clocks.start()
    # per-kernel CUDA events over K eager steps (launch durations for the roofline)
    ms_eager, per_kernel = timed(lambda: layer.step(x, g), True)
    if graph is not None:
        ms, _ = timed(graph.replay, False)
    else:
        ms = ms_eager
    clk = clocks.stop()
    timing_desc = "CUDA-graph replays of the step" if graph is not None else "eager launches"
    value = job_tokens_per_s(world, T, args.steps, ms)
    launches = sum(c for c, _ in per_kernel.values())  # the same kernels, once per step

    # ---- end to end: pinned host inputs in, input gradient out, every step
    e2e = None
    if not args.no_e2e:
        xh = inp["x"].pin_memory()
        gh = inp["g"].pin_memory()
        dxh = torch.empty_like(xh).pin_memory()
        use_graphs = not args.no_graph
        layer.steps_from_host([xh] * 2, [gh] * 2, [dxh] * 2, graphs=use_graphs)  # warm up
        barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        # every step copies its x and dout in from pinned host memory and its dx
        # out; the copies overlap the neighbouring steps' compute
        layer.steps_from_host([xh] * args.steps, [gh] * args.steps, [dxh] * args.steps,
                              graphs=use_graphs)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ems = max_over_ranks(e0.elapsed_time(e1), world, "cuda")
        e2e = {"value": job_tokens_per_s(world, T, args.steps, ems), "unit": "tokens/s",
               "h2d_bytes_per_step": int(xh.numel() * 2 + gh.numel() * 2),
               "d2h_bytes_per_step": int(dxh.numel() * 2)}

    if int(layer.err.item()) != 0:
        raise RuntimeError(f"device error flag {int(layer.err.item())}")

    # ---- roofline of the dominant kernel
    peak_file = load_peaks()
    peaks = roofline_peaks(peak_file)
    tc, tc_src = peaks[2], peaks[3]
    # the secondary workloads time their kernels on their own: burst peak
    tc_burst, tc_burst_src = burst_tc_peak(peak_file)
    work = kernel_work(cfg, T, 4 if args.wgrad == "f32" else 2)
    # the DRAM traffic on record was captured with fp32 weight gradients
    roof, breakdown, grouped_pct = roofline_report(
        per_kernel, work, peaks,
        lambda name: dram_traffic(name, cfg.name) if args.wgrad == "f32" else None,
        executed=dense_executed_flops(cfg, T))

    secondary = None
    if rank == 0 and not args.no_secondary and not (args.tokens or args.experts):
        del layer, graph
        torch.cuda.empty_cache()
        secondary = secondary_workloads(20, 3, tc_burst)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        n = args.cpu_sample_tokens
        secs = oracle_sample_time(inp, n)
        cpu = {"value": n / secs, "unit": "tokens/s", "cores": host_threads(), "kind": "oracle",
               "sample": f"fwd+bwd of the first {n} tokens of the workload, full weights, "
                         f"{secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": cfg.name, "T": T, "d": cfg.d, "l": cfg.l, "E": cfg.E,
                       "k": cfg.k, "S": cfg.S, "f": cfg.f, "wgrad_dtype": args.wgrad,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (2.8 GB of expert weights and >1 GB of "
                             "activations streamed per step); no explicit flush"},
            "roofline": roof,
            "grouped_gemm_pct_bf16_peak": grouped_pct,
            "grouped_gemm_peak": {"tflops": tc, "source": tc_src},
            "secondary": secondary,
            "secondary_peak": {"tflops": tc_burst, "source": tc_burst_src},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "timing": {"value": timing_desc,
                       "kernels": "CUDA events around every launch over K eager steps",
                       "ms_per_step_eager": ms_eager / args.steps},
            "clocks": clk,
            "kernels": breakdown,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- single entry points

def entry_point_case(name, T, E, k, l):
    """A closure that calls one libmoe entry point on synthetic inputs of the
    given sizes; only the buffers that entry point touches are allocated."""
    import torch

    from sparse_moe_layer_topk_gb300 import _lib as M
    from sparse_moe_layer_topk_gb300 import inputs as I
    dev = "cuda"
    if name == "topk":
        L = I.make_logits(1, T, E).to(dev)
        idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        w = torch.empty(T, k, dtype=torch.float32, device=dev)
        s = torch.empty(T, k, dtype=torch.float32, device=dev)
        return lambda: M.moe_topk_from_logits(L, None, T, E, k, idx, w, s)
    ids = I.make_topk_ids(2, T, E, k).to(dev)
    R = T * k
    if name == "permute":
        z = torch.randn(T, l, device=dev).to(torch.bfloat16)
        zp = torch.empty(R, l, dtype=torch.bfloat16, device=dev)
        bufs = [torch.empty(n, dtype=torch.int32, device=dev) for n in (E, E + 1, R, R, E + 1)]
        wsb = M.moe_workspace_size(M.MOE_OP_PERMUTE, T=T, E=E)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        return lambda: M.moe_permute(z, ids, None, T, l, E, k, zp, bufs[0], bufs[1], bufs[2],
                                     bufs[3], bufs[4], None, ws, wsb)
    perm = torch.randperm(R, generator=torch.Generator().manual_seed(3))
    token_of = (perm // k).to(torch.int32).to(dev)
    slot_of = torch.empty(R, dtype=torch.int32)
    slot_of[perm] = torch.arange(R, dtype=torch.int32)
    slot_of = slot_of.to(dev)
    if name == "gather":
        src = torch.randn(T, l, device=dev).to(torch.bfloat16)
        dst = torch.empty(R, l, dtype=torch.bfloat16, device=dev)
        return lambda: M.moe_unpermute_combine_bwd(src, token_of, T, k, l, dst)
    yp = torch.randn(R, l, device=dev).to(torch.bfloat16)
    ysh = torch.randn(T, l, device=dev).to(torch.bfloat16)
    out = torch.empty(T, l, dtype=torch.bfloat16, device=dev)
    return lambda: M.moe_unpermute_combine(yp, slot_of, ysh, T, k, l, out)


def run_case(args):
    """One entry point alone, `--steps` calls after `--warmup`, CUDA-event timed
    (a case for ncu captures of single kernels); prints one JSON line."""
    import torch

    from sparse_moe_layer_topk_gb300 import _lib as M
    from sparse_moe_layer_topk_gb300 import build as B
    B.build_library()
    M.load()
    cfg = workload(args)
    fn = entry_point_case(args.case, cfg.T, cfg.E, cfg.k, cfg.l)
    ms = _event_time(fn, args.steps, max(1, args.warmup), torch.cuda.current_stream())
    print(json.dumps({"case": args.case, "workload": cfg.name, "T": cfg.T, "E": cfg.E,
                      "k": cfg.k, "l": cfg.l, "avg_us": 1000.0 * ms, "calls": args.steps}),
          flush=True)


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    elif args.case:
        run_case(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
