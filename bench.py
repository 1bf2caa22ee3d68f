#!/usr/bin/env python3
"""Benchmark of the MoE feed-forward layer (hidden 4096, expert width 14336,
8 experts, top-2, bf16) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config decode|prefill|skewed]
    python bench.py --impl reference ...      # the CPU oracle, timed as the reference arm

One step = one whole layer forward (router, grouping, both grouped expert
GEMMs, combine) over one batch of T tokens already resident in HBM.  Prints
one JSON line (rank 0).  With N > 1 (torchrun) every rank runs its own batch
against replicated weights: no data-path collective; the timed region is
bracketed by barriers and the slowest rank's time is reported ("weak"
scaling).  Every step streams the layer's 2.8 GB of expert weights, far more
than the 126 MB L2, so no flush is needed between steps.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (d4096 ffn14336 E8 top2 bf16) + % of HBM/TC roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# ---------------------------------------------------------------- distributed

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(value: float, world: int, device) -> float:
    """Largest value over ranks (outside any timed region)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_token_seed(base_seed: int, rank: int) -> int:
    """Each rank draws its own batch of tokens (weights are shared)."""
    return base_seed + 7919 * rank


# ---------------------------------------------------------------- peaks, clocks

GEMM_SOURCES = ("sparse_mixture_experts_58_b300/csrc/gemm_tc.cu",
                "sparse_mixture_experts_58_b300/csrc/gemm_pair.cu",
                "sparse_mixture_experts_58_b300/csrc/ptx.cuh",
                "sparse_mixture_experts_58_b300/csrc/common.cuh")


def uses_pairs(T, k, E) -> bool:
    """Whether the library's tile plan runs the expert GEMMs on CTA pairs
    (at least 128 rows per expert on average, unless overridden)."""
    wide = (T * k) // E >= 128
    if os.environ.get("MOE_PLAN_WIDE"):
        wide = int(os.environ["MOE_PLAN_WIDE"]) != 0
    if os.environ.get("MOE_PLAN_PAIR"):
        return int(os.environ["MOE_PLAN_PAIR"]) != 0
    return wide


def gemm_source_hash() -> str:
    """Hash of the tensor-core GEMM's device sources (ties recorded ncu
    counters to the kernel they were taken on)."""
    import hashlib
    h = hashlib.sha256()
    for p in GEMM_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(key: str):
    """DRAM bytes (read + write) per launch from the committed ncu summary,
    or None when absent or taken on a different kernel source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    ent = d.get(key)
    if not ent or ent.get("source_hash") != gemm_source_hash():
        return None
    return ent.get("bytes_per_launch")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in PEAKS_FALLBACK}, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


class _Nvml:
    """Read-only NVML queries through the driver's libnvidia-ml (ctypes):
    SM clock, its maximum, and the active clock-event reasons."""

    def __init__(self, index):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
            raise RuntimeError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def sm_mhz(self):
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(v))   # 1 = SM clock
        return v.value

    def sm_max_mhz(self):
        v = self.ct.c_uint()
        self.lib.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(v))
        return v.value

    def reasons(self):
        v = self.ct.c_ulonglong()
        self.reasons_fn(self.h, self.ct.byref(v))
        return v.value


class ClockSampler:
    """NVML samples (SM clock, max clock, clock-event reasons) every few ms
    while running; read-only.  Uses the driver's NVML library directly."""

    REASONS = {
        "gpu_idle": 0x1, "applications_clocks_setting": 0x2, "sw_power_cap": 0x4,
        "hw_slowdown": 0x8, "sync_boost": 0x10, "sw_thermal_slowdown": 0x20,
        "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80,
        "display_clock_setting": 0x100,
    }

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples = []
        self.period = period_s
        self.ok = False
        self.max_mhz = None
        try:
            self.nv = _Nvml(index)
            self.max_mhz = self.nv.sm_max_mhz()
            self.ok = True
        except Exception as e:  # no NVML: report that instead of clocks
            self.err = repr(e)
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append((self.nv.sm_mhz(), self.nv.reasons()))
            except Exception:
                pass
            time.sleep(self.period)

    def start(self):
        """Start (or resume) sampling; samples accumulate across start/stop."""
        if self.ok:
            self._stop.clear()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()

    def stop(self):
        if self._t is not None:
            self._stop.set()
            self._t.join()
            self._t = None

    def summary(self):
        if not self.ok:
            return {"error": getattr(self, "err", "nvml unavailable")}
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0}
        mhz = [m for m, _ in self.samples]
        seen = 0
        for _, r in self.samples:
            seen |= r
        reasons = [name for name, bit in self.REASONS.items() if seen & bit and name != "gpu_idle"]
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": min(mhz), "reasons": reasons, "samples": len(mhz)}


# ---------------------------------------------------------------- workload

WORKLOAD_NAMES = {
    "decode": "Mixtral MoE layer, decode: T=16, d=4096, ffn=14336, E=8, top-2, bf16",
    "prefill": "Mixtral MoE layer, prefill: T=4096, d=4096, ffn=14336, E=8, top-2, bf16",
    "skewed": "Mixtral MoE layer, skewed routing: T=8192, bias [+2,+1,0,0,0,0,-1,-2], "
              "5% duplicate tokens, d=4096, ffn=14336, E=8, top-2, bf16",
}


def algorithmic(T, d, ffn, E, k, n_touched, rows=None):
    """Algorithmic FLOPs and HBM bytes of one layer forward (what the method
    must do: the expert rows computed -- T*k, or the kept ones under a
    capacity limit -- the touched experts' weights once, the router weights,
    x in, out)."""
    rows = T * k if rows is None else rows
    flops = rows * 2 * 3 * d * ffn + T * 2 * d * E
    bytes_ = n_touched * 3 * d * ffn * 2 + d * E * 2 + 2 * T * d * 2 + T * E * 4
    return flops, bytes_


def gemm1_algorithmic(rows, d, ffn, n_touched):
    """Gate/up grouped GEMM, per launch: FLOPs and bytes (W1+W3 of touched
    experts, grouped rows in, hidden activations out)."""
    flops = 4 * rows * d * ffn
    bytes_ = n_touched * 2 * d * ffn * 2 + rows * d * 2 + rows * ffn * 2
    return flops, bytes_


# ---------------------------------------------------------------- reference arm

def run_reference(args, rank, world):
    """Times the CPU oracle (as it stands) on the host cores, on bounded
    samples of the same workload.  Rank 0 only."""
    if rank != 0:
        return 0
    import torch

    import oracle
    from sparse_mixture_experts_58_b300 import inputs

    dev = "cuda" if torch.cuda.is_available() else "cpu"
    cfg, overrides = workload_cfg(args, args.config)
    x, layer = inputs.make_workload(cfg["T"], cfg["d"], cfg["ffn"], cfg["E"], cfg["k"],
                                    cfg["dtype"], cfg["seed"], dev, cfg.get("bias"),
                                    cfg.get("dup_frac", 0.0))
    T = x.shape[0]
    k = cfg["k"]
    host = inputs.layer_to_host(layer)
    xh = inputs.to_host(x)
    o = oracle.load()
    cores = o.max_threads()
    n = max(1, min(T, cores))          # one token per host thread per step
    rng = __import__("numpy").random.default_rng(0)

    def step(i):
        rows = rng.choice(T, size=n, replace=False)
        o.moe_forward(xh[rows], *host[:4], k, bias=host[4])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_record(args.config, cfg, overrides, world),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} seeded tokens of the {T}-token batch per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def cpu_baseline(x, layer, k, budget_s=12.0):
    """The oracle as it stands on all host threads, on the benchmark batch,
    repeated until about `budget_s` of CPU wall time."""
    import oracle
    from sparse_mixture_experts_58_b300 import inputs
    o = oracle.load()
    host = inputs.layer_to_host(layer)
    T = x.shape[0]
    n = min(T, 64)
    xh = inputs.to_host(x[:n])
    done, t_total, reps = 0, 0.0, 0
    while t_total < budget_s and reps < 50:
        t0 = time.perf_counter()
        o.moe_forward(xh, *host[:4], k, bias=host[4])
        t_total += time.perf_counter() - t0
        done += n
        reps += 1
    return {"value": done / t_total, "unit": "tokens/s", "cores": o.max_threads(),
            "kind": "oracle",
            "sample": f"first {n} tokens of the batch, {reps} pass(es), {t_total:.1f} s"}


# ---------------------------------------------------------------- our arm

def workload_cfg(args, name):
    """The named workload's shape with the command line's overrides (T, E, k)
    applied; returns (cfg, overrides)."""
    from sparse_mixture_experts_58_b300 import inputs
    cfg = dict(inputs.WORKLOADS[name])
    overrides = []
    for key in ("T", "E", "k"):
        v = getattr(args, key, 0)
        if v:
            cfg[key] = v
            overrides.append(f"{key}={v}")
    if cfg.get("bias") is not None and len(cfg["bias"]) != cfg["E"]:
        cfg["bias"] = (list(cfg["bias"]) + [0.0] * cfg["E"])[:cfg["E"]]
    return cfg, overrides


def config_record(name, cfg, overrides, world):
    """The line's `config`: the workload and its shape only (the same for
    both arms; what a run observes, such as the routing, goes elsewhere)."""
    workload = WORKLOAD_NAMES[name]
    if overrides:
        workload = f"{workload} ({'; '.join(overrides)})"
    T, d, ffn, E, k = cfg["T"], cfg["d"], cfg["ffn"], cfg["E"], cfg["k"]
    return {"workload": workload, "T": T, "d": d, "ffn": ffn, "E": E, "k": k,
            "tokens_per_gpu": T, "parallelism": f"replicas x{world} (no data-path collective)",
            "l2": "no flush: each step streams the touched experts' weights (up to "
                  f"{E * 3 * d * ffn * 2 / 1e9:.2f} GB) > 126 MB L2"}


def route_options(args, T, k, E):
    """Routing options from the command line: (moe.forward keywords,
    descriptions for the workload name)."""
    from sparse_mixture_experts_58_b300 import moe
    cap = moe.capacity(args.capacity_factor, T, k, E) if args.capacity_factor > 0 else 0
    policy = 1 if args.drop_policy == "renorm" else 0
    route_kw = dict(gating=args.gating, capacity=cap, drop_policy=policy if cap else 0)
    notes = []
    if args.gating:
        notes.append("gating: softmax over all experts, then top-k")
    if cap:
        notes.append(f"capacity factor {args.capacity_factor} -> {cap} rows/expert, "
                     f"dropped mass {'renormalised' if policy else 'lost'}")
    for var in ("MOE_PLAN_WIDE", "MOE_PLAN_PAIR", "MOE_PLAN_SPLITS", "MOE_PLAN_BM", "MOE_PDL",
                "MOE_TC_NARROW", "MOE_FUSE_COMBINE", "MOE_GRAPHS"):
        if os.environ.get(var):
            notes.append(f"{var}={os.environ[var]}")
    return route_kw, notes


def bench_layer(args, name, cfg, route_kw, dev, rank, world, local, steps, warmup,
                with_e2e=False, traffic_key=None):
    """One workload: the forward as a CUDA-graph replay of one moe_forward
    call per step (CUDA events on the launching stream, barriers and the
    slowest rank's time), the same call made directly, a per-stage
    breakdown through the stage entry points and, with `with_e2e`, the
    end-to-end figure through the host-buffer entry point.  Returns a dict
    (rank 0's view of the job)."""
    import torch

    from sparse_mixture_experts_58_b300 import inputs, moe

    T, d, ffn, E, k = cfg["T"], cfg["d"], cfg["ffn"], cfg["E"], cfg["k"]
    # weights shared by every rank; tokens per rank
    gen = inputs.generator(cfg["seed"], dev)
    x0, _ = inputs.draw_tokens(gen, T, d, "bf16", dev, cfg.get("dup_frac", 0.0))
    layer = inputs.draw_weights(gen, d, ffn, E, "bf16", dev, cfg.get("bias"))
    if rank > 0:
        x0, _ = inputs.draw_tokens(inputs.generator(rank_token_seed(cfg["seed"], rank), dev),
                                   T, d, "bf16", dev, cfg.get("dup_frac", 0.0))
    x = x0.contiguous()
    out = torch.empty_like(x)
    ws = moe.Workspace(dev)
    bias = layer.bias
    cap = route_kw["capacity"]

    def step():
        moe.forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=bias, out=out,
                    workspace=ws, **route_kw)

    # routing of this batch: kept rows per expert (for the algorithmic counts)
    logits0, _, _ = moe.router(x, layer.Wg, k, bias)
    _, _, kept_counts, _, _, _ = moe.route_from_logits(logits0, k, gating=route_kw["gating"],
                                                       capacity=cap)
    counts = kept_counts.cpu()
    n_touched = int((counts > 0).sum())
    rows_kept = int(counts.sum())

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    # The timed step is the forward captured once into a CUDA graph (the same
    # C-ABI call and kernels; replays cost one graph launch of host time).
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
        for _ in range(warmup):
            graph.replay()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step

    def timed(fn, n, on=stream):
        barrier(world)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(on)
        for _ in range(n):
            fn()
        e1.record(on)
        torch.cuda.synchronize()
        barrier(world)
        return reduce_max(e0.elapsed_time(e1) / 1e3, world, dev)

    clocks = ClockSampler(local)
    clocks.start()
    elapsed_max = timed(run, steps)
    clocks.stop()
    status = moe.device_status(clear=True)
    if status != 0:
        raise RuntimeError(f"device status {status} after the timed region")
    # the same forward called directly (host launch overhead included)
    direct_elapsed = timed(step, steps)

    # -- per-stage breakdown through the stage entry points (same kernels),
    #    events on the launching stream between stages; a sleep kernel first
    #    lets the host queue the whole sequence so the events see GPU time
    stage_names = ["router", "route", "permute", "gate_up_swiglu", "down", "combine"]
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(len(stage_names) + 1)]
    acc = [0.0] * len(stage_names)
    n_rep = max(3, min(steps, 50))
    for rep in range(n_rep + 2):
        torch.cuda._sleep(2_000_000)
        evs[0].record(stream)
        logits, _, _ = moe.router(x, layer.Wg, k, bias)
        evs[1].record(stream)
        _, gates2, _, offsets, perm, inv = moe.route_from_logits(
            logits, k, gating=route_kw["gating"], capacity=cap)
        evs[2].record(stream)
        xp = moe.permute(x, perm, k, rows=rows_kept)
        evs[3].record(stream)
        h = moe.expert_swiglu(xp, offsets, layer.W1, layer.W3)
        evs[4].record(stream)
        y = moe.expert_down(h, offsets, layer.W2, T, k)
        evs[5].record(stream)
        moe.combine(y, gates2, inv, T, k, torch.bfloat16)
        evs[6].record(stream)
        torch.cuda.synchronize()
        if rep >= 2:
            for i in range(len(stage_names)):
                acc[i] += evs[i].elapsed_time(evs[i + 1]) / 1e3
    stage_s = [a / n_rep for a in acc]
    del h, y, xp

    res = {}
    if with_e2e and not (route_kw["gating"] or cap):
        # -- end to end through the C ABI's host-buffer call: every step is one
        #    moe_forward_host_io call with the tokens in pinned host memory and
        #    the output written back to pinned host memory; the library enqueues
        #    the copy in, the layer and the copy out on the stream, so the
        #    copies sit inside each step (nothing overlaps them)
        x_host = x.cpu().pin_memory()
        out_host = torch.empty_like(x_host).pin_memory()
        x_dev, out_dev = torch.empty_like(x), torch.empty_like(x)

        def e2e_step():
            moe.forward_host_io(x_host, layer.Wg, layer.W1, layer.W3, layer.W2, k, bias=bias,
                                out_host=out_host, x_dev=x_dev, out_dev=out_dev, workspace=ws,
                                stream=stream)

        for _ in range(warmup):
            e2e_step()
        torch.cuda.synchronize()
        e2e_elapsed = timed(e2e_step, steps)
        res["e2e"] = {"value": T * world * steps / e2e_elapsed, "unit": "tokens/s",
                      "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                      "d2h_bytes_per_step": out_host.numel() * out_host.element_size(),
                      "how": "per step one moe_forward_host_io call (the C ABI's host-buffer "
                             "entry point), all on one stream: the pinned host tokens are read "
                             "over the bus by the router (batches under 1536 tokens; larger "
                             "ones are copied to the device first), the layer runs, and its "
                             "last kernel writes the output into pinned host memory",
                      "output_matches_device_path": bool(torch.equal(out_host, out.cpu()))}

    peaks, peak_src = load_peaks()
    flops, bytes_ = algorithmic(T, d, ffn, E, k, n_touched, rows=rows_kept)
    t_step = elapsed_max / steps
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    t_roof = max(t_hbm, t_tc)
    layer_bound = "hbm" if t_hbm > t_tc else "tensor"
    g_flops, g_bytes = gemm1_algorithmic(rows_kept, d, ffn, n_touched)
    t_g = stage_s[3]
    g_bound = "hbm" if g_bytes / (peaks["hbm_gbs"] * 1e9) > g_flops / (peaks["bf16_tflops"] * 1e12) else "tensor"
    if g_bound == "hbm":
        achieved, peak, unit = g_bytes / t_g / 1e9, peaks["hbm_gbs"], "GB/s"
    else:
        achieved, peak, unit = g_flops / t_g / 1e12, peaks["bf16_tflops"], "TFLOP/s"
    res.update({
        "value": T * world * steps / elapsed_max,
        "ms_per_step": t_step * 1e3,
        "routing": {"experts_touched": n_touched, "rows_per_expert": counts.tolist(),
                    "rows_computed": rows_kept, "options": route_kw},
        "roofline": {
            "kernel": "grouped gate/up GEMM + SwiGLU (tcgen05, "
                      + ("CTA pairs, tokens as N)" if uses_pairs(T, k, E) else "one CTA per tile)"),
            "bound": g_bound, "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "peak_source": f"{peak_src} (burst)",
            "traffic": recorded_traffic(traffic_key) if traffic_key else None,
            "traffic_source": "profiles/ncu_traffic.json (dram__bytes_read.sum + "
                              "dram__bytes_write.sum, one ncu capture; null if the kernel "
                              "source changed since)",
            "algorithmic_per_launch": {"bytes": g_bytes, "flops": g_flops},
            "launch_us": t_g * 1e6,
        },
        "layer_roofline": {
            "bound": layer_bound, "roofline_us": t_roof * 1e6, "measured_us": t_step * 1e6,
            "frac": t_roof / t_step, "algorithmic_bytes": bytes_, "algorithmic_flops": flops,
            "frac_vs_sustained_tc": (max(t_hbm, flops / (peaks["bf16_tflops_sustained"] * 1e12))
                                     / t_step),
        },
        "stages_us": {n: s * 1e6 for n, s in zip(stage_names, stage_s)},
        "timed_as": "CUDA graph replay of one moe_forward call per step" if graph is not None
                    else "moe_forward called per step",
        "direct_call_tokens_per_s": T * world * steps / direct_elapsed,
        "gpu_launches": moe.forward_launches(T, d, ffn, E, k, moe.BF16) * steps,
        "clocks": clocks.summary(),
    })
    res["_x"], res["_layer"] = x, layer
    return res


def measure(args, rank, world, local):
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    cfg, overrides = workload_cfg(args, args.config)
    T, E, k = cfg["T"], cfg["E"], cfg["k"]
    route_kw, notes = route_options(args, T, k, E)
    config = config_record(args.config, cfg, overrides + notes, world)
    tkey = None if (overrides or notes) else f"gate_up_{args.config}"
    r = bench_layer(args, args.config, cfg, route_kw, dev, rank, world, local, args.steps,
                    args.warmup, with_e2e=True, traffic_key=tkey)
    x, layer = r.pop("_x"), r.pop("_layer")
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x, layer, k)
    del x, layer
    # the tensor-core half of the metric: prefill T=4096 in the same run
    sub = None
    if args.config == "decode" and not (overrides or notes) and not args.no_prefill:
        torch.cuda.empty_cache()
        pcfg, _ = workload_cfg(argparse.Namespace(), "prefill")
        pkw, _ = route_options(argparse.Namespace(capacity_factor=0.0, drop_policy="lose",
                                                  gating=0), pcfg["T"], pcfg["k"], pcfg["E"])
        sub = bench_layer(args, "prefill", pcfg, pkw, dev, rank, world, local,
                          max(args.steps, 10), args.warmup, traffic_key="gate_up_prefill")
        sub.pop("_x")
        sub.pop("_layer")
        sub = {"config": config_record("prefill", pcfg, [], world), "unit": "tokens/s",
               "steps": max(args.steps, 10), **sub}
        torch.cuda.empty_cache()
    if rank != 0:
        return 0
    line = {
        "metric": METRIC,
        "value": r.pop("value"),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": r.pop("ms_per_step"),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded x~N(0,1), weights~N(0,1/fan_in), random init",
        "config": config,
        **r,
    }
    if sub is not None:
        line["prefill"] = sub
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)
    return 0


def measure_sweep(args, rank, world, local):
    """Token-count sweep: for each T, the 32-layer chain
    x <- x + MoE_l(RMSNorm(x)) with independent layer weights (90 GB resident),
    captured as one CUDA graph and replayed; reports per-T chain time, per-layer
    time and the fraction of the per-layer roofline."""
    import torch

    from sparse_mixture_experts_58_b300 import inputs, moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    cfg = inputs.WORKLOADS["sweep"]
    d, ffn, E, k, L = cfg["d"], cfg["ffn"], cfg["E"], cfg["k"], cfg["layers"]
    Ts = [int(t) for t in args.sweep_T.split(",")] if args.sweep_T else list(cfg["Ts"])
    layers = [inputs.sweep_layer(l, d, ffn, E, device=dev, seed0=cfg["layer_seed0"])
              for l in range(L)]
    peaks, peak_src = load_peaks()
    ws = moe.Workspace(dev)
    stream = torch.cuda.current_stream()
    results = []
    clocks = ClockSampler(local)
    tot_tokens, tot_time = 0, 0.0
    for T in Ts:
        x0 = inputs.sweep_tokens(T, d, device=dev, seed=rank_token_seed(cfg["seed"], rank))
        x, xn = x0.clone(), torch.empty_like(x0)
        ws.get(moe.workspace_bytes(T, d, ffn, E, k, moe.BF16))

        # one pre-norm block per layer: x <- x + MoE(RMSNorm(x)), the RMSNorm
        # and the residual add fused into the layer's kernels
        def chain():
            x.copy_(x0)
            for layer in layers:
                moe.block_forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, eps=1e-5,
                                  workspace=ws)

        # experts touched per layer on this batch (for the byte roofline)
        chain()
        torch.cuda.synchronize()
        x.copy_(x0)
        touched = []
        for layer in layers:
            moe.add_rmsnorm(x, None, xn)
            _, idx, _ = moe.router(xn, layer.Wg, k)
            touched.append(int((torch.bincount(idx.flatten().long(), minlength=E) > 0).sum()))
            moe.block_forward(x, layer.Wg, layer.W1, layer.W3, layer.W2, k, eps=1e-5,
                              workspace=ws)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            chain()
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        g.replay()
        torch.cuda.synchronize()
        est = time.perf_counter() - t0
        reps = max(3, min(args.steps, int(0.5 / max(est, 1e-6))))
        barrier(world)
        clocks.start()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        clocks.stop()
        barrier(world)
        t_chain = reduce_max(e0.elapsed_time(e1) / 1e3 / reps, world, dev)
        if moe.device_status(clear=True) != 0:
            raise RuntimeError("device status set during the sweep")
        roof = 0.0
        for n in touched:
            f, b = algorithmic(T, d, ffn, E, k, n)
            b += T * d * 2                     # the residual add reads x once more
            roof += max(b / (peaks["hbm_gbs"] * 1e9), f / (peaks["bf16_tflops"] * 1e12))
        results.append({"T": T, "chain_ms": t_chain * 1e3, "layer_us": t_chain / L * 1e6,
                        "tokens_per_s_32_layers": T * world / t_chain,
                        "roofline_chain_ms": roof * 1e3, "frac": roof / t_chain,
                        "experts_touched_min": min(touched), "reps": reps})
        tot_tokens += T * world
        tot_time += t_chain
        del g
    if rank != 0:
        return 0
    last = results[-1]
    line = {
        "metric": METRIC + " [32-layer token-count sweep]",
        "value": last["tokens_per_s_32_layers"], "unit": "tokens/s (32-layer chain)",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": last["chain_ms"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded x~N(0,1), weights~N(0,1/fan_in), random init",
        "config": {"workload": "token-count sweep: T in " + ",".join(map(str, Ts)) +
                   ", 32 layers with independent weights, x <- x + MoE(RMSNorm(x)) "
                   "(one fused pre-norm block per layer), d=4096, ffn=14336, E=8, top-2, bf16",
                   "l2": "no flush: 90 GB of layer weights stream per chain"},
        "sweep": results,
        "peaks": {"source": peak_src, **peaks},
        "gpu_launches": L * moe.forward_launches(16, d, ffn, E, k, moe.BF16),
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def backward_algorithmic(T, d, ffn, E, k, n_touched):
    """FLOPs and bytes the layer's backward must move.  FLOPs: the gate/up
    projections again (4 T k d ffn), Z = dout W2 (2), dX = dU W1 + dV W3 (4),
    the three weight gradients (6), the router (4 T d E).  Bytes: W1 and W3
    of the touched experts read twice and W2 once, the fp32 weight gradients
    of every expert written (overwritten, zero for an untouched expert), x and
    dout read, dx written, the router matrix and its gradient."""
    flops = 16 * T * k * d * ffn + 4 * T * d * E
    bytes_ = (n_touched * 5 * d * ffn * 2 + E * 3 * d * ffn * 4 + 3 * T * d * 2
              + E * d * (2 + 4))
    return flops, bytes_


def measure_backward(args, rank, world, local):
    """The layer's backward (moe_backward): CUDA-graph replays of one call per
    step on the chosen workload, timed with CUDA events; the roofline counts
    the backward's algorithmic work at the measured peaks."""
    import torch

    from sparse_mixture_experts_58_b300 import inputs, moe

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist_init(world, "nccl")
    cfg = dict(inputs.WORKLOADS[args.config])
    overrides = []
    for key in ("T", "E", "k"):
        v = getattr(args, key)
        if v:
            cfg[key] = v
            overrides.append(f"{key}={v}")
    T, d, ffn, E, k = cfg["T"], cfg["d"], cfg["ffn"], cfg["E"], cfg["k"]
    if cfg.get("bias") is not None and len(cfg["bias"]) != E:
        cfg["bias"] = (list(cfg["bias"]) + [0.0] * E)[:E]
    workload = "backward of the " + WORKLOAD_NAMES[args.config]
    if overrides:
        workload = f"{workload} ({'; '.join(overrides)})"
    gen = inputs.generator(cfg["seed"], dev)
    x0, _ = inputs.draw_tokens(gen, T, d, "bf16", dev, cfg.get("dup_frac", 0.0))
    layer = inputs.draw_weights(gen, d, ffn, E, "bf16", dev, cfg.get("bias"))
    tok_gen = inputs.generator(rank_token_seed(cfg["seed"] + 17, rank), dev)
    if rank > 0:
        x0, _ = inputs.draw_tokens(inputs.generator(rank_token_seed(cfg["seed"], rank), dev),
                                   T, d, "bf16", dev, cfg.get("dup_frac", 0.0))
    x = x0.contiguous()
    dout = torch.randn(T, d, generator=tok_gen, device=dev).to(torch.bfloat16)
    grads = dict(dx=torch.empty_like(x),
                 dWg=torch.empty(E, d, dtype=torch.float32, device=dev),
                 dW1=torch.empty(E, ffn, d, dtype=torch.float32, device=dev),
                 dW3=torch.empty(E, ffn, d, dtype=torch.float32, device=dev),
                 dW2=torch.empty(E, d, ffn, dtype=torch.float32, device=dev))
    ws = moe.Workspace(dev)

    def step():
        moe.backward(x, layer.Wg, layer.W1, layer.W3, layer.W2, dout, k, bias=layer.bias,
                     workspace=ws, grads=grads)

    logits0, _, _ = moe.router(x, layer.Wg, k, layer.bias)
    _, _, counts, _, _, _ = moe.route_from_logits(logits0, k)
    n_touched = int((counts.cpu() > 0).sum())
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    barrier(world)
    elapsed = reduce_max(e0.elapsed_time(e1) / 1e3, world, dev)
    if moe.device_status(clear=True) != 0:
        raise RuntimeError("device status set during the timed region")
    if rank != 0:
        return 0
    peaks, peak_src = load_peaks()
    flops, bytes_ = backward_algorithmic(T, d, ffn, E, k, n_touched)
    t_step = elapsed / args.steps
    t_hbm = bytes_ / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    bound = "hbm" if t_hbm > t_tc else "tensor"
    achieved = (bytes_ / t_step / 1e9) if bound == "hbm" else (flops / t_step / 1e12)
    peak = peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops"]
    line = {
        "metric": "MoE-layer backward tokens/s (d4096 ffn14336 E8 top2 bf16; dx bf16, "
                  "weight gradients fp32)",
        "value": T * world / t_step, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded x~N(0,1), dout~N(0,1), weights~N(0,1/fan_in)",
        "config": {"workload": workload, "T": T, "d": d, "ffn": ffn, "E": E, "k": k,
                   "experts_touched": n_touched,
                   "l2": "no flush: each step reads the weights and writes the fp32 weight "
                         f"gradients ({(E * 3 * d * ffn * 4) / 1e9:.2f} GB) > 126 MB L2"},
        "roofline": {"kernel": "whole backward (12 kernels)", "bound": bound,
                     "achieved": achieved, "peak": peak,
                     "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak,
                     "peak_source": f"{peak_src} (burst)", "traffic": None,
                     "algorithmic_per_step": {"bytes": bytes_, "flops": flops},
                     "roofline_us": max(t_hbm, t_tc) * 1e6},
        "timed_as": "CUDA graph replay of one moe_backward call per step",
        "gpu_launches": 12 * args.steps,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


def relaunch(n: int, argv) -> int:
    """Run this script under torchrun with n ranks on this node (rendezvous on
    127.0.0.1); returns its exit code.  Rank 0 prints the line."""
    import socket
    import subprocess
    sock = socket.socket()
    sock.bind(("127.0.0.1", 0))
    port = sock.getsockname()[1]
    sock.close()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.abspath(__file__), *argv]
    return subprocess.run(cmd).returncode


def measure_dry(args, rank, world):
    """The multi-rank plumbing without a GPU: gloo process group, per-rank
    token batches against shared weights (drawn on the CPU), barriers around
    a timed region of host no-ops and the slowest rank's time.  Measures
    nothing about the layer; the line is marked as a dry run."""
    from sparse_mixture_experts_58_b300 import inputs
    dist_init(world, "gloo")
    T, d = 8, 64
    x, _ = inputs.draw_tokens(inputs.generator(rank_token_seed(0, rank), "cpu"), T, d, "bf16",
                              "cpu")
    layer = inputs.draw_weights(inputs.generator(1000, "cpu"), d, 64, 4, "bf16", "cpu")
    digest = (float(x.float().sum()), float(layer.W1.float().sum()))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        time.sleep(0.001)
    barrier(world)
    elapsed = reduce_max(time.perf_counter() - t0, world, "cpu")
    digests = [digest]
    if world > 1:
        import torch.distributed as dist
        digests = [None] * world
        dist.all_gather_object(digests, digest)
    if rank == 0:
        print(json.dumps({
            "metric": METRIC + " [dry run: no GPU work]", "dry_run": True,
            "value": T * world * args.steps / elapsed, "unit": "host no-op steps x tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "scaling": "weak", "ranks": [{"rank": i, "tokens_sum": dg[0], "w1_sum": dg[1]}
                                         for i, dg in enumerate(digests)]}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", choices=sorted(WORKLOAD_NAMES) + ["sweep"], default="decode")
    ap.add_argument("--sweep-T", default="", help="comma-separated token counts for --config sweep")
    ap.add_argument("--T", type=int, default=0, help="override the workload's token count")
    ap.add_argument("--E", type=int, default=0, help="override the number of experts")
    ap.add_argument("--k", type=int, default=0, help="override the experts per token")
    ap.add_argument("--gating", type=int, default=0, choices=[0, 1],
                    help="0: softmax over the kept logits; 1: softmax over all, then top-k")
    ap.add_argument("--capacity-factor", type=float, default=0.0,
                    help="rows per expert = ceil(factor * T * k / E); 0 = no limit")
    ap.add_argument("--drop-policy", choices=["lose", "renorm"], default="lose")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time direct moe_forward calls instead of a captured CUDA graph")
    ap.add_argument("--backward", action="store_true",
                    help="time the layer's backward (moe_backward) instead of the forward")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the prefill (T=4096) sub-record of the default decode run")
    ap.add_argument("--dry-run", action="store_true",
                    help="rank plumbing only, on CPU over gloo: no GPU work, no kernels "
                         "(the line says so); for tests of --gpus N")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # one process per GPU: relaunch this command under torchrun
        return relaunch(args.gpus, sys.argv[1:] if argv is None else list(argv))
    rank, world, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but the launch gives {world} rank(s)")
    if args.dry_run:
        return measure_dry(args, rank, world)
    if args.impl == "reference":
        if args.config == "sweep":
            args.config = "decode"
        return run_reference(args, rank, world)
    if args.config == "sweep":
        return measure_sweep(args, rank, world, local)
    if args.backward:
        return measure_backward(args, rank, world, local)
    return measure(args, rank, world, local)


if __name__ == "__main__":
    sys.exit(main())
