#!/usr/bin/env python3
"""Benchmark of the GB300 local MoE FFN forward.

One step = one pass of the whole path (route -> dispatch -> SwiGLU experts
-> combine) through the one-call ``moe_forward`` over one batch of the
coarse-grained prefill workload (T=16384 tokens, H=4096, I=14336, E=8
experts, top_k=2, BF16; the largest single-GPU workload) with inputs
resident in HBM. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

* ``value``: tokens/s of the whole job (all ranks), device time from CUDA
  events on the launching stream, L2 flushed (256 MiB write) between steps.
* ``e2e``: the same metric through the one-call C ABI (``moe_forward``) with
  pinned HOST buffers: each step copies x and logits in and y out.
* ``roofline``: the expert grouped GEMM (GEMM1 + GEMM2, the dominant
  kernels) inside the same one-call forward, timed by events recorded around
  its two launches (``moe_forward_ex``), with algorithmic FLOPs (6*H*I per
  assignment) and bytes (touched weights, x_disp, h twice, expert outputs)
  against the measured peak of the roof its intensity hits; ``kernels``
  gives every stage.
* ``cpu_baseline`` (rank 0, N=1): the CPU oracle on a bounded token sample.
* ``--impl reference``: the CPU oracle as the reference arm (rank 0 only).

Multi-GPU: every rank runs an independent replica on its own GPU (no
collective on the data path); the step time is the max over ranks. Under
torchrun each process is one rank; ``--gpus N`` without torchrun relaunches
this script under torch.distributed.run with N ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "MoE fwd tokens/s; expert GEMM TFLOP/s and combine GB/s as % of GB300 peak"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# GB300's nominal HBM3e bandwidth: HBM-bound lines also state their fraction
# of it (frac_nominal) beside the fraction of the measured copy bandwidth
NOMINAL_HBM_GBS = 8000.0
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS, source="fallback")


KERNEL_SOURCES = {"experts": ["experts_tc.cu", "tc_ptx.cuh", "common.cuh"],
                  "experts_bwd": ["experts_tc_bwd.cu", "tc_ptx.cuh", "common.cuh"],
                  "combine_add_rmsnorm": ["combine.cu", "common.cuh"]}


def source_digest(kernel):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "mixture_experts_ffn_topk_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(workload, kernel):
    """Per-launch DRAM bytes from the committed ncu summary, or None when
    the kernel's sources changed since the counters were taken."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
        entry = d.get(workload, {}).get(kernel)
        if not entry or entry.get("source") != source_digest(kernel):
            return None
        return entry["bytes"]
    except (OSError, ValueError, KeyError):
        return None


# ---------------------------------------------------------------- distributed

def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return rank, world, local, dist
    return 0, 1, 0, None


def barrier(dist, device):
    if dist is not None:
        if device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def reduce_max(dist, value, device):
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(step_s_max: float, tokens_per_rank: int, world: int) -> float:
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's step."""
    return tokens_per_rank * world / step_s_max


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """Samples the SM clock and clock-event (throttle) reasons of one GPU while
    the timed region runs: a background thread reads NVML through ctypes
    every millisecond (read-only queries). Falls back to nothing if NVML is
    unavailable."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device: torch.device):
        self.device = device
        self.samples = []
        self.max_mhz = None
        self._stop = None
        self._thread = None

    def _handle(self):
        import ctypes
        nvml = ctypes.CDLL("libnvidia-ml.so.1")
        if nvml.nvmlInit_v2() != 0:
            return None, None
        h = ctypes.c_void_p()
        uuid = getattr(torch.cuda.get_device_properties(self.device), "uuid", None)
        ok = False
        if uuid is not None:
            ok = nvml.nvmlDeviceGetHandleByUUID(("GPU-" + str(uuid)).encode(), ctypes.byref(h)) == 0
        if not ok:
            ok = nvml.nvmlDeviceGetHandleByIndex_v2(self.device.index or 0, ctypes.byref(h)) == 0
        return (nvml, h) if ok else (None, None)

    def __enter__(self):
        import ctypes
        import threading
        try:
            nvml, h = self._handle()
        except OSError:
            nvml, h = None, None
        if nvml is None:
            return self
        mx = ctypes.c_uint()
        if nvml.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = mx.value
        reasons_fn = getattr(nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        self._stop = threading.Event()

        def poll():
            clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
            while not self._stop.is_set():
                if nvml.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and \
                        reasons_fn(h, ctypes.byref(rs)) == 0:
                    self.samples.append((clk.value, rs.value))
                time.sleep(0.001)
        self._thread = threading.Thread(target=poll, daemon=True)
        self._thread.start()
        time.sleep(0.01)
        return self

    def __exit__(self, *exc):
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples),
                "sm_max_mhz": self.max_mhz, "reasons": reasons,
                "samples": len(self.samples), "source": "NVML, 1 ms polling"}


# ---------------------------------------------------------------- our arm

def run_ours(args, rank, world, local, dist):
    import mixture_experts_ffn_topk_gb300 as moe
    from mixture_experts_ffn_topk_gb300 import build, workloads as W

    build.build()
    moe.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    if args.workload == W.COMBINE_NORM.name:
        return run_combine_norm(args, rank, world, local, dist, dev, peaks, flush)
    if args.workload == W.COMBINE_V2.name:
        return run_combine_v2(args, rank, world, dist, dev, peaks, flush)
    if args.workload == "routing_sweep":
        return run_routing_sweep(args, world, dist, dev, peaks, flush)
    if args.workload in TRAINING_WORKLOADS:
        return run_training(args, rank, world, local, dist, dev, peaks, flush)

    cfg = forward_config(args.workload)
    d = W.moe_inputs(cfg, device=dev, seed=cfg.seed + 1000 * rank)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    A = T * k
    x, logits = d["x"], d["logits"]
    y = torch.empty((T, H), dtype=x.dtype, device=dev)
    lay = moe.moe_forward_workspace_layout(T, H, I, E, k, x.dtype, logits.dtype)
    ws_f = torch.empty(lay["total"], dtype=torch.uint8, device=dev)

    sigmoid = cfg.routing == "sigmoid_grouped"
    bias = d.get("bias")
    sg = ({"bias": bias, "groups": cfg.groups, "selected_groups": cfg.selected_groups,
           "group_top_two": cfg.group_top_two, "scale": cfg.scale} if sigmoid else None)

    def forward(x_, lg, y_, ev=None):
        # the one-call forward; with ev = (begin, end) the same call records
        # events right before the first and right after the last expert GEMM
        if ev is not None:
            moe.moe_forward_ex(x_, lg, d["gate"], d["up"], d["down"], k, cfg.renormalize,
                               sigmoid_grouped=sg, experts_begin_event=ev[0],
                               experts_end_event=ev[1], y=y_, workspace=ws_f)
        elif sigmoid:
            moe.moe_forward_sigmoid_grouped(x_, lg, bias, d["gate"], d["up"], d["down"], k,
                                            cfg.groups, cfg.selected_groups, cfg.group_top_two,
                                            cfg.renormalize, cfg.scale, y=y_, workspace=ws_f)
        else:
            moe.moe_forward(x_, lg, d["gate"], d["up"], d["down"], k, cfg.renormalize,
                            y=y_, workspace=ws_f)

    # kernels per forward: the front end (one fused route-and-count kernel,
    # rank, gather for softmax routing below 64 tokens per SM; else route,
    # count, scan, rank, gather), GEMM1, GEMM2, then the finalize or combine
    front = 3 if (not sigmoid and fused_route_dispatch(T, E, k, dev)) else 5
    launches_per_step = front + 2 + 1
    for _ in range(args.warmup):
        forward(x, logits, y)
        flush.fill_(1)
    torch.cuda.synchronize(dev)
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error during warm-up")

    # Timed region 1 (the headline): K passes of the one-call forward, events
    # only at step boundaries so every kernel may start early (PDL).
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk:
        for a, b in pairs:
            a.record(stream)
            forward(x, logits, y)
            b.record(stream)
            flush.fill_(1)   # untimed: between the events of consecutive steps
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    step_ms = [a.elapsed_time(b) for a, b in pairs]
    ms = statistics.mean(step_ms)
    ms_max = reduce_max(dist, ms, dev)
    value = aggregate(ms_max / 1e3, T, world)
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error in the timed region")

    # Timed region 2 (the per-stage breakdown and the expert GEMMs' time):
    # the same one-call forward (moe_forward_ex, same kernels) with events at
    # the step boundaries and around its two expert GEMM launches.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk2:
        for e4 in evs:
            e4[0].record(stream)
            forward(x, logits, y, ev=(e4[1], e4[2]))
            e4[3].record(stream)
            flush.fill_(1)
        torch.cuda.synchronize(dev)
    stage_ms = {name: statistics.mean(e4[j].elapsed_time(e4[j + 1]) for e4 in evs)
                for j, name in enumerate(["route+dispatch", "experts", "combine"])}
    instrumented_ms = statistics.mean(e4[0].elapsed_time(e4[3]) for e4 in evs)

    # Timed region 3: the same one-call forward captured once in a CUDA graph
    # (the memset, the kernels and their programmatic-launch edges) and
    # replayed, so no host work sits between steps.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        forward(x, logits, y)
    for _ in range(args.warmup):
        graph.replay()
        flush.fill_(1)
    gpairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for a, b in gpairs:
        a.record(stream)
        graph.replay()
        b.record(stream)
        flush.fill_(1)
    torch.cuda.synchronize(dev)
    graph_ms = reduce_max(dist, statistics.mean(a.elapsed_time(b) for a, b in gpairs), dev)
    del graph
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error in the graph replays")

    # Timed region 4 (end to end): host buffers in, y out, every step.
    eb = x.element_size()
    x_h = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    x_h.copy_(x)
    l_h = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)
    l_h.copy_(logits)
    ins = [[torch.empty_like(x), torch.empty_like(logits)] for _ in range(2)]
    outs = [[torch.empty_like(y)] for _ in range(2)]
    outs_h = [[torch.empty(y.shape, dtype=y.dtype, pin_memory=True)] for _ in range(2)]

    def e2e_step(slot):
        forward(ins[slot][0], ins[slot][1], outs[slot][0])
    e2e_ms = pipelined_e2e(e2e_step, [x_h, l_h], ins, outs, outs_h, args, dev)
    e2e_ms_max = reduce_max(dist, e2e_ms, dev)
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error in the timed region")

    # Algorithmic work (per forward): 6*H*I FLOPs per assignment in the two
    # expert GEMMs; their bytes are the touched experts' weights, x_disp read,
    # the expert outputs written, and h written and read back.
    counts = ws_f[lay["counts"]:lay["counts"] + 4 * E].view(torch.int32).cpu()
    touched = int((counts > 0).sum())
    flops = 6.0 * H * I * A
    lb, wb = logits.element_size(), logits.element_size()
    gemm_bytes = 3 * touched * I * H * eb + 2 * A * H * eb + 2 * A * I * eb
    route_bytes = T * E * lb + A * (4 + wb) + (E * 4 if bias is not None else 0)
    disp_bytes = A * 12 + E * 8 + T * H * eb + A * H * eb     # x read once, x_disp written
    comb_bytes = A * H * eb + A * (wb + 4) + T * H * eb
    exp_ms = stage_ms["experts"]
    hbm = peaks["hbm_gbs"]
    kernels = {
        "route+dispatch": {"ms": stage_ms["route+dispatch"], "bytes": route_bytes + disp_bytes},
        "experts": {"ms": exp_ms, "flops": flops, "bytes": gemm_bytes,
                    "experts_touched": touched},
        "combine": {"ms": stage_ms["combine"], "bytes": comb_bytes,
                    "how": "finalize of the FP32 accumulator the second GEMM reduced into"
                           if fold_combine(T, H, x) else
                           "slot-order combine of the FP32 expert outputs"},
    }
    for kk in kernels.values():
        kk["gbs"] = kk["bytes"] / (kk["ms"] / 1e3) / 1e9
        kk["frac_hbm"] = kk["gbs"] / hbm
        kk["frac_hbm_nominal"] = kk["gbs"] / NOMINAL_HBM_GBS
    kernels["experts"]["tflops"] = flops / (exp_ms / 1e3) / 1e12
    kernels["experts"]["frac_bf16_peak"] = kernels["experts"]["tflops"] / peaks["bf16_tflops"]
    kernels["experts"]["frac_bf16_sustained"] = (kernels["experts"]["tflops"]
                                                 / peaks["bf16_tflops_sustained"])
    traffic = load_traffic(args.workload, "experts")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == "bf16" else cfg.dtype,
        "data": "synthetic (seeded; random-init expert weights)",
        "config": dict({"workload": cfg.name, "T": T, "H": H, "I": I, "E": E, "top_k": k,
                        "renormalize": cfg.renormalize, "logits_dtype": cfg.logits_dtype,
                        "global_batch": T * world, "parallelism": f"replicas x{world}",
                        "l2": "flushed between steps (256 MiB write)"}, **routing_config(cfg)),
        "e2e": {"value": aggregate(e2e_ms_max / 1e3, T, world), "unit": UNIT,
                "h2d_bytes_per_step": x.numel() * eb + logits.numel() * lb,
                "d2h_bytes_per_step": y.numel() * eb,
                "how": "moe_forward through the C ABI; per step x and logits copied in from "
                       "pinned host memory and y copied out, double-buffered so the copies "
                       "of neighbouring steps (in and out on separate copy streams) overlap "
                       "the compute; no L2 flush (each step streams "
                       f"{3 * touched * I * H * eb / 1e9:.2f} GB of expert weights, more "
                       "than L2)"},
        "graph": {"value": aggregate(graph_ms / 1e3, T, world), "unit": UNIT,
                  "ms_per_step": graph_ms,
                  "how": "the same moe_forward captured once in a CUDA graph and replayed; "
                         "L2 flushed between replays"},
        "instrumented_ms_per_step": instrumented_ms,
        "ms_per_step_median": statistics.median(step_ms),
        "roofline": roofline_entry(flops, gemm_bytes, exp_ms, peaks, traffic),
        "kernels": kernels,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
        "clocks_breakdown": clk2.summary(),
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, d, args.cpu_seconds)
    return line


# Smaller cases of the forward workloads with the same per-expert shapes
# (H, I) and routing, for profiler captures that must hold a few GB at most:
# name -> (workload, overrides). The coarse prefill with 4 experts and 4096
# tokens keeps about 2048 rows per expert; the decode shapes with 32 experts
# keep the Zipf-skewed, weight-streaming decode GEMMs.
SCALED_WORKLOADS = {
    "coarse_prefill_e4_bf16": ("coarse_prefill_bf16", {"T": 4096, "E": 4}),
    "decode_e32_bf16": ("decode_bf16", {"E": 32}),
    "sigmoid_grouped_decode_e32_bf16": ("sigmoid_grouped_decode_bf16", {"E": 32}),
}


def forward_config(name):
    """The MoeConfig of a forward workload or of one of its scaled cases."""
    from mixture_experts_ffn_topk_gb300 import workloads as W
    if name in SCALED_WORKLOADS:
        base, overrides = SCALED_WORKLOADS[name]
        return W.CONFIGS[base].scaled(name=name, **overrides)
    return W.CONFIGS[name]


def fold_combine(T, H, x):
    """Whether moe_forward folds the combine into the second expert GEMM:
    BF16/F16 with an FP32 [T, H] accumulator of at most 64 MiB."""
    return x.dtype != torch.float32 and T * H * 4 <= 64 << 20


# Training step workloads: a forward that keeps the backward's cache, then
# the four backward steps of ruDNN section 12, on a forward workload's shapes.
# name -> (forward workload, overrides); the half case keeps the fine prefill's
# rows per expert (T*k/E = 384) at half the tokens and experts, small enough
# for full profiler captures of the backward kernels
TRAINING_WORKLOADS = {"train_fine_prefill_bf16": ("fine_prefill_bf16", {}),
                      "train_coarse_prefill_bf16": ("coarse_prefill_bf16", {}),
                      "train_fine_prefill_half_bf16": ("fine_prefill_bf16", {"T": 2048, "E": 32}),
                      # the coarse prefill's per-expert shapes, 4 experts of about
                      # 2048 rows: small enough for multi-pass profiler captures
                      "train_coarse_prefill_e4_bf16": ("coarse_prefill_bf16", {"T": 4096, "E": 4})}


def run_training(args, rank, world, local, dist, dev, peaks, flush):
    """One step = route -> dispatch -> router weights (softmax of the fixed
    selection) -> experts forward keeping the cache -> combine, then combine
    backward -> expert backward -> dispatch backward -> router backward, for
    an N(0,1) output gradient. Inputs and weights resident in HBM."""
    import mixture_experts_ffn_topk_gb300 as moe
    from mixture_experts_ffn_topk_gb300 import workloads as W
    base_name, overrides = TRAINING_WORKLOADS[args.workload]
    cfg = W.CONFIGS[base_name].scaled(**overrides) if overrides else W.CONFIGS[base_name]
    d = W.moe_inputs(cfg, device=dev, seed=cfg.seed + 1000 * rank)
    gy = W.training_grad(cfg, device=dev, seed=cfg.seed + 1000 * rank)
    T, H, I, E, k = cfg.T, cfg.H, cfg.I, cfg.E, cfg.top_k
    A = T * k
    x, logits = d["x"], d["logits"]
    dt = x.dtype
    f32 = torch.float32
    b = {"idx": torch.empty((T, k), dtype=torch.int32, device=dev),
         "wr": torch.empty((T, k), dtype=logits.dtype, device=dev),
         "counts": torch.empty(E, dtype=torch.int32, device=dev),
         "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
         "row_of": torch.empty(A, dtype=torch.int32, device=dev),
         "src_of": torch.empty(A, dtype=torch.int32, device=dev),
         "x_disp": torch.empty((A, H), dtype=dt, device=dev),
         "w": torch.empty((T, k), dtype=f32, device=dev),
         "out": torch.empty((A, H), dtype=f32, device=dev),
         "cache": torch.empty(moe.moe_experts_training_cache_size(A, I, dt), dtype=torch.uint8,
                              device=dev),
         "y": torch.empty((T, H), dtype=dt, device=dev),
         "dexp": torch.empty((A, H), dtype=dt, device=dev),
         "dw": torch.empty((T, k), dtype=f32, device=dev),
         "dxd": torch.empty((A, H), dtype=dt, device=dev),
         "dgate": torch.empty((E, I, H), dtype=f32, device=dev),
         "dup": torch.empty((E, I, H), dtype=f32, device=dev),
         "ddown": torch.empty((E, H, I), dtype=f32, device=dev),
         "dx": torch.empty((T, H), dtype=dt, device=dev),
         "dl": torch.empty_like(logits),
         "ws_d": torch.empty(max(1, moe.moe_dispatch_workspace_size(T, k, E)),
                             dtype=torch.uint8, device=dev),
         "ws_b": torch.empty(moe.moe_experts_backward_workspace_size(A, E, H, I, dt),
                             dtype=torch.uint8, device=dev)}
    stream = torch.cuda.current_stream(dev)

    def step(x_, lg, g_, ev=None, dx_out=None, dl_out=None):
        if ev: ev[0].record(stream)
        moe.moe_route(lg, k, cfg.renormalize, expert_indices=b["idx"], weights=b["wr"])
        moe.moe_dispatch(b["idx"], x_, E, counts=b["counts"], offsets=b["offsets"],
                         row_of=b["row_of"], src_of=b["src_of"], x_disp=b["x_disp"],
                         workspace=b["ws_d"])
        moe.moe_router_weights(lg, b["idx"], "softmax", cfg.renormalize, 1.0, weights=b["w"])
        if ev: ev[1].record(stream)
        moe.moe_experts_forward_training(b["x_disp"], b["offsets"], d["gate"], d["up"],
                                         d["down"], out_disp=b["out"], cache=b["cache"])
        if ev: ev[2].record(stream)
        moe.moe_combine(b["out"], b["w"], b["row_of"], y=b["y"])
        moe.moe_combine_backward(b["out"], b["w"], b["row_of"], g_, grad_out_disp=b["dexp"],
                                 grad_weights=b["dw"])
        if ev: ev[3].record(stream)
        moe.moe_experts_backward(b["x_disp"], b["offsets"], d["gate"], d["up"], d["down"],
                                 b["cache"], b["dexp"], grad_x_disp=b["dxd"],
                                 grad_gate=b["dgate"], grad_up=b["dup"], grad_down=b["ddown"],
                                 workspace=b["ws_b"])
        if ev: ev[4].record(stream)
        moe.moe_dispatch_backward(b["dxd"], b["row_of"], T, k,
                                  grad_x=b["dx"] if dx_out is None else dx_out)
        moe.moe_router_backward(lg, b["idx"], b["dw"], "softmax", cfg.renormalize, 1.0,
                                grad_logits=b["dl"] if dl_out is None else dl_out)
        if ev: ev[5].record(stream)

    # route 1, dispatch 4, router weights 1, experts fwd 2, combine 1,
    # combine bwd 1, experts bwd 6 (2 map builds + 4 GEMMs), dispatch bwd 1, router bwd 1
    launches_per_step = 18
    for _ in range(args.warmup):
        step(x, logits, gy)
        flush.fill_(1)
    torch.cuda.synchronize(dev)
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error during warm-up")
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    with ClockSampler(dev) as clk:
        for a, e in pairs:
            a.record(stream)
            step(x, logits, gy)
            e.record(stream)
            flush.fill_(1)
        torch.cuda.synchronize(dev)
    barrier(dist, dev)
    ms = statistics.mean(a.elapsed_time(e) for a, e in pairs)
    ms_max = reduce_max(dist, ms, dev)

    names = ["route+dispatch+weights", "experts_fwd", "combine+combine_bwd", "experts_bwd",
             "dispatch_bwd+router_bwd"]
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for i in range(args.steps):
        step(x, logits, gy, evs[i])
        flush.fill_(1)
    torch.cuda.synchronize(dev)
    stage_ms = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1])
                                   for i in range(args.steps)) for j, n in enumerate(names)}

    # end to end: x, logits and the output gradient in from pinned host
    # memory, the input and logits gradients back out
    hx = torch.empty(x.shape, dtype=dt, pin_memory=True); hx.copy_(x)
    hl = torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True); hl.copy_(logits)
    hg = torch.empty(gy.shape, dtype=dt, pin_memory=True); hg.copy_(gy)
    ins = [[torch.empty_like(x), torch.empty_like(logits), torch.empty_like(gy)] for _ in range(2)]
    outs = [[torch.empty_like(x), torch.empty_like(logits)] for _ in range(2)]
    outs_h = [[torch.empty(x.shape, dtype=dt, pin_memory=True),
               torch.empty(logits.shape, dtype=logits.dtype, pin_memory=True)] for _ in range(2)]

    def e2e_step(slot):
        step(ins[slot][0], ins[slot][1], ins[slot][2], dx_out=outs[slot][0], dl_out=outs[slot][1])
    e2e_ms = pipelined_e2e(e2e_step, [hx, hl, hg], ins, outs, outs_h, args, dev)
    e2e_ms_max = reduce_max(dist, e2e_ms, dev)
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error in the timed region")

    eb = x.element_size()
    touched = int((b["counts"].cpu() > 0).sum())
    bwd_ms = stage_ms["experts_bwd"]
    bwd_flops = 12.0 * H * I * A
    # algorithmic bytes of the expert backward: the touched experts' weights
    # read (dh, dx), the FP32 weight gradients of every expert written, the
    # activations read (do twice, x, h, g and u) and dgu written and read twice
    bwd_bytes = (3 * touched * I * H * eb + 3 * E * I * H * 4
                 + 2 * A * H * eb + A * H * eb + A * I * eb + 2 * A * I * 4
                 + 3 * 2 * A * I * eb + A * H * eb)
    tflops = bwd_flops / (bwd_ms / 1e3) / 1e12
    gbs = bwd_bytes / (bwd_ms / 1e3) / 1e9
    t_tensor = bwd_flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = bwd_bytes / (peaks["hbm_gbs"] * 1e9)
    common = {"kernel": "expert backward (dh + dx + weight-gradient tcgen05 GEMMs)",
              "algorithmic_flops": bwd_flops, "algorithmic_bytes": bwd_bytes,
              "traffic": load_traffic(args.workload, "experts_bwd"),
              "tflops": tflops, "gbs": gbs,
              "frac_bf16_peak": tflops / peaks["bf16_tflops"], "frac_hbm": gbs / peaks["hbm_gbs"]}
    if t_tensor >= t_hbm:
        roof = dict(common, bound="tensor", achieved=tflops, peak=peaks["bf16_tflops"],
                    unit="TFLOP/s", frac=tflops / peaks["bf16_tflops"],
                    peak_source=peaks["source"] + " burst bf16")
    else:
        roof = dict(common, bound="hbm", achieved=gbs, peak=peaks["hbm_gbs"], unit="GB/s",
                    frac=gbs / peaks["hbm_gbs"], frac_nominal=gbs / NOMINAL_HBM_GBS,
                    peak_source=peaks["source"] + " HBM copy")
    fwd_flops = 6.0 * H * I * A
    line = {
        "metric": "MoE training step (forward + first-order backward) tokens/s",
        "value": aggregate(ms_max / 1e3, T, world), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; random-init expert weights; N(0,1) output gradient)",
        "config": dict({"workload": args.workload, "T": T, "H": H, "I": I, "E": E, "top_k": k,
                        "renormalize": cfg.renormalize, "router_scoring": "softmax",
                        "global_batch": T * world, "parallelism": f"replicas x{world}",
                        "l2": "flushed between steps (256 MiB write)"}),
        "e2e": {"value": aggregate(e2e_ms_max / 1e3, T, world), "unit": UNIT,
                "h2d_bytes_per_step": x.numel() * eb + logits.numel() * logits.element_size()
                + gy.numel() * eb,
                "d2h_bytes_per_step": x.numel() * eb + logits.numel() * logits.element_size(),
                "how": "the training step through the C ABI; per step x, logits and the output "
                       "gradient copied in from pinned host memory, the input and logits "
                       "gradients copied out, double-buffered so the copies of neighbouring "
                       "steps (in and out on separate copy streams) overlap the compute; no L2 flush (each step streams the 1.1 GB "
                       "of expert weights and writes 2.2 GB of weight gradients)"},
        "roofline": roof,
        "kernels": {n: {"ms": v} for n, v in stage_ms.items()},
        "experts_fwd_tflops": fwd_flops / (stage_ms["experts_fwd"] / 1e3) / 1e12,
        "experts_touched": touched,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if world == 1 and rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_training_baseline(cfg, d, gy, args.cpu_seconds)
    return line


def cpu_training_baseline(cfg, d, gy, seconds):
    """The oracle's training step on a bounded token sample (one thread):
    forward with the fixed selection and router weights, then the four
    backward steps, for the sampled tokens as a batch of their own."""
    import numpy as np
    import oracle
    from mixture_experts_ffn_topk_gb300 import workloads as W
    lib = oracle.load_library()
    host = {kk: W.to_numpy(v) for kk, v in d.items()}
    g_h = W.to_numpy(gy)
    k, E = cfg.top_k, cfg.E

    def run(tokens):
        lg = host["logits"][tokens]
        x = host["x"][tokens]
        idx, _, _ = oracle.route(lg, cfg.logits_dtype, k, cfg.renormalize, lib)
        counts, offsets, row_of, src_of, _ = oracle.dispatch(idx, E, lib)
        w, _ = oracle.router_weights(lg, cfg.logits_dtype, idx, "softmax", cfg.renormalize, 1.0,
                                     "f32", lib)
        xd = oracle.gather(x, cfg.dtype, k, src_of, tokens.size * k, lib)
        out = oracle.experts_dispatched(xd, cfg.dtype, offsets, host["gate"], host["up"],
                                        host["down"], lib)
        oracle.combine(out, "f64", w, "f32", row_of, k, lib)
        dexp, dw = oracle.combine_backward(out, "f64", w, "f32", row_of, g_h[tokens], cfg.dtype,
                                           k, lib)
        dxd = oracle.experts_backward_dispatched(xd, cfg.dtype, offsets, host["gate"], host["up"],
                                                 host["down"], dexp, "f64", lib)[0]
        oracle.dispatch_backward(dxd, "f64", row_of, k, lib)
        oracle.router_backward(lg, cfg.logits_dtype, idx, dw, "f64", "softmax", cfg.renormalize,
                               1.0, "f64", lib)
    rng = np.random.default_rng(cfg.seed)
    t0 = time.perf_counter()
    run(rng.choice(cfg.T, size=1, replace=False))
    one = max(time.perf_counter() - t0, 1e-3)
    n = int(max(1, min(cfg.T, seconds / one)))
    tokens = rng.choice(cfg.T, size=n, replace=False)
    t0 = time.perf_counter()
    run(tokens)
    wall = time.perf_counter() - t0
    return {"value": n / wall, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} of {cfg.T} tokens of {cfg.name} as one training batch "
                      f"(forward, combine/expert/dispatch/router backward) in {wall:.1f} s"}


def routing_config(cfg):
    """Config keys naming the routing of a workload."""
    if cfg.routing != "sigmoid_grouped":
        return {"routing": "softmax"}
    return {"routing": "sigmoid_grouped", "groups": cfg.groups,
            "selected_groups": cfg.selected_groups, "group_top_two": cfg.group_top_two,
            "scale": cfg.scale, "correction_bias_var": cfg.correction_var}


def fused_route_dispatch(T, E, k, dev):
    """Whether moe_forward routes and counts in one kernel: the library does so
    unless it would route one token per thread (E <= 64, top_k <= 8 and at
    least 64 tokens per SM), and when E <= 1024 and the chunk counts (chunks x
    E) fit the 14336 the last CTA scans in shared memory."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    A = T * k
    chunk = 256
    while chunk < 2048 and chunk < A // (sms * 8):
        chunk *= 2
    thread_route = E <= 64 and k <= 8 and T >= sms * 64
    return not thread_route and E <= 1024 and (A + chunk - 1) // chunk * E <= 14 * 1024


def roofline_entry(flops, nbytes, ms, peaks, traffic):
    """The expert GEMMs (GEMM1 + GEMM2 of the one-call forward, timed by
    events around their launches) against the roof that binds them: their
    arithmetic intensity (algorithmic FLOPs over algorithmic bytes) against
    the ridge of the measured peaks decides; the fraction is the achieved
    rate over that peak."""
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    ai = flops / nbytes
    tflops = flops / (ms / 1e3) / 1e12
    gbs = nbytes / (ms / 1e3) / 1e9
    common = {"kernel": "grouped SwiGLU GEMM (GEMM1 + GEMM2 of moe_forward)",
              "ms": ms, "algorithmic_flops": flops, "algorithmic_bytes": nbytes,
              "arithmetic_intensity": ai, "ridge": ridge, "traffic": traffic,
              "tflops": tflops, "gbs": gbs}
    if ai >= ridge:
        return dict(common, bound="tensor", achieved=tflops, peak=peaks["bf16_tflops"],
                    unit="TFLOP/s", frac=tflops / peaks["bf16_tflops"],
                    frac_sustained=tflops / peaks["bf16_tflops_sustained"],
                    peak_source=peaks["source"] + " burst bf16")
    return dict(common, bound="hbm", achieved=gbs, peak=peaks["hbm_gbs"], unit="GB/s",
                frac=gbs / peaks["hbm_gbs"], frac_nominal=gbs / NOMINAL_HBM_GBS,
                peak_source=peaks["source"] + " HBM copy")


def timed_loop(fn, args, stream, flush):
    for _ in range(max(1, args.warmup)):
        fn()
        flush.fill_(1)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in pairs:
        a.record(stream)
        fn()
        b.record(stream)
        flush.fill_(1)
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in pairs)


def pipelined_e2e(run_step, host_in, dev_in, dev_out, host_out, args, dev):
    """End-to-end steps through the C ABI with host buffers: every step copies
    its inputs from pinned host memory, computes, and copies its result back.
    Two buffer sets, an inbound and an outbound copy stream beside the compute
    stream: step i+1's inputs and step i-1's result cross the link (each way
    on its own copy engine) while step i computes, a serving loop's double
    buffering. host_in[j] -> dev_in[slot][j]; dev_out[slot][j] ->
    host_out[slot][j]; run_step(slot) computes on the current stream. Returns
    milliseconds per step (first copy in to last copy out, over args.steps
    steps, after args.warmup such steps)."""
    comp = torch.cuda.current_stream(dev)
    cp_in, cp_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    h2d_done = [torch.cuda.Event(), torch.cuda.Event()]
    comp_done = [torch.cuda.Event(), torch.cuda.Event()]
    d2h_done = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d(i):
        slot = i % 2
        with torch.cuda.stream(cp_in):
            if i >= 2:
                cp_in.wait_event(comp_done[slot])       # the slot's last reader is done
            for src, dst in zip(host_in, dev_in[slot]):
                dst.copy_(src, non_blocking=True)
            h2d_done[slot].record(cp_in)

    def loop(n):
        h2d(0)
        for i in range(n):
            slot = i % 2
            comp.wait_event(h2d_done[slot])
            if i >= 2:
                comp.wait_event(d2h_done[slot])         # the slot's result has left
            run_step(slot)
            comp_done[slot].record(comp)
            if i + 1 < n:
                h2d(i + 1)
            with torch.cuda.stream(cp_out):
                cp_out.wait_event(comp_done[slot])
                for src, dst in zip(dev_out[slot], host_out[slot]):
                    dst.copy_(src, non_blocking=True)
                d2h_done[slot].record(cp_out)

    loop(max(2, args.warmup))
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(cp_in)
    loop(args.steps)
    end.record(cp_out)
    torch.cuda.synchronize(dev)
    return start.elapsed_time(end) / args.steps


def run_routing_sweep(args, world, dist, dev, peaks, flush):
    """Route and dispatch alone, on the fine prefill's routing shape (E=64,
    top_k=6, BF16 logits N(0,1)) at growing T, to show where they leave the
    launch-bound regime. Dispatch carries 8-element rows so its gather is
    small; its algorithmic bytes are the indices read once, the two maps
    written, and the gathered rows."""
    import mixture_experts_ffn_topk_gb300 as moe
    from mixture_experts_ffn_topk_gb300 import workloads as W
    base = W.CONFIGS["fine_prefill_bf16"]
    stream = torch.cuda.current_stream(dev)
    E, k, Hs = base.E, base.top_k, 8
    rows = []
    with ClockSampler(dev) as clk:
        for T in (4096, 65536, 1 << 20):
            cfg = base.scaled(T=T, H=Hs, I=8)
            d = W.moe_inputs(cfg, device=dev)
            logits, x = d["logits"], d["x"]
            idx = torch.empty((T, k), dtype=torch.int32, device=dev)
            w = torch.empty((T, k), dtype=logits.dtype, device=dev)
            A = T * k
            bufs = {"counts": torch.empty(E, dtype=torch.int32, device=dev),
                    "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
                    "row_of": torch.empty(A, dtype=torch.int32, device=dev),
                    "src_of": torch.empty(A, dtype=torch.int32, device=dev),
                    "x_disp": torch.empty((A, Hs), dtype=x.dtype, device=dev),
                    "workspace": torch.empty(moe.moe_dispatch_workspace_size(T, k, E),
                                             dtype=torch.uint8, device=dev)}
            r_ms = timed_loop(lambda: moe.moe_route(logits, k, False, expert_indices=idx,
                                                    weights=w), args, stream, flush)
            d_ms = timed_loop(lambda: moe.moe_dispatch(idx, x, E, **bufs), args, stream, flush)
            r_bytes = T * E * 2 + A * (4 + 2)
            d_bytes = A * 12 + E * 8 + T * Hs * 2 + A * Hs * 2
            rows.append({"T": T, "route_us": r_ms * 1e3,
                         "route_frac_hbm": r_bytes / (r_ms / 1e3) / 1e9 / peaks["hbm_gbs"],
                         "dispatch_us": d_ms * 1e3,
                         "dispatch_frac_hbm": d_bytes / (d_ms / 1e3) / 1e9 / peaks["hbm_gbs"]})
        # the same dispatch at T = 2^20 moving the fine prefill's 4 KiB rows
        # (H = 2048): the regime of a real gather, where the rows dominate
        # the bytes (idx and logits as above; x drawn on the device)
        T, Hw = 1 << 20, base.H
        A = T * k
        gen = torch.Generator(device=dev)
        gen.manual_seed(base.seed)
        xw = torch.randn((T, Hw), generator=gen, device=dev).to(torch.bfloat16)
        wide = {"counts": torch.empty(E, dtype=torch.int32, device=dev),
                "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
                "row_of": torch.empty(A, dtype=torch.int32, device=dev),
                "src_of": torch.empty(A, dtype=torch.int32, device=dev),
                "x_disp": torch.empty((A, Hw), dtype=torch.bfloat16, device=dev),
                "workspace": torch.empty(moe.moe_dispatch_workspace_size(T, k, E),
                                         dtype=torch.uint8, device=dev)}
        dw_ms = timed_loop(lambda: moe.moe_dispatch(idx, xw, E, **wide), args, stream, flush)
        dw_bytes = A * 12 + E * 8 + T * Hw * 2 + A * Hw * 2
        wide_row = {"T": T, "H": Hw, "dispatch_us": dw_ms * 1e3, "bytes": dw_bytes,
                    "dispatch_frac_hbm": dw_bytes / (dw_ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
        del xw, wide
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error in the routing sweep")
    big = rows[-1]
    T = big["T"]
    return {"metric": METRIC, "value": T * world / (big["route_us"] + big["dispatch_us"]) * 1e6,
            "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": (big["route_us"] + big["dispatch_us"]) / 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded)",
            "config": {"workload": "routing_sweep", "E": E, "top_k": k, "logits_dtype": "bf16",
                       "l2": "flushed between steps (256 MiB write)"},
            "sweep": rows,
            "dispatch_wide_rows": wide_row,
            "roofline": {"bound": "hbm", "kernel": "route (T = 2^20)",
                         "achieved": big["route_frac_hbm"] * peaks["hbm_gbs"],
                         "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": big["route_frac_hbm"],
                         "frac_nominal": big["route_frac_hbm"] * peaks["hbm_gbs"] / NOMINAL_HBM_GBS,
                         "peak_source": peaks["source"], "traffic": None},
            "gpu_launches": (5 * len(rows) + 4) * (args.steps + max(1, args.warmup)),
            "clocks": clk.summary()}


def run_combine_norm(args, rank, world, local, dist, dev, peaks, flush):
    import oracle
    import mixture_experts_ffn_topk_gb300 as moe
    from mixture_experts_ffn_topk_gb300 import workloads as W
    cfg = W.COMBINE_NORM
    d = W.combine_norm_inputs(cfg, device=dev, seed=cfg.seed + 1000 * rank)
    T, H, k = cfg.T, cfg.H, cfg.top_k
    idx, w = moe.moe_route(d["logits"], k, True)
    disp = moe.moe_dispatch(idx, torch.zeros((T, 8), dtype=torch.bfloat16, device=dev), cfg.E)
    row_of = disp["row_of"]
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    xo = torch.empty_like(y)
    rstd = torch.empty(T, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def fn():
        moe.moe_combine_add_rmsnorm(d["out_disp"], w, row_of, d["residual"], d["gamma"],
                                    cfg.eps, y=y, x_out=xo, rstd=rstd)
    with ClockSampler(dev) as clk:
        ms = timed_loop(fn, args, stream, flush)
    ms_max = reduce_max(dist, ms, dev)
    nbytes = (T * k * H * 2 + T * k * (4 + 4) + T * H * 2 + H * 2 + 2 * T * H * 2 + T * 4)
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"metric": METRIC, "value": aggregate(ms_max / 1e3, T, world), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded)",
            "config": {"workload": cfg.name, "T": T, "H": H, "E": cfg.E, "top_k": k,
                       "l2": "flushed between steps (256 MiB write)"},
            "roofline": {"bound": "hbm", "kernel": "combine + Add + RMSNorm", "achieved": gbs,
                         "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": gbs / peaks["hbm_gbs"],
                         "frac_nominal": gbs / NOMINAL_HBM_GBS, "peak_source": peaks["source"],
                         "traffic": load_traffic(cfg.name, "combine_add_rmsnorm")},
            "gpu_launches": args.steps, "clocks": clk.summary()}


def run_combine_v2(args, rank, world, dist, dev, peaks, flush):
    """The local math of the Ascend V2 combine: special experts (zero, copy,
    const), the shared-expert term, a 2-D active mask, then Add + RMSNorm,
    on the combine + norm workload's shapes."""
    import numpy as np
    import mixture_experts_ffn_topk_gb300 as moe
    from mixture_experts_ffn_topk_gb300 import workloads as W
    cfg = W.COMBINE_V2
    d = W.combine_v2_inputs(cfg, device=dev, seed=cfg.seed + 1000 * rank)
    T, H, k, E = cfg.T, cfg.H, cfg.top_k, cfg.E
    special = cfg.zero + cfg.copy + cfg.const
    idx, w = moe.moe_route(d["logits"], k, True)
    disp = moe.moe_dispatch_special(idx, torch.zeros((T, 8), dtype=torch.bfloat16, device=dev),
                                    E, special)
    row_of = disp["row_of"]
    y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    xo = torch.empty_like(y)
    rstd = torch.empty(T, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    mask = d["mask"].to(torch.uint8)      # the C ABI takes bytes; no conversion per call

    def fn():
        moe.moe_combine_v2(d["out_disp"], w, row_of, torch.bfloat16, expert_indices=idx,
                           num_experts=E, zero_experts=cfg.zero, copy_experts=cfg.copy,
                           const_experts=cfg.const, ori_x=d["ori_x"], const_alpha1=d["alpha1"],
                           const_alpha2=d["alpha2"], const_v=d["const_v"],
                           shared_expert_x=d["shared_x"], active_mask=mask,
                           residual=d["residual"], gamma=d["gamma"], eps=cfg.eps, y=y,
                           x_out=xo, rstd=rstd)
    with ClockSampler(dev) as clk:
        ms = timed_loop(fn, args, stream, flush)
    ms_max = reduce_max(dist, ms, dev)
    if moe.moe_device_status() != 0:
        raise RuntimeError("device status error in the timed region")
    # algorithmic bytes: the rows of routed, kept slots; ori_x for tokens with
    # a kept copy / const slot; per-slot ids, weights, maps and mask bytes;
    # shared_x, residual, gamma; y, x_out and rstd written
    ids = idx.cpu().numpy().astype(np.int64)
    keep = mask.cpu().numpy()
    routed_rows = int(((ids < E) & keep).sum())
    needs_ori = ((ids >= E + cfg.zero) & (ids < E + special) & keep).any(axis=1).sum()
    nbytes = (routed_rows * H * 2 + int(needs_ori) * H * 2 + T * k * (4 + 4 + 4 + 1)
              + T * H * 2 * 2 + H * 2 + cfg.const * (H + 2) * 2 + 2 * T * H * 2 + T * 4)
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"metric": METRIC, "value": aggregate(ms_max / 1e3, T, world), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded)",
            "config": {"workload": cfg.name, "T": T, "H": H, "E": E, "top_k": k,
                       "zero_experts": cfg.zero, "copy_experts": cfg.copy,
                       "const_experts": cfg.const, "active_mask": f"2-D, keep {cfg.keep}",
                       "shared_expert": True, "norm": "Add + RMSNorm",
                       "l2": "flushed between steps (256 MiB write)"},
            "roofline": {"bound": "hbm", "kernel": "combine (V2 extras) + Add + RMSNorm",
                         "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "frac_nominal": gbs / NOMINAL_HBM_GBS,
                         "peak_source": peaks["source"], "algorithmic_bytes": nbytes,
                         "traffic": None},
            "gpu_launches": args.steps, "clocks": clk.summary()}


# ---------------------------------------------------------------- CPU oracle

def _oracle_runner(cfg, host):
    """run(tokens): the oracle's whole forward for those tokens, one by one."""
    import oracle
    lib = oracle.load_library()
    sg = None
    if cfg.routing == "sigmoid_grouped":
        sg = {"bias": host.get("bias"), "groups": cfg.groups,
              "selected_groups": cfg.selected_groups, "group_top_two": cfg.group_top_two,
              "scale": cfg.scale}

    def run(tokens):
        oracle.forward_tokens(tokens, host["x"], cfg.dtype, host["logits"], cfg.logits_dtype,
                              host["gate"], host["up"], host["down"], cfg.top_k,
                              cfg.renormalize, lib, sigmoid_grouped=sg)
    return run


def oracle_seconds_per_token(run):
    import numpy as np
    run(np.array([0]))                       # first touch of the weights
    t0 = time.perf_counter()
    run(np.array([1]))
    return max(time.perf_counter() - t0, 1e-4)


def oracle_batch(run, tokens, threads):
    """Wall seconds of the oracle on `tokens`, split over `threads` host
    threads (the C oracle releases the GIL through ctypes)."""
    import concurrent.futures as cf
    import numpy as np
    chunks = [c for c in np.array_split(tokens, threads) if c.size]
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(max_workers=len(chunks)) as ex:
        list(ex.map(run, chunks))
    return time.perf_counter() - t0


def oracle_token_rate(cfg, host, seconds, max_threads=None):
    """Oracle throughput (tokens/s) on a bounded token sample of about
    `seconds` of wall time, split over the host's threads."""
    import numpy as np
    threads = max_threads or os.cpu_count() or 1
    run = _oracle_runner(cfg, host)
    one = oracle_seconds_per_token(run)
    n = int(max(threads, min(cfg.T, seconds * threads / one)))
    n = max(threads, n // threads * threads)
    rng = np.random.default_rng(cfg.seed)
    tokens = rng.choice(cfg.T, size=min(n, cfg.T), replace=False)
    wall = oracle_batch(run, tokens, threads)
    return tokens.size / wall, tokens.size, threads, wall


def host_inputs(cfg, d):
    from mixture_experts_ffn_topk_gb300 import workloads as W
    return {k: W.to_numpy(v) for k, v in d.items()}


def cpu_baseline(cfg, d, seconds):
    host = host_inputs(cfg, d)
    rate, n, threads, wall = oracle_token_rate(cfg, host, seconds)
    return {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{n} of {cfg.T} tokens of {cfg.name}, full forward per token "
                      f"(route, k experts, combine) in {wall:.1f} s"}


REFERENCE_BUDGET_S = 120.0      # wall seconds of oracle work over all steps of the arm


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm, on this arm's workload: each of
    the W + K steps runs the oracle's whole forward on a fresh sample of the
    same number of tokens (all host threads); ms_per_step is the measured wall
    time of a step and value its tokens over that time."""
    if rank != 0:
        return None
    import numpy as np
    from mixture_experts_ffn_topk_gb300 import workloads as W
    if args.workload not in W.CONFIGS and args.workload not in SCALED_WORKLOADS:
        return {"impl": "reference",
                "unavailable": "the oracle reference arm times the one-call forward workloads "
                               f"only, not {args.workload}"}
    cfg = forward_config(args.workload)
    d = W.moe_inputs(cfg, device="cpu")
    host = host_inputs(cfg, d)
    threads = os.cpu_count() or 1
    run = _oracle_runner(cfg, host)
    one = oracle_seconds_per_token(run)
    per_step = min(6.0, max(0.5, REFERENCE_BUDGET_S / (args.steps + args.warmup)))
    n = int(max(threads, min(cfg.T, per_step * threads / one)))
    n = max(threads, n // threads * threads)
    rng = np.random.default_rng(cfg.seed)
    for _ in range(args.warmup):
        oracle_batch(run, rng.choice(cfg.T, size=n, replace=False), threads)
    walls = [oracle_batch(run, rng.choice(cfg.T, size=n, replace=False), threads)
             for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(walls)
    value = n / (ms / 1e3)
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": cfg.dtype, "data": "synthetic (seeded; random-init expert weights)",
            "config": dict({"workload": cfg.name, "T": cfg.T, "H": cfg.H, "I": cfg.I,
                            "E": cfg.E, "top_k": cfg.top_k, "renormalize": cfg.renormalize,
                            "tokens_per_step": n}, **routing_config(cfg)),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"{n} of the workload's {cfg.T} tokens per step (a "
                                       f"fresh seeded sample each step), the oracle's whole "
                                       f"forward per token on {threads} host threads; "
                                       f"{args.steps} timed steps of {ms / 1e3:.2f} s"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def launch_plan(gpus: int, env) -> str:
    """How bench.py runs for --gpus N: "single" (N = 1, no process group),
    "rank" (one rank of a torchrun job of N ranks) or "spawn" (N > 1 without
    torchrun: relaunch under torch.distributed.run with N ranks). A torchrun
    job whose WORLD_SIZE is not N is an error."""
    world = env.get("WORLD_SIZE")
    if world is not None and int(world) > 1:
        if int(world) != gpus:
            raise SystemExit(f"bench.py: --gpus {gpus} but WORLD_SIZE={world}")
        return "rank"
    if gpus > 1:
        return "spawn"
    if gpus < 1:
        raise SystemExit("bench.py: --gpus must be >= 1")
    return "single"


def spawn_ranks(gpus: int, argv) -> int:
    """Run this script as `gpus` ranks of one node (torch.distributed.run on
    127.0.0.1); returns the launcher's exit status."""
    import socket
    import subprocess
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr", "127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="coarse_prefill_bf16")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target CPU seconds of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if launch_plan(args.gpus, os.environ) == "spawn":
        return spawn_ranks(args.gpus, argv)
    rank, world, local, dist = dist_setup(args.gpus)
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
