#!/usr/bin/env python
"""Benchmark of the rollout-side NVFP4 W4A4 + RAC hot path on GB300.

One step = one forward pass of the routed SwiGLU MoE expert layer with W4A4 + RAC in both
expert GEMMs (dispatch, activation quantization + channel selection + residual tail, gather,
gate/up grouped GEMM with SwiGLU, per-expert quantization + selection of h, down grouped GEMM
with routing weights, combine) over one synthetic batch: T = 16384 tokens, hidden 2048,
128 experts, top-8 with Zipf(1.1)-skewed routing, intermediate 768, k = 32 per GEMM.

The JSON line reports whole-job tokens/s (inputs resident in HBM, device-timed), an end-to-end
figure through the same public API with host buffers, the roofline of the dominant kernel
(the gate/up grouped GEMM), the activation quantizer + RAC bandwidth on the 8192 x 4096
activation workload, and the CPU oracle timed on a bounded sample on the host cores.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_FLUSH_BYTES = 512 << 20           # > 2x the 129 MB L2
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FP4_OVER_BF16 = 13.5 / 2.25          # nominal dense ratio (NVFP4 / BF16) on GB300
METRIC = "W4A4+RAC grouped-GEMM TFLOPS & tokens/s; act-quant+RAC HBM GB/s (1×GB300)"


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "gemm_kernel_moe_prefill_dram_traffic.md")
GEMM_SOURCE = os.path.join(ROOT, "nvfp4_w4a4_quantized_quantize_gb300", "csrc", "gemm.cu")


def gemm_traffic_per_launch(launch: str = "gate_up"):
    """DRAM bytes (read + write) of one full-size launch of the grouped GEMM, from the committed
    ncu summary, or None when the kernel source has changed since those counters were taken."""
    import hashlib
    import re
    if not os.path.exists(TRAFFIC_PROFILE):
        return None
    src = hashlib.sha256(open(GEMM_SOURCE, "rb").read()).hexdigest()
    for line in open(TRAFFIC_PROFILE):
        m = re.search(r"traffic: launch=(\w+) dram_read=(\d+) dram_write=(\d+) gemm_cu_sha256=([0-9a-f]+)", line)
        if m and m.group(1) == launch:
            return int(m.group(2)) + int(m.group(3)) if m.group(4) == src else None
    return None


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


# ----------------------------------------------------------------------------- distributed
def dist_setup(backend=None):
    """One process per GPU (torchrun): rank, world size and local rank from the environment;
    NCCL when CUDA is available, else gloo (host-side tests)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank_step: float, world: int, max_ms_per_step: float) -> float:
    """Whole-job rate under weak scaling: every rank processes its own batch of units per step,
    and the job's step time is the slowest rank's."""
    return units_per_rank_step * world / (max_ms_per_step * 1e-3)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling (every 20 ms) over the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "20"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- our arm
class LaunchCounter:
    """Kernels each C-ABI call launches (counted by the binding calls below)."""
    PER_CALL = {"moe_dispatch": 4, "nvfp4_quantize": 2, "rac_select_quantize": 2, "nvfp4_gather_rows": 1,
                "rac_weight_tail": 1, "w4a4_rac_grouped_gemm": 1, "moe_combine": 1}


def _bf16(t_bits, dev):
    import torch
    return torch.from_numpy(np.ascontiguousarray(t_bits).view(np.int16)).view(torch.bfloat16).to(dev)


def run_ours(args, world, rank, local):
    import torch

    from nvfp4_w4a4_quantized_quantize_gb300 import _lib as L
    from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
    from nvfp4_w4a4_quantized_quantize_gb300.layers import MoERacLayer

    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    cfg = wl.CFG_MOE_PREFILL
    # every rank processes its own independent batch (weak scaling, no data-path collective)
    cfg_r = wl.MoELayer(cfg.name, cfg.T, cfg.H, cfg.E, cfg.topk, cfg.I, cfg.k, cfg.seed + 1000 * rank,
                        cfg.routing, cfg.zipf_s, cfg.n_outliers, cfg.outlier_gain, cfg.w_std)
    x_bits, ids, tw, _ = cfg_r.make_tokens()
    w13_bits, w2_bits = wl.MoELayer(**{**cfg.__dict__}).make_weights()
    E, H, I, T, topk, k = cfg.E, cfg.H, cfg.I, cfg.T, cfg.topk, cfg.k
    w13 = _bf16(w13_bits.reshape(E * 2 * I, H), dev).view(E, 2 * I, H)
    w2 = _bf16(w2_bits.reshape(E * H, I), dev).view(E, H, I)
    layer = MoERacLayer(w13, w2, k, topk, T)
    del w13, w2
    x = _bf16(x_bits, dev)
    ids_d = torch.from_numpy(ids).to(dev)
    tw_d = torch.from_numpy(tw).to(dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def step_eager(events=None):
        layer.forward(x, ids_d, tw_d, out, events=events)

    for _ in range(args.warmup):
        flush.zero_()
        step_eager()
    torch.cuda.synchronize()
    st, where = L.device_status()
    if st != 0:
        raise RuntimeError(f"device wait ran out ({where}) during warm-up")

    # the whole layer as one CUDA graph (no host synchronisation inside a forward), with the
    # per-kernel events recorded inside the graph
    # timing events recorded inside the graph must be external (event-record nodes)
    # only the two grouped GEMMs carry timing events in the timed graph (each event is a graph
    # node); the per-stage breakdown is taken from a separate graph after the timed region
    try:
        graph_events = {name: (torch.cuda.Event(enable_timing=True, external=True),
                               torch.cuda.Event(enable_timing=True, external=True))
                        for name in ("gemm_gate_up", "gemm_down")}
    except TypeError:  # torch without external events: per-kernel times come from an eager pass
        graph_events = None
    graph = None
    if not args.eager:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            layer.forward(x, ids_d, tw_d, out)  # warm on the capture stream
            torch.cuda.synchronize()
            with torch.cuda.graph(graph, stream=cap):
                layer.forward(x, ids_d, tw_d, out, events=graph_events)
        if graph_events is None:
            graph_events = {}
        stream.wait_stream(cap)
        for _ in range(args.warmup):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()

    def step(events=None):
        if graph is None:
            step_eager(events)
        else:
            graph.replay()
            if events is not None:
                for k2, (e0, e1) in graph_events.items():
                    events[k2] = (e0, e1)

    # ---- device-timed steps (inputs resident), L2 flushed before every step (untimed)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev_lists = [dict() for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t_wall0 = time.perf_counter()
    kernel_ms = {}
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step(ev_lists[i])
        ends[i].record(stream)
        if graph is not None:
            # graph events are re-recorded by every replay: read them before the next one
            ends[i].synchronize()
            for k2, (e0, e1) in ev_lists[i].items():
                try:
                    kernel_ms.setdefault(k2, []).append(e0.elapsed_time(e1))
                except (RuntimeError, ValueError):  # a stage this layer does not run
                    pass
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    barrier(world)
    clocks = sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    launches_per_step = layer.kernel_launches_per_step()

    # per-kernel durations of the two grouped GEMMs inside the timed steps
    def avg(name):
        if graph is not None:
            v = kernel_ms.get(name, [])
        else:
            v = [ev[name][0].elapsed_time(ev[name][1]) for ev in ev_lists if name in ev]
        return sum(v) / len(v) if v else None

    t_gu, t_dn = avg("gemm_gate_up"), avg("gemm_down")
    stage_ms_rac = stage_times(lambda ev: layer.forward(x, ids_d, tw_d, out, events=ev), flush, max(5, min(args.steps, 50)))
    rows_total = T * topk
    flop_gu = 2.0 * rows_total * (2 * I) * (H + k)
    flop_dn = 2.0 * rows_total * H * (I + k)
    peaks, src = _peaks()
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    ach_gu = flop_gu / (t_gu * 1e-3) / 1e12
    tokens_per_s = job_throughput(T, world, ms_per_step)

    # ---- end-to-end through the public API with host buffers: every step copies its inputs
    # from pinned host memory and its output back (HostPipeline overlaps the copies of
    # neighbouring steps with the current step's kernels)
    from nvfp4_w4a4_quantized_quantize_gb300.pipeline import HostPipeline
    x_h = torch.from_numpy(np.ascontiguousarray(x_bits).view(np.int16)).view(torch.bfloat16).pin_memory()
    ids_h = torch.from_numpy(ids).pin_memory()
    tw_h = torch.from_numpy(tw).pin_memory()
    out_h = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()
    h2d = x_h.numel() * 2 + ids_h.numel() * 4 + tw_h.numel() * 4
    d2h = out_h.numel() * 2
    pipe = HostPipeline(layer, T, use_graph=not args.eager)
    pipe.run(x_h, ids_h, tw_h, out_h, args.warmup)
    barrier(world)
    e2e_ms = pipe.run(x_h, ids_h, tw_h, out_h, args.steps)
    # the result read back to the host is the layer output itself
    assert torch.equal(out_h.view(torch.int16), pipe.last_output(args.steps).cpu().view(torch.int16))
    assert torch.equal(out_h.view(torch.int16), out.cpu().view(torch.int16))
    e2e_tot = max_over_ranks(e2e_ms, world)
    e2e_tps = job_throughput(T, world, e2e_tot / args.steps)
    st, where = L.device_status()
    if st != 0:
        raise RuntimeError(f"device wait ran out ({where}) in the timed region")

    # ---- activation quantizer + RAC on the 8192 x 4096 Student-t workload (HBM-bound)
    act = act_quant_bench(args, L, wl, dev, flush, peaks) if rank == 0 else None
    # ---- baseline rows: the same layer without RAC (k = 0), and the expert GEMMs in bf16
    base = baseline_rows(args, layer, x, ids_d, tw_d, w13_bits, w2_bits, cfg, dev, flush, ms_per_step,
                         t_gu, t_dn, stage_ms_rac) if rank == 0 else None
    trainer = trainer_rows(args, L, dev, flush, peaks) if rank == 0 else None
    del layer
    torch.cuda.empty_cache()
    # ---- the other workloads of the measurement plan: the dense RAC GEMM and the decode step
    dense = dense_rows(args, L, wl, dev, flush, peaks) if rank == 0 else None
    decode = decode_rows(args, L, wl, dev, flush, peaks) if rank == 0 else None
    probe = mma_probe_row(L) if rank == 0 else None

    result = {
        "metric": METRIC,
        "value": round(tokens_per_s, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "nvfp4(e2m1+ue4m3) x nvfp4 -> fp32 acc, bf16 io",
        "data": "synthetic (seeded; MoE routing Zipf(1.1), 1% outlier channels x20, N(0,0.02) weights)",
        "config": {"workload": cfg.name, "tokens": T, "hidden": H, "experts": E, "topk": topk,
                   "intermediate": I, "rac_k": k, "parallelism": f"dp{world} (independent batches)",
                   "l2": "flushed (512 MiB write) before every timed step"},
        "gemm_tflops": round((flop_gu + flop_dn) / (ms_per_step * 1e-3) / 1e12, 2),
        "kernel_ms": {"gemm_gate_up": round(t_gu, 4), "gemm_down": round(t_dn, 4),
                      "timing": "CUDA events around each GEMM inside the timed graph replays"},
        "roofline": {"kernel": "gemm_kernel (gate/up, SwiGLU epilogue)", "bound": "tensor",
                     "achieved": round(ach_gu, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(ach_gu / fp4_peak, 4), "traffic": gemm_traffic_per_launch("gate_up"),
                     "peak_source": f"{src} bf16 burst {peaks['bf16_tflops']} x nominal NVFP4/BF16 ratio 6"},
        "e2e": {"value": round(e2e_tps, 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "launch_mode": "cuda graph (one replay per step)" if graph is not None else "eager stream launches",
        "clocks": clocks,
        "wall_s_timed_region": round(t_wall, 3),
    }
    if act:
        result["act_quant_rac"] = act
    if base:
        result["baselines"] = base
    if trainer:
        result["trainer_side"] = trainer
    if dense:
        result["dense_rac_gemm"] = dense
    if decode:
        result["moe_decode"] = decode
    if probe:
        result["mma_probe"] = probe
    return result, (x_bits, ids, tw, w13_bits, w2_bits, cfg)


def _time_replays(fn, flush, steps, warmup):
    from nvfp4_w4a4_quantized_quantize_gb300.timing import time_graph_replays
    return time_graph_replays(fn, flush, steps, warmup)


def clocked(fn, flush, min_s: float = 0.35, warmup: int = 3):
    """Median ms of CUDA-graph replays of fn (L2 flushed before each, outside the events), replayed
    for at least min_s seconds so that the clock sampler running meanwhile takes several samples."""
    import torch
    t_est = _time_replays(fn, flush, 3, 1)
    per_iter_s = (t_est + 0.12) * 1e-3  # + the 512 MiB flush write
    steps = max(5, int(min_s / per_iter_s))
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    ms = _time_replays(fn, flush, steps, warmup)
    return ms, sampler.stop()


def stage_times(fwd, flush, steps: int):
    """Mean per-stage ms of a layer forward captured in a CUDA graph with external timing events
    (fwd(events) runs the forward with the events dict), L2 flushed before each replay."""
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300.layers import MOE_STAGES
    try:
        ev = {n: (torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True))
              for n in MOE_STAGES}
    except TypeError:
        return {}
    cap = torch.cuda.Stream()
    cap.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(cap):
        fwd(None)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fwd(ev)
    torch.cuda.current_stream().wait_stream(cap)
    used = set()
    acc = {}
    for i in range(steps + 2):
        flush.zero_()
        g.replay()
        torch.cuda.synchronize()
        if i < 2:
            continue
        for n, (a, b) in ev.items():
            try:
                acc.setdefault(n, []).append(a.elapsed_time(b))
                used.add(n)
            except (RuntimeError, ValueError):  # a stage this layer does not run (never recorded)
                pass
    return {n: sum(v) / len(v) for n, v in acc.items() if n in used}


def dense_rows(args, L, wl, dev, flush, peaks):
    """The dense prefill-shaped RAC linear layer (M 4096, K 4096, N 14336, k 64): the whole forward
    (quantize + select + residual and weight tails + GEMM) and the block-scaled GEMM alone, against
    the NVFP4 roofline.  X from the workload generator; W ~ N(0, 0.02^2) drawn on the device."""
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300.layers import RacLinear
    cfg = wl.CFG_DENSE
    x_bits = wl.activations(cfg.M, cfg.K, cfg.seed, cfg.dist, cfg.x_scale, cfg.n_outliers, cfg.outlier_gain)[0]
    gen = torch.Generator(device=dev).manual_seed(cfg.seed + 1)
    w = (torch.randn(cfg.N, cfg.K, device=dev, generator=gen) * cfg.w_std).bfloat16()
    lin = RacLinear(w, cfg.k, cfg.M)
    del w
    x = _bf16(x_bits, dev)
    out = torch.empty(cfg.M, cfg.N, dtype=torch.bfloat16, device=dev)
    ms_fwd, clk_fwd = clocked(lambda: lin.forward(x, out), flush)
    lin.forward(x, out)

    def gemm():
        L.w4a4_rac_grouped_gemm(lin.a.codes, lin.a.sf, lin.a.sf_cols, lin.a.tscale, lin.w.codes, lin.w.sf, lin.w.sf_cols,
                                lin.w.tscale, lin.N, lin.K, lin.k, None, out, rows=cfg.M)
    ms_gemm, clk_gemm = clocked(gemm, flush)
    flop = 2.0 * cfg.M * cfg.N * (cfg.K + cfg.k)
    fp4_peak = peaks["bf16_tflops"] * FP4_OVER_BF16
    tf = flop / (ms_gemm * 1e-3) / 1e12
    del lin, x, out
    torch.cuda.empty_cache()
    return {"workload": cfg.name, "gemm_ms": round(ms_gemm, 4), "gemm_tflops": round(tf, 1),
            "gemm_frac_of_fp4_peak": round(tf / fp4_peak, 4), "fp4_peak_tflops": round(fp4_peak, 1),
            "layer_forward_ms": round(ms_fwd, 4),
            "layer_tflops": round(flop / (ms_fwd * 1e-3) / 1e12, 1), "gemm_flop": flop,
            "clocks_gemm": clk_gemm, "clocks_forward": clk_fwd,
            "timing": "median of CUDA-graph replays, L2 flushed (512 MiB write) before each"}


def decode_rows(args, L, wl, dev, flush, peaks):
    """The decode-shaped MoE step (512 tokens, H 4096, 128 experts, top-8 uniform routing,
    I 1536, k = 64 per GEMM): tokens/s, the grouped GEMMs against the HBM roofline (about 32 routed
    rows per expert, so the GEMMs stream each expert's weights once), and the same layer at k = 0
    and in FP8 W8A8 (the pages' decode comparison).  Tokens from the workload generator; expert
    weights ~ N(0, 0.02^2) drawn on the device."""
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Fp8MoELayer, MoERacLayer
    cfg = wl.CFG_MOE_DECODE
    E, H, I, T, topk, k = cfg.E, cfg.H, cfg.I, cfg.T, cfg.topk, cfg.k
    x_bits, ids, tw, _ = cfg.make_tokens()
    gen = torch.Generator(device=dev).manual_seed(cfg.seed + 11)
    w13 = (torch.randn(E, 2 * I, H, device=dev, generator=gen) * cfg.w_std).bfloat16()
    w2 = (torch.randn(E, H, I, device=dev, generator=gen) * cfg.w_std).bfloat16()
    x = _bf16(x_bits, dev)
    ids_d, tw_d = torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    steps = max(5, min(args.steps, 50))
    res = {"workload": cfg.name}
    layer = MoERacLayer(w13, w2, k, topk, T)
    ms, clk = clocked(lambda: layer.forward(x, ids_d, tw_d, out), flush)
    st = stage_times(lambda ev: layer.forward(x, ids_d, tw_d, out, events=ev), flush, steps)
    # weight bytes the two GEMMs stream (codes + scales of the K + k columns of every expert)
    wb13 = E * 2 * I * ((H + k) // 2 + L.sf_cols(H + k))
    wb2 = E * H * ((I + k) // 2 + L.sf_cols(I + k))
    t_gemm = st.get("gemm_gate_up", 0.0) + st.get("gemm_down", 0.0)
    gbs = (wb13 + wb2) / (t_gemm * 1e-3) / 1e9 if t_gemm else None
    res["w4a4_rac"] = {"ms_per_step": round(ms, 4), "tokens_per_s": round(T / (ms * 1e-3), 1), "clocks": clk,
                       "stage_ms": {n: round(v, 4) for n, v in st.items()},
                       "gemm_weight_bytes": int(wb13 + wb2),
                       "gemm_weight_gbs": round(gbs, 1) if gbs else None,
                       "gemm_frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 4) if gbs else None}
    del layer
    layer0 = MoERacLayer(w13, w2, 0, topk, T)
    ms0, clk0 = clocked(lambda: layer0.forward(x, ids_d, tw_d, out), flush)
    del layer0
    res["w4a4_no_rac"] = {"ms_per_step": round(ms0, 4), "tokens_per_s": round(T / (ms0 * 1e-3), 1), "clocks": clk0}
    f8 = Fp8MoELayer(w13, w2, topk, T)
    ms8, clk8 = clocked(lambda: f8.forward(x, ids_d, tw_d, out), flush)
    del f8, w13, w2
    torch.cuda.empty_cache()
    res["fp8_w8a8"] = {"ms_per_step": round(ms8, 4), "tokens_per_s": round(T / (ms8 * 1e-3), 1), "clocks": clk8}
    res["w4a4_over_fp8"] = round(ms8 / ms0, 3)
    res["w4a4_rac_over_fp8"] = round(ms8 / ms, 3)
    res["rac_cost"] = round((ms - ms0) / ms0, 4)
    res["timing"] = "median of CUDA-graph replays, L2 flushed (512 MiB write) before each"
    return res


def mma_probe_row(L):
    """The measured NVFP4 tensor-core rate (nvq_fp4_mma_rate: back-to-back M128 N256 K64 MMAs on
    every SM, no memory traffic) with the SM clock sampled meanwhile: cycles per MMA = time x
    median SM clock / MMAs."""
    import torch
    sampler = ClockSampler(torch.cuda.current_device())
    L.fp4_mma_rate(4096)
    mmas = 65536
    sampler.start()
    t0 = time.perf_counter()
    rates = []
    while time.perf_counter() - t0 < 0.4:
        rates.append(L.fp4_mma_rate(mmas))
    clk = sampler.stop()
    tf = statistics.median(rates)
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    res = {"tflops": round(tf, 1), "launches": len(rates), "mmas_per_sm": mmas, "clocks": clk}
    if clk.get("sm_mhz"):
        flop_per_mma = 2.0 * 128 * 256 * 64
        res["cycles_per_mma"] = round(flop_per_mma * sms / (tf * 1e12) * clk["sm_mhz"] * 1e6, 1)
    return res


def baseline_rows(args, layer, x, ids_d, tw_d, w13_bits, w2_bits, cfg, dev, flush, ms_rac, t_gu, t_dn, stage_ms_rac):
    """The comparison rows of the measurement plan: the same layer with k = 0 (W4A4 without RAC;
    RAC cost = (t_RAC - t_noRAC) / t_noRAC), and the two expert GEMMs with SwiGLU in bf16 through
    cuBLAS (a per-expert loop over this batch's routed rows, captured in a CUDA graph)."""
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300.layers import MoERacLayer
    E, H, I, T, topk = cfg.E, cfg.H, cfg.I, cfg.T, cfg.topk
    steps = max(5, min(args.steps, 20))
    w13 = _bf16(w13_bits.reshape(E * 2 * I, H), dev).view(E, 2 * I, H)
    w2 = _bf16(w2_bits.reshape(E * H, I), dev).view(E, H, I)
    layer0 = MoERacLayer(w13, w2, 0, topk, T)
    out0 = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ms0, clk0 = clocked(lambda: layer0.forward(x, ids_d, tw_d, out0), flush)
    # the RAC layer with every launch in order on one stream (no side stream)
    layer1 = MoERacLayer(w13, w2, cfg.k, topk, T, side_stream=False)
    out1 = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ms1, clk1 = clocked(lambda: layer1.forward(x, ids_d, tw_d, out1), flush)
    del layer1, out1
    stage0 = stage_times(lambda ev: layer0.forward(x, ids_d, tw_d, out0, events=ev), flush, steps)
    del layer0, out0
    # bf16 expert GEMMs on the routed rows of this batch (the rows gathered outside the timing)
    off = layer.grp_off.cpu().tolist()
    cnt = layer.grp_rows.cpu().tolist()
    src = layer.row_src.long()
    xs, ys = [], []
    for e in range(E):
        r = src[off[e]:off[e] + cnt[e]]
        xs.append(x[r // topk].contiguous() if cnt[e] else None)
        ys.append(torch.empty(cnt[e], H, dtype=torch.bfloat16, device=dev) if cnt[e] else None)

    def bf16_gemms():
        for e in range(E):
            if xs[e] is not None:
                g = xs[e] @ w13[e].t()
                h = torch.nn.functional.silu(g[:, :I]) * g[:, I:]
                torch.matmul(h, w2[e].t(), out=ys[e])

    ms_bf = _time_replays(bf16_gemms, flush, steps, 3)
    rows = T * topk
    flop_k0 = 2.0 * rows * (2 * I) * H + 2.0 * rows * H * I
    del xs, ys
    # FP8 W8A8 block-scaled baseline (E4M3, power-of-two scale per 1 x 128 / 128 x 128 tile): the
    # whole layer, and each of its two grouped GEMMs alone
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib as L
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Fp8MoELayer
    f8 = Fp8MoELayer(w13, w2, topk, T)
    del w13, w2
    out8 = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    ms8 = _time_replays(lambda: f8.forward(x, ids_d, tw_d, out8), flush, steps, 3)
    f8.forward(x, ids_d, tw_d, out8)
    t8_gu = _time_replays(lambda: L.fp8_blockscaled_grouped_gemm(
        f8.a_routed.codes, f8.a_routed.sf, f8.a_routed.sf_cols, f8.w13.codes, f8.w13.sf, f8.w13.sf_cols, 2 * I, H, f8.h,
        groups=E, grp_off=f8.grp_off, grp_rows=f8.grp_rows, rows=f8.cap, epilogue=L.NVQ_EPI_SWIGLU), flush, steps, 3)
    t8_dn = _time_replays(lambda: L.fp8_blockscaled_grouped_gemm(
        f8.a2.codes, f8.a2.sf, f8.a2.sf_cols, f8.w2.codes, f8.w2.sf, f8.w2.sf_cols, H, I, f8.y, groups=E,
        grp_off=f8.grp_off, grp_rows=f8.grp_rows, rows=f8.cap, epilogue=L.NVQ_EPI_ROW_SCALE, row_w=f8.row_w),
        flush, steps, 3)
    peaks, src = _peaks()
    fp8_peak = peaks["bf16_tflops"] * 2.0
    flop_gu8 = 2.0 * rows * (2 * I) * H
    del f8, out8
    torch.cuda.empty_cache()
    breakdown = {n: {"k32_ms": round(stage_ms_rac[n], 4), "k0_ms": round(stage0.get(n, 0.0), 4),
                     "rac_ms": round(stage_ms_rac[n] - stage0.get(n, 0.0), 4)} for n in stage_ms_rac}
    return {
        "w4a4_no_rac_layer": {"ms_per_step": round(ms0, 4), "tokens_per_s": round(T / (ms0 * 1e-3), 1),
                              "rac_cost": round((ms_rac - ms0) / ms0, 4), "clocks": clk0},
        "w4a4_rac_layer_one_stream": {"ms_per_step": round(ms1, 4), "tokens_per_s": round(T / (ms1 * 1e-3), 1),
                                      "clocks": clk1},
        "rac_cost_breakdown": {"stages": breakdown,
                               "note": "per-stage device time (CUDA events inside the graph, mean over replays) of the "
                                       "layer at k = 32 per GEMM and at k = 0; the side-stream stages (tokens, weight "
                                       "tails) overlap the main stream's, so the stages do not sum to the step"},
        "bf16_expert_gemms": {"ms": round(ms_bf, 4), "tflops": round(flop_k0 / (ms_bf * 1e-3) / 1e12, 1),
                              "impl": "cuBLAS per-expert loop (gate/up, SwiGLU, down) in a CUDA graph"},
        "w4a4_rac_expert_gemms": {"ms": round(t_gu + t_dn, 4),
                                  "useful_tflops": round(flop_k0 / ((t_gu + t_dn) * 1e-3) / 1e12, 1),
                                  "speedup_vs_bf16": round(ms_bf / (t_gu + t_dn), 3)},
        "fp8_w8a8_layer": {"ms_per_step": round(ms8, 4), "tokens_per_s": round(T / (ms8 * 1e-3), 1),
                           "w4a4_over_fp8": round(ms8 / ms0, 3), "w4a4_rac_over_fp8": round(ms8 / ms_rac, 3),
                           "gemm_gate_up_ms": round(t8_gu, 4), "gemm_down_ms": round(t8_dn, 4),
                           "gate_up_tflops": round(flop_gu8 / (t8_gu * 1e-3) / 1e12, 1),
                           "gate_up_frac_of_fp8_peak": round(flop_gu8 / (t8_gu * 1e-3) / 1e12 / fp8_peak, 4),
                           "fp8_peak_tflops": round(fp8_peak, 1),
                           "peak_source": f"{src} bf16 burst x nominal FP8/BF16 ratio 2",
                           "impl": "Fp8MoELayer: E4M3, power-of-two scale per 1x128 / 128x128 tile, tcgen05 kind::mxf8f6f4"},
    }


def trainer_rows(args, L, dev, flush, peaks):
    """Trainer-side rows: weight_qdq (QDQ_W of Eq. (12)) over all expert weights of the decode
    workload shape (W13 [128, 3072, 4096] + W2 [128, 4096, 1536], 2.42 G elements, with the bf16
    W-hat), against the HBM roofline; and a W4A16 QAT linear layer (forward + backward at
    M = 4096, K = 4096, N = 14336) against the same layer in plain bf16."""
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Operand
    from nvfp4_w4a4_quantized_quantize_gb300.qat import QATLinear
    gen = torch.Generator(device=dev).manual_seed(5)
    res = {}
    total_ms, elems = 0.0, 0
    clks = []
    for (G, N, K) in ((128, 3072, 4096), (128, 4096, 1536)):
        w = (torch.randn(G, N, K, device=dev, generator=gen) * 0.02).bfloat16()
        op = Operand.empty(G * N, K, 0, G, device=dev)
        w_hat = torch.empty(G, N, K, dtype=torch.bfloat16, device=dev)

        def qdq():
            L.weight_qdq(w, G, N, K, op.codes, op.sf, op.sf_cols, op.tscale, w_hat=w_hat, w_hat_dtype=L.NVQ_BF16)
        ms_g, clk_g = clocked(qdq, flush, min_s=0.3)
        total_ms += ms_g
        clks.append(clk_g)
        elems += G * N * K
        del w, op, w_hat
        torch.cuda.empty_cache()
    alg = elems * (2 + 0.5625 + 2)
    res["weight_qdq"] = {"workload": "W13 [128,3072,4096] + W2 [128,4096,1536], bf16 W-hat", "elements": elems,
                         "ms": round(total_ms, 4), "algorithmic_bytes": int(alg),
                         "gbs": round(alg / (total_ms * 1e-3) / 1e9, 1),
                         "frac_of_measured_hbm": round(alg / (total_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
                         "clocks": clks}
    torch.manual_seed(6)
    M, K, N = 4096, 4096, 14336
    x = torch.randn(M, K, device=dev).bfloat16().requires_grad_(True)
    lin = QATLinear(K, N, device=dev)
    gy = torch.randn(M, N, device=dev).bfloat16()
    w_plain = lin.weight.detach().clone().requires_grad_(True)

    def step_qat():
        y = lin(x)
        y.backward(gy)

    def step_bf16():
        y = x @ w_plain.t()
        y.backward(gy)

    ts = {}
    for name, fn in (("qat", step_qat), ("bf16", step_bf16)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        times = []
        for _ in range(10):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            b.synchronize()
            times.append(a.elapsed_time(b))
        ts[name] = statistics.median(times)
    res["qat_linear_4096x4096x14336"] = {"ms_fwd_bwd": round(ts["qat"], 4), "bf16_ms_fwd_bwd": round(ts["bf16"], 4),
                                         "qdq_overhead": round((ts["qat"] - ts["bf16"]) / ts["bf16"], 4)}
    del x, lin, gy, w_plain
    torch.cuda.empty_cache()
    return res


def act_quant_bench(args, L, wl, dev, flush, peaks):
    import torch
    cfg = wl.CFG_ACT
    x_bits, _, _ = cfg.make()
    M, K, k = cfg.M, cfg.K, cfg.k
    x = _bf16(x_bits, dev)
    ld = (K + k) // 2
    sfc = L.sf_cols(K + k)
    codes = torch.empty(M, ld, dtype=torch.uint8, device=dev)
    sf = torch.empty(L.sf_bytes(M, sfc), dtype=torch.uint8, device=dev)
    ts = torch.empty(1, 4, dtype=torch.float32, device=dev)
    scores = torch.empty(K, dtype=torch.int64, device=dev)
    idx = torch.empty(k, dtype=torch.int32, device=dev)
    def quant():
        L.nvfp4_quantize(x, codes, sf, sfc, ts, scores=scores)

    def select():
        L.rac_select_quantize(x, ts, scores, k, codes, sf, sfc, idx)

    def step():
        quant()
        select()

    # CUDA-graph replays (as the layer step), L2 flushed before each: the whole path, and each
    # half alone (the selection replays over the scores the last quantize left)
    t_all, clk = clocked(step, flush)
    t_q = _time_replays(quant, flush, args.steps, args.warmup)
    t_r = _time_replays(select, flush, args.steps, args.warmup)
    algo = M * K * (2 + 0.5 + 1 / 16) + M * k * (2 + 0.5 + 1 / 16) + k * 4
    q_bytes = M * K * (2 + 0.5 + 1 / 16)
    hbm = peaks["hbm_gbs"]
    return {"workload": cfg.name, "algorithmic_bytes": int(algo), "ms": round(t_all, 4),
            "gbs": round(algo / (t_all * 1e-3) / 1e9, 1), "frac_of_measured_hbm": round(algo / (t_all * 1e-3) / 1e9 / hbm, 4),
            "nvfp4_quantize_ms": round(t_q, 4), "nvfp4_quantize_gbs": round(q_bytes / (t_q * 1e-3) / 1e9, 1),
            "rac_select_quantize_ms": round(t_r, 4), "clocks": clk,
            "timing": "median of CUDA-graph replays, L2 flushed (512 MiB write) before each"}


# ----------------------------------------------------------------------------- oracle (CPU)
def oracle_moe_sample(tokens, x_bits, ids, tw, w_q13, w_q2, cfg):
    """The oracle's MoE layer on a sample of tokens, in the paper's order of steps; weights are
    already quantized (quantization of the experts' weights happens once, outside the timing)."""
    import oracle
    k, I, H, topk = cfg.k, cfg.I, cfg.H, cfg.topk
    xs = x_bits[tokens]
    q1 = oracle.rac_quantize(xs, k)
    a1c = np.concatenate([q1.codes, q1.tail_codes], 1)
    a1s = np.concatenate([q1.scales, q1.tail_scales], 1)
    h_rows, h_exp, h_w, h_pos = [], [], [], []
    for ti in range(len(tokens)):
        for s in range(topk):
            e = int(ids[tokens[ti], s])
            wc, ws, wts = w_q13[e]
            tc, tsc = oracle.weight_tail(wc, ws, wts, q1.idx)
            gu = oracle.gemm(a1c[ti:ti + 1], a1s[ti:ti + 1], np.concatenate([wc, tc], 1), np.concatenate([ws, tsc], 1),
                             q1.ts.s_dec, wts.s_dec)[0]
            h = oracle.swiglu(gu[:I], gu[I:])
            h_rows.append(oracle.bf16_round(h.astype(np.float32)))
            h_exp.append(e)
            h_w.append(tw[tokens[ti], s])
            h_pos.append(ti * topk + s)
    h_rows = np.stack(h_rows)
    h_exp = np.array(h_exp)
    y = np.zeros((len(h_rows), H), np.uint16)
    for e in np.unique(h_exp):
        sel = np.nonzero(h_exp == e)[0]
        hq = oracle.rac_quantize(h_rows[sel], k)
        wc, ws, wts = w_q2[e]
        tc, tsc = oracle.weight_tail(wc, ws, wts, hq.idx)
        ye = oracle.gemm(np.concatenate([hq.codes, hq.tail_codes], 1), np.concatenate([hq.scales, hq.tail_scales], 1),
                         np.concatenate([wc, tc], 1), np.concatenate([ws, tsc], 1), hq.ts.s_dec, wts.s_dec)
        ye = ye * np.array(h_w)[sel][:, None]
        y[sel] = oracle.bf16_round(ye.astype(np.float32))
    pos = np.zeros(len(tokens) * topk, np.int64)
    pos[np.array(h_pos)] = np.arange(len(h_pos))
    return oracle.moe_combine(y, pos, topk)


def oracle_setup(tokens, ids, w13_bits, w2_bits):
    import oracle
    experts = sorted({int(e) for t in tokens for e in ids[t]})
    w_q13, w_q2 = {}, {}
    for e in experts:
        t13 = oracle.tensor_scale(w13_bits[e])
        c, s = oracle.quantize(w13_bits[e], t13)
        w_q13[e] = (c, s, t13)
        t2 = oracle.tensor_scale(w2_bits[e])
        c, s = oracle.quantize(w2_bits[e], t2)
        w_q2[e] = (c, s, t2)
    return w_q13, w_q2


def cpu_baseline(inputs, n_tokens=48, n_tokens_1t=4):
    """The oracle on a bounded sample of the batch, on every host core (its GEMM spreads the
    output elements over threads), and on one core for a smaller sample."""
    import oracle
    x_bits, ids, tw, w13_bits, w2_bits, cfg = inputs
    tokens = np.arange(n_tokens)
    w_q13, w_q2 = oracle_setup(tokens, ids, w13_bits, w2_bits)
    cores = oracle.hardware_threads()
    oracle.set_threads(cores)
    t0 = time.perf_counter()
    oracle_moe_sample(tokens, x_bits, ids, tw, w_q13, w_q2, cfg)
    dt = time.perf_counter() - t0
    oracle.set_threads(1)
    t1 = time.perf_counter()
    oracle_moe_sample(tokens[:n_tokens_1t], x_bits, ids, tw, w_q13, w_q2, cfg)
    dt1 = time.perf_counter() - t1
    return {"value": round(n_tokens / dt, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "single_thread_value": round(n_tokens_1t / dt1, 4),
            "sample": f"{n_tokens} tokens ({n_tokens * cfg.topk} routed rows) of the {cfg.name} batch, "
                      f"full layer (quantize, select k={cfg.k}, tails, both GEMMs, SwiGLU, combine) on {cores} host "
                      f"threads, {dt:.1f} s; single-thread value from the first {n_tokens_1t} tokens, {dt1:.1f} s; "
                      f"expert weights pre-quantized outside the timing"}


def run_reference(args, world, rank):
    """The oracle, as it stands, on the host cores: each step one bounded sample of the batch."""
    from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
    if rank != 0:
        return None
    cfg = wl.CFG_MOE_PREFILL
    x_bits, ids, tw, _ = cfg.make_tokens()
    w13_bits, w2_bits = cfg.make_weights()
    import oracle
    per_step = 8
    tokens = np.arange(per_step)
    w_q13, w_q2 = oracle_setup(tokens, ids, w13_bits, w2_bits)
    cores = oracle.hardware_threads()
    oracle.set_threads(cores)
    for _ in range(args.warmup):
        oracle_moe_sample(tokens, x_bits, ids, tw, w_q13, w_q2, cfg)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_moe_sample(tokens, x_bits, ids, tw, w_q13, w_q2, cfg)
    dt = time.perf_counter() - t0
    v = per_step * args.steps / dt
    return {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp32 encode / exact int64 GEMM",
        "data": "synthetic (seeded)",
        "config": {"workload": cfg.name, "tokens": cfg.T, "hidden": cfg.H, "experts": cfg.E, "topk": cfg.topk,
                   "intermediate": cfg.I, "rac_k": cfg.k, "parallelism": f"{cores} host threads"},
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{per_step} tokens ({per_step * cfg.topk} routed rows) of the batch per step, "
                                   f"the oracle's GEMM spread over {cores} host threads"},
        "e2e": {"value": round(v, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def sweep_k(args):
    """The residual channel ratio sweep on one GPU (see the package's sweep module)."""
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300 import sweep
    torch.cuda.set_device(0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    sampler = ClockSampler(0)
    sampler.start()
    res = sweep.run(flush, args.steps, args.warmup)
    return {"sweep": "rac_k_ratio", "steps": args.steps, "warmup": args.warmup,
            "l2": "flushed (512 MiB write) before every replay", "data": "synthetic (seeded)", **res,
            "clocks": sampler.stop()}


def profile_case(name: str):
    """Cases for ncu captures (no timing, no JSON line): 'moe_prefill' runs three eager forwards of
    the bench's full-size MoE layer (for the one-pass launch list only); 'moe_small' runs two MoE layer
    forwards at E=32, T=4096, H=2048, I=768, top-8, k=32 (about 1 GB on the device);
    'act_256mb' quantizes and selects twice on a 32768 x 4096 bf16 activation (256 MB, larger
    than L2), k=64; 'act_8192x4096' runs the activation workload of the bench line three times
    (64 MB, L2 flushed before each); 'fp8_moe_small' runs two forwards of the FP8 W8A8 layer on the
    'moe_small' shapes; 'row_tails_kK' runs the row-path tails once each at k = K: the gate/up
    weight tail of 128 experts (N 1536, K 2048) and the residual tail of h (131072 x 768, 128
    groups)."""
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib as L
    from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
    from nvfp4_w4a4_quantized_quantize_gb300.layers import MoERacLayer, Operand
    dev = "cuda"
    if name == "moe_prefill":
        # the bench's layer step at full size, three eager forwards (for the launch list)
        cfg = wl.CFG_MOE_PREFILL
        x_bits, ids, tw, _ = cfg.make_tokens()
        w13_bits, w2_bits = cfg.make_weights()
        E, H, I, T = cfg.E, cfg.H, cfg.I, cfg.T
        layer = MoERacLayer(_bf16(w13_bits.reshape(E * 2 * I, H), dev).view(E, 2 * I, H),
                            _bf16(w2_bits.reshape(E * H, I), dev).view(E, H, I), cfg.k, cfg.topk, T)
        x = _bf16(x_bits, dev)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        ids_d, tw_d = torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev)
        for _ in range(3):
            layer.forward(x, ids_d, tw_d, out)
    elif name == "moe_small":
        E, T, H, I, k, topk = 32, 4096, 2048, 768, 32, 8
        cfg = wl.MoELayer("moe_small", T=T, H=H, E=E, topk=topk, I=I, k=k, seed=7, routing="zipf", n_outliers=20)
        x_bits, ids, tw, _ = cfg.make_tokens()
        w13_bits, w2_bits = cfg.make_weights()
        layer = MoERacLayer(_bf16(w13_bits.reshape(E * 2 * I, H), dev).view(E, 2 * I, H),
                            _bf16(w2_bits.reshape(E * H, I), dev).view(E, H, I), k, topk, T)
        x = _bf16(x_bits, dev)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        ids_d, tw_d = torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev)
        for _ in range(2):
            layer.forward(x, ids_d, tw_d, out)
    elif name == "fp8_moe_small":
        from nvfp4_w4a4_quantized_quantize_gb300.layers import Fp8MoELayer
        E, T, H, I, topk = 32, 4096, 2048, 768, 8
        cfg = wl.MoELayer("moe_small", T=T, H=H, E=E, topk=topk, I=I, k=0, seed=7, routing="zipf", n_outliers=20)
        x_bits, ids, tw, _ = cfg.make_tokens()
        w13_bits, w2_bits = cfg.make_weights()
        layer = Fp8MoELayer(_bf16(w13_bits.reshape(E * 2 * I, H), dev).view(E, 2 * I, H),
                            _bf16(w2_bits.reshape(E * H, I), dev).view(E, H, I), topk, T)
        x = _bf16(x_bits, dev)
        out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        ids_d, tw_d = torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev)
        for _ in range(2):
            layer.forward(x, ids_d, tw_d, out)
    elif name == "row_tails_kK":
        from nvfp4_w4a4_quantized_quantize_gb300.layers import quantize_weights
        L.set_tail_path(L.NVQ_TAIL_ROWS)
        gen = torch.Generator(device=dev).manual_seed(13)
        G, N, K = 128, 1536, 2048
        op = quantize_weights((torch.randn(G, N, K, device=dev, generator=gen) * 0.02).bfloat16(), K)
        idx = torch.arange(K, dtype=torch.int32, device=dev).unsqueeze(0)
        L.rac_weight_tail(G, N, K, K, idx, op.codes, op.sf, op.sf_cols, op.tscale)
        del op
        M, K2, G2 = 131072, 768, 128
        x = torch.randn(M, K2, device=dev, generator=gen).bfloat16()
        a = Operand.empty(M, K2, K2, G2)
        sc = torch.zeros(G2, K2, dtype=torch.int64, device=dev)
        L.nvfp4_quantize(x, a.codes, a.sf, a.sf_cols, a.tscale, scores=sc, groups=G2)
        idx2 = torch.arange(K2, dtype=torch.int32, device=dev).repeat(G2, 1).contiguous()
        L.rac_residual_tail(x, a.tscale, idx2, K2, a.codes, a.sf, a.sf_cols, groups=G2)
        L.set_tail_path(L.NVQ_TAIL_AUTO)
    elif name == "act_8192x4096":
        # the activation workload of the bench line, three times, L2 flushed before each
        cfg = wl.CFG_ACT
        x_bits, _, _ = cfg.make()
        M, K, k = cfg.M, cfg.K, cfg.k
        x = _bf16(x_bits, dev)
        op = Operand.empty(M, K, k)
        sc = torch.empty(K, dtype=torch.int64, device=dev)
        idx = torch.empty(k, dtype=torch.int32, device=dev)
        flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        for _ in range(3):
            flush.zero_()
            L.nvfp4_quantize(x, op.codes, op.sf, op.sf_cols, op.tscale, scores=sc)
            L.rac_select_quantize(x, op.tscale, sc, k, op.codes, op.sf, op.sf_cols, idx)
    else:
        M, K, k = 32768, 4096, 64
        gen = torch.Generator(device=dev).manual_seed(11)
        x = torch.randn(M, K, device=dev, generator=gen).bfloat16()
        op = Operand.empty(M, K, k)
        sc = torch.empty(K, dtype=torch.int64, device=dev)
        idx = torch.empty(k, dtype=torch.int32, device=dev)
        for _ in range(2):
            L.nvfp4_quantize(x, op.codes, op.sf, op.sf_cols, op.tscale, scores=sc)
            L.rac_select_quantize(x, op.tscale, sc, k, op.codes, op.sf, op.sf_cols, idx)
    torch.cuda.synchronize()
    if L.device_status() != (0, 0):
        raise SystemExit(f"device status {L.device_status()}")
    print("profile case", name, "ok", flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)  # ~0.25 s timed: several clock samples
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch the kernels one by one instead of a CUDA graph")
    ap.add_argument("--sweep-k", action="store_true",
                    help="residual channel ratio sweep (0 to 100 %% of K) at the activation, dense and MoE "
                         "workloads: error and time per ratio, one JSON line, then exit")
    ap.add_argument("--profile-case", choices=["moe_prefill", "moe_small", "fp8_moe_small", "act_256mb", "act_8192x4096",
                                               "row_tails_kK"],
                    help="run a small case twice for an ncu capture and exit (no timing)")
    args = ap.parse_args()
    if args.profile_case:
        profile_case(args.profile_case)
        return
    args.warmup = max(args.warmup, 3)
    if args.sweep_k:
        print(json.dumps(sweep_k(args)), flush=True)
        return
    world, rank, local = dist_setup()
    if args.gpus != world:
        raise SystemExit(f"bench.py: --gpus {args.gpus} but this process group has {world} rank(s); launch N > 1 ranks "
                         f"with: python -m torch.distributed.run --nproc-per-node {args.gpus} --master-addr 127.0.0.1 "
                         f"bench.py --gpus {args.gpus} ...")
    if args.impl == "reference":
        res = run_reference(args, world, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return
    res, inputs = run_ours(args, world, rank, local)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(inputs)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
