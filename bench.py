"""Benchmark of one MoE layer pass (forward + backward) on GB300, printing one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one pass of the whole hot path over one batch: routing, counting/index generation,
permutation, grouped SwiGLU GEMM, combine, and the full backward (combine/routing backward,
grouped GEMM backward incl. weight gradients, un-permute). Inputs are seeded synthetic tensors
resident in HBM before timing starts; the expert weights (768 MiB at the default workload) and the
grouped activations exceed the 129 MB L2, so no flush is needed between steps.

Timing: the K timed steps run back to back with nothing but the pass itself between two CUDA
events on the launching stream; each step is one replay of a CUDA graph of the whole pass (the
library's calls recorded once; --eager launches them call by call instead). Per-kernel times (and the grouped GEMM's roofline) come from a
separate pass of eager steps afterwards, with an event pair around every C-ABI call. The roofline's
bf16 denominator follows the clocks sampled while those kernels ran: the measured burst peak,
unless sw_power_cap was active, then the measured sustained peak; both fractions are printed.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the layer has no
exchange step on one node here): weak scaling, max-over-ranks time, value = all ranks' tokens / time.

--impl reference times the fp64 CPU oracle (as it stands) on a bounded token sample of the same
workload on the host cores; on N > 1 only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import json
import os
import math
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd tokens/s (E=64,k=8,d=2048); grouped-GEMM % BF16 peak"
METRIC_FWD = "MoE layer fwd tokens/s (E=64,k=8,d=2048); grouped-GEMM % BF16 peak"

# DRAM bytes (read + write) of one step's grouped-GEMM launches, from an ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum), stored with the digest of the GEMM sources that
# were captured. The bench reports the figure only while the sources still have that digest: once a
# kernel changes, its traffic is unmeasured (null) until it is captured again.
GEMM_SOURCES = ("gemm_rows.cu", "gemm_tc.cu", "tc_ptx.cuh", "tma_host.cuh", "common.cuh")
GEMM_TRAFFIC = {    # workload -> (bytes per step, source digest)
    "fwdbwd_t8192": (5759519488, "1d603581913ada8f"),
    "fwd_t4096": (1220222464, "1d603581913ada8f"),
}
DEFAULT_WORKLOAD = "fwdbwd_t8192"


def gemm_source_digest():
    """sha256 (first 16 hex digits) over the grouped-GEMM kernel sources, in a fixed order."""
    import hashlib
    h = hashlib.sha256()
    for name in GEMM_SOURCES:
        with open(os.path.join(ROOT, "mixture_experts_layer_histogram_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def gemm_traffic(workload):
    """Measured DRAM bytes per step of the grouped GEMM, or None when no capture matches the sources."""
    rec = GEMM_TRAFFIC.get(workload)
    if rec is None or rec[1] != gemm_source_digest():
        return None
    return rec[0]


def choose_peak(peaks, reasons):
    """The dense bf16 denominator that the sampled clocks justify: the sustained (power-capped)
    figure when sw_power_cap was active while the kernels were timed, else the burst figure."""
    capped = reasons is not None and "sw_power_cap" in reasons
    if capped and peaks.get("bf16_sustained"):
        return peaks["bf16_sustained"], "sustained"
    return peaks["bf16"], "burst"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            p = json.load(fh)
        return dict(hbm=p["hbm_gbs"], bf16=p["bf16_tflops"], bf16_sustained=p.get("bf16_tflops_sustained"),
                    src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sustained=1700.0, src="fallback")


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# Replicas (one per GPU, no data-path collective): the job's time is the slowest rank's, and the
# job processes world x T tokens per step. These helpers take any torch.distributed backend.
def max_over_ranks(ms, world, device):
    """The largest of every rank's `ms` (the value itself when alone)."""
    if world == 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_rank, steps, ms):
    """Whole-job throughput: every rank's tokens over the max-over-ranks time of `steps` steps."""
    return world * tokens_per_rank * steps / (ms * 1e-3)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples, kept only if taken inside the timed window."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.samples = []          # (host time, csv line)
        self.window = None         # (t0, t1) host times of the window summary() describes

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self

        def reader():
            for ln in self.proc.stdout:
                if ln.strip():
                    self.samples.append((time.time(), ln))

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        return self

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, window=None):
        window = window or self.window
        if not self.samples or window is None:
            return None
        t0, t1 = window
        lines = [ln for ts, ln in self.samples if t0 <= ts <= t1 + 0.05]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in lines:
            f = [x.strip() for x in ln.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import moe_inputs
    from mixture_experts_layer_histogram_gb300 import HostPipeline, MoELayer
    from mixture_experts_layer_histogram_gb300 import _lib as L

    world, rank, local = _dist()
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    w = moe_inputs.WORKLOADS[args.workload]
    inp = moe_inputs.make_all(w, dev)
    x, logits, wgu, wd = inp["x"], inp["logits"], inp["w_gate_up"], inp["w_down"]
    g = inp.get("g")
    bwd = w.backward
    layer = MoELayer(w.T, w.d, w.E, w.k, w.f, w.torch_dtype, dev, backward=bwd, recompute=args.recompute,
                     router=args.router, gather=args.gather)
    wr = moe_inputs.make_router_weight(w, dev) if args.router else None
    stream = torch.cuda.current_stream(dev)
    M = w.T * w.k
    gemm_flop = (18.0 if bwd else 6.0) * M * w.d * w.f

    def step(ev=None):
        if ev is None:
            layer.forward(x, None if args.router else logits, wgu, wd, w_router=wr)
            if bwd:
                layer.backward(g, wgu, wd)
            return
        # events around each C-ABI call, on the stream the kernels are launched on
        ev[0].record(stream)
        if args.router:
            L.moe_router_fwd(x, wr, w.k, layer.logits, layer.topk_idx, layer.topk_w, layer.ws_router)
            ev[1].record(stream)
            L.moe_count_index(layer.topk_idx, w.E, layer.counts, layer.offsets, layer.tile_offsets,
                              layer.row_of_slot, layer.token_of_row, layer.ws_index)
        else:   # routing, counting and index generation in one launch
            L.moe_route_count_index(logits, w.k, layer.topk_idx, layer.topk_w, layer.counts, layer.offsets,
                                    layer.tile_offsets, layer.row_of_slot, layer.token_of_row, layer.ws_index)
            ev[1].record(stream)
        ev[2].record(stream)
        if not args.gather:
            L.moe_permute(x, w.k, w.E, layer.row_of_slot, layer.counts, layer.tile_offsets, layer.x_perm)
        ev[3].record(stream)
        ab = layer.ab if bwd and not args.recompute else None   # as MoELayer.forward: stored only for a backward
        if args.gather:
            L.moe_grouped_ffn_fwd_gather(x, layer.token_of_row, wgu, wd, layer.tile_offsets, layer.offsets, ab,
                                         layer.h, layer.y_perm, layer.ws_ffn)
        else:
            L.moe_grouped_ffn_fwd(layer.x_perm, wgu, wd, layer.tile_offsets, layer.offsets, ab, layer.h,
                                  layer.y_perm, layer.ws_ffn)
        ev[4].record(stream)
        L.moe_combine_fwd(layer.y_perm, layer.topk_w, layer.row_of_slot, w.T, w.k, layer.out)
        ev[5].record(stream)
        if not bwd:
            for j in range(6, 10):
                ev[j].record(stream)
            return
        L.moe_combine_bwd(g, layer.y_perm, layer.topk_w, layer.topk_idx, layer.row_of_slot, layer.counts,
                          layer.tile_offsets, w.E, layer.dy_perm, layer.d_topk_w, layer.d_logits)
        ev[6].record(stream)
        if args.gather:
            (L.moe_grouped_ffn_bwd_recompute_gather if args.recompute else L.moe_grouped_ffn_bwd_gather)(
                layer.dy_perm, x, layer.token_of_row, layer.ab, layer.h, wgu, wd, layer.tile_offsets, layer.offsets,
                layer.dab, layer.dx_perm, layer.dw_gate_up, layer.dw_down, layer.ws_ffn)
        else:
            (L.moe_grouped_ffn_bwd_recompute if args.recompute else L.moe_grouped_ffn_bwd)(
                layer.dy_perm, layer.x_perm, layer.ab, layer.h, wgu, wd, layer.tile_offsets, layer.offsets, layer.dab,
                layer.dx_perm, layer.dw_gate_up, layer.dw_down, layer.ws_ffn)
        ev[7].record(stream)
        L.moe_combine_fwd(layer.dx_perm, None, layer.row_of_slot, w.T, w.k, layer.dx)
        ev[8].record(stream)
        if args.router:
            L.moe_router_bwd(x, wr, layer.d_logits, layer.dx, layer.dw_router, layer.ws_router, accumulate_dx=True)
        ev[9].record(stream)

    graph = None
    if args.graph:   # the timed steps replay one captured pass; per-kernel times come from a separate eager pass
        graph = layer.capture(x, None if args.router else logits, wgu, wd, grad_out=g if bwd else None, w_router=wr)
    clk = ClockSampler(dev.index).start()
    for _ in range(args.warmup):
        step() if graph is None else graph.replay()
    torch.cuda.synchronize(dev)
    st = layer.status()
    if any(st):
        raise RuntimeError(f"device status after warm-up: {st}")

    names = ["router_fwd" if args.router else "route_count_index", "count_index", "permute", "grouped_ffn_fwd",
             "combine_fwd", "combine_bwd", "grouped_ffn_bwd", "unpermute", "router_bwd"]
    # timed region: K clean steps (no per-call events inside), device time on the launching stream
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    w0 = time.time()
    t_start.record(stream)
    for i in range(args.steps):
        step() if graph is None else graph.replay()
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    clk.window = (w0, time.time())
    if world > 1:
        dist.barrier()
    elapsed_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    # per-kernel times: a second pass of eager steps, each C-ABI call between two events on the
    # stream its kernels are launched on (the roofline's achieved rate comes from these)
    if args.kernel_steps is None:
        nper = min(2000, max(50, math.ceil(400.0 / max(elapsed_ms / max(args.steps, 1), 1e-3))))
    else:
        nper = max(3, min(args.steps, args.kernel_steps))
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(10)] for _ in range(nper)]
    torch.cuda.synchronize(dev)
    k0 = time.time()
    for i in range(nper):
        step(evs[i])
    torch.cuda.synchronize(dev)
    kernel_window = (k0, time.time())
    clk.stop()
    per = {n: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(nper))
           for j, n in enumerate(names)}
    st = layer.status()
    if any(st):
        raise RuntimeError(f"device status after timing: {st}")

    # ---------------------------------------------------------------- end to end: host buffers
    # Every step uploads its inputs from pinned host memory and downloads its results through the
    # public host-buffer pipeline; uploads and downloads overlap the neighbouring steps' compute.
    pin = dict(x=x.cpu().pin_memory())
    if not args.router:
        pin["logits"] = logits.cpu().pin_memory()
    if bwd:
        pin["g"] = g.cpu().pin_memory()
    pipe = HostPipeline(layer)
    h2d, d2h = pipe.h2d_bytes(), pipe.d2h_bytes()
    for i in range(3):
        pipe.submit(pin, wgu, wd, next_batch=pin if i < 2 else None, w_router=wr)
    pipe.join()
    torch.cuda.synchronize(dev)
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    pipe.h2d.wait_stream(stream)
    for i in range(args.steps):
        pipe.submit(pin, wgu, wd, next_batch=pin if i + 1 < args.steps else None, w_router=wr)
    pipe.join()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world, dev)
    st = layer.status()
    if any(st):
        raise RuntimeError(f"device status after the end-to-end run: {st}")

    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline and bwd:
        cpu_base = oracle_baseline(w, inp, budget_s=args.cpu_seconds)
    if world > 1:
        dist.destroy_process_group()
    if rank != 0:
        return None

    peaks = _peaks()
    ms = elapsed_ms / args.steps
    gemm_ms = per["grouped_ffn_fwd"] + (per["grouped_ffn_bwd"] if bwd else 0.0)
    achieved = gemm_flop / (gemm_ms * 1e-3) / 1e12
    kclk = clk.summary(kernel_window)
    peak, peak_basis = choose_peak(peaks, kclk["reasons"] if kclk else None)
    es = 2 if w.dtype == "bf16" else 4
    mem_bytes = {   # algorithmic bytes per call (rows in the layer dtype; indices and weights 4 B)
        "permute": (w.T * w.d + M * w.d) * es + M * 4,
        "combine_fwd": (M * w.d + w.T * w.d) * es + M * 8,
        "combine_bwd": (w.T * w.d + 2 * M * w.d) * es + M * 16 + w.T * w.E * 4,
        "unpermute": (M * w.d + w.T * w.d) * es + M * 4,
        # router: x and Wr read, logits and the selection written; backward: d_logits, x, Wr read,
        # dx read and written (accumulated), dWr written
        "router_fwd": (w.T * w.d + w.E * w.d) * es + w.T * w.E * 4 + w.T * w.k * 8,
        "router_bwd": (3 * w.T * w.d + 2 * w.E * w.d) * es + w.T * w.E * 4,
    }
    kern = {n: {"ms": round(v, 4)} for n, v in per.items()
            if (bwd or n in names[:5]) and (args.router or n not in ("router_bwd", "count_index"))
            and not (args.gather and n == "permute")}
    for n, b in mem_bytes.items():
        if n not in kern:
            continue
        kern[n]["GBps"] = round(b / (per[n] * 1e-3) / 1e9, 1)
        kern[n]["frac_hbm"] = round(b / (per[n] * 1e-3) / 1e9 / peaks["hbm"], 3)
    kern["grouped_ffn_fwd"]["TFLOPs"] = round(6.0 * M * w.d * w.f / (per["grouped_ffn_fwd"] * 1e-3) / 1e12, 1)
    if bwd:
        kern["grouped_ffn_bwd"]["TFLOPs"] = round(12.0 * M * w.d * w.f / (per["grouped_ffn_bwd"] * 1e-3) / 1e12, 1)
    value = job_tokens_per_s(world, w.T, args.steps, elapsed_ms)
    if w.dtype == "bf16":
        roofline = {"kernel": "grouped SwiGLU GEMM (tcgen05; per step: fwd GATEUP, DOWN" +
                              ("; bwd DH, WGRAD down, DGRAD, WGRAD gate/up)" if bwd else ")"),
                    "bound": "tensor", "achieved": round(achieved, 1), "peak": peak, "unit": "TFLOP/s",
                    "frac": round(achieved / peak, 3),
                    "peak_kind": f"{peaks['src']} bf16 dense, {peak_basis} (" +
                                 ("sw_power_cap active while the kernels were timed" if peak_basis == "sustained"
                                  else "no power cap seen while the kernels were timed") + ")",
                    "frac_vs_burst": round(achieved / peaks["bf16"], 3),
                    "frac_vs_sustained": (round(achieved / peaks["bf16_sustained"], 3)
                                          if peaks.get("bf16_sustained") else None),
                    "kernel_clocks": kclk,
                    "kernel_times": f"events around each C-ABI call, {nper} eager steps after the timed region",
                    "algorithmic_flop_per_step": gemm_flop,
                    # the stored capture is of the plain pass's six GEMM launches; a gathering or a
                    # recomputing pass runs other ones
                    "traffic": None if (args.gather or args.recompute) else gemm_traffic(w.name),
                    "traffic_unit": "DRAM bytes per step (all grouped-GEMM launches)"}
    else:   # true-fp32 FFMA path: bound by the FP32 pipes (152 SMs x 128 lanes x 2 FLOP x 2.07 GHz)
        fp32_peak = 152 * 128 * 2 * 2.07e9 / 1e12
        roofline = {"kernel": "grouped SwiGLU GEMM (SIMT fp32 FFMA)", "bound": "alu", "achieved": round(achieved, 2),
                    "peak": round(fp32_peak, 1), "unit": "TFLOP/s", "frac": round(achieved / fp32_peak, 4),
                    "peak_kind": "nominal FP32 FFMA rate at the maximum SM clock", "algorithmic_flop_per_step": gemm_flop,
                    "traffic": None}
    line = {
        "metric": METRIC if bwd else METRIC_FWD, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded; see moe_inputs.py)",
        "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "f": w.f, "routing": w.routing,
                   "pass": (("fwd+bwd (recompute)" if args.recompute else "fwd+bwd") if bwd else "fwd") +
                           (", router GEMM in the pass" if args.router else "") +
                           (", permutation fused into the GEMM loads" if args.gather else ""),
                   "saved_activations": ("ab and h" if bwd and not args.recompute else
                                         "h only (no backward reads a, b)" if not bwd else
                                         "h only (the backward recomputes a, b)"),
                   "parallelism": f"replicas x{world}", "launch": "cuda graph" if args.graph else "eager",
                   "l2": "inputs larger than L2 (expert weights 768 MiB, grouped activations > 129 MB); no flush"},
        "roofline": roofline,
        "kernels": kern,
        "e2e": {"value": round(job_tokens_per_s(world, w.T, args.steps, e2e_ms), 1), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms / args.steps, 4),
                "api": "HostPipeline.submit (pinned host inputs and results; copies overlap compute; each slot's pass replayed from a CUDA graph)"},
        "gpu_launches": layer.launches(bwd) * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": cpu_base,
    }
    return line


def oracle_baseline(w, inp, budget_s=15.0, per_step_s=None):
    """Time the fp64 oracle (forward + backward incl. weight gradients) on a bounded token sample."""
    import torch

    import oracle
    cpu = {k: v.detach().cpu() for k, v in inp.items()}

    def run(n):
        sl = slice(0, n)
        x, lg, g = cpu["x"][sl].contiguous(), cpu["logits"][sl].contiguous(), cpu["g"][sl].contiguous()
        t0 = time.perf_counter()
        idx, wt = oracle.route_topk(lg, w.k)
        oracle.index(idx, w.E, 128)
        oracle.moe_tokens(x, idx, wt, cpu["w_gate_up"], cpu["w_down"], g)
        oracle.moe_dweights(x, idx, wt, cpu["w_gate_up"], cpu["w_down"], g)
        return time.perf_counter() - t0

    t_probe = run(4)
    n = max(4, min(w.T, int(4 * budget_s / max(t_probe, 1e-3))))
    dt = run(n)
    return {"value": round(n / dt, 3), "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"first {n} tokens of {w.name}, fwd+bwd incl. dW, {dt:.1f} s wall"}


def run_reference(args):
    world, rank, local = _dist()
    if rank != 0:
        return None
    import torch

    import moe_inputs
    import oracle
    w = moe_inputs.WORKLOADS[args.workload]
    inp = moe_inputs.make_all(w, "cpu")
    cpu = inp
    n = args.ref_tokens

    def one():
        sl = slice(0, n)
        x, lg, g = cpu["x"][sl].contiguous(), cpu["logits"][sl].contiguous(), cpu["g"][sl].contiguous()
        idx, wt = oracle.route_topk(lg, w.k)
        oracle.index(idx, w.E, 128)
        oracle.moe_tokens(x, idx, wt, cpu["w_gate_up"], cpu["w_down"], g)
        oracle.moe_dweights(x, idx, wt, cpu["w_gate_up"], cpu["w_down"], g)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = time.perf_counter() - t0
    value = n * args.steps / dt
    cb = {"value": round(value, 3), "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
          "sample": f"first {n} tokens of {w.name} per step, fwd+bwd incl. dW"}
    return {"impl": "reference", "metric": METRIC if w.backward else METRIC_FWD, "value": round(value, 3), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; see moe_inputs.py)",
            "config": {"workload": w.name, "T": w.T, "d": w.d, "E": w.E, "k": w.k, "f": w.f, "routing": w.routing,
                       "pass": "fwd+bwd", "parallelism": "host cores"},
            "cpu_baseline": cb,
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--router", action="store_true",
                    help="the pass starts from x and router weights: router GEMM with fused top-k, and its backward")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="time the steps launched call by call instead of as replays of one CUDA graph of the pass")
    ap.add_argument("--gather", action="store_true",
                    help="fuse the permutation into the grouped GEMMs' token loads (no moe_permute, no x_perm)")
    ap.add_argument("--recompute", action="store_true",
                    help="backward recomputes ab, h from x_perm (selective activation checkpointing)")
    ap.add_argument("--ref-tokens", type=int, default=8)
    ap.add_argument("--kernel-steps", type=int, default=None,
                    help="eager steps of the separate per-kernel timing pass (default: enough for 0.4 s, at "
                         "least 50, so that the clock sampler sees the kernels run)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
