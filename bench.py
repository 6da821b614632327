#!/usr/bin/env python
"""Benchmark of the MoE layer: one step = schedule + forward + backward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dsv3]
                    [--impl mok|reference]

Default workload: the DeepSeek-V3-shaped layer (T=8192, H=7168, I=2048,
E=256, top-8, Zipf-skewed routing), BF16, all experts on one GPU -- the
configuration the tensor-peak target is quoted on.  Inputs are seeded
synthetic tensors resident in HBM; the expert weights alone (22.5 GB) are far
larger than L2, so consecutive steps cannot hit in L2.

Prints ONE JSON line (rank 0).  ``value`` is whole-job algorithmic TFLOP/s
(18*R*H*I FLOPs per step, R = T*k, padding excluded); ``e2e`` is the same
metric with each step's inputs copied from pinned host memory and its results
(out, dX, ds) read back inside the timed region.  ``--impl reference`` times
the float64 CPU oracle (the reference arm of this build) on a bounded sample,
the same slice the line's ``cpu_baseline`` leg repeats.  After the headline
workload the default run also times the two MXFP8 workloads (mid-sized with
Zipf routing, Kimi-K2-shaped) and the library's dense GEMM core, under
``secondary`` and ``dense_core``; ``value``, ``config`` and ``dtype`` stay
the headline's.  Tensor-core fractions are of the measured burst peak (the
timed region is well under a second); the sustained figure is beside it.
Under torchrun every rank runs an independent replica (the layer does not
shard across GPUs); timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE layer fwd+bwd TFLOP/s"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_PHASES = ("fwd_gemm", "bwd_da", "bwd_dx", "bwd_wg13", "bwd_wg2")
HBM_PHASES = ("fwd_combine", "bwd_dx_combine", "fwd_sort", "bwd_sort")
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args_from(argv):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mok", "reference"], default="mok")
    ap.add_argument("--workload", default="dsv3")
    ap.add_argument("--minibatch-rows", type=int, default=0)
    ap.add_argument("--ring-slots", type=int, default=0)
    ap.add_argument("--overlap-sms", type=int, default=0,
                    help="SMs of the short experts' ring launch beside the pair launch (0: the library's rule)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    # MXFP8 workloads timed after the headline one (default run only)
    ap.add_argument("--no-secondary", action="store_true")
    ap.add_argument("--secondary-steps", type=int, default=10)
    # diagnostic: the library's MOK_DEBUG_* bits (alternative launch paths)
    ap.add_argument("--debug-flags", type=int, default=0)
    # bounded-memory backward (forward context of ring_slots minibatches, GEMM1 recomputed)
    ap.add_argument("--replay", action="store_true")
    ap.add_argument("--fused", action="store_true",
                    help="schedule + forward as one launch (mok_forward_fused; MXFP8: after the "
                         "routing-independent quantisation and scale tiling)")
    return ap.parse_args(argv)


def parse_args():
    return parse_args_from(None)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def tensor_peaks(peaks, peaks_src, prec):
    """(peak, sustained peak, note) for the GEMM phases.  ``peak`` is the burst
    figure: the timed region is well under a second of 10-30 ms steps, not
    the seconds-long power-capped loop the sustained figure comes from."""
    burst = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    note = f"{peaks_src} bf16 burst (cuBLAS 8192^3); sustained beside it"
    if prec == "mxfp8":
        # E4M3 contraction: no measured fp8 peak on this machine; the measured bf16
        # figures x the nominal dense fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)
        return 2.0 * burst, 2.0 * sus, f"{peaks_src} bf16 burst x 2 (nominal dense fp8 / bf16 ratio)"
    return burst, sus, note


def flops_per_step(shape):
    # GEMM FLOPs: forward 6*R*H*I (W1|W3: 4RHI, W2: 2RHI), backward 12*R*H*I
    return 18.0 * shape.R * shape.H * shape.I


def phase_flops(shape):
    RHI = float(shape.R) * shape.H * shape.I
    return {"fwd_gemm": 6 * RHI, "bwd_da": 2 * RHI, "bwd_dx": 4 * RHI, "bwd_wg13": 4 * RHI, "bwd_wg2": 2 * RHI,
            "fwd_fused": 6 * RHI}


def phase_min_bytes(shape, prec, active_experts):
    """Compulsory DRAM bytes of each GEMM phase: the weights of the experts
    with routed rows once, each activation operand once, each output once
    (MXFP8 operands at 1 + 1/32 bytes per element, bf16 at 2)."""
    R, T, H, I, E = shape.R, shape.T, shape.H, shape.I, shape.E
    ob = 1.0 + 1.0 / 32 if prec == "mxfp8" else 2.0
    w = active_experts * H * I * ob  # one expert weight matrix
    return {
        "fwd_gemm": 3 * w + T * H * ob + R * 2 * I * 2 + R * H * 2,           # W1|W3|W2, x; ctx [h|u], y
        "bwd_da": w + T * H * ob + R * 2 * I * 2 + R * 2 * I * 2 + R * I * 2
                  + (R * 2 * I * ob if prec == "mxfp8" else 0),               # W2, dout, ctx; dh|du, s*a
        "bwd_dx": 2 * w + R * 2 * I * ob + R * H * 2,                          # W1|W3, dh|du; dX parts
        "bwd_wg13": R * H * ob + R * 2 * I * ob + E * 2 * H * I * 2,           # x, dh|du; dW1, dW3
        "bwd_wg2": R * I * ob + R * H * ob + E * I * H * 2,                    # s*a, dout; dW2
    }


def phase_bytes(shape):
    # algorithmic bytes per run of the HBM-bound kernels (bf16 = 2 B, f32 = 4 B)
    R, T, H = shape.R, shape.T, shape.H
    return {"fwd_combine": R * H * 2 + R * 4 + T * H * 2, "bwd_dx_combine": R * H * 2 + T * H * 2,
            # token-sorted copy of x: R rows read and written (padding rows excluded)
            "fwd_sort": 2 * R * H * 2}


def sort_copies_per_step(args, prec):
    """Token-sorted copies the BF16 backward really makes per step: dout
    always; x only when the forward left no sorted copy of x (the fused
    forward, the gathered ring).  The launch for x runs either way and
    returns at once when the copy is there."""
    if prec != "bf16":
        return None
    f = args.debug_flags
    # a gathered ring (bit 6) runs only where the ring is one single-CTA
    # launch (bit 5, or replay); the serial two-launch debug path (bit 1)
    # gathers too
    gathered = bool(f & 64) and (bool(f & 32) or args.replay)
    forward_sorts_x = not args.fused and not gathered and not (f & 2)
    return 1 if forward_sorts_x else 2


# ---------------------------------------------------------------- clocks
class ClockSampler:
    def __init__(self, device_index):
        self.proc = None
        self.device_index = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.device_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(",") for r in out.strip().splitlines() if r.strip()]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [c.strip() for c in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- traffic
def recorded_traffic(phase, workload):
    """DRAM bytes per launch of a kernel from the committed ncu summary, if it
    was taken on the current source of the kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    src = os.path.join(ROOT, "mixture_experts_layer_side_gb300", "csrc", "gemm.cu")
    try:
        text = open(path).read()
        digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    except OSError:
        return None
    for line in text.splitlines():
        cells = [c.strip() for c in line.strip().strip("|").split("|")]
        if len(cells) >= 4 and cells[0] == phase and cells[1] == workload and cells[3] == digest:
            try:
                return float(cells[2])
            except ValueError:
                return None
    return None


# ---------------------------------------------------------------- oracle
class OracleSample:
    """A bounded sample of the workload for the float64 oracle: same H and I,
    ``tokens`` tokens routed top-``k`` over ``experts`` experts.  Inputs are
    drawn once; ``run()`` times one forward + backward."""

    def __init__(self, shape, tokens, experts, k, seed):
        from mixture_experts_layer_side_gb300.inputs import Shape, make_inputs
        sub = Shape(tokens, shape.H, shape.I, experts, k)
        inp = make_inputs(sub, "uniform", seed=seed, device="cpu")
        self.a = {n: (v.double().numpy() if v.is_floating_point() else v.numpy()) for n, v in inp.items()}
        self.flops = flops_per_step(sub)
        self.desc = (f"float64 NumPy oracle, forward + backward of a {tokens}-token, {experts}-expert, top-{k} "
                     f"slice at H={shape.H}, I={shape.I} (R={tokens * k} routed rows); throughput = the "
                     f"slice's 18*R*H*I FLOPs / its time")

    def run(self):
        from oracle import moe
        a = self.a
        t0 = time.perf_counter()
        moe.forward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"])
        moe.backward(a["x"], a["idx"], a["s"], a["W1"], a["W3"], a["W2"], a["dout"])
        return time.perf_counter() - t0


def host_cores():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count() or 1


# ---------------------------------------------------------------- arms
def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            # host-only ranks (the CPU tests of this launch logic)
            dist.init_process_group("gloo")
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, value):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tflops(world, flops_per_rank_step, ms_per_step):
    """Whole-job throughput: every rank runs the same step on its own replica,
    and ``ms_per_step`` is the slowest rank's time."""
    return world * flops_per_rank_step / (ms_per_step / 1e3) / 1e12


# The one bounded slice of the workload both CPU legs time (the reference arm
# per step, the cpu_baseline leg repeated for about ten seconds): same H and I,
# 256 tokens routed top-2 over 4 experts.
ORACLE_SLICE = dict(tokens=256, experts=4, k=2, seed=11)


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from mixture_experts_layer_side_gb300.inputs import WORKLOADS
    shape, routing, prec = WORKLOADS[args.workload]
    sample = OracleSample(shape, **ORACLE_SLICE)
    flops, desc = sample.flops, sample.desc
    for _ in range(args.warmup):
        sample.run()
    total = sum(sample.run() for _ in range(args.steps))
    value = flops * args.steps / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(args, shape, routing, prec),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(args, shape, routing, prec, layer=None):
    cfg = {"workload": f"{args.workload}: MoE layer T={shape.T} H={shape.H} I={shape.I} E={shape.E} "
                       f"top-{shape.k}, {routing} routing, {prec}",
           "T": shape.T, "H": shape.H, "I": shape.I, "E": shape.E, "k": shape.k, "routing": routing,
           "precision": prec, "global_batch": shape.T, "parallelism": "replicas",
           "l2": "inputs larger than L2 (expert weights alone exceed 129 MB)"}
    if layer is not None:
        cfg["minibatch_rows"] = args.minibatch_rows or "two-wave default"
        cfg["ring_slots"] = args.ring_slots or 4
        if args.debug_flags:
            cfg["debug_flags"] = args.debug_flags
        cfg["overlap_sms"] = args.overlap_sms or "library rule"
        cfg["replay"] = bool(args.replay)
        cfg["fused_forward"] = bool(args.fused)
        cfg["ctx_bytes"] = int(layer.ctx.numel())
    return cfg


def secondary_workload(name, steps, dev, peaks, peaks_src):
    """One more workload timed in the same run (not the headline): its step
    time, per-phase TFLOP/s and fraction of the tensor peak of its precision,
    and the clocks seen while it ran."""
    import torch

    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import WORKLOADS, load_stats, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer

    shape, routing, prec = WORKLOADS[name]
    inp = make_inputs(shape, routing, seed=2000, device=dev)
    layer = MoKLayer(shape, precision=prec, device=dev)
    grads = layer.alloc_grads()
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=dev)
    if prec == "mxfp8":
        wq = layer.quantize_weights(inp["W1"], inp["W3"], inp["W2"])
        w_fwd, w_bwd = wq["fwd"], wq["bwd"]
    else:
        w_fwd = w_bwd = (inp["W1"], inp["W3"], inp["W2"])

    def step():
        layer.build_schedule(inp["idx"])
        layer.forward(inp["x"], inp["s"], *w_fwd, out=out)
        layer.backward(inp["x"], inp["s"], *w_bwd, inp["dout"], grads=grads)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    layer.check()
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(dev.index)
    sampler.start()
    time.sleep(0.3)
    _lib.mok_trace_enable(True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    phases = _lib.mok_trace_read()
    _lib.mok_trace_enable(False)
    layer.check()
    ms = e0.elapsed_time(e1) / steps
    peak, peak_sus, note = tensor_peaks(peaks, peaks_src, prec)
    pf = phase_flops(shape)
    per = {}
    for n, (tot, runs) in phases.items():
        if runs:
            per[n] = {"ms": tot / runs}
            if n in pf:
                tf = pf[n] / (per[n]["ms"] / 1e3) / 1e12
                per[n].update(tflops=tf, frac_of_peak=tf / peak)
    fwd_ms = sum(per.get(n, {"ms": 0})["ms"] for n in ("schedule", "quant", "fwd_gemm", "fwd_combine"))
    stats = load_stats(inp["idx"], shape.E)
    res = {"workload": f"{name}: T={shape.T} H={shape.H} I={shape.I} E={shape.E} top-{shape.k}, {routing} "
                       f"routing, {prec}",
           "dtype": prec, "steps": steps, "ms_per_step": ms, "value": flops_per_step(shape) / (ms / 1e3) / 1e12,
           "unit": UNIT, "tokens_per_s": shape.T / (ms / 1e3), "peak": peak, "peak_source": note,
           "frac_of_peak": flops_per_step(shape) / (ms / 1e3) / 1e12 / peak,
           "phases": per, "clocks": clocks, "load": stats}
    if "quant" in per:
        res["note"] = ("the quant phase (activation quantisation, both passes) is summed into the forward's "
                       f"{fwd_ms:.3f} ms only approximately: it runs in both passes")
    del layer, inp, grads, out
    torch.cuda.empty_cache()
    return res


def dense_core_rates(dev, n=8192, reps=20):
    """The library's tensor-core GEMM on one dense n^3 problem (K-major
    operands), BF16 and MXFP8: the rate its tile pipeline reaches with no
    MoE structure around it (context for the per-phase fractions)."""
    import torch

    from mixture_experts_layer_side_gb300 import _lib
    g = torch.Generator(device=dev).manual_seed(3)
    A = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)
    B = torch.randn((n, n), generator=g, device=dev).to(torch.bfloat16)
    C = torch.empty((n, n), dtype=torch.float32, device=dev)
    scratch = torch.zeros(256 + 2 * n * n // 32, dtype=torch.uint8, device=dev)
    Aq = torch.empty((n, n), dtype=torch.uint8, device=dev)
    Bq = torch.empty((n, n), dtype=torch.uint8, device=dev)
    As = torch.empty((n, n // 32), dtype=torch.uint8, device=dev)
    Bs = torch.empty((n, n // 32), dtype=torch.uint8, device=dev)
    _lib.mok_mxfp8_quantize(A, 1, Aq, As)
    _lib.mok_mxfp8_quantize(B, 1, Bq, Bs)
    runs = {"bf16": lambda: _lib.mok_gemm_bf16(A, 0, B, 0, C, scratch),
            "mxfp8": lambda: _lib.mok_gemm_mxfp8(Aq, As, 0, Bq, Bs, 0, C, scratch)}
    res = {}
    for name, fn in runs.items():
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        res[name] = {"n": n, "ms": ms, "tflops": 2.0 * n ** 3 / (ms / 1e3) / 1e12}
    del A, B, C, scratch, Aq, Bq, As, Bs
    torch.cuda.empty_cache()
    return res


def run_mok(args):
    import torch

    from mixture_experts_layer_side_gb300 import _lib
    from mixture_experts_layer_side_gb300.inputs import WORKLOADS, load_stats, make_inputs
    from mixture_experts_layer_side_gb300.layer import MoKLayer

    world, rank, local = dist_setup(args)
    shape, routing, prec = WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = make_inputs(shape, routing, seed=1000 + rank, device=dev)
    layer = MoKLayer(shape, precision=prec, minibatch_rows=args.minibatch_rows, ring_slots=args.ring_slots,
                     debug_flags=args.debug_flags, replay=args.replay, overlap_sms=args.overlap_sms, device=dev)
    out = torch.empty((shape.T, shape.H), dtype=torch.bfloat16, device=dev)
    grads = layer.alloc_grads()
    stream = torch.cuda.current_stream()
    if prec == "mxfp8":
        # weights are pre-quantised once, outside the step (the pages' ops.mxfp8_quantize)
        wq = layer.quantize_weights(inp["W1"], inp["W3"], inp["W2"])
        w_fwd, w_bwd = wq["fwd"], wq["bwd"]
    else:
        w_fwd = w_bwd = (inp["W1"], inp["W3"], inp["W2"])

    def forward(x, idx, s, o):
        if args.fused:
            layer.forward_fused(idx, x, s, *w_fwd, out=o)
        else:
            layer.build_schedule(idx)
            layer.forward(x, s, *w_fwd, out=o)

    def step(x, idx, s, dout):
        forward(x, idx, s, out)
        layer.backward(x, s, *w_bwd, dout, grads=grads)

    for _ in range(max(args.warmup, 3)):
        step(inp["x"], inp["idx"], inp["s"], inp["dout"])
    torch.cuda.synchronize()
    layer.check()

    # ------------------------------------------------ device-resident timing
    sampler = ClockSampler(dev.index)
    barrier(world)
    torch.cuda.synchronize()
    _lib.mok_trace_enable(True)
    launches0 = _lib.mok_launch_count()
    sampler.start()
    time.sleep(0.3)  # let the sampler take its first sample before the timed region
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step(inp["x"], inp["idx"], inp["s"], inp["dout"])
    ev1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    launches = _lib.mok_launch_count() - launches0
    phases = _lib.mok_trace_read()
    _lib.mok_trace_enable(False)
    layer.check()
    ms = max_over_ranks(world, ev0.elapsed_time(ev1) / args.steps)
    barrier(world)

    fps = flops_per_step(shape)
    value = job_tflops(world, fps, ms)

    # ------------------------------------------------ roofline of the dominant kernel
    peaks, peaks_src = load_peaks()
    pf, pb = phase_flops(shape), phase_bytes(shape)
    per_phase = {n: {"ms": v[0] / max(v[1], 1), "runs": v[1]} for n, v in phases.items() if v[1]}
    dom = max(GEMM_PHASES, key=lambda n: per_phase.get(n, {"ms": 0})["ms"])
    dom_ms = per_phase[dom]["ms"]
    achieved = pf[dom] / (dom_ms / 1e3) / 1e12
    peak, peak_sus, peak_note = tensor_peaks(peaks, peaks_src, prec)
    roofline = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "peak_source": peak_note,
                "peak_sustained": peak_sus, "frac_of_sustained": achieved / peak_sus,
                "traffic": recorded_traffic(dom, args.workload)}
    copies = sort_copies_per_step(args, prec)
    if copies is not None and "bwd_sort" in per_phase:
        # bytes of the copies made, over the time of every launch of the phase
        pb["bwd_sort"] = copies * 2 * shape.R * shape.H * 2 * args.steps / per_phase["bwd_sort"]["runs"]
        per_phase["bwd_sort"]["copies_per_step"] = copies
    for n in per_phase:
        if n in pf:
            per_phase[n]["tflops"] = pf[n] / (per_phase[n]["ms"] / 1e3) / 1e12
            per_phase[n]["frac_of_peak"] = per_phase[n]["tflops"] / peak
        if n in pb:
            gbs = pb[n] / (per_phase[n]["ms"] / 1e3) / 1e9
            per_phase[n]["gbs"] = gbs
            per_phase[n]["frac_of_hbm"] = gbs / float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    # attainable roofline of each GEMM phase: time / max(FLOPs / tensor peak,
    # compulsory bytes / copy bandwidth), with the binding resource named
    stats = load_stats(inp["idx"], shape.E)
    hbm = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    mb = phase_min_bytes(shape, prec, shape.E - stats["empty_experts"])
    for n in GEMM_PHASES:
        if n in per_phase:
            t_flop = pf[n] / (peak * 1e12) * 1e3
            t_byte = mb[n] / (hbm * 1e9) * 1e3
            floor = max(t_flop, t_byte)
            per_phase[n].update(min_bytes=mb[n], floor_ms=floor, bound="tensor" if t_flop >= t_byte else "hbm",
                                attainable_frac=floor / per_phase[n]["ms"])
    sched_share = per_phase.get("schedule", {"ms": 0})["ms"] / ms
    cfg_line = workload_config(args, shape, routing, prec, layer)

    # ------------------------------------------------ router on either side of the layer (not in the metric)
    router = None
    if prec == "bf16":
        from mixture_experts_layer_side_gb300.layer import MoKRouter
        rt = MoKRouter(shape, device=dev)
        g = torch.Generator(device=dev).manual_seed(77)
        Wr = (0.05 * torch.randn((shape.H, shape.E), generator=g, device=dev)).to(torch.bfloat16)
        rds = torch.randn((shape.T, shape.k), generator=g, device=dev)
        ridx, rs = rt.forward(inp["x"], Wr)
        for _ in range(3):
            rt.forward(inp["x"], Wr)
            rt.backward(inp["x"], Wr, ridx, rs, rds)
        torch.cuda.synchronize()
        rt.check()
        _lib.mok_trace_enable(True)
        for _ in range(args.steps):
            rt.forward(inp["x"], Wr)
            rt.backward(inp["x"], Wr, ridx, rs, rds)
        torch.cuda.synchronize()
        rph = _lib.mok_trace_read()
        _lib.mok_trace_enable(False)
        rt.check()
        rf = 2.0 * shape.T * shape.H * shape.E
        router = {}
        for name, fl in (("router_fwd", rf), ("router_bwd", 2 * rf)):
            ms_r = rph[name][0] / max(rph[name][1], 1)
            router[name] = {"ms": ms_r, "tflops": fl / (ms_r / 1e3) / 1e12}
        router["note"] = "logits GEMM + top-k softmax; logit gradient + dWr and dx GEMMs (outside the layer metric)"
        del rt

    # ------------------------------------------------ end to end through the C ABI, host buffers
    e2e = None
    if not args.no_e2e:
        # Every step's inputs come from pinned host memory and its results (out,
        # dX, ds) go back to it.  Two device buffer sets let step i+1's
        # inputs arrive, and step i-1's results leave, on copy streams while
        # step i computes -- what a training loop feeding the layer does.
        host = {n: inp[n].cpu().pin_memory() for n in ("x", "idx", "s", "dout")}
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hdX = torch.empty(grads["dX"].shape, dtype=torch.bfloat16).pin_memory()
        hds = torch.empty(grads["ds"].shape, dtype=torch.float32).pin_memory()
        h2d_st, d2h_st = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        sets = []
        for _ in range(2):
            b = {n: torch.empty_like(inp[n]) for n in host}
            b["out"] = torch.empty_like(out)
            b["grads"] = dict(grads, dX=torch.empty_like(grads["dX"]), ds=torch.empty_like(grads["ds"]))
            b["loaded"], b["computed"], b["drained"] = (torch.cuda.Event() for _ in range(3))
            sets.append(b)

        def load(i):
            b = sets[i % 2]
            with torch.cuda.stream(h2d_st):
                h2d_st.wait_event(b["drained"])  # the set's previous results have left
                for n in host:
                    b[n].copy_(host[n], non_blocking=True)
                b["loaded"].record(h2d_st)

        def e2e_steps(n):
            go = torch.cuda.Event()
            go.record(stream)
            h2d_st.wait_event(go)
            load(0)
            for i in range(n):
                b = sets[i % 2]
                if i + 1 < n:
                    load(i + 1)
                stream.wait_event(b["loaded"])
                forward(b["x"], b["idx"], b["s"], b["out"])
                layer.backward(b["x"], b["s"], *w_bwd, b["dout"], grads=b["grads"])
                b["computed"].record(stream)
                with torch.cuda.stream(d2h_st):
                    d2h_st.wait_event(b["computed"])
                    hout.copy_(b["out"], non_blocking=True)
                    hdX.copy_(b["grads"]["dX"], non_blocking=True)
                    hds.copy_(b["grads"]["ds"], non_blocking=True)
                    b["drained"].record(d2h_st)
            for b in sets:
                stream.wait_event(b["drained"])

        e2e_steps(2)
        torch.cuda.synchronize()
        barrier(world)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e2e_steps(args.steps)
        e1.record(stream)
        torch.cuda.synchronize()
        layer.check()
        ems = max_over_ranks(world, e0.elapsed_time(e1) / args.steps)
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = sum(t.numel() * t.element_size() for t in (hout, hdX, hds))
        e2e = {"value": job_tflops(world, fps, ems), "unit": UNIT, "ms_per_step": ems,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "scope": "activations: x, idx, s, dout copied in and out, dX, ds read back every step; the "
                        "expert weights and their gradients stay resident in HBM (the caller's parameters "
                        "and gradient buffers), as in a training loop"}

    # ------------------------------------------------ MXFP8 and dense-core context (rank 0, one GPU only)
    secondary, dense = None, None
    if rank == 0 and world == 1 and not args.no_secondary and args.workload == "dsv3":
        # free the headline workload's buffers first (about 60 GB)
        layer = inp = grads = out = None
        if not args.no_e2e:
            sets = host = hout = hdX = hds = None
        torch.cuda.empty_cache()
        secondary = [secondary_workload(w, args.secondary_steps, dev, peaks, peaks_src)
                     for w in ("mid_mxfp8_zipf", "kimi_mxfp8")]
        dense = dense_core_rates(dev)

    # ------------------------------------------------ CPU baseline (rank 0, one GPU only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # repeat the slice until about 10 s of CPU work has accumulated (30 s cap)
        sample = OracleSample(shape, **ORACLE_SLICE)
        total, reps = 0.0, 0
        while total < 10.0 and reps < 200:
            total += sample.run()
            reps += 1
        cpu = {"value": sample.flops * reps / total / 1e12, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": f"{sample.desc}; {reps} repetitions", "seconds": total}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": prec, "data": "synthetic (seeded, resident in HBM)",
            "config": cfg_line,
            "tokens_per_s": world * shape.T / (ms / 1e3),
            "gpu_launches": launches,
            "roofline": roofline,
            "phases": per_phase,
            "schedule_share": sched_share,
            "router": router,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clocks,
            "load": stats,
            "secondary": secondary,
            "dense_core": dense,
            "peaks_source": peaks_src,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_mok(args)


if __name__ == "__main__":
    sys.exit(main())
