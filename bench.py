"""Throughput of the MXFP8 SwiGLU MLP (fwd + bwd) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

One step = one forward + backward of the whole MLP (quantize x and the
weights, w13 GEMM, fused SwiGLU + dual quantization, w2 GEMM; then the
backward GEMMs, fused SwiGLU backward and both weight gradients) through
the C ABI, inputs resident in HBM.  Prints ONE JSON line (rank 0).

Workloads (seeded synthetic data, shapes of the pages' MXFP8 fused-MLP
workloads): moe_64e (default: 64 fine-grained routed experts, d=7168,
h=2048, 16384 tokens x top-8, the largest configuration on one GPU),
moe_16e (grouped, default recipe) and llama3_8b_ffn (dense, M=8192,
d=4096, h=14336, wgrad_with_hp recipe; also measured, device-timed, as an
extra key of every default run).

Reported beside the device-timed value:
  e2e           the same step through the public API with host buffers:
                x and dout copied in from pinned memory, and out, dx, dw1,
                dw3 and dw2 copied back, every step (the weights stay
                resident on the device: `resident_bytes`).
  roofline      the dominant kernel (the MXFP8 tcgen05 GEMM): algorithmic
                FLOPs of its launches / their CUDA-event durations, measured
                in a per-kernel pass of the same step (the same kernels
                launched one by one with events between them), against the
                measured burst bf16 peak x 2 (each launch is timed alone).
  cpu_baseline  the CPU oracle on a bounded sample of the workload.
  --impl reference runs that oracle sample as the reference arm.
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

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                  "source": "fallback"}
MXFP8_OVER_BF16 = 2.0   # nominal dense fp8 / bf16 tensor ratio (4.5 / 2.25 PFLOP/s)
MXFP8_NOMINAL_TFLOPS = 4500.0   # GB300 dense MXFP8, nominal
L2_BYTES = 129 * 1024 * 1024
# dram__bytes_read.sum + dram__bytes_write.sum of the MXFP8 GEMM launches of
# one step, from one ncu capture, next to the bytes those launches must move
# (operands read once, outputs written once).  `src` is the digest of the
# GEMM sources the capture ran (gemm_source_digest()); when the sources have
# changed since, the figure no longer describes the kernel and is reported
# as null.
MXFP8_GEMM_TRAFFIC = {
    "moe_64e": {"bytes": 25570545920, "algo": 23233806336, "src": "078049afee56878b",
                "note": "ncu capture of the six GEMM launches of one step "
                        "(profiles/gemm_traffic_moe_64e_step.md): 1.10x the algorithmic bytes"},
}


def gemm_source_digest():
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh"):
        with open(os.path.join(ROOT, "block_scaled_mlp_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            out = dict(FALLBACK_PEAKS)
            for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
                if k in d and d[k]:
                    out[k] = float(d[k])
            out["source"] = "measured"
            return out
        except Exception:
            pass
    return dict(FALLBACK_PEAKS)


# ------------------------------------------------------------------ workload


def make_workload(name):
    w = dict(synth.WORKLOADS[name])
    if w["kind"] == "dense":
        inp = synth.dense_mlp_inputs(w["M"], w["d"], w["h"], w["seed"])
        inp["offs"] = None
        w["tokens"] = w["M"]
        w["M_total"] = w["M"]
    else:
        if w["counts"] == "zipf":
            counts = synth.zipf_group_counts(w["E"], w["tokens"], w["s"], w["seed"], w["n_empty"])
        else:
            counts = synth.dirichlet_group_counts(w["E"], w["tokens"], w["alpha"], w["seed"], w["n_empty"])
        inp = synth.grouped_mlp_inputs(counts, w["d"], w["h"], w["seed"])
        w["M_total"] = int(inp["offs"][-1])
        w["counts_arr"] = counts
    w.setdefault("recipe", "rceil")
    w["flops"] = 18.0 * w["tokens"] * w["d"] * w["h"]   # real routed rows, padding excluded
    return w, inp


def _cpulist(text):
    cpus = set()
    for part in text.strip().split(","):
        if part:
            a, _, b = part.partition("-")
            cpus.update(range(int(a), int(b or a) + 1))
    return cpus


def bind_to_gpu_cpus(dev):
    """Run on the host CPUs local to the GPU (its PCI device's local_cpulist),
    so that pinned host buffers are allocated next to the GPU's host link.
    Best effort: returns the CPU list, or None when it cannot be read."""
    try:
        p = torch.cuda.get_device_properties(dev)
        bus = f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        cpus = _cpulist(open(f"/sys/bus/pci/devices/{bus}/local_cpulist").read())
        if not cpus:
            return None
        if len(cpus) < len(os.sched_getaffinity(0)):
            os.sched_setaffinity(0, cpus)
        # reported also when the process already runs on exactly these CPUs
        # (a box with one NUMA node: nothing to bind)
        return f"{min(cpus)}-{max(cpus)}" if max(cpus) - min(cpus) + 1 == len(cpus) else sorted(cpus)
    except Exception:
        return None


def max_over_ranks(ms: float, world: int, dev) -> float:
    """The slowest rank's time (ms per step): every rank contributes its own
    CUDA-event time and all of them get the maximum (replicas: N independent
    copies of the step, whole-job throughput = N x work / this time)."""
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def workload_config(name, w, world):
    """The line's `config`: the workload and its sizes (both arms print it)."""
    d, h = w["d"], w["h"]
    E = 0 if w["kind"] == "dense" else int(w["E"])
    return {"workload": name, "M_total": int(w["M_total"]), "tokens": int(w["tokens"]), "d": d, "h": h,
            "E": E or None, "recipe": w["recipe"], "flops_per_step": w["flops"],
            "l2": f"inputs larger than L2 (weights {3 * d * h * 2 * max(E, 1) / 1e6:.0f} MB bf16)",
            "parallelism": f"replicas x{world}"}


def whole_job_tflops(flops_per_rank: float, world: int, ms_max: float) -> float:
    return flops_per_rank * world / (ms_max * 1e-3) / 1e12


def to_dev(a, dev):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)


# ------------------------------------------------------------------ clocks


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx_, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 6:
                continue
            try:
                sm.append(float(f[0]))
                mx_.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx_) if mx_ else None,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ GPU arm


def run_gpu(args, rank, world, dev):
    import block_scaled_mlp_gb300 as mx

    w, inp = make_workload(args.workload)
    recipe = mx.RECIPE_RCEIL_WGRAD_HP if w["recipe"] == "wgrad_hp" else mx.RECIPE_RCEIL
    t = {k: to_dev(inp[k], dev) for k in ("x", "w1", "w3", "w2", "dout")}
    offs = None if inp["offs"] is None else torch.from_numpy(inp["offs"]).to(dev)
    if rank != 0 or args.no_cpu_baseline:
        inp = None   # the host copies serve only rank 0's CPU-baseline sample
    M, d, h = w["M_total"], w["d"], w["h"]
    E = 0 if offs is None else offs.numel()
    cb, sb = mx.mlp_workspace_size(M, d, h, E, recipe)
    ctx = torch.empty(cb, dtype=torch.uint8, device=dev)
    scratch = torch.empty(sb, dtype=torch.uint8, device=dev)
    out = torch.empty((M, d), dtype=torch.bfloat16, device=dev)
    grads = (torch.empty((M, d), dtype=torch.bfloat16, device=dev), torch.empty_like(t["w1"]),
             torch.empty_like(t["w3"]), torch.empty_like(t["w2"]))
    err = mx.ErrorWord(dev)
    stream = torch.cuda.current_stream(dev)
    L = mx.lib()
    P = mx._ptr

    def step(x, dout, y=out, dx=grads[0]):
        rc = L.mx_mlp_fwd(P(x), P(t["w1"]), P(t["w3"]), P(t["w2"]), M, d, h, P(offs), max(E, 1), 128, recipe,
                          P(ctx), P(scratch), P(y), err.ptr(), mx._stream())
        mx._check(rc)
        rc = L.mx_mlp_bwd(P(ctx), P(dout), P(x), P(t["w1"]), P(t["w3"]), P(t["w2"]), M, d, h, P(offs), max(E, 1),
                          128, recipe, P(scratch), P(dx), P(grads[1]), P(grads[2]), P(grads[3]), err.ptr(),
                          mx._stream())
        mx._check(rc)

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # warmup
    for _ in range(args.warmup):
        step(t["x"], t["dout"])
    torch.cuda.synchronize(dev)
    err.check()

    # ---- device-timed region (inputs resident in HBM; working set > L2)
    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step(t["x"], t["dout"])
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    err.check()
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    value = whole_job_tflops(w["flops"], world, ms_max)
    # own kernels per step: 12 when the w13 GEMM carries SwiGLU and the
    # quantization of y (wgrad_with_hp recipes, and the MXFP8-wgrad recipes
    # at d >= 4096), else 13 (a separate SwiGLU launch)
    launches_per_step = 12 if (w["recipe"] == "wgrad_hp" or d >= 4096) else 13

    # ---- end to end through the public API with host buffers: every step
    # copies its inputs (x, dout) in from pinned host memory and all of its
    # results (out, dx, dw1, dw3, dw2) back; the weights stay resident.
    # Double-buffered like a training input pipeline: step i+1's inputs go
    # up on one copy stream and earlier steps' results come down on another
    # while step i computes; the timed region spans the first upload to the
    # last download.
    host_cpus = bind_to_gpu_cpus(dev)
    hx = t["x"].cpu().pin_memory()
    hd = t["dout"].cpu().pin_memory()
    res_dev = [(out,) + grads, tuple(torch.empty_like(a) for a in (out,) + grads)]
    res_host = [torch.empty(a.shape, dtype=a.dtype).pin_memory() for a in res_dev[0]]
    xin = [(torch.empty_like(t["x"]), torch.empty_like(t["dout"])) for _ in range(2)]
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()
    x_ready, dout_ready, in_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    fwd_done, out_ready, out_free = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def upload(k):
        with torch.cuda.stream(up):
            xin[k][0].copy_(hx, non_blocking=True)
            x_ready[k].record(up)
            xin[k][1].copy_(hd, non_blocking=True)
            dout_ready[k].record(up)

    def step_into(k, r):
        # the forward needs x only; dout may still be on its way up
        x, dout = xin[k]
        stream.wait_event(x_ready[k])
        rc = L.mx_mlp_fwd(P(x), P(t["w1"]), P(t["w3"]), P(t["w2"]), M, d, h, P(offs), max(E, 1), 128, recipe,
                          P(ctx), P(scratch), P(r[0]), err.ptr(), mx._stream())
        mx._check(rc)
        fwd_done[k].record(stream)
        stream.wait_event(dout_ready[k])
        rc = L.mx_mlp_bwd(P(ctx), P(dout), P(x), P(t["w1"]), P(t["w3"]), P(t["w2"]), M, d, h, P(offs), max(E, 1),
                          128, recipe, P(scratch), P(r[1]), P(r[2]), P(r[3]), P(r[4]), err.ptr(), mx._stream())
        mx._check(rc)

    def pipelined(n):
        up.wait_stream(stream)
        down.wait_stream(stream)
        upload(0)
        for i in range(n):
            k = i % 2
            if i + 1 < n:
                if i >= 1:
                    up.wait_event(in_free[(i + 1) % 2])    # step i-1 no longer reads that buffer
                upload((i + 1) % 2)
            if i >= 2:
                stream.wait_event(out_free[k])              # step i-2's results are down
            step_into(k, res_dev[k])
            in_free[k].record(stream)
            out_ready[k].record(stream)
            with torch.cuda.stream(down):
                # out leaves as soon as the forward has written it, the
                # gradients once the backward is done
                down.wait_event(fwd_done[k])
                res_host[0].copy_(res_dev[k][0], non_blocking=True)
                down.wait_event(out_ready[k])
                for hdst, dsrc in zip(res_host[1:], res_dev[k][1:]):
                    hdst.copy_(dsrc, non_blocking=True)
                out_free[k].record(down)
        stream.wait_stream(down)

    # untimed passes of the same pipeline first, so that the timed region
    # does not hold the first copies through freshly allocated pinned buffers
    pipelined(max(2, min(args.warmup, 3)))
    torch.cuda.synchronize(dev)
    err.check()
    barrier()
    torch.cuda.synchronize(dev)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record(stream)
    pipelined(args.steps)
    a1.record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    err.check()
    ms_e2e = max_over_ranks(a0.elapsed_time(a1) / args.steps, world, dev)
    e2e_value = whole_job_tflops(w["flops"], world, ms_e2e)
    h2d = (hx.numel() + hd.numel()) * 2
    d2h = sum(a.numel() * a.element_size() for a in res_host)
    resident = sum(t[k].numel() * 2 for k in ("w1", "w3", "w2"))

    # ---- per-kernel pass: the same kernels launched one by one with events
    kern = kernel_breakdown(mx, w, t, offs, recipe, dev, max(1, min(args.steps, 10)))
    peaks = load_peaks()
    mx_peak = peaks["bf16_tflops"] * MXFP8_OVER_BF16
    g = kern["mx_gemm"]
    achieved = g["flops"] / (g["ms"] * 1e-3) / 1e12
    tr = MXFP8_GEMM_TRAFFIC.get(args.workload)
    digest = gemm_source_digest()
    fresh = tr is not None and tr["src"] == digest
    roofline = {"kernel": "gemm_kernel<MXFP8> (tcgen05 block-scaled)", "bound": "tensor",
                "achieved": round(achieved, 1), "peak": round(mx_peak, 1), "unit": "TFLOP/s",
                "frac": round(achieved / mx_peak, 4),
                "frac_of_nominal": round(achieved / MXFP8_NOMINAL_TFLOPS, 4),
                "traffic": tr["bytes"] if fresh else None,
                "traffic_unit": "DRAM bytes per step over the step's MXFP8 GEMM launches (ncu)",
                "algorithmic_bytes": tr["algo"] if tr else None,
                "traffic_note": (tr["note"] if fresh else
                                 ("no capture of the current GEMM sources" if tr is None or not fresh else None)),
                "peak_source": f"{peaks['source']} bf16 burst {peaks['bf16_tflops']} x {MXFP8_OVER_BF16} "
                               f"(nominal fp8/bf16 ratio; each GEMM launch is timed alone); "
                               f"frac_of_nominal against {MXFP8_NOMINAL_TFLOPS} TFLOP/s dense MXFP8"}
    mem = kern["mem"]
    mem_gbs = mem["bytes"] / (mem["ms"] * 1e-3) / 1e9

    res = {
        "metric": "MXFP8 MLP fwd+bwd TFLOP/s",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "mxfp8-e4m3 (fp32 accumulate)" + (" + bf16 wgrad" if recipe else ""),
        "data": "synthetic (seeded; bf16 N(0,1) activations, N(0,0.02) weights)",
        "config": workload_config(args.workload, w, world),
        "roofline": roofline,
        "quant_swiglu": {"achieved_gbs": round(mem_gbs, 1), "peak_gbs": peaks["hbm_gbs"],
                         "frac": round(mem_gbs / peaks["hbm_gbs"], 4),
                         "kernels": "quantize x/dout (row+col) + fused SwiGLU fwd/bwd",
                         "peak_source": peaks["source"]},
        "kernels_ms_per_step": {k: round(v["ms"], 4) for k, v in kern.items() if isinstance(v, dict)},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "resident_bytes": resident,
                "resident": "w1, w3, w2 (bf16) stay on the device; x, dout up and out, dx, dw1, dw3, dw2 down "
                            "every step", "host_cpus": host_cpus},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk,
    }
    if w["kind"] == "grouped":
        res["dispatch"] = dispatch_measure(mx, w, dev, peaks["hbm_gbs"])
        res["fp8_tensorwise_grouped"] = fp8_grouped_measure(mx, t, offs, dev, peaks, mx_peak)
    if not args.no_extra and rank == 0 and args.workload != "llama3_8b_ffn":
        res["llama3_8b_ffn"] = extra_workload_measure(mx, "llama3_8b_ffn", dev)
    if w["kind"] == "dense" and not args.no_quant_sweep and rank == 0:
        res["linear_lm_head"] = linear_measure(mx, dev, mx_peak)
    if not args.no_quant_sweep and rank == 0:
        res["quant_sweep"] = quant_sweep_measure(mx, dev, peaks["hbm_gbs"])
    return res, w, inp


def extra_workload_measure(mx, name, dev, steps=10, warmup=3):
    """Device-timed fwd+bwd of another workload (inputs resident, CUDA
    events around `steps` steps after `warmup` untimed ones)."""
    w, inp = make_workload(name)
    recipe = mx.RECIPE_RCEIL_WGRAD_HP if w["recipe"] == "wgrad_hp" else mx.RECIPE_RCEIL
    t = {k: to_dev(inp[k], dev) for k in ("x", "w1", "w3", "w2", "dout")}
    offs = None if inp["offs"] is None else torch.from_numpy(inp["offs"]).to(dev)

    def step():
        o_, c_ = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs, recipe=recipe)
        mx.mlp_bwd(c_, t["dout"])
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1) / steps
    del t
    torch.cuda.empty_cache()
    return {"value": round(w["flops"] / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(ms, 4),
            "steps": steps, "warmup": warmup, "recipe": w["recipe"],
            "timing": "device (CUDA events), inputs resident, outputs allocated per step by the binding"}


def _event_ms(fn, iters):
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / iters


def fp8_grouped_measure(mx, t, offs, dev, peaks, fp8_peak, iters=5):
    """The FP8 per-tensor recipe on the workload's forward w1 GEMM shape:
    amax of x and of each expert's w1, the cast of both (rows), and the
    M-grouped GEMM x . w1[e]^T (E4M3 operands, no block scales).  GEMM
    TFLOP/s against the fp8 peak; amax + cast GB/s against HBM."""
    x, w1 = t["x"], t["w1"]
    M, d = x.shape
    E, h = w1.shape[0], w1.shape[1]
    ax, aw = mx.fp8_amax(x), mx.fp8_amax(w1, batch_axes=1)
    xq = mx.fp8_quantize(x, ax, mx.ROW)["q_row"]
    wq = mx.fp8_quantize(w1, aw, mx.ROW)["q_row"]

    def cast():
        mx.fp8_amax(x)
        mx.fp8_amax(w1, batch_axes=1)
        mx.fp8_quantize(x, ax, mx.ROW)
        mx.fp8_quantize(w1, aw, mx.ROW)
    cast_ms = _event_ms(cast, iters)
    gemm_ms = _event_ms(lambda: mx.fp8_grouped_mm(mx.GROUP_M, xq, ax, wq, aw, offs), iters)
    flops = 2.0 * M * h * d                       # padded rows included: the kernel computes them
    cast_bytes = (x.numel() + w1.numel()) * (2 + 2 + 1)   # amax read, cast read, codes written
    tf = flops / (gemm_ms * 1e-3) / 1e12
    gbs = cast_bytes / (cast_ms * 1e-3) / 1e9
    return {"shape": f"[{M}, {d}] x [{E}, {h}, {d}]^T M-grouped", "gemm_ms": round(gemm_ms, 4),
            "gemm_tflops": round(tf, 1), "gemm_frac": round(tf / fp8_peak, 4),
            "amax_cast_ms": round(cast_ms, 4), "amax_cast_gbs": round(gbs, 1),
            "amax_cast_frac": round(gbs / peaks["hbm_gbs"], 4)}


def dispatch_measure(mx, w, dev, hbm_gbs, iters=10):
    """The token-group padding that precedes a grouped step: routing ids of
    the workload's group counts -> padded layout (mx_token_group_pad), token
    rows -> padded activations and padded results -> routed order
    (mx_gather_rows).  HBM-bound; bytes = rows read + rows written."""
    counts, k, d, E = w["counts_arr"], w["topk"], w["d"], w["E"]
    ids = torch.as_tensor(synth.routed_expert_ids(counts, w["seed"] + 100), device=dev)
    R = ids.numel()
    T = R // k
    m_cap = mx.token_group_capacity(R, E)
    x = torch.randn((T, d), device=dev, dtype=torch.float32).to(torch.bfloat16)
    offs, dst, src = mx.token_group_pad(ids, E, m_cap)
    xp = mx.gather_rows(x, src, div=k)
    pad_ms = _event_ms(lambda: mx.token_group_pad(ids, E, m_cap), iters)
    gat_ms = _event_ms(lambda: mx.gather_rows(x, src, div=k), iters)
    unp_ms = _event_ms(lambda: mx.gather_rows(xp, dst, div=1), iters)
    g_bytes = (R + m_cap) * d * 2
    u_bytes = 2 * R * d * 2
    gbs = (g_bytes + u_bytes) / ((gat_ms + unp_ms) * 1e-3) / 1e9
    return {"routed_rows": R, "topk": k, "padded_rows": m_cap, "pad_ms": round(pad_ms, 4),
            "gather_ms": round(gat_ms, 4), "unpad_ms": round(unp_ms, 4), "gather_gbs": round(gbs, 1),
            "frac": round(gbs / hbm_gbs, 4), "bytes": "gather (R + M_cap) d 2, unpad 2 R d 2"}


def quant_sweep_measure(mx, dev, hbm_gbs, iters=5):
    """The quantize sweep (N x N bf16, N(0,1) with 1% outliers x100) by axis:
    algorithmic GB/s of mx_quantize against the HBM peak.  Outputs are
    allocated once; every timed launch follows a write of a 256 MB buffer
    (L2 flushed, so the smaller sizes read from HBM too) and is bracketed by
    its own CUDA events on the launching stream."""
    out = {}
    L, P = mx.lib(), mx._ptr
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for n in (4096, 8192, 16384, 32768):
        x = torch.randn((n, n), device=dev, dtype=torch.float32)
        x = torch.where(torch.rand_like(x) < 0.01, x * 100, x).to(torch.bfloat16)
        q_row = torch.empty((n, n), dtype=torch.uint8, device=dev)
        q_col = torch.empty((n, n), dtype=torch.uint8, device=dev)
        s_row = torch.zeros(mx.mma_scale_bytes(n, n), dtype=torch.uint8, device=dev)
        s_col = torch.zeros(mx.mma_scale_bytes(n, n), dtype=torch.uint8, device=dev)
        for name, ax, per in (("row", mx.ROW, 2 + 1.03125), ("col", mx.COL, 2 + 1.03125),
                              ("both", mx.BOTH, 2 + 2 * 1.03125)):
            qr, sr = (P(q_row), P(s_row)) if ax & mx.ROW else (None, None)
            qc, sc = (P(q_col), P(s_col)) if ax & mx.COL else (None, None)

            def launch():
                mx._check(L.mx_quantize_mode(P(x), n, n, ax, mx.SCALE_MMA, mx.SCALE_RCEIL, qr, sr, qc, sc,
                                             stream.cuda_stream))
            launch()
            times = []
            for _ in range(iters):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                launch()
                e1.record(stream)
                e1.synchronize()
                times.append(e0.elapsed_time(e1))
            ms = sum(times) / len(times)
            gbs = n * n * per / (ms * 1e-3) / 1e9
            out[f"{n}_{name}"] = {"gbs": round(gbs, 1), "frac": round(gbs / hbm_gbs, 4)}
        del x, q_row, q_col, s_row, s_col
        torch.cuda.empty_cache()
    return out


def linear_measure(mx, dev, mx_peak, iters=3):
    """The per-linear MXFP8 path at a Llama-3 lm_head (8192 tokens, 4096 ->
    128256), default recipe: forward + backward TFLOP/s (6 M K N FLOP)."""
    M, K, N = 8192, 4096, 128256
    x = torch.randn((M, K), device=dev).to(torch.bfloat16)
    wt = (torch.randn((N, K), device=dev) * 0.02).to(torch.bfloat16)
    dout = torch.randn((M, N), device=dev).to(torch.bfloat16)
    c, s = mx.ctypes.c_size_t(), mx.ctypes.c_size_t()
    L, P = mx.lib(), mx._ptr
    mx._check(L.mx_linear_workspace_size(M, K, N, mx.RECIPE_RCEIL, mx.ctypes.byref(c), mx.ctypes.byref(s)))
    ctx = torch.empty(c.value, dtype=torch.uint8, device=dev)
    scratch = torch.empty(s.value, dtype=torch.uint8, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    dx, dw = torch.empty_like(x), torch.empty_like(wt)

    def step():
        mx._check(L.mx_linear_fwd(P(x), P(wt), M, K, N, mx.RECIPE_RCEIL, P(ctx), P(scratch), P(out), None,
                                  mx._stream()))
        mx._check(L.mx_linear_bwd(P(ctx), P(dout), P(wt), M, K, N, mx.RECIPE_RCEIL, P(scratch), P(dx), P(dw), None,
                                  mx._stream()))
    ms = _event_ms(step, iters)
    tf = 6.0 * M * K * N / (ms * 1e-3) / 1e12
    return {"shape_MKN": [M, K, N], "ms_fwd_bwd": round(ms, 3), "tflops": round(tf, 1),
            "frac": round(tf / mx_peak, 4), "recipe": "rceil"}


def kernel_breakdown(mx, w, t, offs, recipe, dev, steps):
    """Per-kernel CUDA-event timing of the step's kernels, launched one by
    one through the per-op entry points (bit-identical to the composite)."""
    hp = recipe == mx.RECIPE_RCEIL_WGRAD_HP
    d, h, M = w["d"], w["h"], w["M_total"]
    grouped = offs is not None
    W1, W3, W2 = (t[k] if grouped else t[k][None] for k in ("w1", "w3", "w2"))
    E = W1.shape[0]
    # weights quantized once, packed as the composite packs them (untimed)
    w13q, w13s, w13qc, w13sc, w2q, w2s, w2qc, w2sc = ([] for _ in range(8))
    for e in range(E):
        a, b, c = mx.quantize(W1[e].contiguous()), mx.quantize(W3[e].contiguous()), mx.quantize(W2[e].contiguous())
        w13q.append(torch.cat([a["q_row"], b["q_row"]]))
        w13s.append(torch.cat([a["s_row"], b["s_row"]]))
        w13qc.append(torch.cat([a["q_col"], b["q_col"]], 1))
        w13sc.append(torch.cat([a["s_col"].view(d // 128, h // 128, 512), b["s_col"].view(d // 128, h // 128, 512)],
                               1).reshape(-1))
        w2q.append(c["q_row"]); w2s.append(c["s_row"]); w2qc.append(c["q_col"]); w2sc.append(c["s_col"])
    pk = [torch.stack(v) if grouped else v[0] for v in (w13q, w13s, w13qc, w13sc, w2q, w2s, w2qc, w2sc)]
    w13q, w13s, w13qc, w13sc, w2q, w2s, w2qc, w2sc = pk
    x, dout = t["x"], t["dout"]
    x_t = x.t().contiguous() if hp else None
    dout_t = dout.t().contiguous() if hp else None
    tokens = w["tokens"]
    f = {"mx_gemm": 0.0, "bf16_gemm": 0.0}
    acc = {"mx_gemm": [0.0, 0.0], "bf16_gemm": [0.0, 0.0], "mem": [0.0, 0.0]}
    stream = torch.cuda.current_stream(dev)

    def timed(kind, flops_or_bytes, fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        r = fn()
        b.record(stream)
        pending.append((kind, flops_or_bytes, a, b))
        return r

    def mm(aq, as_, bq, bs):
        return mx.grouped_mm(mx.GROUP_M, aq, as_, bq, bs, offs) if grouped else mx.scaled_mm(aq, as_, bq, bs)

    def wg(aq, as_, bq, bs):
        return mx.grouped_mm(mx.GROUP_K, aq, as_, bq, bs, offs) if grouped else mx.scaled_mm(aq, as_, bq, bs)

    mdh = 2.0 * tokens * d * h
    for it in range(steps + 1):
        pending = []
        xq = timed("mem", M * d * (2 + 2 * 1.03125), lambda: mx.quantize(x, mx.BOTH))
        h13 = timed("mx_gemm", 2 * mdh, lambda: mm(xq["q_row"], xq["s_row"], w13q, w13s))
        y = timed("mem", M * h * (4 + (1.03125 if hp else 2.0625)),
                  lambda: mx.swiglu_quant(h13, mx.ROW if hp else mx.BOTH))
        timed("mx_gemm", mdh, lambda: mm(y["q_row"], y["s_row"], w2q, w2s))
        dq = timed("mem", M * d * (2 + 2 * 1.03125), lambda: mx.quantize(dout, mx.BOTH))
        dy = timed("mx_gemm", mdh, lambda: mm(dq["q_row"], dq["s_row"], w2qc, w2sc))
        if hp:
            dh = timed("mem", M * h * (6 + 2 * 1.03125 + 6), lambda: mx.swiglu_quant_bwd(dy, h13, mx.ROW,
                                                                                       bf16_transposed=True))
            timed("bf16_gemm", mdh, lambda: mx.bf16_wgrad(dout_t, dh["y_t"], offs))
            timed("bf16_gemm", 2 * mdh, lambda: mx.bf16_wgrad(dh["dh13_t"], x_t, offs))
        else:
            dh = timed("mem", M * h * (6 + 4 * 1.03125), lambda: mx.swiglu_quant_bwd(dy, h13, mx.BOTH))
            timed("mx_gemm", mdh, lambda: wg(dq["q_col"], dq["s_col"], y["q_col"], y["s_col"]))
            timed("mx_gemm", 2 * mdh, lambda: wg(dh["q_col"], dh["s_col"], xq["q_col"], xq["s_col"]))
        timed("mx_gemm", 2 * mdh, lambda: mm(dh["q_row"], dh["s_row"], w13qc, w13sc))
        torch.cuda.synchronize(dev)
        if it == 0:
            continue  # warm-up pass
        for kind, work, a, b in pending:
            acc[kind][0] += work
            acc[kind][1] += a.elapsed_time(b)
    out = {"steps": steps}
    for k, (work, ms) in acc.items():
        if ms > 0:
            out[k] = {"flops" if k != "mem" else "bytes": work / steps, "ms": ms / steps}
    out["mx_gemm"]["flops"] = acc["mx_gemm"][0] / steps
    out["mem"]["bytes"] = acc["mem"][0] / steps
    return out


# ------------------------------------------------------------------ CPU oracle


def oracle_sample(w, inp, tokens, hidden, keep=False):
    """A bounded sample of the workload for the CPU oracle: the first
    `tokens` routed rows and the first `hidden` hidden units (all of d).
    With keep=True also returns the sample's inputs and the oracle's
    results."""
    from oracle import mx_oracle as o
    x = inp["x"][:tokens]
    dout = inp["dout"][:tokens]
    if inp["offs"] is None:
        w1, w3, w2 = inp["w1"][:hidden], inp["w3"][:hidden], inp["w2"][:, :hidden]
        offs = None
    else:
        # the sample stays inside the first non-empty group
        first = int(np.nonzero(np.diff(np.concatenate([[0], inp["offs"]])))[0][0])
        start = 0 if first == 0 else int(inp["offs"][first - 1])
        x = inp["x"][start:start + tokens]
        dout = inp["dout"][start:start + tokens]
        w1, w3 = inp["w1"][first, :hidden], inp["w3"][first, :hidden]
        w2 = inp["w2"][first][:, :hidden]
        offs = None
    rec = "wgrad_hp" if w["recipe"] == "wgrad_hp" else "rceil"
    t0 = time.perf_counter()
    f = o.mlp_fwd(x, w1, w3, w2, offs=offs, recipe=rec)
    b = o.mlp_bwd(x, w1, w3, w2, dout, offs=offs, recipe=rec, fwd=f)
    dt = time.perf_counter() - t0
    flops = 18.0 * tokens * w["d"] * hidden
    if keep:
        return flops, dt, dict(x=x, w1=w1, w3=w3, w2=w2, dout=dout, fwd=f, bwd=b)
    return flops, dt


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args, world=1):
    w, inp = make_workload(args.workload)
    tokens, hidden = 64, 512
    for _ in range(args.warmup):
        oracle_sample(w, inp, tokens, hidden)
    tot_f, tot_t = 0.0, 0.0
    for _ in range(args.steps):
        fl, dt = oracle_sample(w, inp, tokens, hidden)
        tot_f += fl
        tot_t += dt
    value = tot_f / tot_t / 1e12
    sample = f"{tokens} tokens x {hidden} hidden units (all d={w['d']}) of {args.workload}, fwd+bwd"
    return {
        "impl": "reference",
        "metric": "MXFP8 MLP fwd+bwd TFLOP/s",
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64 (exact MXFP8 oracle)",
        "data": "synthetic",
        "config": workload_config(args.workload, w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline(args, w, inp, dev=None):
    """The CPU oracle on a bounded sample of the workload, timed; with a
    device, also the numerics of the GPU path on the same sample (SQNR
    against the oracle's per-GEMM MXFP8 chain and against the unquantized
    fp64 MLP, as the fused-MLP page's test suite tracks them)."""
    tokens, hidden = (256, 1024) if w["kind"] == "dense" else (256, 512)
    fl, dt, smp = oracle_sample(w, inp, tokens, hidden, keep=True)
    res = {"value": fl / dt / 1e12, "unit": "TFLOP/s", "cores": cpu_cores(), "kind": "oracle",
           "seconds": round(dt, 2),
           "sample": f"{tokens} tokens x {hidden} hidden units (all d={w['d']}) of {args.workload}, fwd+bwd"}
    if dev is not None:
        res["numerics"] = sample_numerics(w, smp, dev)
    return res


def sample_numerics(w, smp, dev):
    """SQNR (dB) of out, dx, dw1, dw3, dw2 from the GPU path on the oracle
    sample, against the oracle's per-GEMM MXFP8 chain (fp64 before each
    bf16 rounding) and against the textbook fp64 SwiGLU MLP (no
    quantization), plus the normwise error against the chain."""
    import block_scaled_mlp_gb300 as mx
    from oracle import mx_oracle as o
    recipe = mx.RECIPE_RCEIL_WGRAD_HP if w["recipe"] == "wgrad_hp" else mx.RECIPE_RCEIL
    t = {k: to_dev(smp[k], dev) for k in ("x", "w1", "w3", "w2", "dout")}
    out, ctx = mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], recipe=recipe)
    dx, dw1, dw3, dw2 = mx.mlp_bwd(ctx, t["dout"])
    torch.cuda.synchronize(dev)
    f, b = smp["fwd"], smp["bwd"]
    h = smp["w1"].shape[0]
    X, W1, W3, W2, D = (o.bf16_to_f64(smp[k]) for k in ("x", "w1", "w3", "w2", "dout"))
    g, u = X @ W1.T, X @ W3.T
    sg = 1.0 / (1.0 + np.exp(-g))
    y = g * sg * u
    dy = D @ W2
    dg, du = dy * u * sg * (1.0 + g * (1.0 - sg)), dy * g * sg
    plain = {"out": y @ W2.T, "dx": dg @ W1 + du @ W3, "dw1": dg.T @ X, "dw3": du.T @ X, "dw2": D.T @ y}
    chain = {"out": f["out_f"], "dx": b["dx_f"], "dw1": b["dw13_f"][:h], "dw3": b["dw13_f"][h:],
             "dw2": b["dw2_f"]}
    got = {"out": out, "dx": dx, "dw1": dw1, "dw3": dw3, "dw2": dw2}

    def sqnr(a, ref):
        den = float(np.sum((a - ref) ** 2))
        return None if den == 0.0 else round(10.0 * np.log10(float(np.sum(ref ** 2)) / den), 2)
    r = {"sqnr_vs_mxfp8_chain_db": {}, "sqnr_vs_unquantized_db": {}, "normwise_vs_chain": {}}
    for k, v in got.items():
        a = o.bf16_to_f64(v.cpu().view(torch.int16).numpy().view(np.uint16))
        r["sqnr_vs_mxfp8_chain_db"][k] = sqnr(a, chain[k])
        r["sqnr_vs_unquantized_db"][k] = sqnr(a, plain[k])
        r["normwise_vs_chain"][k] = float(f"{o.normwise_rel_err(a, chain[k]):.3e}")
    return r


# ------------------------------------------------------------------ profiling cases


def run_profile_case(args):
    """One kernel on a small case (a few hundred MB on the device, larger
    than L2), launched --iters times: the command the committed ncu
    summaries were captured with."""
    import block_scaled_mlp_gb300 as mx
    dev = torch.device("cuda", 0)
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    c = args.profile_case
    M = 8192

    def rnd(*shape, std=1.0):
        return (torch.randn(shape, generator=g, device=dev) * std).to(torch.bfloat16)

    if c in ("quant", "quant_row", "quant_col"):
        x = rnd(M, 8192)
        ax = {"quant": mx.BOTH, "quant_row": mx.ROW, "quant_col": mx.COL}[c]
        fn = lambda: mx.quantize(x, ax)
        work, unit = M * 8192 * (2 + (2 if ax == mx.BOTH else 1) * 1.03125), "B"
    elif c in ("swiglu_fwd", "swiglu_fwd_row"):
        h13 = rnd(M, 2 * 8192, std=1.3)
        ax = mx.ROW if c.endswith("row") else mx.BOTH
        fn = lambda: mx.swiglu_quant(h13, ax)
        work, unit = M * 8192 * (4 + (1.03125 if ax == mx.ROW else 2.0625)), "B"
    elif c in ("swiglu_bwd", "swiglu_bwd_hp"):
        h13, dy = rnd(M, 2 * 8192, std=1.3), rnd(M, 8192)
        if c == "swiglu_bwd":
            fn = lambda: mx.swiglu_quant_bwd(dy, h13, mx.BOTH)
            work = M * 8192 * (6 + 4 * 1.03125)
        else:
            fn = lambda: mx.swiglu_quant_bwd(dy, h13, mx.ROW, bf16_transposed=True)
            work = M * 8192 * (6 + 2 * 1.03125 + 6)
        unit = "B"
    elif c == "dispatch":   # MoE 64E routing: 16384 tokens x top-8 over 64 experts, d = 7168
        E, k, T, d = 64, 8, 16384, 7168
        ids = torch.as_tensor(synth.topk_expert_ids(T, E, k, 17), device=dev)
        x = rnd(T, d)
        m_cap = mx.token_group_capacity(T * k, E)

        def fn():
            offs, dst, src = mx.token_group_pad(ids, E, m_cap)
            mx.gather_rows(x, src, div=k)
        work, unit = (T * k + m_cap) * d * 2, "B"
    elif c == "gemm_group_k":  # MoE 16E dW13: [E=16] x [2h=16384, d=5120] over 33536 padded routed rows
        w = synth.WORKLOADS["moe_16e"]
        counts = synth.zipf_group_counts(w["E"], w["tokens"], w["s"], w["seed"], w["n_empty"])
        offs = torch.as_tensor(synth.offsets_from_counts(synth.pad_counts(counts)), device=dev)
        Mt, N, K = int(offs[-1]), 2 * w["h"], w["d"]
        codes = lambda *sh: torch.randint(0, 126, sh, generator=g, device=dev, dtype=torch.uint8)
        aq, bq = codes(N, Mt), codes(K, Mt)
        as_ = torch.full((mx.mma_scale_bytes(N, Mt),), 127, dtype=torch.uint8, device=dev)
        bs = torch.full((mx.mma_scale_bytes(K, Mt),), 120, dtype=torch.uint8, device=dev)
        fn = lambda: mx.grouped_mm(mx.GROUP_K, aq, as_, bq, bs, offs)
        work, unit = 2.0 * Mt * N * K, "FLOP"
    elif c in ("gemm_group_m_fp8", "gemm_group_m_mx"):
        # MoE 64E forward w13 GEMM: [M_total = 139264 padded rows, d = 7168] x
        # [64 experts, 2h = 4096, 7168], FP8 per-tensor or MXFP8 operands
        w = synth.WORKLOADS["moe_64e"]
        counts = synth.dirichlet_group_counts(w["E"], w["tokens"], w["alpha"], w["seed"], w["n_empty"])
        offs = torch.as_tensor(synth.offsets_from_counts(synth.pad_counts(counts)), device=dev)
        Mt, N, K, E = int(offs[-1]), 2 * w["h"], w["d"], w["E"]
        codes = lambda *sh: torch.randint(0, 126, sh, generator=g, device=dev, dtype=torch.uint8)
        aq, bq = codes(Mt, K), codes(E, N, K)
        if c == "gemm_group_m_fp8":
            aa = torch.full((1,), 448.0, device=dev)
            ab = torch.full((E,), 448.0, device=dev)
            fn = lambda: mx.fp8_grouped_mm(mx.GROUP_M, aq, aa, bq, ab, offs)
        else:
            as_ = torch.full((mx.mma_scale_bytes(Mt, K),), 127, dtype=torch.uint8, device=dev)
            bs = torch.full((E * mx.mma_scale_bytes(N, K),), 120, dtype=torch.uint8, device=dev)
            fn = lambda: mx.grouped_mm(mx.GROUP_M, aq, as_, bq, bs, offs)
        work, unit = 2.0 * Mt * N * K, "FLOP"
    elif c == "moe64_gemms":
        # the six MXFP8 GEMMs of a MoE 64E step, one after another (random
        # codes, uniform scales), each timed on its own: prints one line each
        w = synth.WORKLOADS["moe_64e"]
        counts = synth.dirichlet_group_counts(w["E"], w["tokens"], w["alpha"], w["seed"], w["n_empty"])
        offs = torch.as_tensor(synth.offsets_from_counts(synth.pad_counts(counts)), device=dev)
        Mt, d, h, E = int(offs[-1]), w["d"], w["h"], w["E"]
        codes = lambda *sh: torch.randint(0, 126, sh, generator=g, device=dev, dtype=torch.uint8)
        sc = lambda rows, cols, v: torch.full((mx.mma_scale_bytes(rows, cols),), v, dtype=torch.uint8, device=dev)
        shapes = [("w13", "M", 2 * h, d), ("w2", "M", d, h), ("dy", "M", h, d), ("dx", "M", d, 2 * h),
                  ("dw2", "K", d, h), ("dw13", "K", 2 * h, d)]
        for name, mode, N, K in shapes:
            if mode == "M":
                aq, bq = codes(Mt, K), codes(E, N, K)
                as_, bs = sc(Mt, K, 127), torch.cat([sc(N, K, 120)] * E)
                fn = lambda: mx.grouped_mm(mx.GROUP_M, aq, as_, bq, bs, offs)
            else:
                aq, bq = codes(N, Mt), codes(K, Mt)
                as_, bs = sc(N, Mt, 127), sc(K, Mt, 120)
                fn = lambda: mx.grouped_mm(mx.GROUP_K, aq, as_, bq, bs, offs)
            fn()
            torch.cuda.synchronize()
            ms = _event_ms(fn, args.iters)
            print(json.dumps({"case": f"moe64_{name}", "ms": round(ms, 4),
                              "rate": round(2.0 * Mt * N * K / (ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s"}))
            del aq, bq, as_, bs
        return
    elif c == "moe64_fwd":   # MoE 64E forward through mx_mlp_fwd (default recipe)
        w, inp = make_workload("moe_64e")
        t = {k: to_dev(inp[k], dev) for k in ("x", "w1", "w3", "w2")}
        offs = torch.from_numpy(inp["offs"]).to(dev)
        fn = lambda: mx.mlp_fwd(t["x"], t["w1"], t["w3"], t["w2"], offs=offs, recipe=mx.RECIPE_RCEIL)
        work, unit = w["flops"] / 3.0, "FLOP"
    elif c == "mlp_fwd_dense":   # default-recipe forward, M=8192, d=4096, h=8192: the fused w13 GEMM
        d, h = 4096, 8192        # (h13 + rowwise and columnwise MXFP8 y) is its first gemm_kernel launch
        x, w1, w3, w2 = rnd(M, d), rnd(h, d, std=0.02), rnd(h, d, std=0.02), rnd(d, h, std=0.02)
        fn = lambda: mx.mlp_fwd(x, w1, w3, w2, recipe=mx.RECIPE_RCEIL)
        work, unit = 6.0 * M * d * h, "FLOP"
    elif c in ("gemm_mx", "gemm_bf16", "gemm_mx_cublas"):
        N, K = 8192, 4096
        if c == "gemm_mx":
            a, b = mx.quantize(rnd(M, K), mx.ROW), mx.quantize(rnd(N, K, std=0.02), mx.ROW)
            fn = lambda: mx.scaled_mm(a["q_row"], a["s_row"], b["q_row"], b["s_row"])
        elif c == "gemm_mx_cublas":   # the library MXFP8 GEMM on the same operands, for comparison only
            a, b = mx.quantize(rnd(M, K), mx.ROW), mx.quantize(rnd(N, K, std=0.02), mx.ROW)
            A, B = a["q_row"].view(torch.float8_e4m3fn), b["q_row"].view(torch.float8_e4m3fn)
            sa, sb = a["s_row"].view(torch.float8_e8m0fnu), b["s_row"].view(torch.float8_e8m0fnu)
            fn = lambda: torch._scaled_mm(A, B.t(), sa, sb, out_dtype=torch.bfloat16)
        else:
            at, bt = rnd(N, M), rnd(K, M, std=0.02)   # bf16 wgrad: [N, tokens] x [K, tokens]
            fn = lambda: mx.bf16_wgrad(at, bt)
        work, unit = 2.0 * M * N * K, "FLOP"
    else:
        raise SystemExit(f"unknown case {c}")
    for _ in range(2):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.iters
    rate = work / (ms * 1e-3) / (1e9 if unit == "B" else 1e12)
    print(json.dumps({"case": c, "ms": round(ms, 4), "rate": round(rate, 1),
                      "unit": "GB/s" if unit == "B" else "TFLOP/s"}))


# ------------------------------------------------------------------ main


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="moe_64e", choices=sorted(k for k in synth.WORKLOADS if k != "tiny_dense"))
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-quant-sweep", action="store_true", help="skip the quantize-sweep GB/s object")
    ap.add_argument("--no-extra", action="store_true", help="skip the extra llama3_8b_ffn measurement")
    ap.add_argument("--profile-case", default=None,
                    choices=["quant", "quant_row", "quant_col", "swiglu_fwd", "swiglu_fwd_row", "swiglu_bwd",
                             "swiglu_bwd_hp", "gemm_mx", "gemm_bf16", "gemm_group_k", "dispatch",
                             "mlp_fwd_dense", "gemm_mx_cublas", "gemm_group_m_fp8", "gemm_group_m_mx", "moe64_gemms", "moe64_fwd"])
    ap.add_argument("--iters", type=int, default=3)
    args = ap.parse_args()
    if args.profile_case:
        run_profile_case(args)
        return
    args.warmup = max(args.warmup, 3) if args.impl == "native" else args.warmup

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, world)))
        return

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    res, w, inp = run_gpu(args, rank, world, dev)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(args, w, inp, dev)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))


if __name__ == "__main__":
    main()
