#!/usr/bin/env python
"""Benchmark: grouped GEMM TFLOP/s for one MoE expert layer, fwd + dgrad + wgrad.

Workload (default): the DeepSeek-V4-Flash-shaped BF16 MoE layer -- hidden 4096,
256 routed experts, top-6 of softmax over seeded logits for 4096 tokens
(M = 24576 rows), FC1 4096 -> 2x2048 with SwiGLU fused, FC2 2048 -> 4096,
weights ~ N(0, 0.02).  One step = the six grouped-GEMM launches of
precision_grouped_gemm_gb300.layer (fc1 fwd+SwiGLU, fc2 fwd, fc2 dgrad+SwiGLU
backward, fc2 wgrad, fc1 dgrad, fc1 wgrad).

Prints one JSON line.  `value` counts 2*M*N*K flops per GEMM (padding rows the
MMA wastes are not counted) over all ranks divided by the slowest rank's time.
`extra` adds the same measurement for the MXFP8 DeepSeek-shaped, GPT-OSS-shaped
BF16 and Zipf-routed MXFP4 layers (--workload makes any of them the main line),
the DeepSeek-shaped FP8 tensor-wise (current scaling) layer, the fp32 main_grad
accumulation and the single-GPU MoE permute / combine.
--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload instead (the only other code path this file runs).
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from precision_grouped_gemm_gb300 import workloads as wl  # noqa: E402

METRIC = "grouped GEMM TFLOP/s fwd+dgrad+wgrad, % of GB300 dense BF16/MXFP8 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="pgg", choices=["pgg", "reference"])
    p.add_argument("--workload", default=wl.DSV4_BF16.name, choices=sorted(wl.WORKLOADS))
    p.add_argument("--e2e-steps", type=int, default=4)
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-extra", action="store_true", help="skip the other workloads' summary")
    p.add_argument("--extra-steps", type=int, default=30)
    p.add_argument("--experts-cap", type=int, default=0,
                   help="keep only the first N experts (same per-expert shapes; small profiling case)")
    p.add_argument("--only-extra", default=None, choices=["wgrad_accumulate_fp32", "moe_glue"],
                   help="run only this one of the extra measurements (--extra-steps calls; with "
                        "--experts-cap for the accumulate) and print its JSON: a profiling case")
    return p.parse_args()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        with open(self.path) as f:
            text = f.read()
        os.unlink(self.path)
        return parse_clock_samples(text)


def parse_clock_samples(text: str) -> dict:
    """Summarise `nvidia-smi --query-gpu=<ClockSampler.Q> --format=csv,noheader,nounits` lines:
    median SM clock, max clock, max power, and every throttle reason seen active."""
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = set()
    sm, mx, pw = [], [], []
    for line in text.splitlines():
        p = [x.strip() for x in line.split(",")]
        if len(p) < 9:
            continue
        try:
            sm.append(float(p[1])); mx.append(float(p[2])); pw.append(float(p[3]))
        except ValueError:
            continue
        for n, v in zip(names, p[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------

def layer_flops(lens, w):
    return 18.0 * float(lens.sum()) * w.inter * w.hidden


# ----------------------------------------------------------------------------
# CPU oracle timing (baseline leg and reference arm)
# ----------------------------------------------------------------------------

def _oracle_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [d.get("num_threads") for d in threadpool_info() if d.get("user_api") == "blas"]
        if n and n[0]:
            return int(n[0])
    except Exception:
        pass
    return os.cpu_count() or 1


class OracleSample:
    """The fp64 oracle on whole experts of the workload, one expert per call."""

    def __init__(self, w):
        from oracle import grouped_gemm as og
        self.og = og
        self.w = w
        self.lens, self.row_token = w.group_lens()
        self.off = np.concatenate([[0], np.cumsum(self.lens)])

    def inputs(self, e):
        w, a, b = self.w, int(self.off[e]), int(self.off[e + 1])
        rows = torch.from_numpy(self.row_token[a:b])
        X = wl.gen_bf16(wl.KEY_X, rows, w.hidden, 1.0, w.seed)
        W1 = wl.gen_matrix(wl.KEY_W1, 2 * w.inter, w.hidden, w.w_std, w.seed, row0=e * 2 * w.inter)
        W2 = wl.gen_matrix(wl.KEY_W2, w.hidden, w.inter, w.w_std, w.seed, row0=e * w.hidden)
        dY = wl.gen_matrix(wl.KEY_DY, b - a, w.hidden, 1.0, w.seed, row0=a)
        to_bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
        return [to_bits(t) for t in (X, W1, W2, dY)], b - a

    def run(self, bits, n):
        og = self.og
        X, W1, W2, dY = [og.bf16_to_f64(x) for x in bits]
        W1 = W1.reshape(1, 2 * self.w.inter, self.w.hidden)
        W2 = W2.reshape(1, self.w.hidden, self.w.inter)
        lens = np.array([n], dtype=np.int32)
        A, H = og.grouped_fc1_swiglu(X, W1, lens)
        og.grouped_gemm_fwd(A, W2, lens)
        dH = og.grouped_fc2_dgrad_swiglu_bwd(dY, W2, H, lens)
        og.grouped_gemm_wgrad(A, dY, lens)
        og.grouped_gemm_dgrad(dH, W1, lens)
        og.grouped_gemm_wgrad(X, dH, lens)

    def flops(self, n):
        return 18.0 * n * self.w.inter * self.w.hidden


def cpu_baseline(w, seconds):
    s = OracleSample(w)
    done_flops, t_total, experts = 0.0, 0.0, 0
    for e in range(w.experts):
        if s.lens[e] == 0:
            continue
        bits, n = s.inputs(e)
        t0 = time.perf_counter()
        s.run(bits, n)
        t_total += time.perf_counter() - t0
        done_flops += s.flops(n)
        experts += 1
        if t_total >= seconds:
            break
    return {"value": done_flops / t_total / 1e12, "unit": "TFLOP/s", "cores": _oracle_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle (numpy) on the first {experts} non-empty experts of {w.name} "
                      f"({done_flops / 1e9:.1f} GFLOP of the layer's fwd+dgrad+wgrad, {t_total:.1f} s), "
                      f"one expert per call, inputs decoded from bf16 inside the timed region"}


def run_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    s = OracleSample(w)
    nz = [e for e in range(w.experts) if s.lens[e] > 0]
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    cache = {}

    def step(k):
        e = nz[k % len(nz)]
        if e not in cache:
            cache[e] = s.inputs(e)
        bits, n = cache[e]
        t0 = time.perf_counter()
        s.run(bits, n)
        return time.perf_counter() - t0, s.flops(n)

    for k in range(args.warmup):
        step(k)
    # one expert per step; budget only decides whether that already fits
    tt, ff = 0.0, 0.0
    for k in range(args.steps):
        dt, f = step(args.warmup + k)
        tt += dt
        ff += f
    value = ff / tt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tt / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded counter-based generator; routing by top-k of softmax over generated logits)",
        "config": {"workload": w.name, "parallelism": "replicas" if args.gpus > 1 else "single",
                   "step": "the layer's fwd+dgrad+wgrad on one whole expert per step (bounded sample)",
                   "per_step_budget_s": budget},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": _oracle_threads(), "kind": "oracle",
                         "sample": "one whole expert per step, cycling over the non-empty experts"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# the CUDA path
# ----------------------------------------------------------------------------

def kernel_traffic(workload, name):
    """DRAM bytes per launch from the committed ncu summary, if the sources of the kernel's
    family still match the ones the counters were taken on."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    from precision_grouped_gemm_gb300.build import source_digest
    k = d.get("workloads", {}).get(workload, {}).get(name)
    if k is None:
        return None
    family = k.get("family")
    if family is None or d.get("source_digests", {}).get(family) != source_digest(family):
        return None
    return k.get("dram_bytes_per_launch")


PEAK_RATIO = {"bf16": 1.0, "e4m3": 2.0, "e2m1": 6.0, "fp8": 2.0}  # dense tensor peak vs bf16 (nominal ratios)
ARITH = {"fp8": "e4m3"}  # the operand type a layer format computes in, where the names differ
# library kernels per call where a call launches more than one (none at present: an FP8 tensor
# scale is one kernel after a memset; the memsets around kernels are not counted)
KERNELS_PER_CALL = {}


def setup_workload(w, device, cap=0):
    """Inputs and the step function for workload w.

    Returns (lens, bufs, step, names, work, io, err): step(bufs, between) runs one layer
    step on a buffer set; io(bufs) gives that set's (inputs, outputs) tensor lists; a
    second independent set comes from bufs.clone_empty() (for the pipelined e2e run)."""
    from precision_grouped_gemm_gb300.layer import (FP8_STEP_NAMES, MX_STEP_NAMES, STEP_NAMES, Fp8LayerBuffers,
                                                    MxLayerBuffers, build_layer_inputs, expert_layer_step,
                                                    fp8_layer_step, fp8_layer_work, layer_work, mx_layer_step,
                                                    mx_layer_work)
    lens, _, buf = build_layer_inputs(w, device, cap, allocate=(w.fmt == "bf16"))
    M, G, Hd, I = int(lens.sum()), len(lens), w.hidden, w.inter
    if w.fmt == "bf16":
        work = layer_work(M, G, Hd, I)
        io = lambda b: ([b.X, b.W1, b.W2, b.dY, b.group_lens], [b.Y, b.dX, b.dW1, b.dW2])
        return lens, buf, expert_layer_step, STEP_NAMES, work, io, buf.err
    if w.fmt == "fp8":
        fb = Fp8LayerBuffers.build(buf.X, buf.W1, buf.W2, buf.dY, buf.group_lens, host_lens=lens)
        del buf
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        work = fp8_layer_work(M, G, Hd, I, fb.M_pad)
        io = lambda b: ([b.X, b.dY, b.group_lens, b.W1q, b.W1t, b.s_w1, b.W2q, b.W2t, b.s_w2],
                        [b.bufs["Y"], b.bufs["dX"], b.bufs["dW1"], b.bufs["dW2"]])
        return lens, fb, fp8_layer_step, FP8_STEP_NAMES, work, io, fb.bufs["err"]
    mb = MxLayerBuffers.build(w.fmt, buf.X, buf.W1, buf.W2, buf.dY, buf.group_lens, host_lens=lens)
    del buf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    work = mx_layer_work(w.fmt, M, G, Hd, I, mb.M_pad)
    io = lambda b: ([b.X, b.dY, b.group_lens, *b.W1q, *b.W1t, *b.W2q, *b.W2t],
                    [b.bufs["Y"], b.bufs["dX"], b.bufs["dW1"], b.bufs["dW2"]])
    return lens, mb, mx_layer_step, MX_STEP_NAMES, work, io, mb.bufs["err"]


def measure(w, steps, warmup, device, peaks, cap=0, e2e_steps=0, world=1, sample_clocks=True):
    import precision_grouped_gemm_gb300 as pgg
    lens, bufs, step_fn, names, work, io, err = setup_workload(w, device, cap)
    step = lambda between=None: step_fn(bufs, between)
    ins, outs = io(bufs)
    flops = layer_flops(lens, w)
    warmup = max(3, warmup)
    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    if pgg.read_error(err) != 0:
        raise RuntimeError(f"{w.name}: device error word set during warm-up")
    K = steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(names) + 1)] for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device()) if sample_clocks else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for k in range(K):
        row = ev[k]
        step(lambda i, row=row: row[i].record())
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop() if sampler else None
    ms = reduce_max_time(t0.elapsed_time(t1), world, device)
    if pgg.read_error(err) != 0:
        raise RuntimeError(f"{w.name}: device error word set during the timed region")
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    tc = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]) * PEAK_RATIO[w.fmt]
    per = {}
    for i, name in enumerate(names):
        d = [ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(K)]
        avg = sum(d) / len(d)
        f, b = work[name]
        per[name] = {"ms": avg, "tflops": f / avg / 1e9, "gbs": b / avg / 1e6, "algo_bytes": b, "flops": f}
    dom = max(per, key=lambda n: per[n]["ms"])
    f, b = work[dom]
    bound = "hbm" if b / (hbm * 1e9) >= f / (tc * 1e12) else "tensor"
    if bound == "hbm":
        achieved, peak, unit = per[dom]["gbs"], hbm, "GB/s"
        src = "hbm_gbs"
    else:
        achieved, peak, unit = per[dom]["tflops"], tc, "TFLOP/s"
        src = "bf16_tflops_sustained" + (f" x {PEAK_RATIO[w.fmt]:g} (nominal {w.fmt}/bf16 ratio)"
                                         if w.fmt != "bf16" else "")
    attain = sum(max(work[n][1] / (hbm * 1e9), work[n][0] / (tc * 1e12)) for n in names)
    res = {
        "value": job_value(world, flops, ms, K), "unit": "TFLOP/s", "ms_per_step": ms / K, "steps": K,
        "warmup": warmup, "dtype": ARITH.get(w.fmt, w.fmt), "rows_M": int(lens.sum()), "group_lens_min": int(lens.min()),
        "group_lens_max": int(lens.max()), "groups_under_128": int((lens < 128).sum()),
        "empty_groups": int((lens == 0).sum()),
        "pct_of_dense_peak": flops / (ms / K) / 1e9 / (peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
                                                       * PEAK_RATIO[w.fmt]),
        "pct_of_attainable_roofline": (attain * 1e3) / (ms / K),
        "roofline": {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                     "frac": achieved / peak, "traffic": kernel_traffic(w.name, dom),
                     "peak_source": f"{load_peaks()[1]} ({src})", "algo_bytes_per_launch": b,
                     "flops_per_launch": f},
        "kernels": per, "gpu_launches": sum(KERNELS_PER_CALL.get(n, 1) for n in names) * K, "clocks": clocks,
        "weights_gb": sum(t.numel() * t.element_size() for t in ins[1:3]) / 1e9 if w.fmt == "bf16" else None,
    }
    if e2e_steps:
        res["e2e"] = run_e2e(step_fn, bufs, io, flops, e2e_steps)
    del ins, outs, step, bufs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def reduce_max_time(ms, world, device):
    """The timed region's length as the slowest rank saw it (all ranks get the max)."""
    if world <= 1:
        return ms
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world, flops_per_step, ms_total, steps):
    """Whole-job TFLOP/s: every rank runs its own replica of the step (weak scaling)."""
    return world * flops_per_step / (ms_total / steps) / 1e9


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


EXTRA = [wl.DSV4_MXFP8, wl.GPTOSS_BF16, wl.ZIPF_MXFP4, wl.DSV4_FP8]


def measure_wgrad_accumulate(device, peaks, steps, cap=0):
    """FC1 wgrad of the DeepSeek-shaped layer accumulated into an fp32 main_grad
    [256, 4096, 4096] (the first `cap` experts when cap > 0): algorithmic bytes = X + dH +
    fp32 read + write of main_grad."""
    import precision_grouped_gemm_gb300 as pgg
    from precision_grouped_gemm_gb300.layer import build_layer_inputs
    w = wl.DSV4_BF16
    lens, _, b = build_layer_inputs(w, device, cap, allocate=False)
    M, G, Hd, I = int(lens.sum()), len(lens), w.hidden, w.inter
    del b.W1, b.W2
    dH = wl.gen_matrix(wl.KEY_DH, M, 2 * I, 0.25, w.seed, device=device)
    acc = torch.zeros((G, 2 * I, Hd), dtype=torch.float32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    call = lambda: pgg.grouped_gemm_wgrad_accumulate(b.X, dH, b.group_lens, acc, err=err)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(steps):
        call()
    t1.record()
    torch.cuda.synchronize()
    if pgg.read_error(err) != 0:
        raise RuntimeError("device error word set in the wgrad accumulate run")
    ms = t0.elapsed_time(t1) / steps
    flops = 2.0 * M * 2 * I * Hd
    nbytes = 2.0 * M * Hd + 2.0 * M * 2 * I + 8.0 * G * 2 * I * Hd
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    res = {"call": f"pgg_grouped_gemm_wgrad_accumulate (fc1 shape: dW_f32[{G}, 4096, 4096] += dH_g^T X_g)",
           "ms": ms, "tflops": flops / ms / 1e9, "gbs": nbytes / ms / 1e6,
           "roofline": {"bound": "hbm", "achieved": nbytes / ms / 1e6, "peak": hbm, "unit": "GB/s",
                        "frac": nbytes / ms / 1e6 / hbm, "algo_bytes_per_launch": nbytes,
                        "traffic": None if cap else kernel_traffic("wgrad_accumulate_fp32", "fc1_wgrad_accumulate")}}
    del acc, dH, b
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def measure_moe_glue(device, peaks, steps):
    """The single-GPU MoE glue on the DeepSeek-shaped routing (4096 tokens, top-6 of
    256 experts, hidden 4096): permute, weighted combine and combine backward, each
    timed over `steps` back-to-back calls.  Algorithmic bytes: permute = X read once
    + Xs written + ids/pos; combine = Ys read + out written; backward = dOut + Ys
    read + dYs written."""
    import precision_grouped_gemm_gb300 as pgg
    w = wl.DSV4_BF16
    T, k, E, H = w.tokens, w.topk, w.experts, w.hidden
    ids = torch.from_numpy(w.topk_ids().astype(np.int32)).to(device)
    X = wl.gen_matrix(wl.KEY_X, T, H, 1.0, w.seed, device=device)
    wts = wl.gen_f32(wl.KEY_LOGITS, torch.arange(T, device=device), k, 1.0, w.seed + 7).abs().contiguous()
    Xs, lens, pos = pgg.moe_permute(ids, X, E)
    ws = torch.empty(pgg.moe_permute_workspace_size(T, E) // 4, dtype=torch.int32, device=device)
    dOut = wl.gen_matrix(wl.KEY_DY, T, H, 1.0, w.seed, device=device)
    out = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    dYs, dw = torch.empty_like(Xs), torch.empty((T, k), dtype=torch.float32, device=device)
    err = torch.zeros(1, dtype=torch.int32, device=device)
    R = T * k
    calls = {
        "permute": (lambda: pgg.moe_permute(ids, X, E, Xs, lens, pos, ws, err),
                    2.0 * T * H + 2.0 * R * H + 8.0 * R + 4.0 * E, 4),
        "combine": (lambda: pgg.moe_combine(Xs, pos, wts, out), 2.0 * R * H + 2.0 * T * H + 8.0 * R, 1),
        "combine_bwd": (lambda: pgg.moe_combine_bwd(dOut, Xs, pos, wts, dYs, dw),
                        2.0 * T * H + 4.0 * R * H + 12.0 * R, 1),
    }
    hbm = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    res = {"workload": f"tokens {T}, top-{k} of {E} experts, hidden {H}, bf16 rows, fp32 weights"}
    for name, (call, nbytes, launches) in calls.items():
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record()
        for _ in range(steps):
            call()
        t1.record()
        torch.cuda.synchronize()
        ms = t0.elapsed_time(t1) / steps
        res[name] = {"ms": ms, "launches": launches, "algo_bytes": nbytes, "gbs": nbytes / ms / 1e6,
                     "frac_of_measured_hbm": nbytes / ms / 1e6 / hbm}
    if pgg.read_error(err) != 0:
        raise RuntimeError("device error word set in the MoE glue run")
    del X, Xs, dOut, out, dYs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def run_pgg(args, w):
    import precision_grouped_gemm_gb300 as pgg
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    pgg.init(local)
    peaks, _ = load_peaks()
    if args.only_extra:
        if args.only_extra == "wgrad_accumulate_fp32":
            r = measure_wgrad_accumulate(device, peaks, args.extra_steps, args.experts_cap)
        else:
            r = measure_moe_glue(device, peaks, args.extra_steps)
        if rank == 0:
            print(json.dumps({"only_extra": args.only_extra, **r}), flush=True)
        return
    main = measure(w, args.steps, args.warmup, device, peaks, args.experts_cap,
                   0 if args.no_e2e else args.e2e_steps, world)
    extra = {}
    if not args.no_extra and not args.experts_cap:
        for ew in EXTRA:
            if ew.name != w.name:
                r = measure(ew, args.extra_steps, 3, device, peaks, 0, 0, world, sample_clocks=False)
                extra[ew.name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "dtype", "pct_of_dense_peak",
                                                    "pct_of_attainable_roofline", "roofline", "rows_M",
                                                    "group_lens_min", "group_lens_max", "groups_under_128",
                                                    "empty_groups", "steps")}
                extra[ew.name]["kernels_ms"] = {k: round(v["ms"], 4) for k, v in r["kernels"].items()}
        extra["wgrad_accumulate_fp32"] = measure_wgrad_accumulate(device, peaks, args.extra_steps)
        extra["moe_glue"] = measure_moe_glue(device, peaks, args.extra_steps)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)
    line = {
        "metric": METRIC, "value": main["value"], "unit": "TFLOP/s", "n_gpus": world, "steps": main["steps"],
        "warmup": main["warmup"], "ms_per_step": main["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": ARITH.get(w.fmt, w.fmt),
        "data": "synthetic (seeded counter-based generator; routing by top-k of softmax over generated logits)",
        "config": {"workload": w.name + (f"_first{args.experts_cap}experts" if args.experts_cap else ""),
                   "tokens": w.tokens, "experts": args.experts_cap or w.experts, "top_k": w.topk,
                   "hidden": w.hidden, "intermediate": w.inter, "rows_M": main["rows_M"],
                   "group_lens_min": main["group_lens_min"], "group_lens_max": main["group_lens_max"],
                   "l2": "inputs larger than L2 (all expert weights streamed every step), no flush",
                   "parallelism": "replicas" if world > 1 else "single"},
        "pct_of_dense_bf16_peak": main["pct_of_dense_peak"],
        "pct_of_attainable_roofline": main["pct_of_attainable_roofline"],
        "roofline": main["roofline"], "kernels": main["kernels"], "gpu_launches": main["gpu_launches"],
        "clocks": main["clocks"], "e2e": main.get("e2e"), "cpu_baseline": cpu, "extra": extra,
    }
    # last key: one short line per extra workload, so that every number survives a reader that
    # keeps only the end of the output
    line["extra_summary"] = extra_summary(extra)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def extra_summary(extra: dict) -> str:
    """The extra measurements as one compact string (workload: value, ms/step, % of dense peak,
    % of the attainable roofline, dominant call and its roofline fraction)."""
    parts = []
    for name, r in extra.items():
        if "value" in r:
            rf = r["roofline"]
            parts.append(f"{name}: {r['value']:.1f} TFLOP/s {r['ms_per_step']:.3f} ms "
                         f"{100 * r['pct_of_dense_peak']:.1f}% dense {100 * r['pct_of_attainable_roofline']:.1f}% "
                         f"attainable, {rf['kernel']} {rf['bound']} {100 * rf['frac']:.1f}%")
        elif name == "wgrad_accumulate_fp32":
            parts.append(f"{name}: {r['ms']:.3f} ms {100 * r['roofline']['frac']:.1f}% hbm")
        elif name == "moe_glue":
            parts.append(name + ": " + ", ".join(f"{k} {1e3 * r[k]['ms']:.1f} us {100 * r[k]['frac_of_measured_hbm']:.1f}% hbm"
                                                 for k in ("permute", "combine", "combine_bwd")))
    return "; ".join(parts)


def run_e2e(step_fn, bufs, io, flops, n):
    """The same metric through the public API with host buffers.  Every step copies its
    inputs from pinned host memory to the device, runs the layer's calls and copies its
    results back to pinned host memory, all inside the timed region.  Two device buffer
    sets alternate so that step k's results stream out (D2H stream) while step k+1's
    inputs stream in (H2D stream) and compute (current stream) runs."""
    sets = [bufs, bufs.clone_empty()]
    ins0, outs0 = io(bufs)
    h_in = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins0]
    for h, t in zip(h_in, ins0):
        h.copy_(t)
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs0]
    bi = sum(t.numel() * t.element_size() for t in ins0)
    bo = sum(t.numel() * t.element_size() for t in outs0)
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    E = lambda: torch.cuda.Event()
    done_out = [None, None]  # D2H of a set finished -> its buffers may be overwritten

    def one(k):
        b = sets[k & 1]
        ins, outs = io(b)
        with torch.cuda.stream(s_in):
            if done_out[k & 1] is not None:
                s_in.wait_event(done_out[k & 1])
            for d, h in zip(ins, h_in):
                d.copy_(h, non_blocking=True)
            e_in = E(); e_in.record(s_in)
        comp.wait_event(e_in)
        step_fn(b)
        e_c = E(); e_c.record(comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(e_c)
            for h, d in zip(h_out, outs):
                h.copy_(d, non_blocking=True)
            done_out[k & 1] = E(); done_out[k & 1].record(s_out)

    for k in range(2):
        one(k)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for k in range(n):
        one(k)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1) / n
    del sets[1]
    return {"value": flops / ms / 1e9, "unit": "TFLOP/s", "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            "ms_per_step": ms, "steps": n,
            "overlap": "two device buffer sets; H2D, compute and D2H on three streams"}


def main():
    args = parse_args()
    w = wl.WORKLOADS[args.workload]
    if not w.swiglu:
        raise SystemExit("bench.py times the expert-layer workloads")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_pgg(args, w)


if __name__ == "__main__":
    main()
