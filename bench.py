#!/usr/bin/env python
"""Benchmark of the GBLA layer hot path on GB300.

One step = one pass of the whole hot path over one batch: gbla_forward
(training mode: conv, projections + gate, state reduction + combine, readout
with the RmsNorm gate) followed by gbla_backward (query side, key side,
projection GEMMs, conv backward, parameter-gradient sums).  Inputs are seeded
synthetic tensors of the workload's shape, resident in HBM before timing.

Prints one JSON line (rank 0).  --impl reference times the fp64 CPU oracle on
a bounded sample of the same workload instead.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
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

METRIC = "GBLA tokens/s fwd & fwd+bwd at L=2k–32k; achieved HBM GB/s vs peak"
L2_BYTES = 129 * 2 ** 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes per launch from ncu captures (dram__bytes_read.sum + dram__bytes_write.sum),
# keyed by launch name with its variant, "step[variant]": (bytes, workload name, sha1 of
# the kernel's source file when captured).  A source change since the capture makes the
# figure stale: it is then reported as null.
NCU_TRAFFIC: dict = {
    "projection gemm[tc]": (281015296, "GBLA layer bf16 B=32 L=2048 d=512 H=8 d_h=64", "7a83a7a9d951"),
    "dx~ gemm[tc]": (329495040, "GBLA layer bf16 B=32 L=2048 d=512 H=8 d_h=64", "7a83a7a9d951"),
    "dW gemm[tc]": (347428608, "GBLA layer bf16 B=32 L=2048 d=512 H=8 d_h=64", "7a83a7a9d951"),
    "bwd_q[tc]": (316208896, "GBLA layer bf16 B=32 L=2048 d=512 H=8 d_h=64", "fb0d0c90244c"),
    "readout[tc]": (170566400, "GBLA layer bf16 B=32 L=2048 d=512 H=8 d_h=64", "c281bb0f589d"),
    "bwd_kv[tc]": (231275776, "GBLA layer bf16 B=32 L=2048 d=512 H=8 d_h=64", "f0e90d3dc144"),
}
KERNEL_SOURCE = {"projection gemm[tc]": "gemm_tc.cu", "dx~ gemm[tc]": "gemm_tc.cu", "dW gemm[tc]": "gemm_tc.cu",
                 "reduce[tc]": "reduce_tc.cu", "reduce[mma]": "core_bf16.cu", "readout[tc]": "readout_tc.cu",
                 "bwd_q[tc]": "bwd_q_tc.cu", "bwd_kv[tc]": "bwd_kv_tc.cu", "conv[bulk]": "conv.cu",
                 "conv bwd[bulk]": "conv.cu", "param grads": "layer_misc.cu"}


def source_sha(key: str) -> str | None:
    """The hash of the source file of a launch ("step[variant]"): traffic
    measured on another revision of the kernel does not apply."""
    f = KERNEL_SOURCE.get(key)
    if f is None:
        return None
    p = os.path.join(ROOT, "generative_retrieval_encoder_gb300", "csrc", f)
    return hashlib.sha1(open(p, "rb").read()).hexdigest()[:12]


def workloads():
    from generative_retrieval_encoder_gb300 import workloads as W
    return {"train2k": W.FWD_2K, "long32k": W.LONG_32K, "train8k": W.TRAIN_8K, "varlen": W.VARLEN}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d[k]) for k in FALLBACK_PEAKS if k in d}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def algorithmic(wl, T: int, n_wsplit: int | None = None) -> dict:
    """Algorithmic work of one launch of each kernel, as (bound, amount):
    bytes for HBM-bound kernels, flops for tensor contractions."""
    d, H, dh = wl.d, wl.H, wl.dh
    HD, N1 = H * dh, 4 * H * dh + H
    th = T * H
    return {
        "conv": ("hbm", T * d * 4),                         # x in, x~ out (bf16)
        "projection gemm": ("tensor", 2 * T * d * N1),
        "reduce": ("hbm", th * (4 * dh + 4)),               # k, v bf16 + g fp32
        "readout": ("hbm", th * 6 * dh),                    # q, r in; y out
        "bwd_q": ("hbm", th * 10 * dh),                     # q, r, dy in; dq, dr out
        "bwd_kv": ("hbm", th * (8 * dh + 6)),               # k, v, g in; dk, dv, ds out
        "dx~ gemm": ("tensor", 2 * T * N1 * d),
        "dW gemm": ("tensor", 2 * T * d * N1),
        "conv bwd": ("hbm", T * d * 6),                     # x, dx~ in; dx out (bf16)
    }


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        load = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_inputs(wl, device):
    import torch
    from generative_retrieval_encoder_gb300 import gbla
    dt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    cu = wl.cu_seqlens()
    kw = {}
    if cu is not None:
        kw["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32, device=device)
        shape = gbla.make_shape(1, cu[-1], wl.d, wl.H, wl.dh, dtype=wl.dtype, gate=wl.gate, eps=wl.eps, **kw)
    else:
        shape = gbla.make_shape(wl.B, wl.L, wl.d, wl.H, wl.dh, dtype=wl.dtype, gate=wl.gate, eps=wl.eps)
    x = wl.x().to(dt)
    dy = wl.dy().to(dt)
    P = {n: t.to(dt).to(device) for n, t in wl.params().items()}
    return shape, x, dy, P


def cpu_baseline(wl, budget_s: float = 12.0, max_seqs: int = 64):
    """The oracle, as it stands, on whole sequences of the workload (fwd + bwd)
    until about budget_s of CPU time is spent.  Returns (tokens/s, cores, sample)."""
    import numpy as np
    import oracle
    oracle.build()
    lens = wl.lengths() or [wl.L] * wl.B
    P = {n: t.to(_torch_dtype(wl)).double().numpy() for n, t in wl.params().items()}
    rng = np.random.default_rng(0)
    done, t0, nseq = 0, time.perf_counter(), 0
    gm = 1 if wl.gate == "softmax" else 0
    while nseq < min(max_seqs, len(lens)):
        n = int(lens[nseq])
        x = rng.standard_normal((n, wl.d))
        dy = rng.standard_normal((n, wl.H * wl.dh))
        st, ln = oracle.seqs(1, n)
        oracle.gbla_forward(x, P, wl.H, wl.dh, st, ln, gm, wl.eps)
        oracle.gbla_backward(x, P, dy, wl.H, wl.dh, st, ln, gm, wl.eps)
        done += n
        nseq += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return done / el, oracle.num_threads(), f"{nseq} whole sequence(s) ({done} tokens) of the workload, fwd+bwd", el


def _torch_dtype(wl):
    import torch
    return torch.bfloat16 if wl.dtype == "bf16" else torch.float32


def run_reference(args, wl, rank: int):
    if rank != 0:
        return
    import numpy as np
    import oracle
    oracle.build()
    lens = wl.lengths() or [wl.L] * wl.B
    n = int(lens[0]) if wl.lengths() is None else int(sorted(lens)[len(lens) // 2])
    P = {k: t.to(_torch_dtype(wl)).double().numpy() for k, t in wl.params().items()}
    rng = np.random.default_rng(0)
    x = rng.standard_normal((n, wl.d))
    dy = rng.standard_normal((n, wl.H * wl.dh))
    st, ln = oracle.seqs(1, n)
    gm = 1 if wl.gate == "softmax" else 0
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gbla_forward(x, P, wl.H, wl.dh, st, ln, gm, wl.eps)
        oracle.gbla_backward(x, P, dy, wl.H, wl.dh, st, ln, gm, wl.eps)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * sum(times) / len(times)
    value = n / (ms / 1e3)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "step": "forward+backward", "sample": f"one sequence of {n} tokens"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"one {n}-token sequence of the workload per step, fwd+bwd"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def l_scaling(wl, dev, timed, tokens: int = 262144, steps: int = 3):
    """fwd+bwd and forward tokens/s for L = 2k .. 32k at B L = tokens (the
    long-history recipe: repeated low-rank pattern); flat means linear in L."""
    import torch
    from generative_retrieval_encoder_gb300 import gbla
    from generative_retrieval_encoder_gb300.workloads import Workload
    out = {"tokens": tokens, "fwd_bwd_tokens_per_s": {}, "fwd_tokens_per_s": {}}
    for L in (2048, 4096, 8192, 16384, 32768):
        w = Workload(f"scaling L={L}", tokens // L, L, wl.d, wl.H, wl.dh, pattern=True, seed=1003)
        shape, x_h, dy_h, P = make_inputs(w, dev)
        x, dy = x_h.to(dev), dy_h.to(dev)
        y = torch.empty(tokens, w.H * w.dh, dtype=x.dtype, device=dev)
        saved = torch.empty(gbla.gbla_saved_size(shape), dtype=torch.uint8, device=dev)
        ws_f = gbla.workspace(shape, gbla.GBLA_OP_FORWARD, dev)
        ws_b = gbla.workspace(shape, gbla.GBLA_OP_BACKWARD, dev)
        fwd = lambda: gbla.gbla_forward(shape, x, P, y=y, saved=saved, ws=ws_f)
        step = lambda: (fwd(), gbla.gbla_backward(shape, x, P, saved, dy, ws=ws_b))
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        out["fwd_bwd_tokens_per_s"][L] = tokens / (timed(step, steps) * 1e-3)
        out["fwd_tokens_per_s"][L] = tokens / (timed(fwd, steps) * 1e-3)
        del x, dy, y, saved, ws_f, ws_b
        torch.cuda.empty_cache()
    return out


def sa_vs_gbla(wl, dev, timed, flush, peaks, B: int = 8, steps: int = 3):
    """Single-layer forward latency at batch 8 and L = 2k .. 32k (the pages'
    Table 5 setting): the SA blocks' softmax attention (sa_core_forward, Eq. 1;
    TFLOP/s on 4 B H L^2 d_h flops), the GBLA core (bla_core_forward) and the
    whole GBLA layer forward (gbla_forward, inference: no saved activations),
    with the ratio SA / GBLA layer."""
    import torch
    from generative_retrieval_encoder_gb300 import gbla
    from generative_retrieval_encoder_gb300.workloads import Workload
    out = {"B": B, "H": wl.H, "d_h": wl.dh, "d": wl.d, "by_L": {}}
    for L in (2048, 4096, 8192, 16384, 32768):
        w = Workload(f"latency L={L}", B, L, wl.d, wl.H, wl.dh, pattern=True, seed=1004)
        shape, x_h, _, P = make_inputs(w, dev)
        x = x_h.to(dev)
        T = B * L
        r = torch.Generator().manual_seed(1005)
        q, k, v = (torch.randn(T, w.H * w.dh, generator=r).to(torch.bfloat16).to(dev) for _ in range(3))
        g = (torch.rand(T, w.H, generator=r) * 0.98 + 0.01).to(dev)
        o = torch.empty_like(q)
        y = torch.empty(T, w.H * w.dh, dtype=x.dtype, device=dev)
        ws_s = gbla.workspace(shape, gbla.GBLA_OP_SA_FORWARD, dev)
        ws_c = gbla.workspace(shape, gbla.GBLA_OP_CORE_FORWARD, dev)
        ws_f = gbla.workspace(shape, gbla.GBLA_OP_FORWARD, dev)
        fns = {"sa_ms": lambda: gbla.sa_core_forward(shape, q, k, v, o=o, ws=ws_s),
               "gbla_core_ms": lambda: gbla.bla_core_forward(shape, q, k, v, g, o=o, ws=ws_c),
               "gbla_layer_ms": lambda: gbla.gbla_forward(shape, x, P, y=y, ws=ws_f)}
        e = {}
        for name, fn in fns.items():
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            e[name] = round(timed(fn, steps), 4)
        fl = 4.0 * B * w.H * L * L * w.dh
        e["sa_tflops"] = round(fl / (e["sa_ms"] * 1e-3) / 1e12, 1)
        e["sa_frac_of_bf16"] = round(e["sa_tflops"] / peaks["bf16_tflops_sustained"], 3)
        e["sa_over_gbla_layer"] = round(e["sa_ms"] / e["gbla_layer_ms"], 2)
        out["by_L"][L] = e
        del x, q, k, v, g, o, y, ws_s, ws_c, ws_f
        torch.cuda.empty_cache()
    return out


def profile(fn, flush, reps: int = 3):
    """Per-launch times (library CUDA events on the launching stream) of fn,
    averaged over reps runs: ({step name: ms}, {step name: kernel variant})."""
    from generative_retrieval_encoder_gb300 import gbla
    gbla.gbla_profiling_enable(True)
    gbla.gbla_profiling_read()
    for _ in range(reps):
        flush.fill_(1.0)
        fn()
    rec = gbla.gbla_profiling_read()
    gbla.gbla_profiling_enable(False)
    per, variant = {}, {}
    for n, ms in rec:
        base = n.split("[")[0]
        per.setdefault(base, []).append(ms)
        if "[" in n:
            variant[base] = n[len(base) + 1:-1]
    return {n: sum(v) / reps for n, v in per.items()}, variant


def roof_entry(name, ms, amount, bound, peaks, variant=None):
    """One kernel's line: time, achieved rate on its algorithmic work, fraction of the measured peak."""
    e = {"ms": round(ms, 4)}
    if variant:
        e["variant"] = variant
    if amount is not None:
        ach = amount / (ms * 1e-3) / (1e9 if bound == "hbm" else 1e12)
        e["achieved"] = round(ach, 1)
        e["unit"] = "GB/s" if bound == "hbm" else "TFLOP/s"
        e["frac"] = round(ach / (peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops_sustained"]), 3)
    return e


def other_workloads(dev, timed, flush, peaks, steps: int = 5):
    """fwd+bwd and forward tokens/s of the other workloads (B=8 L=32768 long
    history, B=16 L=8192 training, 256 varlen sequences at d=1024, d_h=128),
    with the top kernels and their roofline fractions."""
    import torch
    from generative_retrieval_encoder_gb300 import gbla
    out = {}
    for name, wl in workloads().items():
        if name == "train2k":
            continue
        shape, x_h, dy_h, P = make_inputs(wl, dev)
        T = gbla.rows(shape)
        x, dy = x_h.to(dev), dy_h.to(dev)
        del x_h, dy_h
        y = torch.empty(T, wl.H * wl.dh, dtype=x.dtype, device=dev)
        saved = torch.empty(gbla.gbla_saved_size(shape), dtype=torch.uint8, device=dev)
        ws_f = gbla.workspace(shape, gbla.GBLA_OP_FORWARD, dev)
        ws_b = gbla.workspace(shape, gbla.GBLA_OP_BACKWARD, dev)
        fwd = lambda: gbla.gbla_forward(shape, x, P, y=y, saved=saved, ws=ws_f)
        step = lambda: (fwd(), gbla.gbla_backward(shape, x, P, saved, dy, ws=ws_b))
        for _ in range(3):
            step()
        torch.cuda.synchronize()
        kern, variant = profile(step, flush, reps=2)
        alg = algorithmic(wl, T)
        tops = sorted(((n, ms) for n, ms in kern.items() if n in alg), key=lambda kv: -kv[1])[:4]
        tokens = wl.valid_tokens()
        ms_step, ms_fwd = timed(step, steps), timed(fwd, steps)
        out[name] = {"workload": wl.name, "tokens": tokens, "ms_per_step": round(ms_step, 3),
                     "fwd_bwd_tokens_per_s": tokens / (ms_step * 1e-3), "fwd_tokens_per_s": tokens / (ms_fwd * 1e-3),
                     "top_kernels": {n: roof_entry(n, ms, alg[n][1], alg[n][0], peaks, variant.get(n)) for n, ms in tops}}
        del x, dy, y, saved, ws_f, ws_b
        torch.cuda.empty_cache()
    return out


def core_lines(wl, dev, timed, flush, peaks, steps: int = 10):
    """The gated core alone (bla_core_forward / bla_core_backward) and the core
    under LION's decay masks (bla_decay_core_forward) on the workload's
    tokens and heads: tokens/s and HBM rate on their algorithmic bytes per
    token-head (core forward 8 d_h + 4: q, k, v, g in, o out; backward
    14 d_h + 8: q, k, v, g, do in, dq, dk, dv, dg out; decay forward
    8 d_h + 8: q, k, v, g, lambda in, o out); and the SA blocks' softmax
    attention (sa_core_forward) with its tensor rate."""
    import torch
    from generative_retrieval_encoder_gb300 import gbla
    B, L, H, dh = wl.B, wl.L, wl.H, wl.dh
    T = B * L
    shape = gbla.make_shape(B, L, H * dh, H, dh)
    r = torch.Generator().manual_seed(1234)
    q, k, v, d_o = (torch.randn(T, H * dh, generator=r).to(torch.bfloat16).to(dev) for _ in range(4))
    g = (torch.rand(T, H, generator=r) * 0.98 + 0.01).to(dev)
    lam = (0.85 + 0.15 * torch.rand(T, H, generator=r)).to(dev)
    o = torch.empty_like(q)
    ws_f = gbla.workspace(shape, gbla.GBLA_OP_CORE_FORWARD, dev)
    ws_b = gbla.workspace(shape, gbla.GBLA_OP_CORE_BACKWARD, dev)
    ws_d = gbla.workspace(shape, gbla.GBLA_OP_DECAY_FORWARD, dev)
    ws_s = gbla.workspace(shape, gbla.GBLA_OP_SA_FORWARD, dev)
    fwd = lambda: gbla.bla_core_forward(shape, q, k, v, g, o=o, ws=ws_f)
    bwd = lambda: gbla.bla_core_backward(shape, q, k, v, g, d_o, ws=ws_b)
    dec = lambda: gbla.bla_decay_core_forward(shape, q, k, v, g, lam, o=o, ws=ws_d)
    sa = lambda: gbla.sa_core_forward(shape, q, k, v, o=o, ws=ws_s)
    for fn in (fwd, bwd, dec, sa):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    th = T * H
    out = {"shape": f"B={B} L={L} H={H} d_h={dh} bf16"}
    for name, fn, per_th in (("core_forward", fwd, 8 * dh + 4), ("core_backward", bwd, 14 * dh + 8),
                             ("decay_core_forward", dec, 8 * dh + 8)):
        ms = timed(fn, steps)
        kern, variant = profile(fn, flush)
        out[name] = {"ms": round(ms, 4), "tokens_per_s": T / (ms * 1e-3),
                     "algorithmic_bytes": th * per_th, "achieved_GBps": round(th * per_th / (ms * 1e-3) / 1e9, 1),
                     "frac": round(th * per_th / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                     "kernels": {n: roof_entry(n, t, None, None, peaks, variant.get(n))
                                 for n, t in sorted(kern.items(), key=lambda kv: -kv[1]) if n != "memset"}}
    ms = timed(sa, steps)  # the SA blocks' softmax attention (Eq. 1): tensor-bound, 4 B H L^2 d_h flops
    fl = 4.0 * B * H * L * L * dh
    out["sa_forward"] = {"ms": round(ms, 4), "tokens_per_s": T / (ms * 1e-3), "tflops": round(fl / (ms * 1e-3) / 1e12, 1),
                         "frac": round(fl / (ms * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"], 3),
                         "peak": "measured (cuBLAS bf16, sustained)"}
    del q, k, v, d_o, g, lam, o, ws_f, ws_b, ws_d, ws_s
    torch.cuda.empty_cache()
    return out


def rank_max(v: float, world: int, device) -> float:
    """The largest v over the ranks: a job's time is that of its slowest rank."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: the units every rank processed (replicas of the
    same per-GPU work) over the slowest rank's time in milliseconds."""
    return units_per_rank * world / (ms * 1e-3)


def run_ours(args, wl, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist
    from generative_retrieval_encoder_gb300 import build as B
    from generative_retrieval_encoder_gb300 import gbla

    B.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    shape, x_h, dy_h, P = make_inputs(wl, dev)
    T = gbla.rows(shape)
    tokens = wl.valid_tokens()
    x = x_h.to(dev)
    dy = dy_h.to(dev)
    y = torch.empty(T, wl.H * wl.dh, dtype=x.dtype, device=dev)
    saved = torch.empty(gbla.gbla_saved_size(shape), dtype=torch.uint8, device=dev)
    ws_f = gbla.workspace(shape, gbla.GBLA_OP_FORWARD, dev)
    ws_b = gbla.workspace(shape, gbla.GBLA_OP_BACKWARD, dev)
    f32 = dict(dtype=torch.float32, device=dev)
    d, H, dh = wl.d, wl.H, wl.dh
    grads = {"dx": torch.empty_like(x), "dconv_w": torch.empty(d, 4, **f32), "dconv_b": torch.empty(d, **f32),
             "dW_q": torch.empty(d, H * dh, **f32), "dW_k": torch.empty(d, H * dh, **f32),
             "dW_v": torch.empty(d, H * dh, **f32), "dW_r": torch.empty(d, H * dh, **f32),
             "dw_g": torch.empty(d, H, **f32), "db_g": torch.empty(H, **f32), "drms_w": torch.empty(dh, **f32)}
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)

    def fwd():
        gbla.gbla_forward(shape, x, P, y=y, saved=saved, ws=ws_f)

    def step():
        fwd()
        gbla.gbla_backward(shape, x, P, saved, dy, ws=ws_b, out=grads)

    def timed(fn, k):
        total = 0.0
        for _ in range(k):
            flush.fill_(1.0)  # evicts L2 between steps (outside the events)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            total += e0.elapsed_time(e1)
        return total / k

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    def max_over_ranks(v):
        return rank_max(v, world, dev)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    # per-launch times (CUDA events on the launching stream, from the library)
    gbla.gbla_profiling_enable(True)
    gbla.gbla_profiling_read()
    prof_steps = 3
    for _ in range(prof_steps):
        flush.fill_(1.0)
        step()
    rec = gbla.gbla_profiling_read()
    gbla.gbla_profiling_enable(False)
    per, variant = {}, {}
    for n, ms in rec:
        base = n.split("[")[0]  # launch names carry the kernel variant that ran, e.g. "bwd_q[tc]"
        per.setdefault(base, []).append(ms)
        if "[" in n:
            variant[base] = n[len(base) + 1:-1]
    launches_per_step = len([n for n, _ in rec if n != "memset"]) // prof_steps
    kern = {n: sum(v) / prof_steps for n, v in per.items()}

    # the timed region: K steps, barrier + synchronize on both sides, max over ranks
    with ClockSampler(local_rank) as clk:
        barrier()
        ms_step = timed(step, args.steps)
        barrier()
    ms_step = max_over_ranks(ms_step)
    barrier()
    ms_fwd = max_over_ranks(timed(fwd, args.steps))

    # end to end through the public API with host buffers: every step copies
    # its inputs (x, dy) host -> device from pinned memory, runs forward +
    # backward and reads its results back: the layer output y, the input
    # gradient dx and the parameter gradients.  As a training loop that
    # prefetches its next batch, the copy of step k + 1's inputs runs on a
    # second stream, into a second pair of input buffers, while step k
    # computes; K steps are timed back to back (their working set, ~0.8 GB,
    # is far larger than L2).
    xp, dyp = x_h.pin_memory(), dy_h.pin_memory()
    host_g = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in grads.items()}
    host_g["y"] = torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
    # step k's outputs go device -> host on a third stream while step k + 1
    # computes into the other of two output sets
    outs = [dict(grads, y=y), {k: torch.empty_like(v) for k, v in dict(grads, y=y).items()}]
    xb, dyb = [x, torch.empty_like(x)], [dy, torch.empty_like(dy)]
    copy_stream = torch.cuda.Stream(device=dev)
    d2h_stream = torch.cuda.Stream(device=dev)

    def e2e_run(k):
        main = torch.cuda.current_stream()
        copied = [torch.cuda.Event(), torch.cuda.Event()]
        freed = [torch.cuda.Event(), torch.cuda.Event()]
        done = [torch.cuda.Event(), torch.cuda.Event()]
        read = [torch.cuda.Event(), torch.cuda.Event()]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def load(b):
            with torch.cuda.stream(copy_stream):
                xb[b].copy_(xp, non_blocking=True)
                dyb[b].copy_(dyp, non_blocking=True)
                copied[b].record(copy_stream)

        e0.record(main)
        copy_stream.wait_stream(main)
        d2h_stream.wait_stream(main)
        load(0)
        for i in range(k):
            c = i % 2
            if i + 1 < k:
                if i >= 1:
                    copy_stream.wait_event(freed[1 - c])  # step i - 1 is done with that pair
                load(1 - c)
            main.wait_event(copied[c])
            if i >= 2:
                main.wait_event(read[c])  # step i - 2's outputs have left this output set
            o = outs[c]
            gbla.gbla_forward(shape, xb[c], P, y=o["y"], saved=saved, ws=ws_f)
            gbla.gbla_backward(shape, xb[c], P, saved, dyb[c], ws=ws_b, out=o)
            freed[c].record(main)
            done[c].record(main)
            d2h_stream.wait_event(done[c])
            with torch.cuda.stream(d2h_stream):
                for n, v in host_g.items():
                    v.copy_(o[n], non_blocking=True)
                read[c].record(d2h_stream)
        main.wait_stream(d2h_stream)
        e1.record(main)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / k

    e2e_run(2)
    barrier()
    ms_e2e = max_over_ranks(e2e_run(max(3, args.steps)))
    h2d = x.numel() * x.element_size() + dy.numel() * dy.element_size()
    d2h = sum(v.numel() * v.element_size() for v in host_g.values())

    # linearity in L: the same number of tokens (B L = 262144) at L = 2k .. 32k
    scaling = l_scaling(wl, dev, timed) if args.scaling else None
    peaks, peak_src = load_peaks()
    extra = other_workloads(dev, timed, flush, peaks) if args.scaling and wl.name == workloads()["train2k"].name else None
    core = core_lines(wl, dev, timed, flush, peaks) if wl.dh == 64 and wl.dtype == "bf16" and wl.lengths() is None else None
    sa_lat = sa_vs_gbla(wl, dev, timed, flush, peaks) if args.scaling and wl.name == workloads()["train2k"].name else None

    if rank != 0:
        return
    alg = algorithmic(wl, T)
    if any(variant.get(n) not in (None, "tc") for n in ("readout", "bwd_q", "bwd_kv")) and wl.dh == 64:
        print(f"warning: a d_h = 64 state kernel ran without tcgen05: {variant}", file=sys.stderr)
    dom = max((n for n in kern if n in alg), key=lambda n: kern[n])
    bound, amount = alg[dom]
    achieved = amount / (kern[dom] * 1e-3) / (1e9 if bound == "hbm" else 1e12)
    peak = peaks["hbm_gbs"] if bound == "hbm" else peaks["bf16_tflops_sustained"]
    traffic = None
    dkey = f"{dom}[{variant[dom]}]" if dom in variant else dom
    t = NCU_TRAFFIC.get(dkey)
    if t and t[1] == wl.name and t[2] == source_sha(dkey):
        traffic = t[0]
    roof = {"kernel": dom, "bound": bound, "achieved": achieved, "peak": peak,
            "unit": "GB/s" if bound == "hbm" else "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
            "peak_source": peak_src + (" (HBM copy)" if bound == "hbm" else " (cuBLAS bf16, sustained)"),
            "algorithmic_per_launch": amount, "ms_per_launch": kern[dom]}
    per_kernel = {}
    for n, ms in sorted(kern.items(), key=lambda kv: -kv[1]):
        e = {"ms": round(ms, 4), "share": round(ms / sum(kern.values()), 4)}
        if n in variant:
            e["variant"] = variant[n]
        if n in alg:
            b, a = alg[n]
            e["achieved"] = round(a / (ms * 1e-3) / (1e9 if b == "hbm" else 1e12), 1)
            e["unit"] = "GB/s" if b == "hbm" else "TFLOP/s"
            e["frac"] = round(e["achieved"] / (peaks["hbm_gbs"] if b == "hbm" else peaks["bf16_tflops_sustained"]), 3)
        per_kernel[n] = e
    cpu = None
    if world == 1:
        v, cores, sample, el = cpu_baseline(wl)
        cpu = {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
               "seconds": round(el, 1)}
    line = {"metric": METRIC, "value": job_rate(tokens, world, ms_step), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": {"workload": wl.name, "step": "forward+backward", "tokens_per_gpu": tokens,
                       "l2": "flushed between timed steps (write of 2x L2 outside the events)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "fwd_tokens_per_s": job_rate(tokens, world, ms_fwd), "ms_fwd": ms_fwd,
            "roofline": roof, "kernels": per_kernel, "cpu_baseline": cpu,
            "e2e": {"value": job_rate(tokens, world, ms_e2e), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": ms_e2e,
                    "pipeline": "step k+1's H2D and step k-1's D2H on two more streams under step k's compute"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
            "l_scaling": scaling,
            "other_workloads": extra,
            "cores": core,
            "sa_vs_gbla": sa_lat}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="train2k", choices=sorted(workloads()))
    ap.add_argument("--no-scaling", dest="scaling", action="store_false",
                    help="skip the L = 2k .. 32k linearity sweep")
    args = ap.parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = workloads()[args.workload]
    if args.impl == "reference":
        run_reference(args, wl, rank)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_ours(args, wl, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
