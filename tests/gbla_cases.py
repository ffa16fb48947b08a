"""Helpers shared by the GPU parity tests: seeded inputs (via the workloads
module), the CUDA path through the C-ABI binding, the oracle on the same
values, and the error measures of the tolerance contract:

* fp32 I/O: max |gpu - ref| <= 1e-4 * max |ref scale|
* bf16 I/O (fp32 accumulation): max |gpu - ref| <= 2e-2 * max |ref scale|

where the scale is max |v| for the core output o (the statement of the
tolerance), and max |ref| of the compared tensor for everything else.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from generative_retrieval_encoder_gb300 import gbla
from generative_retrieval_encoder_gb300.workloads import Workload

TOL = {"f32": 1e-4, "bf16": 2e-2}


def tdt(dtype: str) -> torch.dtype:
    return torch.float32 if dtype == "f32" else torch.bfloat16


def dev(t: torch.Tensor, dtype: str) -> torch.Tensor:
    return t.to(tdt(dtype)).cuda().contiguous()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def max_err(gpu, ref, scale=None) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    s = float(np.abs(ref).max()) if scale is None else float(scale)
    return float(np.abs(gpu - ref).max()) / max(s, 1e-30)


def seq_layout(B, L, seq_lens=None, lengths=None):
    """(shape kwargs, oracle (start, len), n_rows) for dense/padded/varlen."""
    if lengths is not None:
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
        st, ln = oracle.seqs(cu_seqlens=cu)
        return {"cu_seqlens": torch.tensor(cu, dtype=torch.int32).cuda()}, (st, ln), int(cu[-1]), (1, int(cu[-1]))
    st, ln = oracle.seqs(B, L, seq_lens=seq_lens)
    kw = {}
    if seq_lens is not None:
        kw["seq_lens"] = torch.tensor(seq_lens, dtype=torch.int32).cuda()
    return kw, (st, ln), B * L, (B, L)


def valid_rows(st, ln, T):
    m = np.zeros(T, dtype=bool)
    for a, n in zip(st, ln):
        m[a:a + n] = True
    return m


def core_case(dtype, B, L, H, dh, seed, seq_lens=None, lengths=None):
    kw, (st, ln), T, (Bs, Ls) = seq_layout(B, L, seq_lens, lengths)
    r = torch.Generator().manual_seed(seed)
    q = torch.randn(T, H * dh, generator=r)
    k = torch.randn(T, H * dh, generator=r)
    v = torch.randn(T, H * dh, generator=r)
    g = torch.rand(T, H, generator=r) * 0.98 + 0.01
    d_o = torch.randn(T, H * dh, generator=r)
    shape = gbla.make_shape(Bs, Ls, 64, H, dh, dtype=dtype, **kw)
    D = {n: dev(t, dtype) for n, t in (("q", q), ("k", k), ("v", v), ("d_o", d_o))}
    D["g"] = g.cuda()
    R = {n: f64(t) for n, t in D.items()}
    return shape, D, R, (st, ln), T


def layer_case(wl: Workload):
    """Device inputs (io dtype) and the exact fp64 values the oracle sees."""
    kw, (st, ln), T, (Bs, Ls) = seq_layout(wl.B, wl.L, wl.seq_lens, wl.lengths())
    shape = gbla.make_shape(Bs, Ls, wl.d, wl.H, wl.dh, dtype=wl.dtype, gate=wl.gate, eps=wl.eps, **kw)
    x = dev(wl.x(), wl.dtype)
    P = {n: dev(t, wl.dtype) for n, t in wl.params().items()}
    dy = dev(wl.dy(), wl.dtype)
    R = {"x": f64(x), "dy": f64(dy), "P": {n: f64(t) for n, t in P.items()}}
    return shape, x, P, dy, R, (st, ln), T


def launch_names(fn) -> list[str]:
    """Runs fn() with the library's per-launch profiler on and returns the
    launch names it recorded, each carrying the kernel variant that ran
    (e.g. "bwd_q[tc]": tcgen05; "bwd_q[mma]": the mma.sync fallback)."""
    gbla.gbla_profiling_enable(True)
    gbla.gbla_profiling_read()
    try:
        fn()
        return [n for n, _ in gbla.gbla_profiling_read()]
    finally:
        gbla.gbla_profiling_enable(False)


# The steps that run on the 5th-generation tensor cores (tcgen05) in the bf16
# layer at d_h = 64: any fallback to another variant is a regression.
TC_STEPS_DH64 = ("projection gemm", "readout", "bwd_q", "bwd_kv", "dx~ gemm", "dW gemm")
# ... and the state reduction, where the gate holds values (sigmoid gate, core
# API); under the softmax gate it runs the mma.sync kernel (chunk maxima).
TC_STEPS_DH64_SIGMOID = TC_STEPS_DH64 + ("reduce",)
# At d_h = 128: the GEMMs, the readout and both backward steps.
TC_STEPS_DH128 = ("projection gemm", "readout", "bwd_q", "bwd_kv", "dx~ gemm", "dW gemm")


def assert_tc_variants(names, steps=TC_STEPS_DH64):
    ran = {n.split("[")[0]: n for n in names}
    for step in steps:
        assert step in ran, (step, names)
        assert ran[step] == step + "[tc]", (step, ran[step], names)


def oracle_layer(R, wl: Workload, st, ln, backward=False):
    gm = 1 if wl.gate == "softmax" else 0
    out = oracle.gbla_forward(R["x"], R["P"], wl.H, wl.dh, st, ln, gm, wl.eps)
    if backward:
        out["grads"] = oracle.gbla_backward(R["x"], R["P"], R["dy"], wl.H, wl.dh, st, ln, gm, wl.eps)
    return out
