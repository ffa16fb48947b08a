"""Parity at the full workload sizes, in the launch configuration that
bench.py times.

* B=32 L=2048 d=512 H=8 d_h=64 (the bench workload) and B=16 L=8192 (the
  training workload): one forward + backward of the whole batch on the GPU,
  compared with the oracle on the whole batch: y and dx on every row, and
  every parameter gradient, whose sums over all 65536 / 131072 rows include
  the dW split over rows and the fixed-order sums that the bench times.
* B=8 L=32768 long-history forward (repeated low-rank pattern): y of all
  eight sequences.
* 256 varlen sequences of 64..16384 rows, d=1024, H=8, d_h=128, training
  step: the oracle recomputes a short, a middling and the longest sequence
  (sequences are independent, so their y and dx are checked row for row); the
  parameter gradients are checked on a GPU rerun of those sequences alone
  against the oracle on the same sequences (the whole batch would take the
  oracle most of an hour).

Every run also checks, from the library's launch names, that the steps with
a tcgen05 kernel for the shape ran it (no silent fallback).

Workloads (seeded, synthetic; the pages' private long listening histories are
stood in for by their shapes)."""
import numpy as np
import pytest
import torch

import oracle
from generative_retrieval_encoder_gb300 import build, gbla
from generative_retrieval_encoder_gb300 import workloads as W
from gbla_cases import TC_STEPS_DH64, TC_STEPS_DH64_SIGMOID, TC_STEPS_DH128, TOL, assert_tc_variants, f64, launch_names, max_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

GRADS = ("dconv_w", "dconv_b", "dW_q", "dW_k", "dW_v", "dW_r", "dw_g", "db_g", "drms_w")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gbla.lib()


def _inputs(wl):
    dt = torch.bfloat16
    cu = wl.cu_seqlens()
    if cu is not None:
        shape = gbla.make_shape(1, cu[-1], wl.d, wl.H, wl.dh, gate=wl.gate, eps=wl.eps,
                                cu_seqlens=torch.tensor(cu, dtype=torch.int32).cuda())
    else:
        shape = gbla.make_shape(wl.B, wl.L, wl.d, wl.H, wl.dh, gate=wl.gate, eps=wl.eps)
    x = wl.x().to(dt).cuda()
    P = {n: t.to(dt).cuda() for n, t in wl.params().items()}
    dy = wl.dy().to(dt).cuda()
    return shape, x, P, dy, cu


def _check(got, ref, tol, what):
    e = max_err(got, ref)
    assert e <= tol, (what, e)


def _gate(wl):
    return 1 if wl.gate == "softmax" else 0


def _run(shape, x, P, dy, backward):
    out = {}

    def fn():
        out["y"], saved = gbla.gbla_forward(shape, x, P, saved=backward or None)
        if backward:
            out["g"] = gbla.gbla_backward(shape, x, P, saved, dy)
        torch.cuda.synchronize()

    return out, launch_names(fn)


@pytest.mark.parametrize("name", ["train2k", "train8k"])
def test_training_step_whole_batch(name):
    wl = {"train2k": W.FWD_2K, "train8k": W.TRAIN_8K}[name]
    shape, x, P, dy, _ = _inputs(wl)
    out, names = _run(shape, x, P, dy, backward=True)
    # the state reduction runs on tcgen05 from 20 256-row tiles an SM on
    # (131072 x 8 / 256 = 4096 tiles), on mma.sync below (train2k: 2048)
    assert_tc_variants(names, TC_STEPS_DH64_SIGMOID if name == "train8k" else TC_STEPS_DH64)
    Pr = {n: f64(t) for n, t in P.items()}
    st, ln = oracle.seqs(wl.B, wl.L)
    xr, dyr = f64(x), f64(dy)
    ref = oracle.gbla_forward(xr, Pr, wl.H, wl.dh, st, ln, _gate(wl), wl.eps)
    tol = TOL["bf16"]
    _check(f64(out["y"]), ref["y"], tol, (name, "y"))
    del ref
    og = oracle.gbla_backward(xr, Pr, dyr, wl.H, wl.dh, st, ln, _gate(wl), wl.eps)
    g = out["g"]
    _check(f64(g["dx"]), og["dx"], tol, (name, "dx"))
    for n in GRADS:
        _check(f64(g[n]), og[n], tol, (name, n))


def test_long_history_forward_all_sequences():
    wl = W.LONG_32K
    shape, x, P, dy, _ = _inputs(wl)
    out, names = _run(shape, x, P, dy, backward=False)
    assert_tc_variants(names, ("projection gemm", "reduce", "readout"))
    Pr = {n: f64(t) for n, t in P.items()}
    st, ln = oracle.seqs(wl.B, wl.L)
    ref = oracle.gbla_forward(f64(x), Pr, wl.H, wl.dh, st, ln, _gate(wl), wl.eps)
    y = f64(out["y"])
    for b in range(wl.B):
        a, e = b * wl.L, (b + 1) * wl.L
        _check(y[a:e], ref["y"][a:e], TOL["bf16"], ("long32k", b, "y"))


def test_varlen_training_step():
    wl = W.VARLEN
    shape, x, P, dy, cu = _inputs(wl)
    lens = np.diff(cu)
    order = np.argsort(lens, kind="stable")
    picks = [int(order[len(order) // 10]), int(order[len(order) // 2]), int(order[-1])]  # ... and the longest
    out, names = _run(shape, x, P, dy, backward=True)
    assert_tc_variants(names, TC_STEPS_DH128)
    y, g = out["y"], out["g"]
    tol = TOL["bf16"]
    Pr = {n: f64(t) for n, t in P.items()}
    rows = [(int(cu[b]), int(cu[b + 1])) for b in picks]
    for a, e in rows:
        st, ln = oracle.seqs(1, e - a)
        ref = oracle.gbla_forward(f64(x[a:e]), Pr, wl.H, wl.dh, st, ln, _gate(wl), wl.eps)
        og = oracle.gbla_backward(f64(x[a:e]), Pr, f64(dy[a:e]), wl.H, wl.dh, st, ln, _gate(wl), wl.eps)
        _check(f64(y[a:e]), ref["y"], tol, ("varlen", a, e, "y"))
        _check(f64(g["dx"][a:e]), og["dx"], tol, ("varlen", a, e, "dx"))
    # parameter gradients: rerun the sampled sequences alone on the GPU
    sub = torch.cat([torch.arange(a, e) for a, e in rows]).cuda()
    sl = [e - a for a, e in rows]
    cu2 = torch.tensor(np.concatenate([[0], np.cumsum(sl)]), dtype=torch.int32).cuda()
    s2 = gbla.make_shape(1, int(sum(sl)), wl.d, wl.H, wl.dh, gate=wl.gate, eps=wl.eps, cu_seqlens=cu2)
    x2, dy2 = x[sub].contiguous(), dy[sub].contiguous()
    out2, _ = _run(s2, x2, P, dy2, backward=True)
    st, ln = oracle.seqs(cu_seqlens=cu2.cpu().numpy())
    og = oracle.gbla_backward(f64(x2), Pr, f64(dy2), wl.H, wl.dh, st, ln, _gate(wl), wl.eps)
    for n in GRADS:
        _check(f64(out2["g"][n]), og[n], tol, ("varlen", n))
    # the subset's rows are the same computation as inside the full batch
    off = 0
    for a, e in rows:
        _check(f64(out2["y"][off:off + e - a]), f64(y[a:e]), 1e-2, ("varlen", a, "subset y"))
        off += e - a
