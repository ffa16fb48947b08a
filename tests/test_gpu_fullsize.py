"""Parity at the full workload sizes, in the launch configuration that
bench.py times: the whole batch runs on the GPU, and the oracle recomputes a
few whole sequences of it (sequences are independent, so their outputs and
input gradients are checked row for row).  Parameter gradients are sums over
all sequences; they are checked on a GPU rerun of the sampled sequences alone
against the oracle on the same sequences.

Workloads (seeded, synthetic; the pages' private long listening histories are
stood in for by their shapes):
  B=32 L=2048 d=512 H=8 d_h=64 forward;  B=8 L=32768 long-history forward
  (repeated low-rank pattern);  B=16 L=8192 training step;  256 varlen
  sequences of 64..16384 rows, d=1024, H=8, d_h=128, training step."""
import numpy as np
import pytest
import torch

import oracle
from generative_retrieval_encoder_gb300 import build, gbla
from generative_retrieval_encoder_gb300 import workloads as W
from gbla_cases import TOL, f64, max_err

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


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


def _ranges(wl, cu, picks):
    if cu is not None:
        return [(cu[b], cu[b + 1]) for b in picks]
    return [(b * wl.L, (b + 1) * wl.L) for b in picks]


def _check_rows(got, ref, tol, what):
    e = max_err(got, ref)
    assert e <= tol, (what, e)


def _oracle_seq(wl, x, P, dy, a, e, backward):
    Pr = {n: f64(t) for n, t in P.items()}
    st, ln = oracle.seqs(1, e - a)
    out = oracle.gbla_forward(f64(x[a:e]), Pr, wl.H, wl.dh, st, ln, 0, wl.eps)
    g = oracle.gbla_backward(f64(x[a:e]), Pr, f64(dy[a:e]), wl.H, wl.dh, st, ln, 0, wl.eps) if backward else None
    return out, g


@pytest.mark.parametrize("name,picks", [("train2k", [0, 31]), ("long32k", [7])])
def test_forward_full_size(name, picks):
    wl = {"train2k": W.FWD_2K, "long32k": W.LONG_32K}[name]
    shape, x, P, dy, cu = _inputs(wl)
    y, _ = gbla.gbla_forward(shape, x, P)
    torch.cuda.synchronize()
    for a, e in _ranges(wl, cu, picks):
        out, _ = _oracle_seq(wl, x, P, dy, a, e, False)
        _check_rows(f64(y[a:e]), out["y"], TOL["bf16"], (name, a, "y"))


@pytest.mark.parametrize("name,picks", [("train8k", [3]), ("varlen", None)])
def test_training_step_full_size(name, picks):
    wl = {"train8k": W.TRAIN_8K, "varlen": W.VARLEN}[name]
    shape, x, P, dy, cu = _inputs(wl)
    if picks is None:  # varlen: a short, a middling and a long sequence
        lens = np.diff(cu)
        order = np.argsort(lens)
        picks = [int(order[len(order) // 10]), int(order[len(order) // 2]), int(order[int(len(order) * 0.7)])]
    y, saved = gbla.gbla_forward(shape, x, P, saved=True)
    g = gbla.gbla_backward(shape, x, P, saved, dy)
    torch.cuda.synchronize()
    tol = TOL["bf16"]
    rows = _ranges(wl, cu, picks)
    for a, e in rows:
        out, og = _oracle_seq(wl, x, P, dy, a, e, True)
        _check_rows(f64(y[a:e]), out["y"], tol, (name, a, "y"))
        _check_rows(f64(g["dx"][a:e]), og["dx"], tol, (name, a, "dx"))
    # parameter gradients: rerun the sampled sequences alone on the GPU
    sub = torch.cat([torch.arange(a, e) for a, e in rows]).cuda()
    lens = [e - a for a, e in rows]
    cu2 = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32).cuda()
    s2 = gbla.make_shape(1, int(sum(lens)), wl.d, wl.H, wl.dh, gate=wl.gate, eps=wl.eps, cu_seqlens=cu2)
    x2, dy2 = x[sub].contiguous(), dy[sub].contiguous()
    y2, saved2 = gbla.gbla_forward(s2, x2, P, saved=True)
    g2 = gbla.gbla_backward(s2, x2, P, saved2, dy2)
    torch.cuda.synchronize()
    Pr = {n: f64(t) for n, t in P.items()}
    st, ln = oracle.seqs(cu_seqlens=cu2.cpu().numpy())
    og = oracle.gbla_backward(f64(x2), Pr, f64(dy2), wl.H, wl.dh, st, ln, 0, wl.eps)
    for n in ("dconv_w", "dconv_b", "dW_q", "dW_k", "dW_v", "dW_r", "dw_g", "db_g", "drms_w"):
        _check_rows(f64(g2[n]), og[n], tol, (name, n))
    # the subset's rows are the same computation as inside the full batch
    off = 0
    for a, e in rows:
        _check_rows(f64(y2[off:off + e - a]), f64(y[a:e]), 1e-2, (name, a, "subset y"))
        off += e - a
