"""Parity of the bla_core entry points (Eq. 5/6, forward and backward) with
the fp64 oracle, through the C ABI, on seeded inputs: dense, padded and
varlen batches, ragged tails, single-token and empty sequences, every
supported d_h, both I/O dtypes; plus determinism and the device-side check
of bad sequence data."""
import numpy as np
import pytest
import torch

import oracle
from generative_retrieval_encoder_gb300 import build, gbla
from gbla_cases import TOL, core_case, f64, launch_names, max_err, valid_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gbla.lib()
    # the tcgen05 kernels wherever they apply, also on the small shapes here
    # (by default the state reduction takes them only from 20 tiles an SM on)
    gbla.gbla_set_kernel_policy(gbla.GBLA_POLICY_TC)
    yield
    gbla.gbla_set_kernel_policy(gbla.GBLA_POLICY_AUTO)


# (dtype, B, L, H, dh, seq_lens, varlen lengths)
CASES = [
    ("f32", 2, 7, 2, 32, None, None),
    ("f32", 3, 300, 2, 4, None, None),
    ("f32", 1, 1, 1, 16, None, None),
    ("f32", 2, 513, 1, 128, None, None),
    ("f32", 3, 200, 2, 64, [200, 1, 77], None),
    ("f32", 1, 0, 2, 32, None, [5, 0, 300, 1, 64]),
    ("bf16", 2, 7, 2, 64, None, None),
    ("bf16", 1, 1, 1, 64, None, None),
    ("bf16", 3, 1000, 2, 64, None, None),
    ("bf16", 2, 513, 2, 32, None, None),
    ("bf16", 2, 777, 1, 128, None, None),
    ("bf16", 3, 300, 2, 64, [300, 1, 157], None),
    ("bf16", 1, 0, 2, 64, None, [5, 0, 700, 1, 64, 129]),
    ("bf16", 1, 0, 1, 128, None, [3, 1500, 0, 31]),
    ("bf16", 1, 0, 4, 32, None, [64] * 9 + [1000]),
]


def _ids(c):
    return f"{c[0]}-B{c[1]}-L{c[2]}-H{c[3]}-dh{c[4]}" + ("-pad" if c[5] else "") + ("-varlen" if c[6] else "")


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_core_forward_matches_oracle(case):
    dtype, B, L, H, dh, sl, lens = case
    shape, D, R, (st, ln), T = core_case(dtype, B, L, H, dh, seed=CASES.index(case), seq_lens=sl, lengths=lens)
    o, den, state = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"], den=True, state=True)
    torch.cuda.synchronize()
    ro, rden, rstate = oracle.core_forward(R["q"], R["k"], R["v"], R["g"], st, ln, H, dh)
    m = valid_rows(st, ln, T)
    tol = TOL[dtype]
    go = f64(o)
    assert np.isfinite(go).all()
    if m.any():
        assert max_err(go[m], ro[m], scale=np.abs(R["v"][m]).max()) <= tol
        assert max_err(f64(den)[m], rden[m]) <= tol
    assert (go[~m] == 0).all() and (f64(den)[~m] == 0).all()
    nz = ln > 0
    if nz.any():
        assert max_err(f64(state)[nz], rstate[nz]) <= tol
    assert (f64(state)[~nz] == 0).all()


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_core_backward_matches_oracle(case):
    dtype, B, L, H, dh, sl, lens = case
    shape, D, R, (st, ln), T = core_case(dtype, B, L, H, dh, seed=CASES.index(case) + 100, seq_lens=sl, lengths=lens)
    dq, dk, dv, dg = gbla.bla_core_backward(shape, D["q"], D["k"], D["v"], D["g"], D["d_o"])
    torch.cuda.synchronize()
    ref = oracle.core_backward(R["q"], R["k"], R["v"], R["g"], R["d_o"], st, ln, H, dh)
    m = valid_rows(st, ln, T)
    tol = TOL[dtype]
    # dq, dk, dg vanish identically for one-token sequences (o_i = v_i there):
    # floor the scale at the gradients' natural size |d_o| |v|.
    floor = 1e-3 * np.abs(R["d_o"]).max() * np.abs(R["v"]).max()
    for name, got, want in zip(("dq", "dk", "dv", "dg"), (dq, dk, dv, dg), ref):
        got = f64(got)
        assert np.isfinite(got).all(), name
        if m.any():
            scale = max(np.abs(want[m]).max(), floor)
            assert max_err(got[m], want[m], scale) <= tol, (name, max_err(got[m], want[m], scale))
        assert (got[~m] == 0).all(), name


@pytest.mark.parametrize("dtype,dh", [("f32", 32), ("bf16", 64), ("bf16", 128)])
def test_core_is_deterministic(dtype, dh):
    shape, D, R, _, _ = core_case(dtype, 2, 3000, 2, dh, seed=5)
    a = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"], den=True, state=True)
    b = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"], den=True, state=True)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    a = gbla.bla_core_backward(shape, D["q"], D["k"], D["v"], D["g"], D["d_o"])
    b = gbla.bla_core_backward(shape, D["q"], D["k"], D["v"], D["g"], D["d_o"])
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_varlen_sequence_alone_equals_inside_batch():
    """A sequence's outputs do not depend on the other sequences of the batch
    (within rounding: the chunking of the state sums depends on the batch)."""
    lens = [100, 2000, 37]
    shape, D, R, (st, ln), T = core_case("bf16", 1, 0, 2, 64, seed=9, lengths=lens)
    o, _, state = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"], state=True)
    a, e = 100, 2100
    s1 = gbla.make_shape(1, e - a, 64, 2, 64)
    o1, _, st1 = gbla.bla_core_forward(s1, *(D[n][a:e].contiguous() for n in ("q", "k", "v", "g")), state=True)
    assert max_err(f64(o)[a:e], f64(o1), scale=np.abs(R["v"]).max()) <= 1e-2
    assert max_err(f64(state)[1], f64(st1)[0]) <= 1e-5


def _status(shape, D):
    ws = gbla.workspace(shape, gbla.GBLA_OP_CORE_FORWARD)
    gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"], ws=ws)
    return gbla.gbla_check_device_status(ws), ws


def test_device_check_flags_bad_cu_seqlens_without_faulting():
    _, D, _, _, _ = core_case("bf16", 1, 10, 1, 64, seed=3)
    for cu in ([0, 5, 3, 10], [0, 5, 9], [1, 5, 10]):
        s = gbla.make_shape(1, 10, 64, 1, 64, cu_seqlens=torch.tensor(cu, dtype=torch.int32).cuda())
        st, _ = _status(s, D)
        assert st == gbla.GBLA_ERR_DEVICE_CHECK, cu
    s = gbla.make_shape(2, 5, 64, 1, 64, seq_lens=torch.tensor([5, 9], dtype=torch.int32).cuda())
    assert _status(s, D)[0] == gbla.GBLA_ERR_DEVICE_CHECK
    s = gbla.make_shape(2, 5, 64, 1, 64, seq_lens=torch.tensor([5, 2], dtype=torch.int32).cuda())
    assert _status(s, D)[0] == gbla.GBLA_OK
    # the context stays usable
    ok = gbla.make_shape(1, 10, 64, 1, 64, cu_seqlens=torch.tensor([0, 4, 10], dtype=torch.int32).cuda())
    assert _status(ok, D)[0] == gbla.GBLA_OK


def test_nan_inputs_propagate_without_crash():
    shape, D, _, _, _ = core_case("bf16", 1, 200, 1, 64, seed=4)
    D["v"][17, 3] = float("nan")
    o, _, _ = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"])
    torch.cuda.synchronize()
    assert torch.isnan(o[:, 3]).all()


# (policy, variant the bf16 core readout runs under it); shapes with a ragged
# tail, a one-token sequence and, at d_h = 128, varlen lengths
READOUT_CASES = [
    ("tc", 64, [700, 1, 300], None),
    ("mma", 64, [700, 1, 300], None),
    ("tc", 128, None, [3, 1500, 0, 31, 129]),
    ("mma", 128, None, [3, 1500, 0, 31, 129]),
]


@pytest.mark.parametrize("case", READOUT_CASES, ids=[f"{c[0]}-dh{c[1]}" for c in READOUT_CASES])
def test_core_forward_readout_variants(case):
    """The core forward's readout on tcgen05 (phi applied to q in shared
    memory) and, under GBLA_POLICY_MMA, on mma.sync: each matches the oracle,
    and the variant that ran is the one asked for."""
    variant, dh, sl, lens = case
    B, L = (3, 700) if sl else (1, 0)
    shape, D, R, (st, ln), T = core_case("bf16", B, L, 2, dh, seed=400 + READOUT_CASES.index(case), seq_lens=sl,
                                         lengths=lens)
    gbla.gbla_set_kernel_policy(gbla.GBLA_POLICY_TC if variant == "tc" else gbla.GBLA_POLICY_MMA)
    try:
        res = {}
        names = launch_names(lambda: res.update(zip(("o", "den", "state"),
                                                     gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"],
                                                                           den=True))))
        torch.cuda.synchronize()
    finally:
        gbla.gbla_set_kernel_policy(gbla.GBLA_POLICY_TC)
    assert f"readout[{variant}]" in names, names
    ro, rden, _ = oracle.core_forward(R["q"], R["k"], R["v"], R["g"], st, ln, 2, dh)
    m = valid_rows(st, ln, T)
    go, gden = f64(res["o"]), f64(res["den"])
    assert max_err(go[m], ro[m], scale=np.abs(R["v"][m]).max()) <= TOL["bf16"]
    assert max_err(gden[m], rden[m]) <= TOL["bf16"]
    assert (go[~m] == 0).all() and (gden[~m] == 0).all()


# (policy, d_h, B, L, seq_lens, varlen lengths) of the bf16 core backward
BACKWARD_VARIANT_CASES = [
    ("tc", 64, 3, 700, [700, 1, 300], None),
    ("mma", 64, 3, 700, [700, 1, 300], None),
    ("tc", 64, 1, 0, None, [5, 0, 1500, 1, 64, 129, 384]),
    ("tc", 128, 1, 0, None, [3, 1500, 0, 31, 129]),
]


@pytest.mark.parametrize("case", BACKWARD_VARIANT_CASES,
                         ids=[f"{c[0]}-dh{c[1]}-" + ("varlen" if c[5] else "pad") for c in BACKWARD_VARIANT_CASES])
def test_core_backward_variants(case):
    """The core backward on tcgen05 (phi applied to q and k in shared memory;
    the query side at d_h = 64, the key side at 64 and 128) and, under
    GBLA_POLICY_MMA, on mma.sync: each matches the oracle, and the kernels
    that ran are the ones asked for."""
    variant, dh, B, L, sl, lens = case
    shape, D, R, (st, ln), T = core_case("bf16", B, L, 2, dh, seed=500 + BACKWARD_VARIANT_CASES.index(case),
                                         seq_lens=sl, lengths=lens)
    gbla.gbla_set_kernel_policy(gbla.GBLA_POLICY_TC if variant == "tc" else gbla.GBLA_POLICY_MMA)
    try:
        res = {}
        names = launch_names(lambda: res.update(zip(("dq", "dk", "dv", "dg"), gbla.bla_core_backward(
            shape, D["q"], D["k"], D["v"], D["g"], D["d_o"]))))
        torch.cuda.synchronize()
    finally:
        gbla.gbla_set_kernel_policy(gbla.GBLA_POLICY_TC)
    assert f"bwd_kv[{variant}]" in names, names
    assert f"bwd_q[{variant if dh == 64 else 'mma'}]" in names, names
    ref = oracle.core_backward(R["q"], R["k"], R["v"], R["g"], R["d_o"], st, ln, 2, dh)
    m = valid_rows(st, ln, T)
    floor = 1e-3 * np.abs(R["d_o"]).max() * np.abs(R["v"]).max()  # one-token sequences: see above
    for name, want in zip(("dq", "dk", "dv", "dg"), ref):
        got = f64(res[name])
        assert np.isfinite(got).all(), name
        if m.any():
            scale = max(np.abs(want[m]).max(), floor)
            assert max_err(got[m], want[m], scale) <= TOL["bf16"], (name, max_err(got[m], want[m], scale))
        assert (got[~m] == 0).all(), name
