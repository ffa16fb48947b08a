"""Parity of the core under LION's decay masks (bla_decay_core_forward; "Linear
Attention for Efficient Bidirectional Sequence Modeling", mask construction,
Lion-d / Lion-s; with the gate of Gated Bidirectional Linear Attention, Eq. 5)
with the fp64 oracle's masked definition, through the C ABI: dense, padded and
varlen batches with ragged tails, empty and one-token sequences, chunk
boundaries (128 rows) crossed many times; constant (Lion-d) and per-token
(Lion-s) decays, no decay (equal to the GBLA core) and full decay (o = v).

Tolerance: bf16 I/O with fp32 accumulation, max |gpu - ref| <= 2e-2 max |v|
for o and 2e-2 max |den| for den."""
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


def _lam(kind, T, H, seed):
    r = np.random.default_rng(seed)
    if kind == "lion-d":
        return np.full((T, H), 0.97)
    if kind == "lion-s":
        return r.uniform(0.85, 1.0, (T, H))
    if kind == "none":
        return np.ones((T, H))
    if kind == "strong":
        return r.uniform(0.0, 0.5, (T, H))
    raise ValueError(kind)


# (B, L, H, seq_lens, varlen lengths, decay)
CASES = [
    (2, 300, 2, None, None, "lion-s"),
    (2, 300, 2, None, None, "lion-d"),
    (1, 1, 1, None, None, "lion-s"),
    (3, 700, 2, [700, 1, 257], None, "lion-s"),
    (1, 0, 2, None, [5, 0, 300, 1, 64, 129, 1000], "lion-s"),
    (1, 0, 1, None, [128, 256, 127, 129], "lion-d"),
    (2, 513, 2, None, None, "none"),
    (2, 400, 1, None, None, "strong"),
]


def _ids(c):
    return f"B{c[0]}-L{c[1]}-H{c[2]}" + ("-pad" if c[3] else "") + ("-varlen" if c[4] else "") + f"-{c[5]}"


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_decay_core_matches_oracle(case):
    B, L, H, sl, lens, kind = case
    shape, D, R, (st, ln), T = core_case("bf16", B, L, H, 64, seed=CASES.index(case) + 200, seq_lens=sl, lengths=lens)
    lam = torch.tensor(_lam(kind, T, H, CASES.index(case)), dtype=torch.float32).cuda()
    out = {}
    names = launch_names(lambda: out.update(zip(("o", "den"), gbla.bla_decay_core_forward(
        shape, D["q"], D["k"], D["v"], D["g"], lam, den=True))))
    torch.cuda.synchronize()
    assert [n for n in names if n.startswith("decay")] == ["decay states[mma]", "decay scan", "decay out[mma]"], names
    ro, rden = oracle.decay_core_forward(R["q"], R["k"], R["v"], R["g"], f64(lam), st, ln, H, 64)
    m = valid_rows(st, ln, T)
    go, gden = f64(out["o"]), f64(out["den"])
    assert np.isfinite(go).all() and np.isfinite(gden).all()
    if m.any():
        assert max_err(go[m], ro[m], scale=np.abs(R["v"]).max()) <= TOL["bf16"]
        assert max_err(gden[m], rden[m]) <= TOL["bf16"]
    assert (go[~m] == 0).all() and (gden[~m] == 0).all()
    if kind == "none":  # no decay: the GBLA core itself
        o2, _, _ = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"])
        assert max_err(go[m], f64(o2)[m], scale=np.abs(R["v"]).max()) <= TOL["bf16"]


def test_decay_core_full_decay_returns_values():
    """lambda = 0: M = I, so o_i = v_i (within bf16 rounding)."""
    shape, D, R, (st, ln), T = core_case("bf16", 2, 300, 2, 64, seed=250)
    lam = torch.zeros(T, 2, dtype=torch.float32).cuda()
    o, _ = gbla.bla_decay_core_forward(shape, D["q"], D["k"], D["v"], D["g"], lam)
    torch.cuda.synchronize()
    assert max_err(f64(o), R["v"], scale=np.abs(R["v"]).max()) <= TOL["bf16"]


def test_decay_core_bench_shape_sampled_sequences():
    """The bench's shape (B = 32, L = 2048, H = 8, d_h = 64), Lion-s decays:
    two whole sequences against the oracle (sequences are independent)."""
    B, L, H = 32, 2048, 8
    shape, D, R, _, T = core_case("bf16", B, L, H, 64, seed=251)
    lam = torch.tensor(_lam("lion-s", T, H, 251), dtype=torch.float32).cuda()
    o, den = gbla.bla_decay_core_forward(shape, D["q"], D["k"], D["v"], D["g"], lam, den=True)
    torch.cuda.synchronize()
    lr = f64(lam)
    for b in (0, 31):
        a, e = b * L, (b + 1) * L
        st, ln = oracle.seqs(1, L)
        ro, rden = oracle.decay_core_forward(R["q"][a:e], R["k"][a:e], R["v"][a:e], R["g"][a:e], lr[a:e], st, ln, H, 64)
        assert max_err(f64(o)[a:e], ro, scale=np.abs(R["v"][a:e]).max()) <= TOL["bf16"], b
        assert max_err(f64(den)[a:e], rden) <= TOL["bf16"], b


def test_decay_core_is_deterministic():
    shape, D, R, _, T = core_case("bf16", 2, 1000, 2, 64, seed=252)
    lam = torch.tensor(_lam("lion-s", T, 2, 252), dtype=torch.float32).cuda()
    a = gbla.bla_decay_core_forward(shape, D["q"], D["k"], D["v"], D["g"], lam, den=True)
    b = gbla.bla_decay_core_forward(shape, D["q"], D["k"], D["v"], D["g"], lam, den=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
