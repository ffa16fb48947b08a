"""Parity of the SA blocks' attention (sa_core_forward: the bidirectional
softmax attention of Eq. 1, "Gated Bidirectional Linear Attention for
Generative Retrieval", Core method 1) with the fp64 oracle, through the C ABI:
dense, padded and varlen batches, ragged key and query tails (the kernel
takes 256 queries and 128 keys at a time), one-token and empty sequences,
long sequences, and determinism.

Tolerance: bf16 I/O with fp32 accumulation (the weights enter the second
contraction in bf16), max |gpu - ref| <= 2e-2 max |v| over the valid rows."""
import numpy as np
import pytest
import torch

import oracle
from generative_retrieval_encoder_gb300 import build, gbla
from gbla_cases import TOL, core_case, dev, f64, launch_names, max_err, valid_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gbla.lib()


# (B, L, H, seq_lens, varlen lengths)
CASES = [
    (2, 300, 2, None, None),
    (1, 1, 1, None, None),
    (1, 256, 1, None, None),
    (3, 700, 2, [700, 1, 257], None),
    (1, 0, 2, None, [5, 0, 300, 1, 64, 129, 1000, 256, 255]),
    (2, 2048, 2, None, None),
]


def _ids(c):
    return f"B{c[0]}-L{c[1]}-H{c[2]}" + ("-pad" if c[3] else "") + ("-varlen" if c[4] else "")


@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_sa_matches_oracle(case):
    B, L, H, sl, lens = case
    shape, D, R, (st, ln), T = core_case("bf16", B, L, H, 64, seed=600 + CASES.index(case), seq_lens=sl,
                                         lengths=lens)
    res = {}
    names = launch_names(lambda: res.update(o=gbla.sa_core_forward(shape, D["q"], D["k"], D["v"])))
    torch.cuda.synchronize()
    assert "sa[tc]" in names, names
    ro, _ = oracle.sa_forward(R["q"], R["k"], R["v"], st, ln, H, 64)
    m = valid_rows(st, ln, T)
    go = f64(res["o"])
    assert np.isfinite(go).all()
    if m.any():
        assert max_err(go[m], ro[m], scale=np.abs(R["v"][m]).max()) <= TOL["bf16"]
    assert (go[~m] == 0).all()


def test_sa_long_sequence():
    """One sequence of 16384 tokens (128 key tiles, 64 query blocks) against
    the oracle on every row."""
    L, H = 16384, 1
    shape, D, R, (st, ln), T = core_case("bf16", 1, L, H, 64, seed=650)
    o = f64(gbla.sa_core_forward(shape, D["q"], D["k"], D["v"]))
    torch.cuda.synchronize()
    ro, _ = oracle.sa_forward(R["q"], R["k"], R["v"], st, ln, H, 64)
    assert max_err(o, ro, scale=np.abs(R["v"]).max()) <= TOL["bf16"]


def test_sa_bench_size_sampled_rows():
    """The launch the benchmark times at its largest size, B = 8 sequences of
    L = 32768 tokens, H = 8, d_h = 64, against the oracle at 96 sampled
    (query, head) pairs: first and last rows of the first and last sequence,
    rows on both sides of the kernel's 128-key and 256-query tile edges, and
    random rows (every other row's sum over 32768 keys is out of the oracle's
    reach at this size)."""
    B, L, H, dh = 8, 32768, 8, 64
    T = B * L
    r = torch.Generator().manual_seed(660)
    D = {n: dev(torch.randn(T, H * dh, generator=r), "bf16") for n in ("q", "k", "v")}
    shape = gbla.make_shape(B, L, H * dh, H, dh)
    go = gbla.sa_core_forward(shape, D["q"], D["k"], D["v"])
    torch.cuda.synchronize()
    rng = np.random.default_rng(661)
    edges = [0, 127, 128, 255, 256, 511, 512, L - 1]
    rows = np.array([b * L + e for b in (0, B - 1) for e in edges] + rng.integers(0, T, 80).tolist())
    heads = rng.integers(0, H, len(rows))
    R = {n: f64(D[n]) for n in ("q", "k", "v")}
    st, ln = oracle.seqs(B, L)
    ref = oracle.sa_rows(R["q"], R["k"], R["v"], st, ln, H, dh, rows, heads)
    got = np.stack([f64(go[int(i), int(h) * dh:(int(h) + 1) * dh]) for i, h in zip(rows, heads)])
    assert np.isfinite(got).all()
    assert max_err(got, ref, scale=np.abs(R["v"]).max()) <= TOL["bf16"]


def test_sa_is_deterministic_and_equals_sequence_alone():
    shape, D, R, (st, ln), T = core_case("bf16", 1, 0, 2, 64, seed=651, lengths=[100, 2000, 37])
    a = gbla.sa_core_forward(shape, D["q"], D["k"], D["v"])
    b = gbla.sa_core_forward(shape, D["q"], D["k"], D["v"])
    assert torch.equal(a, b)
    s0, n0 = int(st[1]), int(ln[1])
    shape1 = gbla.make_shape(1, n0, 64, 2, 64, dtype="bf16")
    one = gbla.sa_core_forward(shape1, D["q"][s0:s0 + n0].contiguous(), D["k"][s0:s0 + n0].contiguous(),
                               D["v"][s0:s0 + n0].contiguous())
    torch.cuda.synchronize()
    assert torch.equal(one, a[s0:s0 + n0])
