"""The fp64 oracle against the hand-worked examples in tests/golden.

Each case there is a small input worked out by hand from the equation it cites
(Gated Bidirectional Linear Attention for Generative Retrieval, Core method:
Eq. 4 conv, Eq. 5/6 gated core, Eq. 7 gated RMSNorm); its expected values are
exact rationals or closed forms, written in the file with their derivation.
"""
import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.txt")
_ENV = {"__builtins__": {}, "log": math.log, "exp": math.exp, "sqrt": math.sqrt}


def _matrix(text: str) -> np.ndarray:
    rows = [[float(eval(e, _ENV)) for e in r.split(",")] for r in text.split(";")]
    return np.array(rows, dtype=np.float64)


def load_cases(path: str = GOLDEN) -> dict:
    """{name: {"cite": str, "shape": {key: str}, key: matrix, ...}}"""
    cases, cur = {}, None
    for raw in open(path):
        line = raw.strip()
        if not line or line.startswith("#"):
            continue
        if line.startswith("[") and line.endswith("]"):
            cur = cases.setdefault(line[1:-1], {"shape": {}})
        elif line.startswith("cite:"):
            cur["cite"] = line[5:].strip()
        elif line.startswith("shape:"):
            cur["shape"] = dict(kv.split("=") for kv in line[6:].split())
        else:
            key, _, val = line.partition("=")
            cur[key.strip()] = _matrix(val)
    return cases


CASES = load_cases()


def test_every_case_cites_the_page():
    assert CASES, "no worked examples found"
    for name, c in CASES.items():
        cite = c.get("cite", "")
        assert "Gated Bidirectional Linear Attention" in cite, name
        if name.startswith("decay_"):
            assert "Linear Attention for Efficient Bidirectional Sequence Modeling" in cite, name


@pytest.mark.parametrize("name", [n for n in CASES if n.startswith("decay_")])
def test_decay_core_worked_example(name):
    c = CASES[name]
    H, dh = int(c["shape"]["H"]), int(c["shape"]["dh"])
    T = c["q"].shape[0]
    start, ln = oracle.seqs(B=1, L=T)
    o, den = oracle.decay_core_forward(c["q"], c["k"], c["v"], c["g"], c["lam"], start, ln, H, dh)
    np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(den, c["den"], rtol=1e-14, atol=0)
    np.testing.assert_allclose(oracle.decay_core_rnn(c["q"], c["k"], c["v"], c["g"], c["lam"], start, ln, H, dh),
                               c["o"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("name", [n for n in CASES if n.startswith("core_")])
def test_core_worked_example(name):
    c = CASES[name]
    H, dh = int(c["shape"]["H"]), int(c["shape"]["dh"])
    T = c["q"].shape[0]
    start, ln = oracle.seqs(B=1, L=T)
    o, den, _ = oracle.core_forward(c["q"], c["k"], c["v"], c["g"], start, ln, H, dh)
    np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(den, c["den"], rtol=1e-14, atol=0)
    # the single-query form of Eq. 5 gives the same hand-worked values
    np.testing.assert_allclose(oracle.core_explicit(c["q"], c["k"], c["v"], c["g"], start, ln, H, dh), c["o"],
                               rtol=0, atol=1e-14)


@pytest.mark.parametrize("name", [n for n in CASES if n.startswith("conv_")])
def test_conv_worked_example(name):
    c = CASES[name]
    lens = c["lens"].astype(np.int64).ravel()
    cu = np.concatenate([[0], np.cumsum(lens)])
    start, ln = oracle.seqs(cu_seqlens=cu)
    xt = oracle.conv1d(c["x"], c["w"], c["b"].ravel(), start, ln)
    np.testing.assert_allclose(xt, c["xt"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("name", [n for n in CASES if n.startswith("layer_")])
def test_layer_worked_example(name):
    c = CASES[name]
    sh = c["shape"]
    H, dh = int(sh["H"]), int(sh["dh"])
    params = {"conv_w": c["conv_w"], "W_q": c["W_q"], "W_k": c["W_k"], "W_v": c["W_v"], "W_r": c["W_r"],
              "w_g": c["w_g"], "rms_w": c["rms_w"].ravel()}
    T = c["x"].shape[0]
    start, ln = oracle.seqs(B=1, L=T)
    out = oracle.gbla_forward(c["x"], params, H, dh, start, ln, gate_mode=0 if sh["gate"] == "sigmoid" else 1,
                              eps=float(sh["eps"]))
    for key in ("g", "o", "y"):
        if key in c:
            np.testing.assert_allclose(out[key], c[key], rtol=0, atol=1e-14, err_msg=f"{name}: {key}")


@pytest.mark.parametrize("name", [n for n in CASES if n.startswith("sa_")])
def test_sa_worked_example(name):
    c = CASES[name]
    H, dh = int(c["shape"]["H"]), int(c["shape"]["dh"])
    T = c["q"].shape[0]
    start, ln = oracle.seqs(B=1, L=T)
    o, lse = oracle.sa_forward(c["q"], c["k"], c["v"], start, ln, H, dh)
    np.testing.assert_allclose(o, c["o"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, c["lse"], rtol=1e-14, atol=0)
