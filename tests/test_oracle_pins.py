"""Pins of the fp64 oracle against what the pages and the mathematics fix.

None of these compares the oracle with itself restated: each check is a second
form of the method the pages give (the O(L^2) single-query sum of Eq. 5, LION's
bidirectional RNN), a closed form or invariant of Eq. 5-7, a library routine
(PyTorch conv1d / rms_norm / silu / elu / softmax / autograd, all in fp64), or
central finite differences.  A dropped term, a wrong sign or index, or a
transposed operand anywhere in the oracle fails at least one of them.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

pytestmark = pytest.mark.filterwarnings("ignore")


def _rand_core(T, H, dh, seed):
    r = np.random.default_rng(seed)
    return (r.standard_normal((T, H * dh)), r.standard_normal((T, H * dh)),
            r.standard_normal((T, H * dh)), r.uniform(0.05, 1.0, (T, H)))


SHAPES = [(1, 1, 1, 4), (1, 2, 2, 4), (2, 3, 2, 8), (1, 7, 1, 16), (3, 64, 2, 8), (2, 5, 1, 32)]


# ------------------------------------------------------------------ the core

@pytest.mark.parametrize("B,L,H,dh", SHAPES)
def test_state_form_equals_explicit_quadratic_form(B, L, H, dh):
    """Eq. 6 (state, O(L d_h^2)) equals Eq. 5 (single query, O(L^2))."""
    q, k, v, g = _rand_core(B * L, H, dh, 1)
    st, ln = oracle.seqs(B, L)
    o, den, state = oracle.core_forward(q, k, v, g, st, ln, H, dh)
    o2 = oracle.core_explicit(q, k, v, g, st, ln, H, dh)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("B,L,H,dh", SHAPES)
def test_lion_bidirectional_rnn_equals_full_form(B, L, H, dh):
    """LION Theorem 3.1 with an all-ones mask and the -1/2 k_i v_i^T diagonal
    correction gives the same output as the full (global-sum) form."""
    q, k, v, g = _rand_core(B * L, H, dh, 2)
    st, ln = oracle.seqs(B, L)
    o, _, _ = oracle.core_forward(q, k, v, g, st, ln, H, dh)
    o2 = oracle.core_lion_rnn(q, k, v, g, st, ln, H, dh)
    np.testing.assert_allclose(o, o2, rtol=1e-11, atol=1e-11)


def test_single_token_returns_its_value():
    """L = 1: the only weight is 1, so o_1 = v_1."""
    q, k, v, g = _rand_core(3, 2, 16, 3)
    st, ln = oracle.seqs(3, 1)
    o, _, _ = oracle.core_forward(q, k, v, g, st, ln, 2, 16)
    np.testing.assert_allclose(o, v, rtol=1e-14, atol=1e-14)


def test_constant_value_and_shift():
    """Weights are non-negative and sum to 1: v == c gives o == c, and v + c
    shifts o by c."""
    T, H, dh = 40, 2, 8
    q, k, v, g = _rand_core(T, H, dh, 4)
    st, ln = oracle.seqs(2, 20)
    c = np.random.default_rng(5).standard_normal(H * dh)
    o_c, _, _ = oracle.core_forward(q, k, np.tile(c, (T, 1)), g, st, ln, H, dh)
    np.testing.assert_allclose(o_c, np.tile(c, (T, 1)), rtol=1e-13, atol=1e-13)
    o, _, _ = oracle.core_forward(q, k, v, g, st, ln, H, dh)
    o_s, _, _ = oracle.core_forward(q, k, v + c, g, st, ln, H, dh)
    np.testing.assert_allclose(o_s, o + c, rtol=1e-12, atol=1e-12)


def test_outputs_are_convex_combinations():
    """Every o_{i,e} lies in [min_j v_{j,e}, max_j v_{j,e}] of its sequence."""
    B, L, H, dh = 3, 50, 2, 8
    q, k, v, g = _rand_core(B * L, H, dh, 6)
    st, ln = oracle.seqs(B, L)
    o, den, _ = oracle.core_forward(q, k, v, g, st, ln, H, dh)
    assert (den > 0).all()
    for b in range(B):
        vs = v[b * L:(b + 1) * L]
        os_ = o[b * L:(b + 1) * L]
        assert (os_ >= vs.min(0) - 1e-12).all() and (os_ <= vs.max(0) + 1e-12).all()


def test_key_permutation_invariance():
    """Permuting the (k_j, v_j, g_j) triples leaves every o_i unchanged."""
    L, H, dh = 33, 2, 8
    q, k, v, g = _rand_core(L, H, dh, 7)
    st, ln = oracle.seqs(1, L)
    o, _, _ = oracle.core_forward(q, k, v, g, st, ln, H, dh)
    p = np.random.default_rng(8).permutation(L)
    o2, _, _ = oracle.core_forward(q, k[p], v[p], g[p], st, ln, H, dh)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)


def test_gate_scale_invariance():
    """o is invariant under g -> c g (c > 0); this is why the softmax
    normaliser of Eq. 5 cancels."""
    L, H, dh = 25, 2, 8
    q, k, v, g = _rand_core(2 * L, H, dh, 9)
    st, ln = oracle.seqs(2, L)
    o, _, _ = oracle.core_forward(q, k, v, g, st, ln, H, dh)
    o2, _, _ = oracle.core_forward(q, k, v, 37.5 * g, st, ln, H, dh)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)


def test_ungated_core_equals_eq3_einsum():
    """With g == 1 the core is Eq. 3: (phi(Q)(phi(K)^T V)) / (phi(Q)(phi(K)^T 1)),
    here evaluated with torch fp64 elu and einsum."""
    L, H, dh = 31, 2, 16
    q, k, v, _ = _rand_core(L, H, dh, 10)
    st, ln = oracle.seqs(1, L)
    o, _, _ = oracle.core_forward(q, k, v, np.ones((L, H)), st, ln, H, dh)
    Q = F.elu(torch.tensor(q).view(L, H, dh)) + 1
    K = F.elu(torch.tensor(k).view(L, H, dh)) + 1
    V = torch.tensor(v).view(L, H, dh)
    num = torch.einsum("ihe,hef->ihf", Q, torch.einsum("jhe,jhf->hef", K, V))
    den = torch.einsum("ihe,he->ih", Q, K.sum(0))
    np.testing.assert_allclose(o, (num / den[..., None]).reshape(L, H * dh).numpy(), rtol=1e-12, atol=1e-12)


def test_sequences_are_independent():
    """Packed sequences give the same outputs as each sequence alone."""
    H, dh = 2, 8
    lens = [5, 1, 17, 9]
    T = sum(lens)
    q, k, v, g = _rand_core(T, H, dh, 11)
    cu = np.concatenate([[0], np.cumsum(lens)])
    st, ln = oracle.seqs(cu_seqlens=cu)
    o, _, state = oracle.core_forward(q, k, v, g, st, ln, H, dh)
    for b, (a, e) in enumerate(zip(cu[:-1], cu[1:])):
        s1, l1 = oracle.seqs(1, e - a)
        o1, _, st1 = oracle.core_forward(q[a:e], k[a:e], v[a:e], g[a:e], s1, l1, H, dh)
        np.testing.assert_array_equal(o[a:e], o1)
        np.testing.assert_array_equal(state[b], st1[0])


# --------------------------------------------------------------- the layer

def _tiny_layer(seed, d=8, H=2, dh=4, gamma=True):
    r = np.random.default_rng(seed)
    s = 1.0 / np.sqrt(d)
    P = {"conv_w": r.standard_normal((d, 4)) * 0.5, "conv_b": r.standard_normal(d) * s,
         "W_q": r.standard_normal((d, H * dh)) * s, "W_k": r.standard_normal((d, H * dh)) * s,
         "W_v": r.standard_normal((d, H * dh)) * s, "W_r": r.standard_normal((d, H * dh)) * s,
         "w_g": r.standard_normal((d, H)) * s, "b_g": r.standard_normal(H) * s}
    if gamma:
        P["rms_w"] = 1.0 + 0.3 * r.standard_normal(dh)
    return P


def test_conv_equals_torch_depthwise_conv1d():
    """Eq. 4 Conv1d read as depthwise causal kernel 4: torch
    conv1d(groups=d, padding=3)[..., :L] per sequence, fp64."""
    d = 6
    lens = [1, 2, 3, 4, 11]
    cu = np.concatenate([[0], np.cumsum(lens)])
    r = np.random.default_rng(12)
    x = r.standard_normal((cu[-1], d))
    w = r.standard_normal((d, 4))
    b = r.standard_normal(d)
    st, ln = oracle.seqs(cu_seqlens=cu)
    xt = oracle.conv1d(x, w, b, st, ln)
    for a, e in zip(cu[:-1], cu[1:]):
        ref = F.conv1d(torch.tensor(x[a:e]).T[None], torch.tensor(w)[:, None, :], torch.tensor(b),
                       padding=3, groups=d)[0, :, : e - a].T
        np.testing.assert_allclose(xt[a:e], ref.numpy(), rtol=1e-13, atol=1e-13)


def _torch_layer(x, P, H, dh, lens, gate_mode, eps):
    """The layer as a composition of torch fp64 library routines, one sequence
    at a time: conv1d -> matmul -> sigmoid/softmax -> elu+1 -> einsum -> rms_norm -> silu."""
    T, d = x.shape
    ys = []
    cu = np.concatenate([[0], np.cumsum(lens)])
    for a, e in zip(cu[:-1], cu[1:]):
        L = e - a
        xt = F.conv1d(x[a:e].T[None], P["conv_w"][:, None, :], P.get("conv_b"), padding=3, groups=d)[0, :, :L].T
        q = (xt @ P["W_q"]).view(L, H, dh)
        k = (xt @ P["W_k"]).view(L, H, dh)
        v = (xt @ P["W_v"]).view(L, H, dh)
        r = (xt @ P["W_r"]).view(L, H, dh)
        s = xt @ P["w_g"] + P["b_g"]
        g = torch.sigmoid(s) if gate_mode == 0 else torch.softmax(s, dim=0)
        Qf = F.elu(q) + 1
        Kt = g[..., None] * (F.elu(k) + 1)
        S = torch.einsum("jhe,jhf->hef", Kt, v)
        z = Kt.sum(0)
        o = torch.einsum("ihe,hef->ihf", Qf, S) / torch.einsum("ihe,he->ih", Qf, z)[..., None]
        y = F.rms_norm(o, (dh,), weight=P.get("rms_w"), eps=eps) * F.silu(r)
        ys.append(y.reshape(L, H * dh))
    return torch.cat(ys, 0)


@pytest.mark.parametrize("gate_mode", [0, 1])
@pytest.mark.parametrize("lens", [[7], [1, 4, 9], [3, 3]])
def test_layer_forward_and_backward_equal_torch_library_composition(gate_mode, lens):
    """Forward equals the torch fp64 composition; the hand-derived backward
    equals torch autograd through that composition."""
    d, H, dh, eps = 8, 2, 4, 1e-6
    P = _tiny_layer(13 + gate_mode, d, H, dh)
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    r = np.random.default_rng(14)
    x = r.standard_normal((T, d))
    dy = r.standard_normal((T, H * dh))
    st, ln = oracle.seqs(cu_seqlens=cu)
    out = oracle.gbla_forward(x, P, H, dh, st, ln, gate_mode, eps)
    grads = oracle.gbla_backward(x, P, dy, H, dh, st, ln, gate_mode, eps)
    xt = torch.tensor(x, requires_grad=True)
    Pt = {n: torch.tensor(a, requires_grad=True) for n, a in P.items()}
    y = _torch_layer(xt, Pt, H, dh, lens, gate_mode, eps)
    np.testing.assert_allclose(out["y"], y.detach().numpy(), rtol=1e-11, atol=1e-12)
    (y * torch.tensor(dy)).sum().backward()
    np.testing.assert_allclose(grads["dx"], xt.grad.numpy(), rtol=1e-9, atol=1e-11)
    for n, a in Pt.items():
        np.testing.assert_allclose(grads["d" + n], a.grad.numpy(), rtol=1e-9, atol=1e-11, err_msg=n)


def test_rmsnorm_gate_equals_torch_rms_norm_and_silu():
    """Eq. 7 on the oracle's own o and r: y = rms_norm(o) * gamma * silu(r)."""
    d, H, dh, eps = 8, 2, 4, 1e-6
    P = _tiny_layer(15, d, H, dh)
    x = np.random.default_rng(16).standard_normal((12, d))
    st, ln = oracle.seqs(1, 12)
    out = oracle.gbla_forward(x, P, H, dh, st, ln, 0, eps)
    o = torch.tensor(out["o"]).view(12, H, dh)
    r = torch.tensor(out["r"]).view(12, H, dh)
    ref = F.rms_norm(o, (dh,), weight=torch.tensor(P["rms_w"]), eps=eps) * F.silu(r)
    np.testing.assert_allclose(out["y"], ref.reshape(12, H * dh).numpy(), rtol=1e-13, atol=1e-13)


def test_softmax_gate_equals_unnormalised_exp_gate():
    """Under Eq. 5 the softmax normaliser cancels: the core with g = softmax(s)
    equals the core with g = exp(s - c) for any c."""
    d, H, dh = 8, 2, 4
    P = _tiny_layer(17, d, H, dh)
    x = np.random.default_rng(18).standard_normal((10, d))
    st, ln = oracle.seqs(1, 10)
    out = oracle.gbla_forward(x, P, H, dh, st, ln, 1, 1e-6)
    np.testing.assert_allclose(out["g"].sum(0), np.ones(H), rtol=1e-13)
    o2, _, _ = oracle.core_forward(out["q"], out["k"], out["v"], np.exp(out["s"] - 3.0), st, ln, H, dh)
    np.testing.assert_allclose(out["o"], o2, rtol=1e-12, atol=1e-12)


def test_padding_rows_are_zero_and_valid_rows_match_dense():
    d, H, dh = 8, 2, 4
    P = _tiny_layer(19, d, H, dh)
    B, L, lens = 3, 6, [6, 2, 4]
    x = np.random.default_rng(20).standard_normal((B * L, d))
    st, ln = oracle.seqs(B, L, seq_lens=lens)
    out = oracle.gbla_forward(x, P, H, dh, st, ln)
    for b, n in enumerate(lens):
        assert (out["y"][b * L + n:(b + 1) * L] == 0).all()
        s1, l1 = oracle.seqs(1, n)
        o1 = oracle.gbla_forward(x[b * L:b * L + n], P, H, dh, s1, l1)
        np.testing.assert_array_equal(out["y"][b * L:b * L + n], o1["y"])


# ------------------------------------------------------- finite differences

def _fd_check(f, arrays, grads, h=1e-6, rtol=1e-6):
    """Central differences of the scalar f() for every element of every array."""
    for name, a in arrays.items():
        num = np.zeros_like(a)
        flat = a.reshape(-1)
        for i in range(flat.size):
            old = flat[i]
            flat[i] = old + h
            fp = f()
            flat[i] = old - h
            fm = f()
            flat[i] = old
            num.reshape(-1)[i] = (fp - fm) / (2 * h)
        scale = max(np.abs(num).max(), 1e-3)
        err = np.abs(num - grads[name]).max() / scale
        assert err <= rtol, f"{name}: relative error {err:.3e}"


@pytest.mark.parametrize("lens,H,dh", [([5], 1, 4), ([1, 6], 2, 4), ([3, 4, 2], 2, 2)])
def test_core_backward_finite_differences(lens, H, dh):
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    q, k, v, g = _rand_core(T, H, dh, 21)
    d_o = np.random.default_rng(22).standard_normal((T, H * dh))
    st, ln = oracle.seqs(cu_seqlens=cu)
    dq, dk, dv, dg = oracle.core_backward(q, k, v, g, d_o, st, ln, H, dh)
    arrs = {"q": q, "k": k, "v": v, "g": g}
    f = lambda: float((oracle.core_forward(q, k, v, g, st, ln, H, dh)[0] * d_o).sum())
    _fd_check(f, arrs, {"q": dq, "k": dk, "v": dv, "g": dg})


@pytest.mark.parametrize("gate_mode", [0, 1])
@pytest.mark.parametrize("lens,d,H,dh", [([6], 4, 1, 4), ([2, 5], 6, 2, 4), ([1, 3, 4, 2], 4, 2, 2),
                                         ([9], 8, 2, 4)])
def test_layer_backward_finite_differences(gate_mode, lens, d, H, dh):
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = int(cu[-1])
    P = _tiny_layer(23, d, H, dh)
    r = np.random.default_rng(24)
    x = r.standard_normal((T, d))
    dy = r.standard_normal((T, H * dh))
    st, ln = oracle.seqs(cu_seqlens=cu)
    grads = oracle.gbla_backward(x, P, dy, H, dh, st, ln, gate_mode)
    arrs = {"x": x, **P}
    gmap = {"x": grads["dx"], **{n: grads["d" + n] for n in P}}
    f = lambda: float((oracle.gbla_forward(x, P, H, dh, st, ln, gate_mode)["y"] * dy).sum())
    _fd_check(f, arrs, gmap)


def test_backward_homogeneity_invariants():
    """o is degree-0 homogeneous in q~_i and in the set {k~_j}, and rows of the
    weight matrix sum to 1, so (Euler):  sum_j g_j dg_j = 0 per (seq, head);
    sum_e q~_{i,e} dq~_{i,e} = 0 per token; sum_j dv_j = sum_i do_i."""
    B, L, H, dh = 2, 23, 2, 8
    q, k, v, g = _rand_core(B * L, H, dh, 25)
    d_o = np.random.default_rng(26).standard_normal((B * L, H * dh))
    st, ln = oracle.seqs(B, L)
    dq, dk, dv, dg = oracle.core_backward(q, k, v, g, d_o, st, ln, H, dh)
    qt = np.where(q > 0, q + 1, np.exp(q))
    dphi = np.where(q > 0, 1.0, np.exp(q))
    dqt = dq / dphi
    for b in range(B):
        sl = slice(b * L, (b + 1) * L)
        np.testing.assert_allclose((g[sl] * dg[sl]).sum(0), 0, atol=1e-11)
        np.testing.assert_allclose(dv[sl].sum(0), d_o[sl].sum(0), rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose((qt * dqt).reshape(B * L, H, dh).sum(-1), 0, atol=1e-11)


# ------------------------------------------------- LION decay masks (Lion-d, Lion-s)

@pytest.mark.parametrize("B,L,H,dh", SHAPES)
@pytest.mark.parametrize("kind", ["lion-s", "lion-d"])
def test_decay_core_definition_equals_bidirectional_rnn(B, L, H, dh, kind):
    """LION Theorem 3.1 with the decays as state transitions (forward and
    backward scans, -1/2 k_i v_i^T each) equals the masked definition with
    M = M^F + M^B - I."""
    q, k, v, g = _rand_core(B * L, H, dh, 21)
    r = np.random.default_rng(22)
    lam = r.uniform(0.2, 1.0, (B * L, H)) if kind == "lion-s" else np.full((B * L, H), 0.8)
    st, ln = oracle.seqs(B, L)
    o, den = oracle.decay_core_forward(q, k, v, g, lam, st, ln, H, dh)
    np.testing.assert_allclose(oracle.decay_core_rnn(q, k, v, g, lam, st, ln, H, dh), o, rtol=1e-11, atol=1e-11)
    assert (den > 0).all()


def test_decay_core_with_no_decay_is_the_gbla_core():
    """lambda = 1 everywhere is the all-ones mask: Eq. 5 exactly."""
    q, k, v, g = _rand_core(90, 2, 8, 23)
    st, ln = oracle.seqs(cu_seqlens=[0, 40, 41, 90])
    o, den = oracle.decay_core_forward(q, k, v, g, np.ones((90, 2)), st, ln, 2, 8)
    o2, den2, _ = oracle.core_forward(q, k, v, g, st, ln, 2, 8)
    np.testing.assert_allclose(o, o2, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(den, den2, rtol=1e-12)


def test_decay_core_full_decay_returns_each_value():
    """lambda = 0: every product off the diagonal holds a zero, M = I, o = v."""
    q, k, v, g = _rand_core(30, 2, 4, 24)
    st, ln = oracle.seqs(3, 10)
    o, _ = oracle.decay_core_forward(q, k, v, g, np.zeros((30, 2)), st, ln, 2, 4)
    np.testing.assert_allclose(o, v, rtol=1e-14, atol=1e-14)


def test_lion_d_is_symmetric_under_reversal():
    """A constant decay gives M_ij = lambda^|i-j|, symmetric in i and j: the
    outputs of a reversed sequence are the reversed outputs.  (A selective
    decay shifts by one position under reversal, so this holds for Lion-d.)"""
    q, k, v, g = _rand_core(25, 2, 8, 25)
    lam = np.full((25, 2), 0.7)
    st, ln = oracle.seqs(1, 25)
    o, _ = oracle.decay_core_forward(q, k, v, g, lam, st, ln, 2, 8)
    rev = lambda a: np.ascontiguousarray(a[::-1])
    o2, _ = oracle.decay_core_forward(rev(q), rev(k), rev(v), rev(g), lam, st, ln, 2, 8)
    np.testing.assert_allclose(rev(o2), o, rtol=1e-12, atol=1e-12)


def test_decay_core_outputs_are_convex_combinations_and_sequences_independent():
    """Mask entries and weights are >= 0, so o_i lies between the smallest and
    largest v_j of its sequence; a packed sequence equals itself alone."""
    q, k, v, g = _rand_core(60, 1, 4, 26)
    lam = np.random.default_rng(27).uniform(0.0, 1.0, (60, 1))
    st, ln = oracle.seqs(cu_seqlens=[0, 25, 60])
    o, _ = oracle.decay_core_forward(q, k, v, g, lam, st, ln, 1, 4)
    for a, n in zip(st, ln):
        seg = v[a:a + n]
        assert (o[a:a + n] >= seg.min(0) - 1e-12).all() and (o[a:a + n] <= seg.max(0) + 1e-12).all()
        s1, l1 = oracle.seqs(1, int(n))
        alone, _ = oracle.decay_core_forward(q[a:a + n], k[a:a + n], v[a:a + n], g[a:a + n], lam[a:a + n], s1, l1, 1, 4)
        np.testing.assert_allclose(o[a:a + n], alone, rtol=1e-13, atol=1e-13)


# --------------------------------------------------------------------------
# Bidirectional softmax attention (GBLA notes, "Core method" 1, Eq. 1)


def _rand_qkv(T, H, dh, seed):
    r = np.random.default_rng(seed)
    return tuple(r.standard_normal((T, H * dh)) for _ in range(3))


@pytest.mark.parametrize("lens", [[7], [1, 33, 5], [64, 64]])
def test_sa_equals_torch_scaled_dot_product_attention(lens):
    """Eq. 1 per sequence equals the library's scaled-dot-product attention
    (torch, fp64, no mask, scale 1/sqrt(d_h)), head by head."""
    H, dh = 2, 16
    T = sum(lens)
    q, k, v = _rand_qkv(T, H, dh, 31)
    st, ln = oracle.seqs(cu_seqlens=np.concatenate([[0], np.cumsum(lens)]).tolist())
    o, lse = oracle.sa_forward(q, k, v, st, ln, H, dh)
    for s, n in zip(st, ln):
        for h in range(H):
            sl = slice(h * dh, (h + 1) * dh)
            t = lambda a: torch.tensor(a[s:s + n, sl])[None, None]
            ref = F.scaled_dot_product_attention(t(q), t(k), t(v))[0, 0].numpy()
            np.testing.assert_allclose(o[s:s + n, sl], ref, rtol=1e-12, atol=1e-12)
            scores = t(q)[0, 0] @ t(k)[0, 0].T / np.sqrt(dh)
            np.testing.assert_allclose(lse[s:s + n, h], torch.logsumexp(scores, dim=1).numpy(), rtol=1e-12)


def test_sa_rows_equal_torch_scaled_dot_product_attention():
    """The sampled-row form (Eq. 1 at chosen query, head pairs, for sequences
    too long for every row) equals the library's scaled-dot-product attention
    at each pair, over ragged packed sequences; a row in no sequence (padding
    past the last one) gives zeros."""
    H, dh = 3, 16
    lens = [1, 37, 130, 64]
    T = sum(lens) + 5  # five padding rows at the end
    q, k, v = _rand_qkv(T, H, dh, 37)
    cu = np.concatenate([[0], np.cumsum(lens)])
    st, ln = oracle.seqs(cu_seqlens=cu.tolist())
    rng = np.random.default_rng(38)
    rows = np.concatenate([[0, 1, 37, 38, 167, 168, 231, T - 1], rng.integers(0, T, 24)])
    heads = rng.integers(0, H, len(rows))
    o = oracle.sa_rows(q, k, v, st, ln, H, dh, rows, heads)
    for p, (i, h) in enumerate(zip(rows, heads)):
        b = np.searchsorted(cu, i, side="right") - 1
        if b >= len(lens):
            assert (o[p] == 0).all()
            continue
        s, n = cu[b], lens[b]
        sl = slice(h * dh, (h + 1) * dh)
        tq = torch.tensor(q[i:i + 1, sl])[None, None]
        tk, tv = (torch.tensor(a[s:s + n, sl])[None, None] for a in (k, v))
        ref = F.scaled_dot_product_attention(tq, tk, tv)[0, 0, 0].numpy()
        np.testing.assert_allclose(o[p], ref, rtol=1e-12, atol=1e-12)


def test_sa_single_key_and_identical_keys():
    """One key: the weight is 1, o = v.  Identical keys: equal weights, o is
    the mean of the values of the sequence."""
    q, k, v = _rand_qkv(13, 2, 8, 32)
    st, ln = oracle.seqs(cu_seqlens=[0, 1, 13])
    kk = k.copy()
    kk[1:13] = kk[1]
    o, _ = oracle.sa_forward(q, kk, v, st, ln, 2, 8)
    np.testing.assert_allclose(o[0], v[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(o[1:13], np.broadcast_to(v[1:13].mean(axis=0), (12, 16)), rtol=1e-12, atol=1e-12)


def test_sa_hard_limit_selects_the_best_key():
    """Scaling the queries up makes the weights one-hot on each query's
    largest score: o_i tends to v of that key (checked at a large scale)."""
    q, k, v = _rand_qkv(20, 1, 8, 33)
    st, ln = oracle.seqs(1, 20)
    o, _ = oracle.sa_forward(q * 1e4, k, v, st, ln, 1, 8)
    best = np.argmax(q @ k.T, axis=1)
    np.testing.assert_allclose(o, v[best], rtol=0, atol=1e-9)


def test_sa_key_permutation_convexity_and_independence():
    """Permuting the keys and values of a sequence together leaves o unchanged;
    each output coordinate lies between the sequence's smallest and largest
    value coordinate; a packed sequence equals itself alone."""
    q, k, v = _rand_qkv(50, 2, 8, 34)
    st, ln = oracle.seqs(cu_seqlens=[0, 20, 50])
    o, _ = oracle.sa_forward(q, k, v, st, ln, 2, 8)
    perm = np.concatenate([np.random.default_rng(35).permutation(20), 20 + np.random.default_rng(36).permutation(30)])
    o2, _ = oracle.sa_forward(q, k[perm], v[perm], st, ln, 2, 8)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-12)
    for s, n in zip(st, ln):
        assert (o[s:s + n] <= v[s:s + n].max(axis=0) + 1e-12).all()
        assert (o[s:s + n] >= v[s:s + n].min(axis=0) - 1e-12).all()
    st1, ln1 = oracle.seqs(1, 30)
    o3, _ = oracle.sa_forward(q[20:], k[20:], v[20:], st1, ln1, 2, 8)
    np.testing.assert_allclose(o3, o[20:], rtol=1e-13, atol=1e-13)
