"""GBLA oracle: a plain fp64 CPU statement of the GBLA layer (C, OpenMP over
independent (sequence, head) pairs), wrapped with ctypes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never imports, links or calls it; it shares no code with the CUDA path.

What each function computes, with the passage it follows, is documented in
``gbla_oracle.c`` ("Gated Bidirectional Linear Attention for Generative
Retrieval", section "Core method", Eq. 2-7; LION notes, Theorem 3.1).

Sequences are given as ``(start, len)`` int64 arrays: rows ``start[b] ..
start[b] + len[b] - 1`` of every ``[T, *]`` array form sequence ``b``; rows in no
sequence are padding (outputs 0).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gbla_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None
_lock = threading.Lock()

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile the oracle with the host gcc (plain C, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
                               "-Wno-unused-parameter", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            seq = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, _I64]
            lib.oracle_core_forward.argtypes = seq + [_D] * 7
            lib.oracle_core_explicit.argtypes = seq + [_D] * 5
            lib.oracle_core_lion_rnn.argtypes = seq + [_D] * 5
            lib.oracle_core_backward.argtypes = seq + [_D] * 9
            lib.oracle_decay_core_explicit.argtypes = seq + [_D] * 7
            lib.oracle_decay_core_rnn.argtypes = seq + [_D] * 6
            lib.oracle_sa_forward.argtypes = seq + [_D] * 5
            lib.oracle_sa_rows.argtypes = seq + [_D] * 3 + [ctypes.c_int, _I64, ctypes.POINTER(ctypes.c_int), _D]
            lib.oracle_conv1d.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, _I64, _I64] + [_D] * 4
            layer = ([ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _I64, _I64]
                     + [_D] * 10 + [ctypes.c_int, ctypes.c_double])
            lib.oracle_gbla_forward.argtypes = layer + [_D] * 11
            lib.oracle_gbla_forward.restype = ctypes.c_int
            lib.oracle_gbla_backward.argtypes = layer + [_D] * 11
            lib.oracle_gbla_backward.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def _p(a):
    if a is None:
        return None
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(_D)


def _f64(a):
    if a is None:
        return None
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def seqs(B: int | None = None, L: int | None = None, seq_lens=None, cu_seqlens=None):
    """(start, len) int64 arrays for the three batch forms.

    dense: B sequences of L rows; padding: sequence b owns rows b*L .. b*L +
    seq_lens[b] - 1 of its L-row slot; varlen: sequence b is cu[b] .. cu[b+1]-1.
    """
    if cu_seqlens is not None:
        cu = np.asarray(cu_seqlens, dtype=np.int64)
        return np.ascontiguousarray(cu[:-1]), np.ascontiguousarray(np.diff(cu))
    start = np.arange(B, dtype=np.int64) * L
    ln = np.full(B, L, dtype=np.int64) if seq_lens is None else np.asarray(seq_lens, dtype=np.int64)
    return np.ascontiguousarray(start), np.ascontiguousarray(ln)


def _seqargs(start, ln):
    start = np.ascontiguousarray(start, dtype=np.int64)
    ln = np.ascontiguousarray(ln, dtype=np.int64)
    return start, ln, start.ctypes.data_as(_I64), ln.ctypes.data_as(_I64)


def core_forward(q, k, v, g, start, ln, H: int, dh: int):
    """Eq. 5/6 state form.  q, k, v [T, H*dh]; g [T, H] gate values.
    Returns (o [T, H*dh], den [T, H], state [n_seq, H, dh, dh+1])."""
    q, k, v, g = map(_f64, (q, k, v, g))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    o = np.zeros((T, H * dh)); den = np.zeros((T, H)); st = np.zeros((len(start), H, dh, dh + 1))
    _load().oracle_core_forward(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), _p(g), _p(o), _p(den), _p(st))
    return o, den, st


def core_explicit(q, k, v, g, start, ln, H: int, dh: int):
    """Eq. 5 single-query O(L^2) form (never forms the state)."""
    q, k, v, g = map(_f64, (q, k, v, g))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    o = np.zeros((T, H * dh))
    _load().oracle_core_explicit(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), _p(g), _p(o))
    return o


def core_lion_rnn(q, k, v, g, start, ln, H: int, dh: int):
    """LION bidirectional RNN (Theorem 3.1) with an all-ones mask."""
    q, k, v, g = map(_f64, (q, k, v, g))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    o = np.zeros((T, H * dh))
    _load().oracle_core_lion_rnn(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), _p(g), _p(o))
    return o


def decay_core_forward(q, k, v, g, lam, start, ln, H: int, dh: int):
    """The core under LION's decay masks (oracle_decay_core_explicit): lam [T, H]
    holds lambda_t in [0, 1].  Returns (o [T, H*dh], den [T, H])."""
    q, k, v, g, lam = map(_f64, (q, k, v, g, lam))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    o = np.zeros((T, H * dh)); den = np.zeros((T, H))
    _load().oracle_decay_core_explicit(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), _p(g), _p(lam), _p(o),
                                       _p(den))
    return o, den


def decay_core_rnn(q, k, v, g, lam, start, ln, H: int, dh: int):
    """The same through LION's bidirectional RNN with the decays (Theorem 3.1)."""
    q, k, v, g, lam = map(_f64, (q, k, v, g, lam))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    o = np.zeros((T, H * dh))
    _load().oracle_decay_core_rnn(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), _p(g), _p(lam), _p(o))
    return o


def sa_forward(q, k, v, start, ln, H: int, dh: int):
    """Bidirectional softmax attention, Eq. 1 (oracle_sa_forward): returns
    (o [T, H*dh], lse [T, H]); rows in no sequence are zero."""
    q, k, v = map(_f64, (q, k, v))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    o = np.zeros((T, H * dh)); lse = np.zeros((T, H))
    _load().oracle_sa_forward(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), _p(o), _p(lse))
    return o, lse


def sa_rows(q, k, v, start, ln, H: int, dh: int, rows, heads):
    """Eq. 1 at chosen (query row, head) pairs only (oracle_sa_rows): o [n, dh],
    zeros for a row in no sequence."""
    q, k, v = map(_f64, (q, k, v))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    r = np.ascontiguousarray(rows, dtype=np.int64)
    hh = np.ascontiguousarray(heads, dtype=np.int32)
    assert r.shape == hh.shape and r.ndim == 1
    o = np.zeros((len(r), dh))
    _load().oracle_sa_rows(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), len(r),
                           r.ctypes.data_as(_I64), hh.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), _p(o))
    return o


def core_backward(q, k, v, g, d_o, start, ln, H: int, dh: int):
    """Backward of core_forward for <d_o, o>.  Returns (dq, dk, dv, dg)."""
    q, k, v, g, d_o = map(_f64, (q, k, v, g, d_o))
    T = q.shape[0]
    start, ln, ps, pl = _seqargs(start, ln)
    dq = np.zeros((T, H * dh)); dk = np.zeros((T, H * dh)); dv = np.zeros((T, H * dh)); dg = np.zeros((T, H))
    _load().oracle_core_backward(T, H, dh, len(start), ps, pl, _p(q), _p(k), _p(v), _p(g), _p(d_o),
                                 _p(dq), _p(dk), _p(dv), _p(dg))
    return dq, dk, dv, dg


def conv1d(x, w, b, start, ln):
    """Eq. 4 depthwise causal Conv1d, kernel 4.  x [T, d], w [d, 4], b [d] or None."""
    x, w, b = _f64(x), _f64(w), _f64(b)
    T, d = x.shape
    start, ln, ps, pl = _seqargs(start, ln)
    xt = np.zeros((T, d))
    _load().oracle_conv1d(T, d, len(start), ps, pl, _p(x), _p(w), _p(b), _p(xt))
    return xt


PARAM_NAMES = ("conv_w", "conv_b", "W_q", "W_k", "W_v", "W_r", "w_g", "b_g", "rms_w")


def _layer_args(x, params, H, dh, start, ln, gate_mode, eps):
    x = _f64(x)
    P = {n: _f64(params.get(n)) for n in PARAM_NAMES}
    T, d = x.shape
    start, ln, ps, pl = _seqargs(start, ln)
    args = [T, d, H, dh, len(start), ps, pl, _p(x), _p(P["conv_w"]), _p(P["conv_b"]), _p(P["W_q"]),
            _p(P["W_k"]), _p(P["W_v"]), _p(P["W_r"]), _p(P["w_g"]), _p(P["b_g"]), _p(P["rms_w"]),
            int(gate_mode), float(eps)]
    return x, P, T, d, args, (start, ln)


def gbla_forward(x, params, H: int, dh: int, start, ln, gate_mode: int = 0, eps: float = 1e-6):
    """Full layer forward.  Returns a dict with y and every intermediate
    (xt, q, k, v, r, s, g, o, den, state)."""
    x, P, T, d, args, keep = _layer_args(x, params, H, dh, start, ln, gate_mode, eps)
    n = len(keep[0])
    out = {"y": np.zeros((T, H * dh)), "xt": np.zeros((T, d)), "q": np.zeros((T, H * dh)),
           "k": np.zeros((T, H * dh)), "v": np.zeros((T, H * dh)), "r": np.zeros((T, H * dh)),
           "s": np.zeros((T, H)), "g": np.zeros((T, H)), "o": np.zeros((T, H * dh)),
           "den": np.zeros((T, H)), "state": np.zeros((n, H, dh, dh + 1))}
    names = ("y", "xt", "q", "k", "v", "r", "s", "g", "o", "den", "state")
    rc = _load().oracle_gbla_forward(*args, *[_p(out[k]) for k in names])
    if rc != 0:
        raise MemoryError("oracle_gbla_forward: out of memory")
    return out


def gbla_backward(x, params, dy, H: int, dh: int, start, ln, gate_mode: int = 0, eps: float = 1e-6):
    """Full layer backward for <dy, y>.  Returns dx and one gradient per parameter
    (keys d<name>)."""
    x, P, T, d, args, keep = _layer_args(x, params, H, dh, start, ln, gate_mode, eps)
    dy = _f64(dy)
    g = {"dx": np.zeros((T, d)), "dconv_w": np.zeros((d, 4)), "dconv_b": np.zeros(d),
         "dW_q": np.zeros((d, H * dh)), "dW_k": np.zeros((d, H * dh)), "dW_v": np.zeros((d, H * dh)),
         "dW_r": np.zeros((d, H * dh)), "dw_g": np.zeros((d, H)), "db_g": np.zeros(H),
         "drms_w": np.zeros(dh)}
    names = ("dx", "dconv_w", "dconv_b", "dW_q", "dW_k", "dW_v", "dW_r", "dw_g", "db_g", "drms_w")
    rc = _load().oracle_gbla_backward(*args, _p(dy), *[_p(g[k]) for k in names])
    if rc != 0:
        raise MemoryError("oracle_gbla_backward: out of memory")
    return g
