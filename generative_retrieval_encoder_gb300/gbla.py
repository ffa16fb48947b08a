"""Thin Python binding of libgbla.so (include/gbla.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  PyTorch supplies device memory (outputs, workspace) and the current
CUDA stream.  There is no CPU path: if the library is missing this module
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libgbla.so")

GBLA_OK, GBLA_ERR_INVALID_ARG, GBLA_ERR_UNSUPPORTED, GBLA_ERR_WORKSPACE, GBLA_ERR_CUDA, GBLA_ERR_DEVICE_CHECK = \
    0, -1, -2, -3, -4, -5
GBLA_ERR_DEVICE_TIMEOUT = -6
GBLA_POLICY_AUTO, GBLA_POLICY_TC, GBLA_POLICY_MMA = 0, 1, 2
GBLA_F32, GBLA_BF16 = 0, 1
GBLA_GATE_SIGMOID, GBLA_GATE_SOFTMAX = 0, 1
GBLA_OP_FORWARD, GBLA_OP_BACKWARD, GBLA_OP_CORE_FORWARD, GBLA_OP_CORE_BACKWARD, GBLA_OP_DECAY_FORWARD = 0, 1, 2, 3, 4
GBLA_OP_SA_FORWARD = 5

EXPORTS = ("gbla_workspace_size", "gbla_saved_size", "gbla_validate_shape", "gbla_forward", "gbla_backward",
           "bla_core_forward", "bla_core_backward", "gbla_check_device_status", "gbla_status_string",
           "gbla_last_error", "gbla_version", "gbla_profiling_enable", "gbla_profiling_read",
           "bla_core_forward_noalloc", "bla_core_noalloc_check_device_status", "gbla_diag_bounded_wait",
           "gbla_set_kernel_policy", "bla_decay_core_forward", "sa_core_forward")
NOALLOC_SCRATCH_BYTES = 64 << 20


class GblaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = lib().gbla_status_string(status).decode()
        if status == GBLA_ERR_CUDA:
            msg += " (" + lib().gbla_last_error().decode() + ")"
        super().__init__(f"{what}: {msg}")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int), ("H", ctypes.c_int),
                ("d_h", ctypes.c_int), ("cu_seqlens", ctypes.c_void_p), ("num_seqs", ctypes.c_int),
                ("seq_lens", ctypes.c_void_p), ("io_dtype", ctypes.c_int), ("gate", ctypes.c_int),
                ("rms_eps", ctypes.c_float)]


_lib = None


def lib() -> ctypes.CDLL:
    """Loads libgbla.so (built by build.py).  Raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libgbla.so not built ({LIB_PATH}); run generative_retrieval_encoder_gb300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        vp, sz, f = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p
        sp = ctypes.POINTER(Shape)
        L.gbla_workspace_size.argtypes = [sp, ctypes.c_int]
        L.gbla_workspace_size.restype = sz
        L.gbla_saved_size.argtypes = [sp]
        L.gbla_saved_size.restype = sz
        L.gbla_validate_shape.argtypes = [sp]
        L.gbla_validate_shape.restype = ctypes.c_int
        L.gbla_forward.argtypes = [sp] + [vp] * 13 + [sz, vp]
        L.gbla_forward.restype = ctypes.c_int
        L.gbla_backward.argtypes = [sp] + [vp] * 13 + [f] * 9 + [vp, sz, vp]
        L.gbla_backward.restype = ctypes.c_int
        L.bla_core_forward.argtypes = [sp] + [vp] * 8 + [sz, vp]
        L.bla_core_forward.restype = ctypes.c_int
        L.bla_core_backward.argtypes = [sp] + [vp] * 10 + [sz, vp]
        L.bla_core_backward.restype = ctypes.c_int
        L.bla_decay_core_forward.argtypes = [sp] + [vp] * 8 + [sz, vp]
        L.bla_decay_core_forward.restype = ctypes.c_int
        L.sa_core_forward.argtypes = [sp] + [vp] * 5 + [sz, vp]
        L.sa_core_forward.restype = ctypes.c_int
        L.bla_core_forward_noalloc.argtypes = [sp] + [vp] * 8
        L.bla_core_forward_noalloc.restype = ctypes.c_int
        L.bla_core_noalloc_check_device_status.argtypes = [vp]
        L.bla_core_noalloc_check_device_status.restype = ctypes.c_int
        L.gbla_diag_bounded_wait.argtypes = [vp, sz, ctypes.c_uint, vp]
        L.gbla_diag_bounded_wait.restype = ctypes.c_int
        L.gbla_set_kernel_policy.argtypes = [ctypes.c_int]
        L.gbla_set_kernel_policy.restype = ctypes.c_int
        L.gbla_check_device_status.argtypes = [vp, vp]
        L.gbla_check_device_status.restype = ctypes.c_int
        L.gbla_status_string.argtypes = [ctypes.c_int]
        L.gbla_status_string.restype = ctypes.c_char_p
        L.gbla_last_error.restype = ctypes.c_char_p
        L.gbla_version.restype = ctypes.c_int
        L.gbla_profiling_enable.argtypes = [ctypes.c_int]
        L.gbla_profiling_enable.restype = None
        L.gbla_profiling_read.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_float),
                                          ctypes.c_int]
        L.gbla_profiling_read.restype = ctypes.c_int
        _lib = L
    return _lib


def make_shape(B: int, L: int, d: int, H: int, d_h: int, dtype: str = "bf16", gate: str = "sigmoid",
               eps: float = 1e-6, cu_seqlens: torch.Tensor | None = None,
               seq_lens: torch.Tensor | None = None) -> Shape:
    """Builds a gbla_shape.  cu_seqlens / seq_lens are int32 CUDA tensors (kept
    alive by the returned object).  With cu_seqlens, B = 1 and L = total rows."""
    s = Shape()
    s.B, s.L, s.d, s.H, s.d_h = B, L, d, H, d_h
    s.io_dtype = GBLA_F32 if dtype in ("f32", "fp32", torch.float32) else GBLA_BF16
    s.gate = GBLA_GATE_SOFTMAX if gate == "softmax" else GBLA_GATE_SIGMOID
    s.rms_eps = eps
    s._keep = []
    if cu_seqlens is not None:
        assert cu_seqlens.dtype == torch.int32 and cu_seqlens.is_cuda
        s.cu_seqlens = cu_seqlens.data_ptr()
        s.num_seqs = cu_seqlens.numel() - 1
        s._keep.append(cu_seqlens)
    if seq_lens is not None:
        assert seq_lens.dtype == torch.int32 and seq_lens.is_cuda
        s.seq_lens = seq_lens.data_ptr()
        s._keep.append(seq_lens)
    return s


def io_dtype(shape: Shape) -> torch.dtype:
    return torch.float32 if shape.io_dtype == GBLA_F32 else torch.bfloat16


def rows(shape: Shape) -> int:
    return shape.L if shape.cu_seqlens else shape.B * shape.L


def n_seq(shape: Shape) -> int:
    return shape.num_seqs if shape.cu_seqlens else shape.B


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(status: int, what: str):
    if status != GBLA_OK:
        raise GblaError(status, what)


def gbla_workspace_size(shape: Shape, op: int) -> int:
    return lib().gbla_workspace_size(ctypes.byref(shape), op)


def gbla_saved_size(shape: Shape) -> int:
    return lib().gbla_saved_size(ctypes.byref(shape))


def gbla_validate_shape(shape: Shape) -> int:
    return lib().gbla_validate_shape(ctypes.byref(shape))


def workspace(shape: Shape, op: int, device="cuda") -> torch.Tensor:
    n = gbla_workspace_size(shape, op)
    if n == 0:
        _check(gbla_validate_shape(shape) or GBLA_ERR_INVALID_ARG, "gbla_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


PARAMS = ("conv_w", "conv_b", "W_q", "W_k", "W_v", "W_r", "w_g", "b_g", "rms_w")


def gbla_forward(shape: Shape, x: torch.Tensor, params: dict, y: torch.Tensor | None = None,
                 saved: torch.Tensor | bool | None = None, ws: torch.Tensor | None = None):
    """Layer forward.  Returns (y, saved); pass saved=True to allocate the
    activation buffer that gbla_backward needs."""
    if y is None:
        y = torch.empty(rows(shape), shape.H * shape.d_h, dtype=io_dtype(shape), device=x.device)
    if saved is True:
        saved = torch.empty(gbla_saved_size(shape), dtype=torch.uint8, device=x.device)
    if ws is None:
        ws = workspace(shape, GBLA_OP_FORWARD, x.device)
    P = [params.get(n) for n in PARAMS]
    st = lib().gbla_forward(ctypes.byref(shape), _ptr(x), *[_ptr(p) for p in P], _ptr(y),
                            _ptr(saved if isinstance(saved, torch.Tensor) else None), _ptr(ws), ws.numel(), _stream())
    _check(st, "gbla_forward")
    return y, (saved if isinstance(saved, torch.Tensor) else None)


def gbla_backward(shape: Shape, x: torch.Tensor, params: dict, saved: torch.Tensor, dy: torch.Tensor,
                  ws: torch.Tensor | None = None, out: dict | None = None) -> dict:
    """Layer backward for <dy, y>.  Returns dx (io dtype) and fp32 parameter
    gradients d<name>."""
    dev = x.device
    d, H, dh = shape.d, shape.H, shape.d_h
    f = dict(dtype=torch.float32, device=dev)
    g = out if out is not None else {
        "dx": torch.empty_like(x), "dconv_w": torch.empty(d, 4, **f), "dconv_b": torch.empty(d, **f),
        "dW_q": torch.empty(d, H * dh, **f), "dW_k": torch.empty(d, H * dh, **f),
        "dW_v": torch.empty(d, H * dh, **f), "dW_r": torch.empty(d, H * dh, **f),
        "dw_g": torch.empty(d, H, **f), "db_g": torch.empty(H, **f), "drms_w": torch.empty(dh, **f)}
    if ws is None:
        ws = workspace(shape, GBLA_OP_BACKWARD, dev)
    P = [params.get(n) for n in PARAMS]
    names = ("dconv_w", "dconv_b", "dW_q", "dW_k", "dW_v", "dW_r", "dw_g", "db_g", "drms_w")
    st = lib().gbla_backward(ctypes.byref(shape), _ptr(x), *[_ptr(p) for p in P], _ptr(saved), _ptr(dy),
                             _ptr(g["dx"]), *[_ptr(g.get(n)) for n in names], _ptr(ws), ws.numel(), _stream())
    _check(st, "gbla_backward")
    return g


def bla_core_forward(shape: Shape, q, k, v, g, o=None, den=None, state=None, ws=None):
    """The gated BLA core alone: returns (o, den, state); den/state are filled
    when tensors are passed (True allocates them)."""
    dev = q.device
    if o is None:
        o = torch.empty_like(q)
    if den is True:
        den = torch.empty(rows(shape), shape.H, dtype=torch.float32, device=dev)
    if state is True:
        state = torch.empty(n_seq(shape), shape.H, shape.d_h, shape.d_h + 1, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(shape, GBLA_OP_CORE_FORWARD, dev)
    st = lib().bla_core_forward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(o),
                                _ptr(den if isinstance(den, torch.Tensor) else None),
                                _ptr(state if isinstance(state, torch.Tensor) else None), _ptr(ws), ws.numel(),
                                _stream())
    _check(st, "bla_core_forward")
    return o, den, state


def bla_decay_core_forward(shape: Shape, q, k, v, g, lam, o=None, den=None, ws=None):
    """The core under LION's decay masks (see gbla.h): returns (o, den)."""
    dev = q.device
    if o is None:
        o = torch.empty_like(q)
    if den is True:
        den = torch.empty(rows(shape), shape.H, dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(shape, GBLA_OP_DECAY_FORWARD, dev)
    st = lib().bla_decay_core_forward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(lam), _ptr(o),
                                      _ptr(den if isinstance(den, torch.Tensor) else None), _ptr(ws), ws.numel(),
                                      _stream())
    _check(st, "bla_decay_core_forward")
    return o, den


def sa_core_forward(shape: Shape, q, k, v, o=None, ws=None):
    """The bidirectional softmax attention of the SA blocks (Eq. 1, see gbla.h): returns o."""
    if o is None:
        o = torch.empty_like(q)
    if ws is None:
        ws = workspace(shape, GBLA_OP_SA_FORWARD, q.device)
    st = lib().sa_core_forward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(ws), ws.numel(),
                               _stream())
    _check(st, "sa_core_forward")
    return o


def bla_core_forward_noalloc(shape: Shape, q, k, v, g, o, den=None, state=None) -> int:
    """bla_core_forward with the library's fixed 64 MiB device scratch instead
    of a workspace, for callers that cannot allocate; o (and den / state when
    given) must already exist.  Returns the status (GBLA_ERR_WORKSPACE when the
    shape needs more scratch than the fixed array holds)."""
    return lib().bla_core_forward_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(o),
                                          _ptr(den), _ptr(state), _stream())


def bla_core_backward(shape: Shape, q, k, v, g, d_o, ws=None):
    """Backward of bla_core_forward for <d_o, o>: returns (dq, dk, dv, dg)."""
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dg = torch.empty(rows(shape), shape.H, dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(shape, GBLA_OP_CORE_BACKWARD, q.device)
    st = lib().bla_core_backward(ctypes.byref(shape), _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(d_o), _ptr(dq),
                                 _ptr(dk), _ptr(dv), _ptr(dg), _ptr(ws), ws.numel(), _stream())
    _check(st, "bla_core_backward")
    return dq, dk, dv, dg


def gbla_check_device_status(ws: torch.Tensor) -> int:
    return lib().gbla_check_device_status(_ptr(ws), _stream())


def bla_core_noalloc_check_device_status() -> int:
    """The error word of the last bla_core_forward_noalloc call on the current device."""
    return lib().bla_core_noalloc_check_device_status(_stream())


def gbla_diag_bounded_wait(ws: torch.Tensor, polls: int = 4096) -> int:
    """Runs the kernels' bounded mbarrier wait out on purpose (see gbla.h)."""
    return lib().gbla_diag_bounded_wait(_ptr(ws), ws.numel(), polls, _stream())


def gbla_set_kernel_policy(policy: int) -> None:
    """GBLA_POLICY_AUTO (default), GBLA_POLICY_TC or GBLA_POLICY_MMA for this thread's later calls (see gbla.h)."""
    _check(lib().gbla_set_kernel_policy(policy), "gbla_set_kernel_policy")


def gbla_profiling_enable(on: bool) -> None:
    lib().gbla_profiling_enable(1 if on else 0)


def gbla_profiling_read(cap: int = 4096) -> list[tuple[str, float]]:
    """(launch name, milliseconds) for every launch since the last read."""
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_float * cap)()
    n = lib().gbla_profiling_read(names, ms, cap)
    return [(names[i].decode(), float(ms[i])) for i in range(min(n, cap))]
