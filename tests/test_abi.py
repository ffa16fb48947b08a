"""The C-ABI library loads, exports every symbol include/gbla.h declares, and
rejects bad arguments on the host with a status before launching anything
(no GPU needed for any of these)."""
import ctypes
import os
import re

import pytest

from generative_retrieval_encoder_gb300 import build, gbla

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return gbla.lib()


def header_functions():
    src = open(os.path.join(ROOT, "include", "gbla.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M))


def test_library_exports_every_declared_symbol(L):
    names = header_functions()
    assert {"gbla_forward", "gbla_backward", "bla_core_forward", "bla_core_backward"} <= names
    for n in names:
        assert hasattr(L, n), n
    assert set(gbla.EXPORTS) == names


def test_status_strings_and_version(L):
    for s in (0, -1, -2, -3, -4, -5, -6):
        assert L.gbla_status_string(s).startswith(b"GBLA_")
    assert L.gbla_version() >= 100


def test_shape_validation(L):
    ok = gbla.make_shape(32, 2048, 512, 8, 64)
    assert gbla.gbla_validate_shape(ok) == gbla.GBLA_OK
    assert gbla.gbla_validate_shape(gbla.make_shape(2, 256, 64, 2, 32, dtype="f32")) == gbla.GBLA_OK
    assert gbla.gbla_validate_shape(gbla.make_shape(1, 16, 64, 1, 48)) == gbla.GBLA_ERR_UNSUPPORTED
    assert gbla.gbla_validate_shape(gbla.make_shape(1, 16, 64, 1, 6, dtype="f32")) == gbla.GBLA_ERR_UNSUPPORTED
    assert gbla.gbla_validate_shape(gbla.make_shape(0, 16, 64, 1, 64)) == gbla.GBLA_ERR_INVALID_ARG
    assert gbla.gbla_validate_shape(gbla.make_shape(1, 0, 64, 1, 64)) == gbla.GBLA_ERR_INVALID_ARG
    bad = gbla.make_shape(1, 16, 64, 1, 64)
    bad.gate = 7
    assert gbla.gbla_validate_shape(bad) == gbla.GBLA_ERR_INVALID_ARG
    both = gbla.make_shape(1, 16, 64, 1, 64)
    both.cu_seqlens, both.num_seqs, both.seq_lens = 256, 1, 512  # fake device addresses, never read
    assert gbla.gbla_validate_shape(both) == gbla.GBLA_ERR_INVALID_ARG
    vb = gbla.make_shape(2, 16, 64, 1, 64)
    vb.cu_seqlens, vb.num_seqs = 256, 1
    assert gbla.gbla_validate_shape(vb) == gbla.GBLA_ERR_INVALID_ARG  # varlen needs B == 1


def test_workspace_sizes_grow_with_shape(L):
    small = gbla.make_shape(2, 256, 64, 2, 32)
    big = gbla.make_shape(32, 2048, 512, 8, 64)
    for op in range(4):
        assert 0 < gbla.gbla_workspace_size(small, op) < gbla.gbla_workspace_size(big, op)
    assert gbla.gbla_workspace_size(small, 9) == 0
    assert gbla.gbla_saved_size(big) > 32 * 2048 * (512 + 4 * 512) * 2


def test_host_argument_errors_launch_nothing(L):
    """Null / misaligned pointers, too-small or misaligned workspaces and
    unsupported layer widths come back as statuses (nothing reaches CUDA)."""
    s = gbla.make_shape(2, 64, 64, 2, 32)
    fake = ctypes.c_void_p(1 << 20)       # aligned, never dereferenced: host checks fail first
    odd = ctypes.c_void_p((1 << 20) + 2)  # misaligned
    n = gbla.gbla_workspace_size(s, gbla.GBLA_OP_FORWARD)
    args = [fake] * 11
    st = L.gbla_forward(ctypes.byref(s), None, *args, fake, n, None)
    assert st == gbla.GBLA_ERR_INVALID_ARG
    st = L.gbla_forward(ctypes.byref(s), odd, *args, fake, n, None)
    assert st == gbla.GBLA_ERR_INVALID_ARG
    st = L.gbla_forward(ctypes.byref(s), fake, *args, fake, n - 1, None)
    assert st == gbla.GBLA_ERR_WORKSPACE
    st = L.gbla_forward(ctypes.byref(s), fake, *args, ctypes.c_void_p((1 << 20) + 16), n, None)
    assert st == gbla.GBLA_ERR_WORKSPACE
    st = L.gbla_forward(ctypes.byref(s), fake, *args, None, n, None)
    assert st == gbla.GBLA_ERR_WORKSPACE
    s2 = gbla.make_shape(2, 64, 96, 2, 32)  # d % 64 != 0 on the bf16 path
    st = L.gbla_forward(ctypes.byref(s2), fake, *args, fake, 1 << 30, None)
    assert st == gbla.GBLA_ERR_UNSUPPORTED
    n = gbla.gbla_workspace_size(s, gbla.GBLA_OP_CORE_FORWARD)
    st = L.bla_core_forward(ctypes.byref(s), fake, fake, None, fake, fake, None, None, fake, n, None)
    assert st == gbla.GBLA_ERR_INVALID_ARG
    n = gbla.gbla_workspace_size(s, gbla.GBLA_OP_CORE_BACKWARD)
    st = L.bla_core_backward(ctypes.byref(s), *[fake] * 9, fake, n - 256, None)
    assert st == gbla.GBLA_ERR_WORKSPACE
    n = gbla.gbla_workspace_size(s, gbla.GBLA_OP_BACKWARD)
    st = L.gbla_backward(ctypes.byref(s), *[fake] * 10, None, fake, fake, *[None] * 9, fake, n, None)
    assert st == gbla.GBLA_ERR_INVALID_ARG  # saved missing
    assert L.gbla_check_device_status(None, None) == gbla.GBLA_ERR_WORKSPACE


def test_decay_and_sa_entry_points_host_errors(L):
    """bla_decay_core_forward and sa_core_forward: workspace sizes that grow
    with the shape, and null or misaligned pointers, short workspaces and
    unsupported shapes refused as statuses before any CUDA call."""
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 2)
    s = gbla.make_shape(2, 300, 128, 2, 64)
    big = gbla.make_shape(8, 4096, 512, 8, 64)
    for op in (gbla.GBLA_OP_DECAY_FORWARD, gbla.GBLA_OP_SA_FORWARD):
        assert 0 < gbla.gbla_workspace_size(s, op) <= gbla.gbla_workspace_size(big, op)
    n = gbla.gbla_workspace_size(s, gbla.GBLA_OP_SA_FORWARD)
    assert L.sa_core_forward(ctypes.byref(s), None, fake, fake, fake, fake, n, None) == gbla.GBLA_ERR_INVALID_ARG
    assert L.sa_core_forward(ctypes.byref(s), fake, fake, odd, fake, fake, n, None) == gbla.GBLA_ERR_INVALID_ARG
    assert L.sa_core_forward(ctypes.byref(s), fake, fake, fake, None, fake, n, None) == gbla.GBLA_ERR_INVALID_ARG
    assert L.sa_core_forward(ctypes.byref(s), fake, fake, fake, fake, fake, n - 1, None) == gbla.GBLA_ERR_WORKSPACE
    assert L.sa_core_forward(ctypes.byref(s), fake, fake, fake, fake, None, n, None) == gbla.GBLA_ERR_WORKSPACE
    for bad in (gbla.make_shape(2, 300, 64, 2, 32), gbla.make_shape(2, 300, 128, 2, 64, dtype="f32")):
        st = L.sa_core_forward(ctypes.byref(bad), fake, fake, fake, fake, fake, 1 << 30, None)
        assert st == gbla.GBLA_ERR_UNSUPPORTED  # bf16 and d_h = 64 only
    n = gbla.gbla_workspace_size(s, gbla.GBLA_OP_DECAY_FORWARD)
    args = lambda q=fake, lam=fake: (q, fake, fake, fake, lam, fake, None)
    assert L.bla_decay_core_forward(ctypes.byref(s), *args(lam=None), fake, n, None) == gbla.GBLA_ERR_INVALID_ARG
    assert L.bla_decay_core_forward(ctypes.byref(s), *args(q=odd), fake, n, None) == gbla.GBLA_ERR_INVALID_ARG
    assert L.bla_decay_core_forward(ctypes.byref(s), *args(), fake, n - 1, None) == gbla.GBLA_ERR_WORKSPACE
    s32 = gbla.make_shape(2, 300, 64, 2, 32)
    st = L.bla_decay_core_forward(ctypes.byref(s32), *args(), fake, 1 << 30, None)
    assert st == gbla.GBLA_ERR_UNSUPPORTED


def test_diag_and_noalloc_host_errors(L):
    """Host-side errors of the diagnostic and the no-allocation entry points:
    statuses, no launch, no out-of-range access of the per-device address
    cache (which is keyed by device, with no fixed device count)."""
    fake = ctypes.c_void_p(1 << 20)
    assert L.gbla_diag_bounded_wait(None, 1 << 20, 16, None) == gbla.GBLA_ERR_WORKSPACE
    assert L.gbla_diag_bounded_wait(ctypes.c_void_p((1 << 20) + 16), 1 << 20, 16, None) == gbla.GBLA_ERR_WORKSPACE
    assert L.gbla_diag_bounded_wait(fake, 8, 16, None) == gbla.GBLA_ERR_WORKSPACE
    assert L.gbla_diag_bounded_wait(fake, 1 << 20, 0, None) == gbla.GBLA_ERR_INVALID_ARG
    assert L.gbla_diag_bounded_wait(fake, 1 << 20, (1 << 20) + 1, None) == gbla.GBLA_ERR_INVALID_ARG
    big = gbla.make_shape(1024, 64, 64, 16, 128)
    st = L.bla_core_forward_noalloc(ctypes.byref(big), fake, fake, fake, fake, fake, None, None, None)
    assert st == gbla.GBLA_ERR_WORKSPACE  # needs more than the fixed array; refused before any CUDA call
    small = gbla.make_shape(2, 64, 64, 2, 32)
    st = L.bla_core_forward_noalloc(ctypes.byref(small), None, None, None, None, None, None, None, None)
    import torch
    if torch.cuda.is_available():  # the array's address is found, then the null pointers are refused
        assert st == gbla.GBLA_ERR_INVALID_ARG
    else:  # no device: the address lookup fails and is reported, nothing else runs
        assert st == gbla.GBLA_ERR_CUDA
        assert L.bla_core_noalloc_check_device_status(None) == gbla.GBLA_ERR_CUDA
