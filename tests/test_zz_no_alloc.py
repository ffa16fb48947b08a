"""bla_core_forward_noalloc, the core forward for callers that cannot
allocate device memory (a plugin inside a framework that owns every device
buffer, a serving loop where an allocation would stall the other streams):
its scratch is a fixed 64 MiB device array inside the library instead of a
caller workspace.

Checks, through the C ABI, that two calls in a row (different inputs, and a
different shape in between) give the same o, den and state as the workspace
entry point bla_core_forward, within the bf16 / fp32 tolerances of the other
parity tests, and as the fp64 oracle; the d_h = 128 layout (the largest state
per head) under the 64 MiB limit; that bad cu_seqlens are reported through the
array's own error word; and that a shape needing more scratch than the array
holds is refused with GBLA_ERR_WORKSPACE.  The file is named so that pytest
collects it last; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

import oracle
from generative_retrieval_encoder_gb300 import build, gbla
from gbla_cases import TOL, core_case, f64, max_err, valid_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gbla.lib()


def _both(dtype, B, L, H, dh, seed, lengths=None):
    shape, D, R, (st, ln), T = core_case(dtype, B, L, H, dh, seed=seed, lengths=lengths)
    assert gbla.gbla_workspace_size(shape, gbla.GBLA_OP_CORE_FORWARD) <= gbla.NOALLOC_SCRATCH_BYTES
    ref = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"], den=True, state=True)
    o = torch.full_like(D["q"], float("nan"))
    den = torch.full_like(ref[1], float("nan"))
    state = torch.full_like(ref[2], float("nan"))
    s = gbla.bla_core_forward_noalloc(shape, D["q"], D["k"], D["v"], D["g"], o, den, state)
    torch.cuda.synchronize()
    assert s == gbla.GBLA_OK, gbla.lib().gbla_status_string(s)
    assert gbla.bla_core_noalloc_check_device_status() == gbla.GBLA_OK
    tol = TOL[dtype]
    vmax = np.abs(R["v"]).max()
    # against the workspace entry point
    assert max_err(f64(o), f64(ref[0]), scale=vmax) <= tol
    assert max_err(f64(den), f64(ref[1])) <= tol
    assert max_err(f64(state), f64(ref[2])) <= tol
    # against the fp64 oracle
    ro, rden, rstate = oracle.core_forward(R["q"], R["k"], R["v"], R["g"], st, ln, shape.H, dh)
    m = valid_rows(st, ln, T)
    assert max_err(f64(o)[m], ro[m], scale=vmax) <= tol
    assert max_err(f64(den)[m], rden[m]) <= tol
    nz = ln > 0
    assert max_err(f64(state)[nz], rstate[nz]) <= tol


@pytest.mark.parametrize("dtype,dh", [("bf16", 64), ("f32", 32), ("bf16", 128)])
def test_noalloc_matches_workspace_entry_point_and_oracle_twice(dtype, dh):
    _both(dtype, 4, 1500, 2, dh, seed=31)
    _both(dtype, 1, 0, 2, dh, seed=32, lengths=[700, 1, 0, 2048])  # second call, other shape and inputs
    _both(dtype, 4, 1500, 2, dh, seed=33)


def test_noalloc_reports_bad_cu_seqlens_through_its_error_word():
    _, D, _, _, _ = core_case("bf16", 1, 10, 1, 64, seed=3)
    o = torch.empty_like(D["q"])
    for cu in ([0, 5, 3, 10], [1, 5, 10]):
        s = gbla.make_shape(1, 10, 64, 1, 64, cu_seqlens=torch.tensor(cu, dtype=torch.int32).cuda())
        assert gbla.bla_core_forward_noalloc(s, D["q"], D["k"], D["v"], D["g"], o) == gbla.GBLA_OK
        assert gbla.bla_core_noalloc_check_device_status() == gbla.GBLA_ERR_DEVICE_CHECK, cu
    # the next good call clears the word
    s = gbla.make_shape(1, 10, 64, 1, 64, cu_seqlens=torch.tensor([0, 4, 10], dtype=torch.int32).cuda())
    assert gbla.bla_core_forward_noalloc(s, D["q"], D["k"], D["v"], D["g"], o) == gbla.GBLA_OK
    assert gbla.bla_core_noalloc_check_device_status() == gbla.GBLA_OK


def test_noalloc_refuses_shapes_beyond_its_scratch():
    shape = gbla.make_shape(1024, 64, 64, 16, 128)  # 16384 (sequence, head) states of 128 x 136 floats
    assert gbla.gbla_validate_shape(shape) == gbla.GBLA_OK
    assert gbla.gbla_workspace_size(shape, gbla.GBLA_OP_CORE_FORWARD) > gbla.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    g = torch.empty(16, dtype=torch.float32, device="cuda")
    st = gbla.bla_core_forward_noalloc(shape, t, t, t, g, t)
    assert st == gbla.GBLA_ERR_WORKSPACE
