"""bla_core_forward_noalloc, the core forward for callers that cannot
allocate device memory (a plugin inside a framework that owns every device
buffer, a serving loop where an allocation would stall the other streams):
its scratch is a fixed 64 MiB device array inside the library instead of a
caller workspace.

Checks, through the C ABI, that two calls in a row (different inputs, and a
different shape in between) give the same o, den and state as the workspace
entry point bla_core_forward, within the bf16 / fp32 tolerances of the other
parity tests, and that a shape needing more scratch than the array holds is
refused with GBLA_ERR_WORKSPACE.  The file is named so that pytest collects it
last; it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from generative_retrieval_encoder_gb300 import build, gbla
from gbla_cases import TOL, core_case, f64, max_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    gbla.lib()


def _both(dtype, B, L, H, dh, seed, lengths=None):
    shape, D, R, _, _ = core_case(dtype, B, L, H, dh, seed=seed, lengths=lengths)
    ref = gbla.bla_core_forward(shape, D["q"], D["k"], D["v"], D["g"], den=True, state=True)
    o = torch.full_like(D["q"], float("nan"))
    den = torch.full_like(ref[1], float("nan"))
    state = torch.full_like(ref[2], float("nan"))
    st = gbla.bla_core_forward_noalloc(shape, D["q"], D["k"], D["v"], D["g"], o, den, state)
    torch.cuda.synchronize()
    assert st == gbla.GBLA_OK, gbla.lib().gbla_status_string(st)
    tol = TOL[dtype]
    assert max_err(f64(o), f64(ref[0]), scale=np.abs(R["v"]).max()) <= tol
    assert max_err(f64(den), f64(ref[1])) <= tol
    assert max_err(f64(state), f64(ref[2])) <= tol


@pytest.mark.parametrize("dtype,dh", [("bf16", 64), ("f32", 32)])
def test_noalloc_matches_workspace_entry_point_twice(dtype, dh):
    _both(dtype, 4, 1500, 2, dh, seed=31)
    _both(dtype, 1, 0, 2, dh, seed=32, lengths=[700, 1, 0, 2048])  # second call, other shape and inputs
    _both(dtype, 4, 1500, 2, dh, seed=33)


def test_noalloc_refuses_shapes_beyond_its_scratch():
    shape = gbla.make_shape(1024, 64, 64, 16, 128)  # 16384 (sequence, head) states of 128 x 136 floats
    assert gbla.gbla_validate_shape(shape) == gbla.GBLA_OK
    assert gbla.gbla_workspace_size(shape, gbla.GBLA_OP_CORE_FORWARD) > gbla.NOALLOC_SCRATCH_BYTES
    t = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    g = torch.empty(16, dtype=torch.float32, device="cuda")
    st = gbla.bla_core_forward_noalloc(shape, t, t, t, g, t)
    assert st == gbla.GBLA_ERR_WORKSPACE
