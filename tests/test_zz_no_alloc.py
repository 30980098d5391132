"""blr_forward_noalloc, the forward pass for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc (for example a plugin
inside an application that owns every device allocation, or a real-time loop
with a fixed memory budget). blr_forward_noalloc serves them with a fixed
scratch array inside the library instead of a caller workspace. This file
checks it through the C ABI against blr_forward, the entry point with a
caller workspace, on two calls in a row, and checks that a shape too large
for the array is refused without any GPU work. It is collected last so that
a run that stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from binary_rank_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-3


def _inputs(name, M, d_in, d_out, r):
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in t.items()}
    return t, d


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_noalloc_matches_workspace_forward_twice():
    import binary_rank_linear_gb300 as blr
    lib = blr.load()
    assert hasattr(lib, "blr_forward_noalloc")
    shapes = [("small", 300, 320, 448, 96), ("attn", 513, 512, 640, 256)]
    for name, M, d_in, d_out, r in shapes:  # two calls in a row, different shapes and data
        t, d = _inputs(name, M, d_in, d_out, r)
        bu, bv = blr.pack_signs(d["su"]), blr.pack_signs(d["sv"])
        y_na = torch.full((M, d_out), float("nan"), device="cuda")
        blr.forward_noalloc(d["x"], bu, bv, d["g"], d["l"], d["h"], y_na)
        ws = blr.alloc_workspace(M, d_in, d_out, r)
        y_ws = torch.full((M, d_out), float("nan"), device="cuda")
        blr.forward(d["x"], bu, bv, d["g"], d["l"], d["h"], y_ws, ws)
        torch.cuda.synchronize()
        a, b = y_na.cpu().numpy(), y_ws.cpu().numpy()
        assert np.isfinite(a).all()
        assert oracle.rel_err(a, b) <= TOL_OUT
        assert blr.check_status(ws) == 0


def test_noalloc_refuses_shapes_beyond_its_scratch():
    import binary_rank_linear_gb300 as blr
    lib = blr.load()
    fn = lib.blr_forward_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P]
    fn.restype = I
    fake = 1 << 20  # aligned, never dereferenced: the size check comes first
    rc = fn(fake, fake, fake, fake, fake, fake, fake, 0, 65536, 4096, 4096, 1024, None)
    assert rc == blr.BLR_ERR_WORKSPACE
