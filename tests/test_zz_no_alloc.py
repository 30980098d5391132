"""blr_forward_noalloc, the forward pass for callers that cannot allocate.

Some callers of this library cannot call cudaMalloc (for example a plugin
inside an application that owns every device allocation, or a real-time loop
with a fixed memory budget). blr_forward_noalloc serves them with a fixed
scratch array inside the library instead of a caller workspace. This file
checks it through the C ABI against blr_forward, the entry point with a
caller workspace, on calls in a row: both run the same kernels with the same
tile plans on the same data, so y must agree bit for bit, in overwrite and in
accumulate mode; y is also checked against the CPU oracle at the forward's
tolerance, and the array's own status word (blr_noalloc_check_status) must
read 0 after every call. A shape too large for the array is refused without
any GPU work. The file is collected last so that a run that stops at the
first failure has already run every other test; it passes alone too.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from binary_rank_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-3


def _inputs(name, M, d_in, d_out, r, priors=False):
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r), with_priors=priors)
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).cuda() for k, v in t.items()}
    return t, d


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.parametrize("accumulate", [False, True])
def test_noalloc_matches_workspace_forward_twice(accumulate):
    import binary_rank_linear_gb300 as blr
    lib = blr.load()
    assert hasattr(lib, "blr_forward_noalloc") and hasattr(lib, "blr_noalloc_check_status")
    shapes = [("small", 300, 320, 448, 96), ("attn", 513, 512, 640, 256)]
    for name, M, d_in, d_out, r in shapes:  # calls in a row, different shapes and data
        t, d = _inputs(name, M, d_in, d_out, r, priors=accumulate)
        bu, bv = blr.pack_signs(d["su"]), blr.pack_signs(d["sv"])
        start = d["y_prior"] if accumulate else torch.full((M, d_out), float("nan"), device="cuda")
        y_na = start.clone()
        blr.forward_noalloc(d["x"], bu, bv, d["g"], d["l"], d["h"], y_na, accumulate=accumulate)
        assert blr.noalloc_check_status() == 0
        ws = blr.alloc_workspace(M, d_in, d_out, r)
        y_ws = start.clone()
        blr.forward(d["x"], bu, bv, d["g"], d["l"], d["h"], y_ws, ws, accumulate=accumulate)
        assert blr.check_status(ws) == 0
        a, b = y_na.cpu().numpy(), y_ws.cpu().numpy()
        assert np.isfinite(a).all()
        assert np.array_equal(a, b), f"{name}: max |diff| {np.max(np.abs(a - b))}"
        obu, obv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
        want = oracle.forward(t["x"], obu, obv, t["g"], t["l"], t["h"],
                              y_prior=t["y_prior"] if accumulate else None)["y"]
        assert oracle.rel_err(a, want) <= TOL_OUT


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
