"""GPU parity of plane_linear (blr_plane_linear) against the CPU f64 oracle.

Tolerance: normwise relative error <= 2e-3, the layer's own bound for y and
dx (x is staged to f16, relative rounding 2^-11 per element, and the plane is
f16 exactly). On the integer grid (x in {-2..2}, plane in {-1, -1/2, 1/2, 1},
scale 1) every staged value and partial sum is exact in f32, so y must equal
the oracle bit for bit in both directions; that pins the operand roles, the
K-major/MN-major tiles and the output layout.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import binary_rank_linear_gb300 as blr
    blr.load()


def _run(x, plane, transpose=False, y_prior=None, scale=1.0):
    import binary_rank_linear_gb300 as blr
    ntok = x.shape[0]
    n, k = plane.shape
    nout = k if transpose else n
    ws = blr.alloc_plane_workspace(ntok, n, k)
    dx = torch.from_numpy(np.ascontiguousarray(x, np.float32)).cuda()
    dp = torch.from_numpy(np.ascontiguousarray(plane, np.float16)).cuda()
    y = (torch.from_numpy(y_prior.astype(np.float32)).cuda() if y_prior is not None
         else torch.full((ntok, nout), float("nan"), device="cuda"))
    blr.plane_linear(dx, dp, y, ws, transpose=transpose, accumulate=y_prior is not None, scale=scale)
    assert blr.check_status(ws) == 0
    return y.cpu().numpy()


SHAPES = [(128, 256, 256), (70, 384, 256), (1, 64, 96), (333, 160, 288), (513, 1024, 640), (4097, 512, 1056)]


@pytest.mark.parametrize("ntok,n,k", SHAPES[:4])
@pytest.mark.parametrize("transpose", [False, True])
def test_plane_integer_grid_bit_exact(ntok, n, k, transpose):
    rng = np.random.default_rng(ntok + n + k)
    plane = rng.choice(np.array([-1.0, -0.5, 0.5, 1.0], np.float16), size=(n, k))
    x = rng.integers(-2, 3, size=(ntok, n if transpose else k)).astype(np.float32)
    got = _run(x, plane, transpose)
    want = oracle.plane_linear(x, plane, transpose=transpose)
    assert np.array_equal(got, want.astype(np.float32))


@pytest.mark.parametrize("ntok,n,k", SHAPES)
@pytest.mark.parametrize("transpose,scale,mag", [(False, 1.0, 1.0), (True, 1024.0, 1e-4), (True, 1.0, 1.0)])
def test_plane_parity(ntok, n, k, transpose, scale, mag):
    rng = np.random.default_rng(7 * ntok + n)
    plane = (rng.standard_normal((n, k)) * 0.05).astype(np.float16)
    x = (rng.standard_normal((ntok, n if transpose else k)) * mag).astype(np.float32)
    got = _run(x, plane, transpose, scale=scale)
    want = oracle.plane_linear(x, plane, transpose=transpose)
    e = oracle.rel_err(got, want)
    assert np.isfinite(e) and e <= TOL, e


@pytest.mark.parametrize("transpose", [False, True])
def test_plane_accumulate(transpose):
    rng = np.random.default_rng(3)
    ntok, n, k = 300, 320, 192
    plane = (rng.standard_normal((n, k)) * 0.05).astype(np.float16)
    x = rng.standard_normal((ntok, n if transpose else k)).astype(np.float32)
    prior = rng.standard_normal((ntok, k if transpose else n)).astype(np.float32)
    got = _run(x, plane, transpose, y_prior=prior)
    want = oracle.plane_linear(x, plane, transpose=transpose, y_prior=prior)
    assert oracle.rel_err(got, want) <= TOL


def test_plane_attn_sized():
    """An attention-projection-sized frozen linear (8192 tokens, 4096 -> 4096)
    on sampled rows, both directions."""
    rng = np.random.default_rng(11)
    ntok, n, k = 8192, 4096, 4096
    plane = (rng.standard_normal((n, k)) * 0.02).astype(np.float16)
    x = rng.standard_normal((ntok, k)).astype(np.float32)
    rows = np.unique(np.concatenate([[0, ntok - 1], rng.choice(ntok, 40, replace=False)]))
    for transpose in (False, True):
        got = _run(x, plane, transpose)
        want = oracle.plane_linear(x[rows], plane, transpose=transpose)
        assert oracle.rel_err(got[rows], want) <= TOL, transpose
