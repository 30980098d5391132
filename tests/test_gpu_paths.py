"""GPU parity of multi-path layers (blr_forward_paths / blr_backward_paths)
against the CPU f64 oracle: y and dx sum over the paths (tolerance 2e-3),
each path keeps its own dh, dl, dg (5e-3), as the single-path calls do."""
import numpy as np
import pytest
import torch

import oracle
from binary_rank_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import binary_rank_linear_gb300 as blr
    blr.load()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run_paths(x, dy, paths, gscale=0.0, y_prior=None, dx_prior=None):
    import binary_rank_linear_gb300 as blr
    M, d_in = x.shape
    d_out, r = paths[0]["su"].shape
    dp = [{"bu": blr.pack_signs(_dev(p["su"])), "bv": blr.pack_signs(_dev(p["sv"])), "g": _dev(p["g"]),
           "l": _dev(p["l"]), "h": _dev(p["h"])} for p in paths]
    grads = [{"dg": torch.zeros(d_in, device="cuda"), "dl": torch.zeros(r, device="cuda"),
              "dh": torch.zeros(d_out, device="cuda")} for _ in paths]
    ws = blr.alloc_paths_workspace(len(paths), M, d_in, d_out, r)
    y = _dev(y_prior) if y_prior is not None else torch.full((M, d_out), float("nan"), device="cuda")
    dx = _dev(dx_prior) if dx_prior is not None else torch.full((M, d_in), float("nan"), device="cuda")
    blr.forward_paths(_dev(x), dp, y, ws, accumulate=y_prior is not None)
    blr.backward_paths(_dev(x), _dev(dy), dp, dx, grads, ws, gscale=gscale, accumulate=dx_prior is not None)
    for p in range(len(paths)):
        assert blr.check_status(blr.path_workspace(ws, p, M, d_in, d_out, r)) == 0
    return y.cpu().numpy(), dx.cpu().numpy(), [{k: v.cpu().numpy() for k, v in q.items()} for q in grads], ws


def _oracle_paths(x, dy, paths, y_prior=None, dx_prior=None):
    op = [{"bu": oracle.pack_signs(p["su"]), "bv": oracle.pack_signs(p["sv"]), "g": p["g"], "l": p["l"],
           "h": p["h"]} for p in paths]
    return oracle.forward_paths(x, op, y_prior), oracle.backward_paths(x, dy, op, dx_prior)


def _check(x, dy, paths, got, y_prior=None, dx_prior=None):
    y, dx, grads, _ = got
    fw, bw = _oracle_paths(x, dy, paths, y_prior, dx_prior)
    assert oracle.rel_err(y, fw["y"]) <= 2e-3
    assert oracle.rel_err(dx, bw["dx"]) <= 2e-3
    for q, want in zip(grads, bw["paths"]):
        for k in ("dg", "dl", "dh"):
            assert oracle.rel_err(q[k], want[k]) <= 5e-3, k


def test_pages_two_paths():
    """The page's two-path layer: d_out 256, d_in 384, r 128, 70 tokens, gscale 1024."""
    p0, p1 = wl.pages_case(0), wl.pages_case(1)
    got = _run_paths(p0["x"], p0["dy"], [p0, p1], gscale=1024.0)
    _check(p0["x"], p0["dy"], [p0, p1], got)


def _paths_inputs(P, M, d_in, d_out, r):
    """P paths with their own signs and vectors on one x and dy."""
    base = wl.make_inputs(wl.WORKLOADS["small"].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    rng = np.random.default_rng(M + P)
    paths = []
    for _ in range(P):
        q = dict(base)
        q["su"] = np.where(rng.random(base["su"].shape) < 0.5, 1.0, -1.0).astype(np.float32)
        q["sv"] = np.where(rng.random(base["sv"].shape) < 0.5, 1.0, -1.0).astype(np.float32)
        q["g"] = (1 + 0.1 * rng.standard_normal(d_in)).astype(np.float32)
        q["h"] = (1 + 0.1 * rng.standard_normal(d_out)).astype(np.float32)
        q["l"] = (base["l"] * rng.uniform(0.5, 1.5, r)).astype(np.float32)
        paths.append(q)
    return base["x"], base["dy"], paths


@pytest.mark.parametrize("P,M,d_in,d_out,r", [(3, 300, 320, 448, 96), (2, 4600, 1024, 1568, 256),
                                              (4, 129, 192, 96, 64)])
def test_paths_parity(P, M, d_in, d_out, r):
    """P paths with their own signs and vectors on one x and dy."""
    x, dy, paths = _paths_inputs(P, M, d_in, d_out, r)
    _check(x, dy, paths, _run_paths(x, dy, paths))


@pytest.mark.parametrize("P,M,d_in,d_out,r", [(2, 300, 320, 448, 96), (3, 4600, 1024, 1568, 256),
                                              (10, 129, 192, 96, 64), (2, 8192, 512, 4096, 128),
                                              (9, 4600, 256, 1568, 256), (64, 17, 64, 96, 64), (3, 1, 64, 64, 64),
                                              (2, 33, 65536, 64, 64), (2, 40, 64, 32768, 128)])
def test_grouped_paths_match_the_loop(monkeypatch, P, M, d_in, d_out, r):
    """The grouped passes (one launch per stage for up to eight paths; nine
    or ten paths take two groups, the second adding into y and dx, and the
    most paths a call takes, 64, eight groups; CTA-pair tiles at 4600 tokens;
    a single token; the widest d_in and d_out the shape rule admits) against each
    path's single-path calls in turn (BLR_PATHS=loop): y and dx receive the
    same contributions in the same order, and each path's dh, dl, dg the same
    partial sums up to their grouping; both against the oracle."""
    x, dy, paths = _paths_inputs(P, M, d_in, d_out, r)
    got_g = _run_paths(x, dy, paths)
    monkeypatch.setenv("BLR_PATHS", "loop")
    got_l = _run_paths(x, dy, paths)
    assert oracle.rel_err(got_g[0], got_l[0]) <= 1e-6
    assert oracle.rel_err(got_g[1], got_l[1]) <= 1e-6
    for qg, ql in zip(got_g[2], got_l[2]):
        for k in ("dg", "dl", "dh"):
            assert oracle.rel_err(qg[k], ql[k]) <= 1e-5, k
    _check(x, dy, paths, got_g)


@pytest.mark.parametrize("P,M,d_in,d_out,r", [(3, 4600, 1024, 1568, 256), (8, 129, 192, 96, 64),
                                              (2, 2000, 2048, 512, 512)])
def test_grouped_paths_stage_x_in_kernel(monkeypatch, P, M, d_in, d_out, r):
    """The grouped forward with every path's x staged inside the a-product
    (BLR_STAGE=kernel; by default for x of 64 MB or more): the stagers take
    the paths' token tiles path-major, each with its own g, x16 and row
    counters. Against the per-path loop with the same staging and against
    the oracle."""
    monkeypatch.setenv("BLR_STAGE", "kernel")
    x, dy, paths = _paths_inputs(P, M, d_in, d_out, r)
    got_g = _run_paths(x, dy, paths)
    monkeypatch.setenv("BLR_PATHS", "loop")
    got_l = _run_paths(x, dy, paths)
    assert oracle.rel_err(got_g[0], got_l[0]) <= 1e-6
    assert oracle.rel_err(got_g[1], got_l[1]) <= 1e-6
    _check(x, dy, paths, got_g)


def test_grouped_paths_integer_grid():
    """Bit-exact on a grid of small multiples of powers of two (every staged
    operand exact in f16, every product and partial sum exact in f32): three
    paths whose y and dx contributions are added by reduce-add stores in path
    order; a contribution lost to a store that overtook an add, or added
    twice, would show."""
    import binary_rank_linear_gb300 as blr
    M, d_in, d_out, r, P = 2000, 256, 1024, 128, 3
    rng = np.random.default_rng(11)
    x = rng.integers(-2, 3, (M, d_in)).astype(np.float32)
    dy = rng.integers(-2, 3, (M, d_out)).astype(np.float32)
    paths = []
    for _ in range(P):
        paths.append({"su": np.where(rng.random((d_out, r)) < 0.5, 1.0, -1.0).astype(np.float32),
                      "sv": np.where(rng.random((d_in, r)) < 0.5, 1.0, -1.0).astype(np.float32),
                      "g": rng.choice([0.5, 1.0, 2.0], d_in).astype(np.float32),
                      "l": rng.choice([0.25, 0.5], r).astype(np.float32),
                      "h": rng.choice([0.5, 1.0], d_out).astype(np.float32)})
    y, dx, grads, _ = _run_paths(x, dy, paths, gscale=1.0)
    fw, bw = _oracle_paths(x, dy, paths)
    assert np.array_equal(y, fw["y"].astype(np.float32))
    assert np.array_equal(dx, bw["dx"].astype(np.float32))
    for q, want in zip(grads, bw["paths"]):
        for k in ("dg", "dl"):
            assert np.array_equal(q[k], want[k].astype(np.float32)), k
        # dh reads the f16 c tape, whose larger values are rounded
        assert oracle.rel_err(q["dh"], want["dh"]) <= 1e-3
    del blr


def test_paths_accumulate_and_sign_grads():
    """Priors in y and dx (accumulate mode), and each path's sign gradients
    from its slice of the workspace."""
    import binary_rank_linear_gb300 as blr
    p0, p1 = wl.pages_case(0), wl.pages_case(1)
    rng = np.random.default_rng(4)
    yp = rng.standard_normal((70, 256)).astype(np.float32)
    dxp = rng.standard_normal((70, 384)).astype(np.float32)
    got = _run_paths(p0["x"], p0["dy"], [p0, p1], y_prior=yp, dx_prior=dxp)
    _check(p0["x"], p0["dy"], [p0, p1], got, y_prior=yp, dx_prior=dxp)
    ws = got[3]
    for p, path in enumerate((p0, p1)):
        wsp = blr.path_workspace(ws, p, 70, 384, 256, 128)
        sws = blr.alloc_sign_workspace(70, 384, 256, 128)
        gu, gv = torch.empty(256, 128, device="cuda"), torch.empty(384, 128, device="cuda")
        blr.sign_grads(_dev(p0["x"]), _dev(path["g"]), _dev(path["l"]), gu, gv, wsp, sws)
        want = oracle.sign_grads(p0["x"], p0["dy"], oracle.pack_signs(path["su"]), oracle.pack_signs(path["sv"]),
                                 path["g"], path["l"], path["h"])
        assert oracle.rel_err(gu.cpu().numpy(), want["gu"]) <= 3e-3
        assert oracle.rel_err(gv.cpu().numpy(), want["gv"]) <= 3e-3
