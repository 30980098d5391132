"""GPU parity of the sign gradients G_U, G_V (blr_sign_grads) against the
CPU f64 oracle.

Tolerance: normwise relative error <= 3e-3, the bound of the page's own
device-vs-f64 check of the sign gradients (train_mm.rs, test
``blr_sign_grad_matches_host``). On the integer grid (x, dy in {-1, 0, 1},
g = h = 1, l a power of two) every f16 operand and every f32 partial sum is
exact, so G_U and G_V must match the oracle bit for bit; that pins the
transposed staging, the operand roles and the output layout.
"""
import numpy as np
import pytest
import torch

import oracle
from binary_rank_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_SIGN = 3e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import binary_rank_linear_gb300 as blr
    blr.load()


def _run(*a, **k):
    from blr_gpu_run import run_layer
    return run_layer(*a, sign=True, **k)


def _oracle(t, prior=None):
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    sg = oracle.sign_grads(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    if prior is not None:
        sg = {k: sg[k] + prior[k] for k in ("gu", "gv")}
    return sg


def _integer_grid(M, d_in, d_out, r, seed):
    rng = np.random.default_rng(seed)
    return {
        "x": rng.integers(-1, 2, size=(M, d_in)).astype(np.float32),
        "dy": rng.integers(-1, 2, size=(M, d_out)).astype(np.float32),
        "su": np.where(rng.random((d_out, r)) < 0.5, 1.0, -1.0).astype(np.float32),
        "sv": np.where(rng.random((d_in, r)) < 0.5, 1.0, -1.0).astype(np.float32),
        "g": np.ones(d_in, np.float32),
        "h": np.ones(d_out, np.float32),
        "l": rng.choice(np.array([0.5, 1.0, 2.0], np.float32), size=r),
    }


@pytest.mark.parametrize("gscale", [1.0, 0.0])
@pytest.mark.parametrize("M,d_in,d_out,r", [(128, 128, 128, 64), (200, 96, 160, 96), (70, 256, 64, 128),
                                            (333, 384, 256, 288)])
def test_sign_integer_grid_bit_exact(M, d_in, d_out, r, gscale):
    t = _integer_grid(M, d_in, d_out, r, seed=3 * M + r)
    out = _run(t, gscale=gscale)
    want = _oracle(t)
    assert out["status"] == 0
    assert np.array_equal(out["gu"], want["gu"].astype(np.float32))
    assert np.array_equal(out["gv"], want["gv"].astype(np.float32))


SHAPES = [
    ("tiny", 128, 256, 256, 64),
    ("small", 300, 320, 448, 96),
    ("small", 257, 352, 192, 160),
    ("attn", 513, 512, 640, 256),   # r = 256: the 256-rank tiles
    ("attn", 700, 384, 256, 416),   # ragged rank tile (416 = 256 + 160)
    ("ragged", 1, 128, 128, 64),
    ("ragged", 127, 256, 512, 128),
    ("ragged", 129, 192, 96, 64),
]


@pytest.mark.parametrize("name,M,d_in,d_out,r", SHAPES)
@pytest.mark.parametrize("gscale", [0.0, 1024.0])
def test_sign_parity_shapes(name, M, d_in, d_out, r, gscale):
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    if name == "ragged" and gscale > 0:
        gscale = 2.0 ** 30  # the dy ~ 1e-7 workload needs a large fixed scale
    out = _run(t, gscale=gscale)
    want = _oracle(t)
    assert out["status"] == 0, f"device status {out['status']:#x}"
    for k in ("gu", "gv"):
        e = oracle.rel_err(out[k], want[k])
        assert np.isfinite(e) and e <= TOL_SIGN, f"{k}: rel err {e:.3e}"


def test_sign_pages_case():
    """The page's sign-gradient test shape: d_out 256, d_in 384, r 128, 70
    tokens, gscale 1024, both paths."""
    for path in (0, 1):
        p = wl.pages_case(path)
        out = _run(p, gscale=1024.0)
        want = _oracle(p)
        assert out["status"] == 0
        for k in ("gu", "gv"):
            assert oracle.rel_err(out[k], want[k]) <= TOL_SIGN, (path, k)


def test_sign_accumulate():
    w = wl.WORKLOADS["small"].with_shape(M=260, d_in=256, d_out=320, r=128)
    t = wl.make_inputs(w)
    rng = np.random.default_rng(11)
    prior = {"gu": rng.standard_normal((320, 128)).astype(np.float32),
             "gv": rng.standard_normal((256, 128)).astype(np.float32)}
    out = _run(t, sign_prior=prior)
    want = _oracle(t, prior)
    assert out["status"] == 0
    for k in ("gu", "gv"):
        assert oracle.rel_err(out[k], want[k]) <= TOL_SIGN, k


def test_sign_deterministic():
    t = wl.make_inputs(wl.WORKLOADS["small"].with_shape(M=300, d_in=256, d_out=256, r=128))
    a, b = _run(t), _run(t)
    assert np.array_equal(a["gu"], b["gu"]) and np.array_equal(a["gv"], b["gv"])


def test_sign_outputs_stay_in_bounds():
    """Rows past d_out (d_in) of gu (gv) are never written."""
    import binary_rank_linear_gb300 as blr
    from blr_gpu_run import to_dev
    M, d_in, d_out, r = 90, 160, 96, 64
    t = wl.make_inputs(wl.WORKLOADS["tiny"].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    x, dy = to_dev(t["x"]), to_dev(t["dy"])
    g, l, h = to_dev(t["g"]), to_dev(t["l"]), to_dev(t["h"])
    bu, bv = blr.pack_signs(to_dev(t["su"])), blr.pack_signs(to_dev(t["sv"]))
    ws = blr.alloc_workspace(M, d_in, d_out, r)
    sws = blr.alloc_sign_workspace(M, d_in, d_out, r)
    blr.forward(x, bu, bv, g, l, h, torch.empty(M, d_out, device="cuda"), ws)
    z = lambda n: torch.zeros(n, device="cuda")  # noqa: E731
    blr.backward(x, dy, bu, bv, g, l, h, torch.empty(M, d_in, device="cuda"), z(d_in), z(r), z(d_out), ws)
    gu = torch.full((d_out + 5, r), 4321.0, device="cuda")
    gv = torch.full((d_in + 5, r), -99.0, device="cuda")
    blr.sign_grads(x, g, l, gu[:d_out], gv[:d_in], ws, sws)
    assert blr.check_status(ws) == 0
    assert torch.all(gu[d_out:] == 4321.0) and torch.all(gv[d_in:] == -99.0)
    want = _oracle(t)
    assert oracle.rel_err(gu[:d_out].cpu().numpy(), want["gu"]) <= TOL_SIGN


def test_sign_needs_backward():
    """Sign gradients read the backward's staging: a forward alone, or a new
    forward after the backward, is rejected."""
    import binary_rank_linear_gb300 as blr
    from blr_gpu_run import to_dev
    M, d_in, d_out, r = 64, 128, 128, 64
    t = wl.make_inputs(wl.WORKLOADS["tiny"].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    x, dy = to_dev(t["x"]), to_dev(t["dy"])
    g, l, h = to_dev(t["g"]), to_dev(t["l"]), to_dev(t["h"])
    bu, bv = blr.pack_signs(to_dev(t["su"])), blr.pack_signs(to_dev(t["sv"]))
    ws = blr.alloc_workspace(M, d_in, d_out, r)
    sws = blr.alloc_sign_workspace(M, d_in, d_out, r)
    gu, gv = torch.zeros(d_out, r, device="cuda"), torch.zeros(d_in, r, device="cuda")
    y = torch.empty(M, d_out, device="cuda")
    blr.forward(x, bu, bv, g, l, h, y, ws)
    with pytest.raises(blr.BlrError) as e:
        blr.sign_grads(x, g, l, gu, gv, ws, sws)
    assert e.value.code == blr.BLR_ERR_STATE
    z = lambda n: torch.zeros(n, device="cuda")  # noqa: E731
    blr.backward(x, dy, bu, bv, g, l, h, torch.empty(M, d_in, device="cuda"), z(d_in), z(r), z(d_out), ws)
    blr.sign_grads(x, g, l, gu, gv, ws, sws)
    blr.forward(x, bu, bv, g, l, h, y, ws)
    with pytest.raises(blr.BlrError) as e:
        blr.sign_grads(x, g, l, gu, gv, ws, sws)
    assert e.value.code == blr.BLR_ERR_STATE
    assert blr.check_status(ws) == 0


@pytest.mark.parametrize("name,M,d_in,d_out,r", [("tiny", 128, 256, 256, 64), ("small", 2048, 1024, 1024, 256)])
def test_sign_after_fused_small_backward(monkeypatch, name, M, d_in, d_out, r):
    """The fused small-M backward leaves the same staging behind."""
    monkeypatch.setenv("BLR_SMALL_PATH", "fused")
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t)
    want = _oracle(t)
    assert out["status"] == 0
    for k in ("gu", "gv"):
        assert oracle.rel_err(out[k], want[k]) <= TOL_SIGN, k


FULL = ["small", "attn", "ragged", "mlp_up", "mlp_down"]


@pytest.mark.parametrize("name", FULL)
def test_sign_full_size_workload(name):
    """Full-size workloads: sampled rows of G_U and G_V against exact oracle
    values, and on everything the trace identity
    sum_i S_U[i,k] G_U[i,k] = sum_j S_V[j,k] G_V[j,k] = l_k dl_k."""
    w = wl.WORKLOADS[name]
    t = wl.make_inputs(w)
    out = _run(t)
    assert out["status"] == 0
    assert np.isfinite(out["gu"]).all() and np.isfinite(out["gv"]).all()
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    rng = np.random.default_rng(w.wid + 17)
    ru = np.unique(np.concatenate([[0, w.d_out - 1], rng.choice(w.d_out, size=min(w.d_out, 48), replace=False)]))
    rv = np.unique(np.concatenate([[0, w.d_in - 1], rng.choice(w.d_in, size=min(w.d_in, 48), replace=False)]))
    smp = oracle.sign_grads_sampled(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"], ru, rv)
    assert oracle.rel_err(out["gu"][ru], smp["gu"]) <= TOL_SIGN
    assert oracle.rel_err(out["gv"][rv], smp["gv"]) <= TOL_SIGN
    # trace identity against the backward's dl (itself within 5e-3): an
    # error e |G| in G moves each column sum by at most e sqrt(rows) |G[:, k]|
    want = t["l"].astype(np.float64) * out["dl"].astype(np.float64)
    for key, s in (("gu", t["su"]), ("gv", t["sv"])):
        G = out[key].astype(np.float64)
        got = np.sum(s.astype(np.float64) * G, axis=0)
        slack = TOL_SIGN * np.sqrt(G.shape[0]) * np.linalg.norm(G) + 5e-3 * np.linalg.norm(want)
        assert np.linalg.norm(got - want) <= slack, key
