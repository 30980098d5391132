"""GPU parity: the CUDA path (through the C ABI) against the CPU f64 oracle.

Tolerances (normwise relative error, the page's metric): y and dx <= 2e-3;
dh, dl and dg <= 5e-3. Sign packing and expansion are bit-exact. On the
integer grid (x, dy in {-1, 0, 1}, g = h = 1, l a power of two) every f16
operand and every f32 partial sum is exact, so y and dx must match the oracle
bit for bit; that pins the bit-to-rank mappings and the GEMM data layout.
"""
import numpy as np
import pytest
import torch

import oracle
from binary_rank_linear_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL_OUT = 2e-3
TOL_GRAD = 5e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import binary_rank_linear_gb300 as blr
    blr.load()


def _run(*a, **k):
    from blr_gpu_run import run_layer
    return run_layer(*a, **k)


def _check_against_oracle(t, out, gscale_note="", y_prior=None, dx_prior=None, grad_prior=None):
    bu = oracle.pack_signs(t["su"])
    bv = oracle.pack_signs(t["sv"])
    assert np.array_equal(out["bu"], bu) and np.array_equal(out["bv"], bv)
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"], y_prior=y_prior)
    errs = {"y": oracle.rel_err(out["y"], fw["y"])}
    if "dx" in out:
        bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"], dx_prior=dx_prior)
        errs["dx"] = oracle.rel_err(out["dx"], bw["dx"])
        for k in ("dh", "dl", "dg"):
            want = bw[k] + (grad_prior[k] if grad_prior is not None else 0.0)
            errs[k] = oracle.rel_err(out[k], want)
    assert out["status"] == 0, f"device status {out['status']:#x}"
    for k, e in errs.items():
        tol = TOL_OUT if k in ("y", "dx") else TOL_GRAD
        assert np.isfinite(e) and e <= tol, f"{k}: rel err {e:.3e} > {tol} {gscale_note} {errs}"
    return errs


# --------------------------------------------------------- bit-exact parts --
@pytest.mark.parametrize("rows,r", [(1, 64), (37, 40), (300, 256), (513, 95), (64, 1024)])
def test_pack_signs_bit_exact(rows, r):
    import binary_rank_linear_gb300 as blr
    rng = np.random.default_rng(rows + r)
    src = rng.standard_normal((rows, r)).astype(np.float32)
    src[rng.random((rows, r)) < 0.05] = 0.0
    src[rng.random((rows, r)) < 0.02] = -0.0
    src[rng.random((rows, r)) < 0.02] = np.nan
    src[0, 0] = np.inf
    got = blr.pack_signs(torch.from_numpy(src).cuda()).cpu().numpy().view(np.uint32)
    assert np.array_equal(got, oracle.pack_signs(src))


@pytest.mark.parametrize("rows,r", [(3, 40), (129, 64), (50, 1024), (7, 95)])
def test_unpack_signs_bit_exact(rows, r):
    import binary_rank_linear_gb300 as blr
    rng = np.random.default_rng(7 * rows + r)
    bits = rng.integers(0, 2**32, size=(rows, (r + 31) // 32), dtype=np.uint64).astype(np.uint32)
    got = blr.unpack_signs(torch.from_numpy(bits.view(np.int32)).cuda(), r).cpu().numpy().view(np.uint16)
    want = np.where(oracle.unpack_signs(bits, rows, r) > 0, 0x3C00, 0xBC00).astype(np.uint16)
    assert np.array_equal(got, want)


def _integer_grid(M, d_in, d_out, r, seed, one_hot=None):
    rng = np.random.default_rng(seed)
    t = {
        "x": rng.integers(-1, 2, size=(M, d_in)).astype(np.float32),
        "dy": rng.integers(-1, 2, size=(M, d_out)).astype(np.float32),
        "su": np.where(rng.random((d_out, r)) < 0.5, 1.0, -1.0).astype(np.float32),
        "sv": np.where(rng.random((d_in, r)) < 0.5, 1.0, -1.0).astype(np.float32),
        "g": np.ones(d_in, np.float32),
        "h": np.ones(d_out, np.float32),
    }
    if one_hot is None:
        t["l"] = rng.choice(np.array([0.5, 1.0, 2.0], np.float32), size=r)
    else:
        t["l"] = np.zeros(r, np.float32)
        t["l"][one_hot] = 1.0
    return t


@pytest.mark.parametrize("M,d_in,d_out,r", [(128, 128, 128, 64), (200, 96, 160, 96), (70, 256, 64, 128)])
def test_integer_grid_bit_exact(M, d_in, d_out, r):
    t = _integer_grid(M, d_in, d_out, r, seed=M + r)
    out = _run(t, gscale=1.0)
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    assert out["status"] == 0
    assert np.array_equal(out["y"], fw["y"].astype(np.float32))
    assert np.array_equal(out["dx"], bw["dx"].astype(np.float32))
    assert oracle.rel_err(out["dl"], bw["dl"]) == 0.0


@pytest.mark.parametrize("k", [0, 31, 32, 63, 95])
def test_one_hot_rank_bit_exact(k):
    """l = e_k: every output depends on bit k of each bitmap row only."""
    M, d_in, d_out, r = 130, 160, 96, 96
    t = _integer_grid(M, d_in, d_out, r, seed=100 + k, one_hot=k)
    out = _run(t, gscale=1.0)
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    assert np.array_equal(out["y"], fw["y"].astype(np.float32))
    assert np.array_equal(out["dx"], bw["dx"].astype(np.float32))
    for key in ("dh", "dl", "dg"):
        assert np.array_equal(out[key], bw[key].astype(np.float32)), key


# ------------------------------------------------------ tolerance parity ---
SHAPES = [
    # name, M, d_in, d_out, r : several tiles, ragged tails, half k-steps (K % 64 == 32)
    ("tiny", 128, 256, 256, 64),
    ("small", 300, 320, 448, 96),
    ("small", 257, 352, 192, 160),
    ("attn", 513, 512, 640, 256),
    ("ragged", 1, 128, 128, 64),
    ("ragged", 127, 256, 512, 128),
    ("ragged", 129, 192, 96, 64),
    # enough 256 x 256 tiles for the CTA-pair GEMMs of the narrow outputs, ragged
    # M, and a reduction length (d_out = 1568) that ends in a partial k-step
    ("attn", 4600, 1024, 1568, 1280),
    # small M with a wide output: the fused small-M forward, then the general
    # backward (its dy rows are too wide for the fused staging)
    ("small", 200, 128, 9216, 64),
    # the widest rows the streaming dy staging takes (one row per batch, two stages)
    ("small", 150, 128, 16384, 64),
]


@pytest.mark.parametrize("name,M,d_in,d_out,r", SHAPES)
@pytest.mark.parametrize("gscale", [0.0, 1024.0])
def test_parity_shapes(name, M, d_in, d_out, r, gscale):
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    if name == "ragged" and gscale > 0:
        gscale = 2.0 ** 30  # the dy ~ 1e-7 workload needs a large fixed scale
    out = _run(t, gscale=gscale)
    _check_against_oracle(t, out, f"(gscale {gscale})")


def test_accumulate_modes():
    w = wl.WORKLOADS["small"].with_shape(M=200, d_in=256, d_out=320, r=128)
    t = wl.make_inputs(w, with_priors=True)
    rng = np.random.default_rng(5)
    grad_prior = {"dg": rng.standard_normal(256).astype(np.float32),
                  "dl": rng.standard_normal(128).astype(np.float32),
                  "dh": rng.standard_normal(320).astype(np.float32)}
    out = _run(t, y_prior=t["y_prior"], dx_prior=t["dx_prior"], grad_prior=grad_prior)
    _check_against_oracle(t, out, y_prior=t["y_prior"], dx_prior=t["dx_prior"], grad_prior=grad_prior)


def test_pages_two_path_case():
    """The page's own test: two paths summed (path 0 overwrites, path 1
    accumulates), d_out 256, d_in 384, r 128, 70 tokens, gscale 1024."""
    from blr_gpu_run import run_layer
    p0, p1 = wl.pages_case(0), wl.pages_case(1)
    o0 = run_layer(p0, gscale=1024.0)
    o1 = run_layer(p1, gscale=1024.0, y_prior=o0["y"], dx_prior=o0["dx"])
    want_y = np.zeros((70, 256))
    want_dx = np.zeros((70, 384))
    for p, o in ((p0, o0), (p1, o1)):
        bu, bv = oracle.pack_signs(p["su"]), oracle.pack_signs(p["sv"])
        want_y += oracle.forward(p["x"], bu, bv, p["g"], p["l"], p["h"])["y"]
        bw = oracle.backward(p["x"], p["dy"], bu, bv, p["g"], p["l"], p["h"])
        want_dx += bw["dx"]
        for k in ("dh", "dl", "dg"):
            assert oracle.rel_err(o[k], bw[k]) <= 3e-3, k
    assert oracle.rel_err(o1["y"], want_y) <= 2e-3
    assert oracle.rel_err(o1["dx"], want_dx) <= 2e-3


def test_outputs_stay_in_bounds():
    """Rows past M of y and dx are never written (poisoned guard rows survive)."""
    import binary_rank_linear_gb300 as blr
    from blr_gpu_run import to_dev
    M, d_in, d_out, r = 70, 256, 192, 64
    t = wl.make_inputs(wl.WORKLOADS["tiny"].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    ybuf = torch.full((M + 3, d_out), 12345.0, device="cuda")
    dxbuf = torch.full((M + 3, d_in), -777.0, device="cuda")
    x, dy = to_dev(t["x"]), to_dev(t["dy"])
    g, l, h = to_dev(t["g"]), to_dev(t["l"]), to_dev(t["h"])
    bu, bv = blr.pack_signs(to_dev(t["su"])), blr.pack_signs(to_dev(t["sv"]))
    ws = blr.alloc_workspace(M, d_in, d_out, r)
    blr.forward(x, bu, bv, g, l, h, ybuf[:M], ws)
    dg, dl, dh = torch.zeros(d_in, device="cuda"), torch.zeros(r, device="cuda"), torch.zeros(d_out, device="cuda")
    blr.backward(x, dy, bu, bv, g, l, h, dxbuf[:M], dg, dl, dh, ws)
    assert blr.check_status(ws) == 0
    assert torch.all(ybuf[M:] == 12345.0) and torch.all(dxbuf[M:] == -777.0)
    assert torch.isfinite(ybuf[:M]).all() and torch.isfinite(dxbuf[:M]).all()


@pytest.mark.parametrize("M,d_in,d_out,r", [(300, 256, 256, 128), (4600, 1024, 1568, 256)])
def test_reduction_folded_and_separate(monkeypatch, M, d_in, d_out, r):
    """dh, dl and dg reduced in the dx'-product's tail (BLR_REDUCE=fold) and
    by a launch of their own (the default): the same partial rows summed in
    two fixed orders, equal to rounding and both within the tolerance of the
    oracle; y and dx do not depend on it."""
    t = wl.make_inputs(wl.WORKLOADS["small"].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    b = _run(t)
    monkeypatch.setenv("BLR_REDUCE", "fold")
    a = _run(t)
    assert a["status"] == 0 and b["status"] == 0
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["dx"], b["dx"])
    for k in ("dh", "dl", "dg"):
        assert oracle.rel_err(a[k], b[k]) <= 1e-5, k
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    for k in ("dh", "dl", "dg"):
        assert oracle.rel_err(a[k], bw[k]) <= TOL_GRAD, k


@pytest.mark.parametrize("M,d_in,d_out,r,gscale", [
    (8192, 512, 1024, 512, 0.0),        # CTA-pair tiles of the db-product, dynamic scales
    (8000, 256, 2048, 512, 0.0),        # a ragged last token tile
    (8192, 512, 1024, 512, 2.0 ** 8),   # a fixed power-of-two gscale
    (6000, 256, 8448, 512, 0.0),        # rows wider than the streaming prologue's
])
def test_dy_staged_in_the_db_product(monkeypatch, M, d_in, d_out, r, gscale):
    """dy16 staged by the db-product's stager warps after a scale pass
    (BLR_DY_STAGE=kernel) against the backward prologue's staging (=pass):
    the same dy16, scales and tiles, so y, dx, dl and dg are bit-identical and
    dh (summed by the stager warps in another fixed order) and the sign
    gradients (read from the same dy16) equal to rounding, all within the
    oracle's tolerance; the staged product did run, and the
    default is the prologue form."""
    import binary_rank_linear_gb300 as blr
    t = wl.make_inputs(wl.WORKLOADS["small"].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    monkeypatch.setenv("BLR_DY_STAGE", "pass")
    b = _run(t, gscale=gscale, sign=True)
    monkeypatch.setenv("BLR_DY_STAGE", "kernel")
    blr.trace_begin(64)
    a = _run(t, gscale=gscale, sign=True)
    names = [n for n, _ in blr.trace_end()]
    assert "gemm_bwd1s" in names and "bwd_scales" in names, names
    assert a["status"] == 0 and b["status"] == 0
    for k in ("y", "dx", "dl", "dg"):
        assert np.array_equal(a[k], b[k]), k
    assert oracle.rel_err(a["dh"], b["dh"]) <= 1e-5
    # the sign gradients read the staged dy16 and the scales' block maxima
    for k in ("gu", "gv"):
        assert oracle.rel_err(a[k], b[k]) <= 1e-5, k
    _check_against_oracle(t, a)
    monkeypatch.delenv("BLR_DY_STAGE")
    blr.trace_begin(64)
    c = _run(t, gscale=gscale)
    assert "gemm_bwd1s" not in [n for n, _ in blr.trace_end()]
    for k in ("y", "dx", "dh", "dl", "dg"):
        assert np.array_equal(b[k], c[k]), k


def test_deterministic():
    w = wl.WORKLOADS["small"].with_shape(M=300, d_in=256, d_out=256, r=128)
    t = wl.make_inputs(w)
    a, b = _run(t), _run(t)
    for k in ("y", "dx", "dh", "dl", "dg"):
        assert np.array_equal(a[k], b[k]), k


def test_backward_without_forward_is_rejected():
    import binary_rank_linear_gb300 as blr
    M, d_in, d_out, r = 16, 64, 64, 64
    z = lambda *s: torch.zeros(*s, device="cuda")  # noqa: E731
    bits = torch.zeros(64, 2, dtype=torch.int32, device="cuda")
    ws = blr.alloc_workspace(M, d_in, d_out, r)
    with pytest.raises(blr.BlrError) as e:
        blr.backward(z(M, d_in), z(M, d_out), bits, bits, z(d_in), z(r), z(d_out), z(M, d_in),
                     z(d_in), z(r), z(d_out), ws)
    assert e.value.code == blr.BLR_ERR_STATE


def test_backward_needs_the_forwards_inputs_and_a_live_record():
    """The tape record names the forward's inputs: a backward on the same
    workspace with another x (a reused workspace address for another layer of
    the same shape) is refused, and so is any backward after
    blr_workspace_release."""
    import binary_rank_linear_gb300 as blr
    M, d_in, d_out, r = 64, 128, 128, 64
    z = lambda *s: torch.zeros(*s, device="cuda")  # noqa: E731
    bits = torch.zeros(128, 2, dtype=torch.int32, device="cuda")
    x, x2 = z(M, d_in), z(M, d_in)
    g, l, h = torch.ones(d_in, device="cuda"), torch.ones(r, device="cuda"), torch.ones(d_out, device="cuda")
    ws = blr.alloc_workspace(M, d_in, d_out, r)
    blr.forward(x, bits, bits, g, l, h, z(M, d_out), ws)
    with pytest.raises(blr.BlrError) as e:
        blr.backward(x2, z(M, d_out), bits, bits, g, l, h, z(M, d_in), z(d_in), z(r), z(d_out), ws)
    assert e.value.code == blr.BLR_ERR_STATE
    blr.backward(x, z(M, d_out), bits, bits, g, l, h, z(M, d_in), z(d_in), z(r), z(d_out), ws)
    blr.workspace_release(ws)
    with pytest.raises(blr.BlrError) as e:
        blr.backward(x, z(M, d_out), bits, bits, g, l, h, z(M, d_in), z(d_in), z(r), z(d_out), ws)
    assert e.value.code == blr.BLR_ERR_STATE
    assert blr.check_status(ws) == 0


# ------------------------------------------------------- full workloads ----
FULL = ["tiny", "small", "attn", "ragged",
        pytest.param("mlp_up", marks=pytest.mark.slow), pytest.param("mlp_down", marks=pytest.mark.slow)]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """The workloads at full size, in the launch configuration the benchmark
    times: y, dx, dh, dl and dg compared in full, element by element, with the
    oracle's f64 forward and backward on the same inputs; the Euler identities
    on everything."""
    w = wl.WORKLOADS[name]
    t = wl.make_inputs(w)
    out = _run(t)
    assert out["status"] == 0
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    assert np.array_equal(out["bu"], bu) and np.array_equal(out["bv"], bv)
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    errs = {"y": oracle.rel_err(out["y"], fw["y"])}
    del fw
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    errs["dx"] = oracle.rel_err(out["dx"], bw["dx"])
    for k in ("dh", "dl", "dg"):
        errs[k] = oracle.rel_err(out[k], bw[k])
    del bw
    for k, e in errs.items():
        tol = TOL_OUT if k in ("y", "dx") else TOL_GRAD
        assert np.isfinite(e) and e <= tol, f"{name} {k}: rel err {e:.3e} > {tol} {errs}"
    # Euler identities <dh,h> = <dl,l> = <dg,g> = <dx,x> = <dy,y> on every
    # output. A normwise error e in v moves <v,p> by at most e |v| |p|
    # (Cauchy-Schwarz), and likewise for y in <dy,y>: that is the bound.
    dy64, y64 = t["dy"].astype(np.float64), out["y"].astype(np.float64)
    ref = float(np.sum(dy64 * y64))
    ref_slack = TOL_OUT * np.linalg.norm(dy64) * np.linalg.norm(y64)
    pairs = ((out["dh"], t["h"], TOL_GRAD), (out["dl"], t["l"], TOL_GRAD), (out["dg"], t["g"], TOL_GRAD),
             (out["dx"], t["x"], TOL_OUT))
    for vec, par, tol in pairs:
        v64, p64 = vec.astype(np.float64).ravel(), par.astype(np.float64).ravel()
        got = float(np.dot(v64, p64))
        assert abs(got - ref) <= tol * np.linalg.norm(v64) * np.linalg.norm(p64) + ref_slack


@pytest.mark.parametrize("name,M,d_in,d_out,r", [("tiny", 128, 256, 256, 64), ("small", 300, 320, 448, 96),
                                                 ("small", 2048, 1024, 1024, 256), ("ragged", 129, 192, 96, 64)])
def test_fused_small_path(monkeypatch, name, M, d_in, d_out, r):
    """The fused small-M kernels (one cooperative kernel per pass) against the oracle."""
    monkeypatch.setenv("BLR_SMALL_PATH", "fused")
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t, gscale=0.0)
    _check_against_oracle(t, out, "(fused small-M path)")


@pytest.mark.parametrize("src", ["plane", "tmem"])
@pytest.mark.parametrize("name,M,d_in,d_out,r", [("small", 300, 320, 448, 96), ("attn", 4600, 1024, 1568, 1280),
                                                 ("ragged", 2100, 640, 4224, 256), ("small", 200, 128, 9216, 64)])
def test_sign_source_modes(monkeypatch, src, name, M, d_in, d_out, r):
    """Both sources of the sign operand (+-1 f16 planes read by TMA, or bitmap
    words expanded into TMEM), each forced on single-CTA and CTA-pair tiles."""
    monkeypatch.setenv("BLR_SIGN_SRC", src)
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t, gscale=0.0)
    _check_against_oracle(t, out, f"(sign source {src})")


@pytest.mark.parametrize("src", ["plane", "tmem"])
def test_sign_source_integer_grid_bit_exact(monkeypatch, src):
    monkeypatch.setenv("BLR_SIGN_SRC", src)
    M, d_in, d_out, r = 2100, 512, 4096, 160  # CTA-pair tiles in both forms
    t = _integer_grid(M, d_in, d_out, r, seed=77)
    out = _run(t, gscale=1.0)
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    assert out["status"] == 0
    assert np.array_equal(out["y"], fw["y"].astype(np.float32))
    assert np.array_equal(out["dx"], bw["dx"].astype(np.float32))


@pytest.mark.parametrize("name,M,d_in,d_out,r", [("small", 300, 320, 448, 96), ("attn", 4600, 1024, 1568, 1280),
                                                 ("ragged", 127, 256, 512, 128)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_wide_products_token_major(monkeypatch, name, M, d_in, d_out, r, accumulate):
    """The c- and dx'-products run token-major on the dense kernel (BLR_WIDE=token)."""
    monkeypatch.setenv("BLR_WIDE", "token")
    w = wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r)
    t = wl.make_inputs(w, with_priors=accumulate)
    if accumulate:
        out = _run(t, y_prior=t["y_prior"], dx_prior=t["dx_prior"])
        _check_against_oracle(t, out, "(token-major, accumulate)", y_prior=t["y_prior"], dx_prior=t["dx_prior"])
    else:
        out = _run(t)
        _check_against_oracle(t, out, "(token-major)")


@pytest.mark.parametrize("splitk", ["1", "0"])
@pytest.mark.parametrize("name,M,d_in,d_out,r", [("small", 2048, 1024, 1024, 256), ("small", 333, 544, 608, 160),
                                                 ("ragged", 129, 1056, 96, 64), ("attn", 513, 512, 640, 256)])
def test_split_k(monkeypatch, splitk, name, M, d_in, d_out, r):
    """The a- and db-products of problems with few tiles split K over clusters
    of four CTAs (reduced over DSMEM); the same shapes without the split."""
    monkeypatch.setenv("BLR_SPLITK", splitk)
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t, gscale=0.0)
    _check_against_oracle(t, out, f"(split-K {splitk})")


def test_split_k_integer_grid_bit_exact(monkeypatch):
    monkeypatch.setenv("BLR_SPLITK", "1")
    M, d_in, d_out, r = 250, 640, 544, 96  # both r-wide products split (5 and 5 k-steps)
    t = _integer_grid(M, d_in, d_out, r, seed=91)
    out = _run(t, gscale=1.0)
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    assert out["status"] == 0
    assert np.array_equal(out["y"], fw["y"].astype(np.float32))
    assert np.array_equal(out["dx"], bw["dx"].astype(np.float32))
    assert oracle.rel_err(out["dl"], bw["dl"]) == 0.0


@pytest.mark.parametrize("name,M,d_in,d_out,r", [("small", 300, 320, 448, 96), ("attn", 513, 512, 4096, 256),
                                                 ("small", 150, 128, 12288, 64)])
def test_dy_staging_forms(monkeypatch, name, M, d_in, d_out, r):
    """The stand-alone dy staging pass (BLR_STAGE=pass) in its register-staged
    row form (BLR_DY_STAGE=rows) against the oracle on widths the streaming
    form takes by default."""
    monkeypatch.setenv("BLR_STAGE", "pass")
    monkeypatch.setenv("BLR_DY_STAGE", "rows")
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t)
    _check_against_oracle(t, out, "(BLR_DY_STAGE=rows)")


@pytest.mark.parametrize("form", ["flat", "rows", "stream"])
@pytest.mark.parametrize("name,M,d_in,d_out,r", [("small", 300, 320, 448, 96), ("attn", 513, 4096, 512, 256),
                                                 ("small", 77, 12288, 256, 64)])
def test_x_staging_forms(monkeypatch, form, name, M, d_in, d_out, r):
    """Each form of the stand-alone x staging pass (BLR_STAGE=pass):
    grid-stride, row-mapped, streamed through the shared-memory ring, forced
    with BLR_X_STAGE, against the oracle."""
    monkeypatch.setenv("BLR_STAGE", "pass")
    monkeypatch.setenv("BLR_X_STAGE", form)
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t)
    _check_against_oracle(t, out, f"(BLR_X_STAGE={form})")


@pytest.mark.parametrize("name,M,d_in,d_out,r", [("small", 300, 320, 448, 96), ("small", 2048, 1024, 1024, 256)])
def test_128_token_single_tiles(monkeypatch, name, M, d_in, d_out, r):
    """Few-tile products on 128-token single-CTA tiles (BLR_GEMM_BT=128; by
    default they take 64- or 32-token tiles) against the oracle."""
    monkeypatch.setenv("BLR_GEMM_BT", "128")
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t)
    _check_against_oracle(t, out, "(BLR_GEMM_BT=128)")


@pytest.mark.parametrize("M,d_in,d_out,r", [(33, 65536, 32768, 64), (40, 64, 64, 65536)])
def test_maximum_widths(M, d_in, d_out, r):
    """The widest shapes the shape rule admits (d_in and r up to 65536, d_out up
    to 32768) with ragged token counts, against the oracle in full."""
    t = wl.make_inputs(wl.WORKLOADS["small"].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    out = _run(t)
    _check_against_oracle(t, out, "(maximum widths)")


@pytest.mark.parametrize("stage", ["pass", "kernel"])
@pytest.mark.parametrize("name,M,d_in,d_out,r", [("small", 300, 320, 448, 96), ("attn", 4600, 1024, 1568, 1280),
                                                 ("ragged", 2100, 640, 4224, 256), ("small", 1, 64, 64, 64),
                                                 ("small", 200, 128, 9216, 64), ("attn", 3001, 4096, 2048, 512)])
@pytest.mark.parametrize("gscale", [0.0, 1024.0])
def test_stage_forms(monkeypatch, stage, name, M, d_in, d_out, r, gscale):
    """x staged inside the a-product by its stager warps (BLR_STAGE=kernel,
    the default for x of 64 MB or more) or by the stand-alone pass before it
    (BLR_STAGE=pass), on single-CTA and CTA-pair tiles, ragged token counts
    and partial column chunks, against the oracle."""
    monkeypatch.setenv("BLR_STAGE", stage)
    t = wl.make_inputs(wl.WORKLOADS[name].with_shape(M=M, d_in=d_in, d_out=d_out, r=r))
    if name == "ragged" and gscale > 0:
        gscale = 2.0 ** 30
    out = _run(t, gscale=gscale)
    _check_against_oracle(t, out, f"(BLR_STAGE={stage}, gscale {gscale})")


def test_stage_in_kernel_integer_grid_bit_exact(monkeypatch):
    """With exact operands the in-kernel staging gives the oracle's y and dx bit
    for bit (pair tiles, several column chunks, a ragged last token tile)."""
    monkeypatch.setenv("BLR_STAGE", "kernel")
    M, d_in, d_out, r = 2100, 800, 4096, 160
    t = _integer_grid(M, d_in, d_out, r, seed=93)
    out = _run(t, gscale=1.0)
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    assert out["status"] == 0
    assert np.array_equal(out["y"], fw["y"].astype(np.float32))
    assert np.array_equal(out["dx"], bw["dx"].astype(np.float32))
    # (dh is not exact here: it reads the c tape, which holds f16 values)
    assert oracle.rel_err(out["dh"], bw["dh"]) <= TOL_GRAD
