"""Pins of the CPU f64 oracle against facts fixed outside the oracle itself.

Each pin uses an independent route to the same number: hand-written fixtures of
the page's bit convention and pack rule, a dense W_hat built element by element
with plain loops, central finite differences of L = <dy, y> (exact here because
L is linear in each of g, l, h and x), Euler identities, one-hot l, and integer
popcount sums. The planted-mistake tests check that each pin actually catches
the kind of error it is meant to (a flipped bit order, a dropped factor, a
transposed operand, a wrong sign).
"""
import math
import os

import numpy as np
import pytest

import oracle
from binary_rank_linear_gb300 import workloads as wl

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- fixtures --
def _read_convention(golden_dir):
    rows, r = [], None
    with open(os.path.join(golden_dir, "bitmap_convention.txt")) as f:
        lines = [ln.strip() for ln in f if ln.strip() and not ln.startswith("#")]
    words = None
    for ln in lines:
        key, _, rest = ln.partition(" ")
        if key == "r":
            r = int(rest)
        elif key == "row":
            words = [int(w, 16) for w in rest.split()]
        elif key == "signs":
            rows.append((words, [1.0 if ch == "+" else -1.0 for ch in rest]))
    return r, rows


def _read_pack(golden_dir):
    cases, vals = [], None
    with open(os.path.join(golden_dir, "pack_rule.txt")) as f:
        for ln in f:
            ln = ln.strip()
            if not ln or ln.startswith("#"):
                continue
            key, _, rest = ln.partition(" ")
            if key == "values":
                vals = [float(v) for v in rest.split()]
            elif key == "words":
                cases.append((vals, [int(w, 16) for w in rest.split()]))
    return cases


def _tiny(seed=0, M=3, d_in=6, d_out=5, r=40):
    rng = np.random.default_rng(seed)
    su = np.where(rng.random((d_out, r)) < 0.5, 1.0, -1.0).astype(np.float32)
    sv = np.where(rng.random((d_in, r)) < 0.5, 1.0, -1.0).astype(np.float32)
    return {
        "x": rng.standard_normal((M, d_in)).astype(np.float32),
        "dy": rng.standard_normal((M, d_out)).astype(np.float32),
        "su": su, "sv": sv,
        "bu": oracle.pack_signs(su), "bv": oracle.pack_signs(sv),
        "g": (1 + 0.3 * rng.standard_normal(d_in)).astype(np.float32),
        "h": (1 + 0.3 * rng.standard_normal(d_out)).astype(np.float32),
        "l": rng.uniform(0.1, 1.0, r).astype(np.float32),
    }


def _dense_w_loops(su, sv, g, l, h):
    """W_hat[i][j] = h_i g_j sum_k S_U[i,k] l_k S_V[j,k], element by element."""
    d_out, r = su.shape
    d_in = sv.shape[0]
    w = [[0.0] * d_in for _ in range(d_out)]
    for i in range(d_out):
        for j in range(d_in):
            acc = 0.0
            for k in range(r):
                acc += float(su[i][k]) * float(l[k]) * float(sv[j][k])
            w[i][j] = float(h[i]) * acc * float(g[j])
    return w


def _bruteforce_y_dx(t, W):
    x, dy = t["x"].astype(np.float64), t["dy"].astype(np.float64)
    M, d_in = x.shape
    d_out = dy.shape[1]
    y = np.zeros((M, d_out))
    dx = np.zeros((M, d_in))
    for m in range(M):
        for i in range(d_out):
            y[m, i] = sum(W[i][j] * x[m, j] for j in range(d_in))
        for j in range(d_in):
            dx[m, j] = sum(dy[m, i] * W[i][j] for i in range(d_out))
    return y, dx


# ------------------------------------------------------- bitmap convention --
def test_unpack_matches_golden_convention(golden_dir):
    r, rows = _read_convention(golden_dir)
    bits = np.array([w for w, _ in rows], dtype=np.uint32)
    want = np.array([s for _, s in rows])
    got = oracle.unpack_signs(bits, len(rows), r)
    assert got.shape == want.shape
    assert np.array_equal(got, want)


def test_pack_matches_golden_rule(golden_dir):
    for vals, words in _read_pack(golden_dir):
        got = oracle.pack_signs(np.array([vals], dtype=np.float32))
        assert got.dtype == np.uint32
        assert [int(w) for w in got[0]] == words


@pytest.mark.parametrize("rows,r", [(7, 64), (5, 40), (3, 32), (9, 1), (4, 95)])
def test_pack_unpack_roundtrip(rows, r):
    rng = np.random.default_rng(rows * 100 + r)
    s = np.where(rng.random((rows, r)) < 0.5, 1.0, -1.0)
    bits = oracle.pack_signs(s)
    assert bits.shape == (rows, oracle.words_per_row(r))
    assert np.array_equal(oracle.unpack_signs(bits, rows, r), s)
    # unused high bits of the last word are written 0
    if r % 32:
        assert np.all(bits[:, -1] >> np.uint32(r % 32) == 0)


def test_unpack_ignores_bits_past_r():
    bits = np.array([[0xFFFFFFFF, 0xFFFFFF00]], dtype=np.uint32)
    s = oracle.unpack_signs(bits, 1, 40)
    assert np.all(s[0, :32] == 1.0) and np.all(s[0, 32:] == -1.0)


# -------------------------------------------------------- forward/backward --
@pytest.mark.parametrize("seed", [0, 1])
def test_forward_backward_match_bruteforce_dense(seed):
    t = _tiny(seed)
    W = _dense_w_loops(t["su"], t["sv"], t["g"], t["l"], t["h"])
    y_bf, dx_bf = _bruteforce_y_dx(t, W)
    fw = oracle.forward(t["x"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    assert np.allclose(fw["y"], y_bf, rtol=1e-12, atol=1e-12)
    assert np.allclose(bw["dx"], dx_bf, rtol=1e-12, atol=1e-12)


def _loss(t, g=None, l=None, h=None, x=None):
    y = oracle.forward(t["x"] if x is None else x, t["bu"], t["bv"],
                       t["g"] if g is None else g, t["l"] if l is None else l,
                       t["h"] if h is None else h)["y"]
    return float(np.sum(t["dy"].astype(np.float64) * y))


@pytest.mark.parametrize("seed", [2, 3])
def test_gradients_match_central_differences(seed):
    """L = <dy, y> is linear in each of g, l, h, x: the central difference is exact."""
    t = _tiny(seed)
    bw = oracle.backward(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    eps = 0.25
    for name, key in (("g", "dg"), ("l", "dl"), ("h", "dh")):
        base = t[name].astype(np.float64)
        fd = np.empty_like(base)
        for i in range(base.size):
            p, m = base.copy(), base.copy()
            p[i] += eps
            m[i] -= eps
            fd[i] = (_loss(t, **{name: p}) - _loss(t, **{name: m})) / (2 * eps)
        assert np.allclose(bw[key], fd, rtol=1e-10, atol=1e-10), name
    x = t["x"].astype(np.float64)
    fdx = np.empty_like(x)
    for idx in np.ndindex(*x.shape):
        p, m = x.copy(), x.copy()
        p[idx] += eps
        m[idx] -= eps
        fdx[idx] = (_loss(t, x=p) - _loss(t, x=m)) / (2 * eps)
    assert np.allclose(bw["dx"], fdx, rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("name", ["tiny", "small"])
def test_euler_identities(name):
    """y is homogeneous of degree 1 in each of h, l, g and x, so
    <dh,h> = <dl,l> = <dg,g> = <dx,x> = <dy,y> (single path, overwrite mode)."""
    w = wl.WORKLOADS[name].with_shape(M=64)
    t = wl.make_inputs(w)
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    fw = oracle.forward(t["x"], bu, bv, t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    ref = float(np.sum(t["dy"].astype(np.float64) * fw["y"]))
    for vec, par in ((bw["dh"], t["h"]), (bw["dl"], t["l"]), (bw["dg"], t["g"])):
        assert math.isclose(float(np.dot(vec, par.astype(np.float64))), ref, rel_tol=1e-9)
    assert math.isclose(float(np.sum(bw["dx"] * t["x"].astype(np.float64))), ref, rel_tol=1e-9)


@pytest.mark.parametrize("k", [0, 31, 32, 39])
def test_one_hot_l_isolates_rank(k):
    """l = e_k gives W_hat = (h . S_U[:,k]) (g . S_V[:,k])^T: one bit per row of
    each bitmap, so the bit-to-rank mapping is pinned."""
    t = _tiny(5, M=4, d_in=7, d_out=6, r=40)
    l = np.zeros(40, dtype=np.float32)
    l[k] = 1.0
    fw = oracle.forward(t["x"], t["bu"], t["bv"], t["g"], l, t["h"])
    # bit (row, k) read straight from the packed words
    bit_u = np.array([(int(t["bu"][i][k // 32]) >> (k % 32)) & 1 for i in range(6)])
    bit_v = np.array([(int(t["bv"][j][k // 32]) >> (k % 32)) & 1 for j in range(7)])
    su_k = 2.0 * bit_u - 1.0
    sv_k = 2.0 * bit_v - 1.0
    coef = t["x"].astype(np.float64) @ (t["g"].astype(np.float64) * sv_k)
    want = coef[:, None] * (t["h"].astype(np.float64) * su_k)[None, :]
    assert np.allclose(fw["y"], want, rtol=1e-12, atol=1e-12)


def test_popcount_integer_sums():
    """x = 1, g = 1: a_k = 2 * (number of +1 in column k of S_V) - d_in, an integer."""
    d_in, r = 50, 70
    rng = np.random.default_rng(11)
    bv = rng.integers(0, 2**32, size=(d_in, 3), dtype=np.uint64).astype(np.uint32)
    bu = rng.integers(0, 2**32, size=(4, 3), dtype=np.uint64).astype(np.uint32)
    fw = oracle.forward(np.ones((2, d_in), np.float32), bu, bv, np.ones(d_in, np.float32),
                        np.ones(r, np.float32), np.ones(4, np.float32))
    for k in range(r):
        ones = sum(bin(int(bv[j][k // 32]))[2:].zfill(32)[::-1][k % 32] == "1" for j in range(d_in))
        assert fw["a"][0, k] == 2 * ones - d_in
        assert fw["a"][1, k] == 2 * ones - d_in


def test_accumulate_mode_adds_prior():
    t = _tiny(7)
    y0 = np.full((3, 5), 0.75)
    dx0 = np.full((3, 6), -1.25)
    a = oracle.forward(t["x"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    b = oracle.forward(t["x"], t["bu"], t["bv"], t["g"], t["l"], t["h"], y_prior=y0)
    assert np.array_equal(b["y"], a["y"] + y0)
    c = oracle.backward(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    d = oracle.backward(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"], dx_prior=dx0)
    assert np.array_equal(d["dx"], c["dx"] + dx0)


def test_rel_err_metric():
    assert oracle.rel_err([1.0, 2.0], [1.0, 2.0]) == 0.0
    assert math.isclose(oracle.rel_err([3.0, 4.0], [0.0, 0.0]), math.sqrt(25 / 1e-30))
    assert math.isclose(oracle.rel_err([1.1, 0.0], [1.0, 0.0]), 0.1, rel_tol=1e-12)


def test_pages_case_two_paths_pinned():
    """The page's own two-path test shape (d_out 256, d_in 384, r 128, 70 tokens),
    checked path by path against the dense brute force on a token subset."""
    for path in (0, 1):
        t = wl.pages_case(path)
        bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
        fw = oracle.forward(t["x"][:2], bu, bv, t["g"], t["l"], t["h"])
        W = (t["h"].astype(np.float64)[:, None]
             * ((t["su"].astype(np.float64) * t["l"].astype(np.float64)[None, :])
                @ t["sv"].astype(np.float64).T)
             * t["g"].astype(np.float64)[None, :])
        # spot-check entries of W against the element-by-element definition
        for (i, j) in [(0, 0), (17, 300), (255, 383)]:
            ref = sum(float(t["su"][i][k]) * float(t["l"][k]) * float(t["sv"][j][k]) for k in range(128))
            assert math.isclose(W[i, j], float(t["h"][i]) * ref * float(t["g"][j]), rel_tol=1e-12)
        assert np.allclose(fw["y"], t["x"][:2].astype(np.float64) @ W.T, rtol=1e-10, atol=1e-12)


# -------------------------------------------------------- planted mistakes --
def _mutant_unpack_reversed(bits, rows, r):
    w = oracle.words_per_row(r)
    bits = np.asarray(bits, dtype=np.uint32).reshape(rows, w)
    out = np.empty((rows, r))
    for k in range(r):
        out[:, k] = np.where((bits[:, k // 32] >> np.uint32(31 - k % 32)) & 1, 1.0, -1.0)
    return out


def test_planted_bit_order_mistake_is_caught(golden_dir, monkeypatch):
    from oracle import blr_oracle
    r, rows = _read_convention(golden_dir)
    bits = np.array([w for w, _ in rows], dtype=np.uint32)
    want = np.array([s for _, s in rows])
    monkeypatch.setattr(blr_oracle, "unpack_signs", _mutant_unpack_reversed)
    assert not np.array_equal(blr_oracle.unpack_signs(bits, len(rows), r), want)


@pytest.mark.parametrize("mutant", ["drop_l", "permuted_u_rows", "sign_dh"])
def test_planted_formula_mistakes_are_caught(mutant, monkeypatch):
    from oracle import blr_oracle
    t = _tiny(9, M=3, d_in=6, d_out=6, r=40)
    real_matmul = np.matmul
    if mutant == "drop_l":
        orig = blr_oracle.forward

        def fwd(x, bu, bv, g, l, h, y_prior=None):
            return orig(x, bu, bv, g, np.ones_like(l), h, y_prior)
        monkeypatch.setattr(blr_oracle, "forward", fwd)
        W = _dense_w_loops(t["su"], t["sv"], t["g"], t["l"], t["h"])
        y_bf, _ = _bruteforce_y_dx(t, W)
        y = blr_oracle.forward(t["x"], t["bu"], t["bv"], t["g"], t["l"], t["h"])["y"]
        assert not np.allclose(y, y_bf, rtol=1e-6)
    elif mutant == "permuted_u_rows":
        # a wrong row index of S_U (rows reversed) in the backward's db product
        calls = {"n": 0}

        def mm(a, b):
            calls["n"] += 1
            if calls["n"] == 3:          # third product of backward = db
                return real_matmul(a, b[::-1])
            return real_matmul(a, b)
        monkeypatch.setattr(blr_oracle.np, "matmul", mm)
        bw = blr_oracle.backward(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
        monkeypatch.setattr(blr_oracle.np, "matmul", real_matmul)
        W = _dense_w_loops(t["su"], t["sv"], t["g"], t["l"], t["h"])
        _, dx_bf = _bruteforce_y_dx(t, W)
        assert not np.allclose(bw["dx"], dx_bf, rtol=1e-6)
    else:
        bw = blr_oracle.backward(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
        eps = 0.25
        base = t["h"].astype(np.float64)
        fd = np.empty_like(base)
        for i in range(base.size):
            p, m = base.copy(), base.copy()
            p[i] += eps
            m[i] -= eps
            fd[i] = (_loss(t, h=p) - _loss(t, h=m)) / (2 * eps)
        assert np.allclose(bw["dh"], fd, rtol=1e-10)
        assert not np.allclose(-bw["dh"], fd, rtol=1e-6)


def test_sampled_backward_matches_full():
    """The column-sampled evaluation equals the full backward at those columns."""
    w = wl.WORKLOADS["small"].with_shape(M=96, d_in=128, d_out=160, r=64)
    t = wl.make_inputs(w)
    bu, bv = oracle.pack_signs(t["su"]), oracle.pack_signs(t["sv"])
    full = oracle.backward(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"])
    ch, cg = [0, 7, 159, 80], [127, 3, 64]
    smp = oracle.backward_sampled(t["x"], t["dy"], bu, bv, t["g"], t["l"], t["h"], ch, cg)
    assert np.allclose(smp["dl"], full["dl"], rtol=1e-12, atol=1e-14)
    assert np.allclose(smp["dh"], full["dh"][ch], rtol=1e-12, atol=1e-14)
    assert np.allclose(smp["dg"], full["dg"][cg], rtol=1e-12, atol=1e-14)


# ----------------------------------------------------------- sign gradients --
def _flip_bit(bits, rows, r, i, k):
    """Copy of a bitmap with the sign of (row i, rank k) flipped (bit k%32 of word k//32)."""
    w = oracle.words_per_row(r)
    out = np.array(bits, dtype=np.uint32).reshape(rows, w).copy()
    out[i, k // 32] ^= np.uint32(1 << (k % 32))
    return out


@pytest.mark.parametrize("seed", [5, 6])
def test_sign_grads_flip_identity(seed):
    """L = <dy, y> is linear in every single sign, so flipping S[i,k] (value s)
    changes L by exactly -2 s G[i,k]; checked for every sign of a tiny layer
    by re-running the forward with the flipped bitmap."""
    t = _tiny(seed, M=4, d_in=5, d_out=6, r=36)
    sg = oracle.sign_grads(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    l0 = _loss(t)
    d_in, d_out, r = 5, 6, 36
    for side, rows, key, gkey in (("u", d_out, "bu", "gu"), ("v", d_in, "bv", "gv")):
        signs = t["su"] if side == "u" else t["sv"]
        for i in range(rows):
            for k in range(r):
                flipped = dict(t)
                flipped[key] = _flip_bit(t[key], rows, r, i, k)
                dl = _loss(flipped) - l0
                want = -2.0 * float(signs[i, k]) * sg[gkey][i, k]
                assert abs(dl - want) <= 1e-9 * (1.0 + abs(want)), (side, i, k, dl, want)


def test_sign_grads_trace_identity():
    """sum_i S_U[i,k] G_U[i,k] = sum_j S_V[j,k] G_V[j,k] = l_k dl_k: both equal
    l_k sum_t a_tk b_tk, which ties the sign gradients to the backward's dl."""
    t = _tiny(7, M=5, d_in=9, d_out=7, r=40)
    sg = oracle.sign_grads(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    bw = oracle.backward(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    want = t["l"].astype(np.float64) * bw["dl"]
    assert np.allclose(np.sum(t["su"] * sg["gu"], axis=0), want, rtol=1e-12, atol=1e-12)
    assert np.allclose(np.sum(t["sv"] * sg["gv"], axis=0), want, rtol=1e-12, atol=1e-12)


def test_sign_grads_match_loops():
    """The sign gradients against the pages' per-element host formula, written
    as plain Python loops (no matrix products)."""
    t = _tiny(8, M=3, d_in=4, d_out=5, r=33)
    sg = oracle.sign_grads(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    x, dy = t["x"].astype(np.float64), t["dy"].astype(np.float64)
    M, d_in = x.shape
    d_out, r = t["su"].shape
    a = [[sum(x[m, j] * float(t["g"][j]) * float(t["sv"][j, k]) for j in range(d_in)) for k in range(r)]
         for m in range(M)]
    b = [[sum(dy[m, i] * float(t["h"][i]) * float(t["su"][i, k]) for i in range(d_out)) for k in range(r)]
         for m in range(M)]
    for k in range(r):
        for i in range(d_out):
            want = float(t["h"][i]) * float(t["l"][k]) * sum(dy[m, i] * a[m][k] for m in range(M))
            assert math.isclose(sg["gu"][i, k], want, rel_tol=1e-12, abs_tol=1e-12)
        for j in range(d_in):
            want = float(t["g"][j]) * float(t["l"][k]) * sum(x[m, j] * b[m][k] for m in range(M))
            assert math.isclose(sg["gv"][j, k], want, rel_tol=1e-12, abs_tol=1e-12)


@pytest.mark.parametrize("mutant", ["swap_hg", "drop_l", "transpose_b"])
def test_planted_sign_grad_mistakes_are_caught(mutant, monkeypatch):
    """Plausible mistakes in sign_grads fail the flip identity."""
    real = oracle.sign_grads

    def broken(x, dy, bu, bv, g, l, h):
        out = real(x, dy, bu, bv, g, l, h)
        if mutant == "swap_hg":
            out["gu"] = out["gu"] / np.asarray(h, np.float64)[:, None] * np.mean(g)
        elif mutant == "drop_l":
            out["gv"] = out["gv"] / np.asarray(l, np.float64)[None, :]
        else:
            out["gu"] = out["gu"][::-1].copy()
        return out

    monkeypatch.setattr(oracle, "sign_grads", broken)
    with pytest.raises(AssertionError):
        test_sign_grads_flip_identity(5)


def test_sign_grads_sampled_rows():
    """The row-sampled sign gradients equal those rows of the full ones (which
    the flip identity pins), including repeated and edge rows."""
    t = _tiny(9, M=6, d_in=11, d_out=13, r=40)
    full = oracle.sign_grads(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"])
    ru, rv = np.array([0, 5, 5, 12]), np.array([10, 0, 3])
    smp = oracle.sign_grads_sampled(t["x"], t["dy"], t["bu"], t["bv"], t["g"], t["l"], t["h"], ru, rv)
    assert np.allclose(smp["gu"], full["gu"][ru], rtol=1e-13, atol=1e-13)
    assert np.allclose(smp["gv"], full["gv"][rv], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------------------ Adam ---
def _adam_inputs(seed, n=257):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n), rng.standard_normal(n) * 1e-2,
            rng.standard_normal(n) * 1e-3, np.abs(rng.standard_normal(n)) * 1e-4)


def test_adam_matches_torch():
    """No mask, gmul 1, absolute steps: the textbook Adam (torch.optim.Adam, no
    weight decay, eps added to the bias-corrected root), run for several steps
    on the same gradients in f64."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(21)
    n, lr, b1, b2, eps = 300, 3e-3, 0.9, 0.999, 1e-8
    w0 = rng.standard_normal(n)
    grads = [rng.standard_normal(n) * 10.0 ** rng.uniform(-4, 0) for _ in range(6)]
    p = torch.nn.Parameter(torch.tensor(w0, dtype=torch.float64))
    opt = torch.optim.Adam([p], lr=lr, betas=(b1, b2), eps=eps)
    w, m1, m2 = w0.copy(), np.zeros(n), np.zeros(n)
    for step, gvec in enumerate(grads, start=1):
        p.grad = torch.tensor(gvec, dtype=torch.float64)
        opt.step()
        o = oracle.adam_step(w, gvec, m1, m2, lr, step, b1, b2, eps)
        w, m1, m2 = o["w"], o["m1"], o["m2"]
        assert np.allclose(w, p.detach().numpy(), rtol=1e-13, atol=1e-15), step
        st = opt.state[p]
        assert np.allclose(m1, st["exp_avg"].numpy(), rtol=1e-13, atol=0)
        assert np.allclose(m2, st["exp_avg_sq"].numpy(), rtol=1e-13, atol=0)


def test_adam_first_step_closed_form():
    """From zero moments the first bias-corrected moments are gr and gr^2, so the
    step is lr * gr / (|gr| + eps), for any betas."""
    w, g, _, _ = _adam_inputs(3)
    for b1, b2, gmul in ((0.9, 0.999, 1.0), (0.5, 0.9, 0.25), (0.0, 0.0, 4.0)):
        o = oracle.adam_step(w, g, np.zeros_like(w), np.zeros_like(w), 1e-2, 1, b1, b2, 1e-6, gmul=gmul)
        gr = g * gmul
        assert np.allclose(o["w"], w - 1e-2 * gr / (np.abs(gr) + 1e-6), rtol=1e-14, atol=1e-16)
        assert np.allclose(o["m1"], (1 - b1) * gr, rtol=1e-15, atol=0)
        assert np.allclose(o["m2"], (1 - b2) * gr * gr, rtol=1e-15, atol=0)


def test_adam_constant_gradient_closed_form():
    """A constant gradient c from zero moments: both bias-corrected moments are
    exactly c and c^2 at every step, so every step moves by lr*c/(|c|+eps)."""
    rng = np.random.default_rng(4)
    c = rng.standard_normal(50)
    w0 = rng.standard_normal(50)
    w, m1, m2 = w0.copy(), np.zeros(50), np.zeros(50)
    for step in range(1, 8):
        o = oracle.adam_step(w, c, m1, m2, 1e-3, step, 0.8, 0.95, 1e-7)
        w, m1, m2 = o["w"], o["m1"], o["m2"]
        assert np.allclose(w, w0 - step * 1e-3 * c / (np.abs(c) + 1e-7), rtol=1e-12, atol=1e-14)


def test_adam_mask_and_relative_step():
    """Mask 0 freezes an entry (w and both moments); relative steps equal the
    absolute step times max(|w|, floor)."""
    w, g, m1, m2 = _adam_inputs(5)
    mask = (np.arange(w.size) % 3 != 0).astype(np.float64)
    args = (1e-3, 5, 0.9, 0.99, 1e-8)
    full = oracle.adam_step(w, g, m1, m2, *args)
    msk = oracle.adam_step(w, g, m1, m2, *args, mask=mask)
    live = mask != 0
    for k, before in (("w", w), ("m1", m1), ("m2", m2)):
        assert np.array_equal(msk[k][~live], before[~live])
        assert np.array_equal(msk[k][live], full[k][live])
    st = w - full["w"]
    relw = oracle.adam_step(w, g, m1, m2, *args, rel=0.5)["w"]
    # both differences cancel against |w| ~ 1, so about 12 digits survive
    assert np.allclose(w - relw, st * np.maximum(np.abs(w), 0.5), rtol=1e-9, atol=1e-16)


@pytest.mark.parametrize("mutant", ["no_bias_correction", "eps_inside_sqrt", "mask_ignored"])
def test_planted_adam_mistakes_are_caught(mutant, monkeypatch):
    real = oracle.adam_step

    def broken(w, grad, m1, m2, lr, step, b1, b2, eps, mask=None, gmul=1.0, rel=0.0):
        if mutant == "no_bias_correction" and step > 1:
            o = real(w, grad, m1, m2, lr, 1, 0.0, 0.0, eps, mask=mask, gmul=gmul, rel=rel)
            o["m1"], o["m2"] = real(w, grad, m1, m2, lr, step, b1, b2, eps)["m1"], real(
                w, grad, m1, m2, lr, step, b1, b2, eps)["m2"]
            return o
        if mutant == "eps_inside_sqrt":
            o = real(w, grad, m1, m2, lr, step, b1, b2, 0.0, mask=mask, gmul=gmul, rel=rel)
            n1 = b1 * np.asarray(m1) + (1 - b1) * np.asarray(grad) * gmul
            n2 = b2 * np.asarray(m2) + (1 - b2) * (np.asarray(grad) * gmul) ** 2
            st = lr * (n1 / (1 - b1 ** step)) / np.sqrt(n2 / (1 - b2 ** step) + eps)
            o["w"] = np.asarray(w, np.float64) - st
            return o
        return real(w, grad, m1, m2, lr, step, b1, b2, eps, mask=None, gmul=gmul, rel=rel)

    monkeypatch.setattr(oracle, "adam_step", broken)
    with pytest.raises(AssertionError):
        test_adam_matches_torch()
        test_adam_first_step_closed_form()
        test_adam_mask_and_relative_step()


# ---------------------------------------------------------- plane_linear ---
def _plane_case(seed, ntok=5, n=7, k=6):
    rng = np.random.default_rng(seed)
    plane = rng.standard_normal((n, k)).astype(np.float16)
    return rng.standard_normal((ntok, k)), rng.standard_normal((ntok, n)), plane


def test_plane_linear_loops():
    """y[t][i] = sum_j x[t][j] plane[i][j] and its transpose, as plain loops."""
    x, u, p = _plane_case(1)
    y = oracle.plane_linear(x, p)
    yt = oracle.plane_linear(u, p, transpose=True)
    for t in range(x.shape[0]):
        for i in range(p.shape[0]):
            assert math.isclose(y[t, i], sum(x[t, j] * float(p[i, j]) for j in range(p.shape[1])),
                                rel_tol=1e-13, abs_tol=1e-13)
        for j in range(p.shape[1]):
            assert math.isclose(yt[t, j], sum(u[t, i] * float(p[i, j]) for i in range(p.shape[0])),
                                rel_tol=1e-13, abs_tol=1e-13)


def test_plane_linear_adjoint_and_library():
    """<x P^T, u> = <x, u P> (the transpose is the adjoint, which pins which
    index is contracted), and the forward equals torch's linear in f64."""
    torch = pytest.importorskip("torch")
    x, u, p = _plane_case(2, ntok=9, n=13, k=11)
    y = oracle.plane_linear(x, p)
    yt = oracle.plane_linear(u, p, transpose=True)
    assert math.isclose(float(np.sum(y * u)), float(np.sum(x * yt)), rel_tol=1e-12)
    lib = torch.nn.functional.linear(torch.tensor(x), torch.tensor(p.astype(np.float64))).numpy()
    assert np.allclose(y, lib, rtol=1e-13, atol=1e-13)
    prior = np.ones_like(y)
    assert np.allclose(oracle.plane_linear(x, p, y_prior=prior), y + 1.0, rtol=1e-15, atol=1e-15)


@pytest.mark.parametrize("mutant", ["no_transpose", "transposed_plane"])
def test_planted_plane_mistakes_are_caught(mutant, monkeypatch):
    real = oracle.plane_linear

    def broken(x, plane, transpose=False, y_prior=None):
        if mutant == "no_transpose" and transpose:
            return real(x, np.asarray(plane).T, transpose=False, y_prior=y_prior)[:, ::-1]
        if mutant == "transposed_plane":
            q = np.asarray(plane, np.float64).copy()
            q[0, 1], q[1, 0] = q[1, 0], q[0, 1]
            return real(x, q, transpose=transpose, y_prior=y_prior)
        return real(x, plane, transpose=transpose, y_prior=y_prior)

    monkeypatch.setattr(oracle, "plane_linear", broken)
    with pytest.raises(AssertionError):
        test_plane_linear_loops()


# ------------------------------------------------------------ multi-path ---
def _two_paths(seed, M=4, d_in=6, d_out=5, r=36):
    a, b = _tiny(seed, M, d_in, d_out, r), _tiny(seed + 100, M, d_in, d_out, r)
    return a["x"], a["dy"], [a, b]


def test_paths_dense_brute_force():
    """y = x W^T and dx = dy W with W = sum_p diag(h_p) S_U,p diag(l_p) S_V,p^T diag(g_p),
    W built element by element."""
    x, dy, paths = _two_paths(31)
    d_in, d_out, r = 6, 5, 36
    W = np.zeros((d_out, d_in))
    for p in paths:
        for i in range(d_out):
            for j in range(d_in):
                W[i, j] += sum(float(p["h"][i]) * float(p["su"][i, k]) * float(p["l"][k]) * float(p["sv"][j, k])
                               * float(p["g"][j]) for k in range(r))
    fw = oracle.forward_paths(x, paths)
    bw = oracle.backward_paths(x, dy, paths)
    assert np.allclose(fw["y"], x.astype(np.float64) @ W.T, rtol=1e-12, atol=1e-12)
    assert np.allclose(bw["dx"], dy.astype(np.float64) @ W, rtol=1e-12, atol=1e-12)


def test_paths_equal_one_path_of_double_rank():
    """With shared g and h, two rank-r paths are one rank-2r path whose signs
    and l are the two paths' side by side."""
    x, dy, paths = _two_paths(32, r=64)
    a, b = paths
    b = dict(b, g=a["g"], h=a["h"])
    cat = {k: np.concatenate([a[k], b[k]], axis=1) for k in ("su", "sv")}
    bu, bv = oracle.pack_signs(cat["su"]), oracle.pack_signs(cat["sv"])
    lcat = np.concatenate([a["l"], b["l"]])
    one = oracle.forward(x, bu, bv, a["g"], lcat, a["h"])
    two = oracle.forward_paths(x, [a, b])
    assert np.allclose(two["y"], one["y"], rtol=1e-13, atol=1e-13)
    onb = oracle.backward(x, dy, bu, bv, a["g"], lcat, a["h"])
    twb = oracle.backward_paths(x, dy, [a, b])
    assert np.allclose(twb["dx"], onb["dx"], rtol=1e-13, atol=1e-13)
    # per-path gradients: dl splits by path, dg and dh add up over the paths
    assert np.allclose(np.concatenate([twb["paths"][0]["dl"], twb["paths"][1]["dl"]]), onb["dl"], rtol=1e-13)
    assert np.allclose(twb["paths"][0]["dg"] + twb["paths"][1]["dg"], onb["dg"], rtol=1e-12, atol=1e-13)
    assert np.allclose(twb["paths"][0]["dh"] + twb["paths"][1]["dh"], onb["dh"], rtol=1e-12, atol=1e-13)


def test_paths_priors():
    x, dy, paths = _two_paths(33)
    yp = np.ones((4, 5))
    dxp = np.full((4, 6), 2.0)
    assert np.allclose(oracle.forward_paths(x, paths, y_prior=yp)["y"], oracle.forward_paths(x, paths)["y"] + 1.0)
    assert np.allclose(oracle.backward_paths(x, dy, paths, dx_prior=dxp)["dx"],
                       oracle.backward_paths(x, dy, paths)["dx"] + 2.0)
