"""CPU f64 oracle of the binary low-rank (blr) linear layer.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH. Only the test suite,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference leg may
import or call this module. The GPU library never routes through it, and the
two share no code: this file has its own bitmap unpacking, its own packing and
its own arithmetic.

Source: ``train_mm.rs`` of cortiq-engine 0.8.21 (docs.rs source view). Every
function below cites the part of that page it restates:

* module documentation, formula block: the layer
  W_hat = diag(h) . S_U . diag(l) . S_V^T . diag(g) and its six
  forward/backward formulas;
* the ``expand`` kernel's comment: the sign-bitmap convention
  ``[rows][ceil(r/32)]`` u32, bit j of word w is rank 32w+j, a set bit is +1;
* the test helper ``pack_bits``: a sign is packed as 1 iff its value is > 0;
* the test ``blr_layer_matches_host``: the per-token f64 host loop this oracle
  vectorises, and the normwise relative error metric;
* ``blr_backward``'s documentation and the test helper ``host_sign_grads``:
  the sign gradients G_U = diag(h) dy^T a diag(l) and
  G_V = diag(g) x^T b diag(l), b the backward's db;
* the WGSL ``adam`` kernel and its Rust wrapper ``adam``: one Adam step (no
  weight decay) with an optional frozen-entry mask, a gradient multiplier and
  optional steps relative to the parameter's magnitude;
* ``plane_linear`` and ``mm``: a dense frozen linear y = x . plane^T through
  the f16 staging, or its transpose (input gradient) y = x . plane;
* ``Blr`` (a layer is y = sum_p W_hat_p x over its paths) and ``blr_forward``
  / ``blr_backward``'s path loops: path 0 overwrites y and dx, later paths
  add, and each path keeps its own dh, dl, dg.

Precision: inputs are f32 on the page; they are widened to f64 here and every
step runs in f64. There is no staging, no f16 and no scaling in the oracle: the
method reaches the formulas' exact value up to rounding order, so the oracle is
that definition written out. Matrix products use ``numpy.matmul`` as a library
primitive, one product per formula, with no blocking, fusion or reordering.

Parity is pinned (see ``tests/test_oracle.py``) by: a brute-force dense W_hat
built element by element; central finite differences of L = <dy, y> for
dg, dl, dh and dx (exact, since L is linear in each); Euler identities; a
hand-written golden bitmap fixture; one-hot l; and integer popcount sums.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "words_per_row",
    "unpack_signs",
    "pack_signs",
    "forward",
    "backward",
    "backward_sampled",
    "sign_grads",
    "sign_grads_sampled",
    "adam_step",
    "plane_linear",
    "forward_paths",
    "backward_paths",
    "rel_err",
]


def words_per_row(r: int) -> int:
    """Number of u32 words per bitmap row: ceil(r / 32) (``expand`` kernel comment)."""
    return (int(r) + 31) // 32


def unpack_signs(bits: np.ndarray, rows: int, r: int) -> np.ndarray:
    """Sign bitmap -> dense +-1 matrix [rows][r] in f64.

    train_mm.rs, ``expand`` kernel comment: the bitmap is ``[rows][words]``
    u32 with words = ceil(r/32); bit j of word w is rank 32w+j; a set bit is
    +1 and a clear bit is -1. Bits of the last word at ranks >= r are ignored.
    """
    w = words_per_row(r)
    bits = np.asarray(bits, dtype=np.uint32).reshape(rows, w)
    out = np.empty((rows, r), dtype=np.float64)
    for k in range(r):
        word = bits[:, k // 32]
        bit = (word >> np.uint32(k % 32)) & np.uint32(1)
        out[:, k] = np.where(bit == 1, 1.0, -1.0)
    return out


def pack_signs(src: np.ndarray) -> np.ndarray:
    """Dense values [rows][r] -> sign bitmap [rows][ceil(r/32)] u32.

    train_mm.rs, test helper ``pack_bits``: bit (row, k) is set iff
    src[row, k] > 0. Zero, -0.0 and NaN therefore pack as -1. Unused high
    bits of the last word are written 0.
    """
    src = np.asarray(src)
    rows, r = src.shape
    w = words_per_row(r)
    out = np.zeros((rows, w), dtype=np.uint32)
    positive = src > 0
    for k in range(r):
        out[:, k // 32] |= positive[:, k].astype(np.uint32) << np.uint32(k % 32)
    return out


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=np.float64)


def forward(x, bits_u, bits_v, g, l, h, y_prior=None) -> dict:
    """blr forward in f64.

    train_mm.rs, module documentation (forward row of the formula block):
        a = (x (.) g) . S_V        x [M][d_in], S_V [d_in][r]
        c = (a (.) l) . S_U^T      S_U [d_out][r]
        y (+)= h (.) c             y [M][d_out]
    The page's ``Blr`` is "m x n" with m = d_out and n = d_in; S_U is expanded
    from ``bits_u`` over d_out rows and S_V from ``bits_v`` over d_in rows.
    ``y_prior`` given = accumulate mode (the page's later paths), else y is
    overwritten (its first path).

    Returns a dict with y, a and c (f64).
    """
    x = _f64(x)
    g, l, h = _f64(g), _f64(l), _f64(h)
    M, d_in = x.shape
    d_out, r = h.shape[0], l.shape[0]
    s_u = unpack_signs(bits_u, d_out, r)
    s_v = unpack_signs(bits_v, d_in, r)
    a = np.matmul(x * g[None, :], s_v)           # [M][r]
    c = np.matmul(a * l[None, :], s_u.T)         # [M][d_out]
    y = h[None, :] * c
    if y_prior is not None:
        y = _f64(y_prior) + y
    return {"y": y, "a": a, "c": c}


def backward(x, dy, bits_u, bits_v, g, l, h, dx_prior=None) -> dict:
    """blr backward in f64.

    train_mm.rs, module documentation (backward rows of the formula block):
        dh  = sum over tokens of dy (.) c
        db  = (dy (.) h) . S_U
        dl  = sum over tokens of a (.) db
        dx' = (db (.) l) . S_V^T
        dg  = sum over tokens of x (.) dx'
        dx (+)= g (.) dx'
    a and c are the forward's intermediates on the same x and parameters,
    recomputed here. ``dx_prior`` given = accumulate mode, else overwrite.
    The gradients dh, dl, dg are returned as this call's contribution; the GPU
    library adds them into caller vectors, so a test adds any prior itself.

    Returns a dict with dx, dg, dl, dh, db and dxp (f64).
    """
    x, dy = _f64(x), _f64(dy)
    g, l, h = _f64(g), _f64(l), _f64(h)
    fw = forward(x, bits_u, bits_v, g, l, h)
    a, c = fw["a"], fw["c"]
    M, d_in = x.shape
    d_out, r = h.shape[0], l.shape[0]
    s_u = unpack_signs(bits_u, d_out, r)
    s_v = unpack_signs(bits_v, d_in, r)
    dh = np.sum(dy * c, axis=0)
    db = np.matmul(dy * h[None, :], s_u)         # [M][r]
    dl = np.sum(a * db, axis=0)
    dxp = np.matmul(db * l[None, :], s_v.T)      # [M][d_in]
    dg = np.sum(x * dxp, axis=0)
    dx = g[None, :] * dxp
    if dx_prior is not None:
        dx = _f64(dx_prior) + dx
    return {"dx": dx, "dg": dg, "dl": dl, "dh": dh, "db": db, "dxp": dxp}


def backward_sampled(x, dy, bits_u, bits_v, g, l, h, cols_h, cols_g) -> dict:
    """dl in full, and dh and dg at the given output columns, in f64.

    The same backward formulas (train_mm.rs, module documentation), evaluated
    only where asked: dh_i needs c[:, i] = (a (.) l) . S_U[i, :]^T, and dg_j
    needs dx'[:, j] = (db (.) l) . S_V[j, :]^T, so restricting the sign
    matrices to the sampled rows restricts the products to those columns.
    a and db are computed in full (both are token-by-rank). This lets full-size
    workloads be checked against exact values at a fraction of the cost.

    Returns a dict with dl [r], dh [len(cols_h)], dg [len(cols_g)].
    """
    x, dy = _f64(x), _f64(dy)
    g, l, h = _f64(g), _f64(l), _f64(h)
    d_in, d_out, r = x.shape[1], h.shape[0], l.shape[0]
    s_u = unpack_signs(bits_u, d_out, r)
    s_v = unpack_signs(bits_v, d_in, r)
    cols_h = np.asarray(cols_h, dtype=np.int64)
    cols_g = np.asarray(cols_g, dtype=np.int64)
    a = np.matmul(x * g[None, :], s_v)
    db = np.matmul(dy * h[None, :], s_u)
    dl = np.sum(a * db, axis=0)
    c_cols = np.matmul(a * l[None, :], s_u[cols_h].T)
    dh = np.sum(dy[:, cols_h] * c_cols, axis=0)
    dxp_cols = np.matmul(db * l[None, :], s_v[cols_g].T)
    dg = np.sum(x[:, cols_g] * dxp_cols, axis=0)
    return {"dl": dl, "dh": dh, "dg": dg}


def sign_grads(x, dy, bits_u, bits_v, g, l, h) -> dict:
    """Sign gradients of the layer in f64.

    train_mm.rs, ``blr_backward`` documentation and the test helper
    ``host_sign_grads``:
        a = (x (.) g) . S_V,  b = (dy (.) h) . S_U            [M][r]
        G_U[i][k] = h_i l_k sum_t dy[t][i] a[t][k]           [d_out][r]
        G_V[j][k] = g_j l_k sum_t x[t][j]  b[t][k]           [d_in][r]
    i.e. G_U = diag(h) dy^T a diag(l) and G_V = diag(g) x^T b diag(l). With
    L = <dy, y> these are dL/dS_U and dL/dS_V (L is linear in each sign).

    Returns a dict with gu [d_out][r] and gv [d_in][r] (f64).
    """
    x, dy = _f64(x), _f64(dy)
    g, l, h = _f64(g), _f64(l), _f64(h)
    d_in, d_out, r = x.shape[1], h.shape[0], l.shape[0]
    s_u = unpack_signs(bits_u, d_out, r)
    s_v = unpack_signs(bits_v, d_in, r)
    a = np.matmul(x * g[None, :], s_v)
    b = np.matmul(dy * h[None, :], s_u)
    gu = h[:, None] * np.matmul(dy.T, a) * l[None, :]
    gv = g[:, None] * np.matmul(x.T, b) * l[None, :]
    return {"gu": gu, "gv": gv}


def sign_grads_sampled(x, dy, bits_u, bits_v, g, l, h, rows_u, rows_v) -> dict:
    """G_U at the given rows of S_U and G_V at the given rows of S_V, in f64.

    The sign_grads formulas (train_mm.rs, ``blr_backward`` documentation and
    the test helper ``host_sign_grads``) restricted to rows: G_U[i, :] needs
    only dy[:, i], and G_V[j, :] only x[:, j]; a and b are token-by-rank and
    computed in full. For checking full-size workloads at a fraction of the
    cost.

    Returns a dict with gu [len(rows_u)][r] and gv [len(rows_v)][r].
    """
    x, dy = _f64(x), _f64(dy)
    g, l, h = _f64(g), _f64(l), _f64(h)
    d_in, d_out, r = x.shape[1], h.shape[0], l.shape[0]
    s_u = unpack_signs(bits_u, d_out, r)
    s_v = unpack_signs(bits_v, d_in, r)
    rows_u = np.asarray(rows_u, dtype=np.int64)
    rows_v = np.asarray(rows_v, dtype=np.int64)
    a = np.matmul(x * g[None, :], s_v)
    b = np.matmul(dy * h[None, :], s_u)
    gu = h[rows_u, None] * np.matmul(dy[:, rows_u].T, a) * l[None, :]
    gv = g[rows_v, None] * np.matmul(x[:, rows_v].T, b) * l[None, :]
    return {"gu": gu, "gv": gv}


def adam_step(w, grad, m1, m2, lr, step, b1, b2, eps, mask=None, gmul=1.0, rel=0.0) -> dict:
    """One Adam update, elementwise, in f64.

    train_mm.rs, WGSL ``adam`` kernel and its wrapper ``adam``. Entries whose
    mask value is exactly 0 are frozen (nothing changes). For every other
    entry, with t = step (1-based):
        gr = grad * gmul
        m1 <- b1 m1 + (1 - b1) gr
        m2 <- b2 m2 + (1 - b2) gr^2
        st = lr * (m1 / (1 - b1^t)) / (sqrt(m2 / (1 - b2^t)) + eps)
        w  <- w - st * max(|w|, rel)   if rel > 0 (relative step, floored)
        w  <- w - st                   otherwise
    Returns a dict with the new w, m1, m2 (f64).
    """
    w, grad, m1, m2 = _f64(w), _f64(grad), _f64(m1), _f64(m2)
    t = float(step)
    gr = grad * float(gmul)
    n1 = b1 * m1 + (1.0 - b1) * gr
    n2 = b2 * m2 + (1.0 - b2) * gr * gr
    mh = n1 / (1.0 - b1 ** t)
    vh = n2 / (1.0 - b2 ** t)
    st = lr * mh / (np.sqrt(vh) + eps)
    nw = w - st * np.maximum(np.abs(w), rel) if rel > 0 else w - st
    if mask is not None:
        live = _f64(mask) != 0.0
        nw = np.where(live, nw, w)
        n1 = np.where(live, n1, m1)
        n2 = np.where(live, n2, m2)
    return {"w": nw, "m1": n1, "m2": n2}


def plane_linear(x, plane, transpose=False, y_prior=None) -> np.ndarray:
    """A dense frozen linear in f64.

    train_mm.rs, ``plane_linear`` (staging ``cvt`` of x under ``scale``, then
    ``mm`` with output scale 1/scale) and ``mm`` (out[m][n] = act[m][k] .
    plane[n][k]^T): y = (x s) plane^T / s = x plane^T, the scale cancelling
    exactly; with ``transpose`` (the input gradient through the same plane),
    y = x plane. ``plane`` holds f16 values (given as any float array).
    ``y_prior`` adds the result to it (accumulate mode).
    """
    x, p = _f64(x), _f64(plane)
    y = np.matmul(x, p) if transpose else np.matmul(x, p.T)
    return y if y_prior is None else _f64(y_prior) + y


def forward_paths(x, paths, y_prior=None) -> dict:
    """A multi-path layer y = sum_p W_hat_p x, in f64.

    train_mm.rs, ``Blr`` and ``blr_forward`` (its loop over paths: path 0
    overwrites y, later paths add). ``paths`` is a list of dicts with keys
    bu, bv (bitmaps), g, l, h. Returns y and the per-path forward dicts.
    """
    outs = [forward(x, p["bu"], p["bv"], p["g"], p["l"], p["h"]) for p in paths]
    y = sum(o["y"] for o in outs)
    if y_prior is not None:
        y = _f64(y_prior) + y
    return {"y": y, "paths": outs}


def backward_paths(x, dy, paths, dx_prior=None) -> dict:
    """Backward of a multi-path layer, in f64.

    train_mm.rs, ``blr_backward``'s loop over paths: dx = sum_p dx_p (path 0
    overwrites, later paths add) and each path's own dh, dl, dg.
    """
    outs = [backward(x, dy, p["bu"], p["bv"], p["g"], p["l"], p["h"]) for p in paths]
    dx = sum(o["dx"] for o in outs)
    if dx_prior is not None:
        dx = _f64(dx_prior) + dx
    return {"dx": dx, "paths": outs}


def rel_err(got, want) -> float:
    """Normwise relative error sqrt(sum (got-want)^2 / max(sum want^2, 1e-30)).

    train_mm.rs, test ``blr_layer_matches_host`` (its ``rel`` closure).
    """
    got = _f64(got).ravel()
    want = _f64(want).ravel()
    num = float(np.sum((got - want) ** 2))
    den = max(float(np.sum(want * want)), 1e-30)
    return float(np.sqrt(num / den))
