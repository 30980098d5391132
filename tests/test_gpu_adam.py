"""GPU parity of the Adam step (blr_adam) against the CPU f64 oracle.

The kernel computes in f32, as the page's WGSL kernel does; the bounds below
follow from f32 rounding (unit 2^-24 ~ 6e-8) of each operation:
  - a moment b m + (1 - b) v is within 4e-7 (b|m| + (1 - b)|v|) of the exact
    value: a few roundings of terms that may cancel;
  - the step st = lr (m1/bc1) / (sqrt(m2/bc2) + eps) is within 1e-5 |st| plus
    what the m1 error carries through, lr e1 / bc1 / (sqrt(m2/bc2) + eps);
  - w - st f rounds once more at f32 precision of |w| (3e-7 |w|).
Frozen entries must come back bit for bit unchanged.

The hyper-parameters are f32 on the page (uniforms of the WGSL kernel) and in
the C ABI, so the oracle receives the same f32 values, widened: f32(0.999)
makes 1 - b2 differ from 0.001 by 1.3e-5 relative, far above the f32
rounding this test bounds.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import binary_rank_linear_gb300 as blr
    blr.load()


def _state(n, seed):
    rng = np.random.default_rng(seed)
    w = rng.standard_normal(n).astype(np.float32)
    g = (rng.standard_normal(n) * 10.0 ** rng.uniform(-5, 0, n)).astype(np.float32)
    m1 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m2 = (np.abs(rng.standard_normal(n)) * 1e-5).astype(np.float32)
    return w, g, m1, m2


def f32(v):
    return float(np.float32(v))


HP = dict(lr=3e-3, b1=0.9, b2=0.999, eps=1e-8)


def _oracle(w, g, m1, m2, lr, step, b1, b2, eps, **kw):
    kw = {k: (f32(v) if k in ("gmul", "rel") else v) for k, v in kw.items()}
    return oracle.adam_step(w, g, m1, m2, f32(lr), step, f32(b1), f32(b2), f32(eps), **kw)


def _check(got, want, w, g, m1, m2, lr, step, b1, b2, eps, gmul=1.0, rel=0.0, mask=None):
    b1, b2, lr, eps = f32(b1), f32(b2), f32(lr), f32(eps)
    w, gr = w.astype(np.float64), g.astype(np.float64) * f32(gmul)
    e1 = 4e-7 * (b1 * np.abs(m1) + (1 - b1) * np.abs(gr)) + 1e-38
    e2 = 4e-7 * (b2 * np.abs(m2) + (1 - b2) * gr * gr) + 1e-38
    bc1, bc2 = 1 - b1 ** step, 1 - b2 ** step
    den = np.sqrt(want["m2"] / bc2) + eps
    st = lr * (want["m1"] / bc1) / den
    fac = np.maximum(np.abs(w), f32(rel)) if rel > 0 else np.ones_like(w)
    ew = 3e-7 * np.abs(w) + (1e-5 * np.abs(st) + lr * e1 / bc1 / den) * fac + 1e-38
    live = np.ones(w.shape, bool) if mask is None else (mask != 0)
    assert np.all(np.abs(got["m1"] - want["m1"])[live] <= e1[live])
    assert np.all(np.abs(got["m2"] - want["m2"])[live] <= e2[live])
    assert np.all(np.abs(got["w"] - want["w"])[live] <= ew[live])


def _gpu(w, g, m1, m2, **kw):
    import binary_rank_linear_gb300 as blr
    d = {k: torch.from_numpy(v.copy()).cuda() for k, v in (("w", w), ("g", g), ("m1", m1), ("m2", m2))}
    mask = kw.pop("mask", None)
    blr.adam(d["w"], d["g"], d["m1"], d["m2"], mask=torch.from_numpy(mask).cuda() if mask is not None else None, **kw)
    torch.cuda.synchronize()
    return {k: d[k].cpu().numpy() for k in ("w", "m1", "m2")}


@pytest.mark.parametrize("n", [1, 17, 1000, 100003])
@pytest.mark.parametrize("step,gmul,rel", [(1, 1.0, 0.0), (7, 0.5, 0.0), (3, 1.0, 1e-2), (1000, 2.0, 0.5)])
def test_adam_parity(n, step, gmul, rel):
    w, g, m1, m2 = _state(n, n + step)
    got = _gpu(w, g, m1, m2, step=step, gmul=gmul, rel=rel, **HP)
    want = _oracle(w, g, m1, m2, HP["lr"], step, HP["b1"], HP["b2"], HP["eps"], gmul=gmul, rel=rel)
    _check(got, want, w, g, m1, m2, HP["lr"], step, HP["b1"], HP["b2"], HP["eps"], gmul=gmul, rel=rel)


def test_adam_mask_freezes_entries_bit_exactly():
    n = 4099
    w, g, m1, m2 = _state(n, 9)
    mask = (np.arange(n) % 5 != 2).astype(np.float32)
    mask[7] = -0.0  # minus zero is zero: frozen as well
    got = _gpu(w, g, m1, m2, mask=mask, step=4, lr=1e-2, b1=0.8, b2=0.99, eps=1e-6)
    want = _oracle(w, g, m1, m2, 1e-2, 4, 0.8, 0.99, 1e-6, mask=mask)
    frozen = mask == 0
    for k, before in (("w", w), ("m1", m1), ("m2", m2)):
        assert np.array_equal(got[k][frozen], before[frozen]), k
    _check(got, want, w, g, m1, m2, 1e-2, 4, 0.8, 0.99, 1e-6, mask=mask)


def test_adam_trajectory():
    """Five steps in a row on fresh gradients, f32 state carried on the GPU and
    f64 state in the oracle."""
    import binary_rank_linear_gb300 as blr
    n = 5000
    rng = np.random.default_rng(12)
    w0 = rng.standard_normal(n).astype(np.float32)
    dw, dm1, dm2 = (torch.from_numpy(a).cuda() for a in (w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)))
    w, m1, m2 = w0.astype(np.float64), np.zeros(n), np.zeros(n)
    for step in range(1, 6):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        blr.adam(dw, torch.from_numpy(g).cuda(), dm1, dm2, step=step, lr=1e-3)
        o = _oracle(w, g, m1, m2, 1e-3, step, 0.9, 0.999, 1e-8)
        w, m1, m2 = o["w"], o["m1"], o["m2"]
    got = dw.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(got - w) <= 1e-6 * np.abs(w0) + 1e-4 * np.abs(w0 - w) + 1e-30)
    # m1 sums gradients of both signs (terms (1 - b1) g ~ 1e-4): its error is
    # absolute, a few f32 ulps of those terms per step
    assert np.allclose(dm1.cpu().numpy(), m1, rtol=1e-5, atol=1e-10)
