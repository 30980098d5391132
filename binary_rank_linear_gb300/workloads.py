"""Seeded synthetic workloads for the blr layer (shapes and value distributions).

This module holds only random draws and the workload table; it does none of the
layer's arithmetic. Both the GPU tests and the CPU oracle's tests take their
inputs from here, so the two sides see the same arrays.

Signs are drawn as +-1 f32 matrices (S_U [d_out][r], S_V [d_in][r]); packing
them into bitmaps is the library's job (``blr_pack_signs``) on the GPU side and
the oracle's own ``pack_signs`` on the CPU side.

Generator: numpy PCG64 (``numpy.random.default_rng``), one stream per tensor,
seed = 1000 * workload id + tensor id.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

# tensor ids inside a workload's seed block
_T_X, _T_DY, _T_SU, _T_SV, _T_G, _T_H, _T_L, _T_YP, _T_DXP = range(1, 10)


@dataclass(frozen=True)
class Workload:
    """One synthetic blr layer: sizes plus the recipe of its value distributions."""

    name: str
    wid: int            # seed block
    M: int              # tokens
    d_in: int
    d_out: int
    r: int
    dy_scale: float     # dy ~ N(0,1) * dy_scale
    p_plus: float       # P(sign = +1)
    gh_sigma: float     # g, h = 1 + gh_sigma * N(0,1)
    l_kind: str         # "exp1": 0.05 e^{-i/r}; "exp2": 0.02 e^{-2i/r}; "unif": U(1e-3, 1e-1)
    note: str = ""

    def with_shape(self, M=None, d_in=None, d_out=None, r=None, name=None) -> "Workload":
        """Same distributions at another shape (for parity cases the oracle finishes fast)."""
        return Workload(
            name=name or self.name,
            wid=self.wid,
            M=self.M if M is None else M,
            d_in=self.d_in if d_in is None else d_in,
            d_out=self.d_out if d_out is None else d_out,
            r=self.r if r is None else r,
            dy_scale=self.dy_scale,
            p_plus=self.p_plus,
            gh_sigma=self.gh_sigma,
            l_kind=self.l_kind,
            note=self.note,
        )

    @property
    def flops(self) -> float:
        """Algorithmic FLOP of one forward+backward: four products of 2*M*r*d each."""
        return 4.0 * self.M * self.r * (self.d_in + self.d_out)

    @property
    def canonical_bytes(self) -> float:
        """Algorithmic HBM bytes of one forward+backward (overwrite mode).

        x read twice (forward, and backward for dg), y written, dy read, dx
        written, the f32 tape a [M][r] written and read, both bitmaps read in
        the forward and in the backward. Vectors are negligible.
        """
        M, di, do, r = self.M, self.d_in, self.d_out, self.r
        words = (r + 31) // 32
        return 4.0 * M * (3 * di + 2 * do + 2 * r) + 2.0 * (di + do) * words * 4


WORKLOADS = {
    "tiny": Workload("tiny", 0, 128, 256, 256, 64, 1.0, 0.5, 0.1, "exp1",
                     "M=128 tokens, 256->256, r=64"),
    "small": Workload("small", 1, 2048, 1024, 1024, 256, 1e-3, 0.5, 0.1, "exp1",
                      "M=2048 (4 windows x 512), 1024->1024, r=256"),
    "attn": Workload("attn", 2, 8192, 4096, 4096, 1024, 1e-4, 0.5, 0.1, "exp2",
                     "M=8192 (16 windows x 512), 4096->4096, r=1024"),
    "mlp_up": Workload("mlp_up", 3, 16384, 4096, 12288, 1024, 1e-4, 0.5, 0.1, "exp2",
                       "SwiGLU up: M=16384 (8 windows x 2048), 4096->12288, r=1024"),
    "mlp_down": Workload("mlp_down", 4, 16384, 12288, 4096, 1024, 1e-4, 0.5, 0.1, "exp2",
                         "SwiGLU down: M=16384, 12288->4096, r=1024"),
    "ragged": Workload("ragged", 5, 4000, 2048, 32768, 512, 1e-7, 0.9, 0.3, "unif",
                       "M=4000 (ragged), 2048->32768, r=512, dy ~1e-7, 90% +1 signs"),
}


# Steps made of several layers, each with its own seeded inputs: the SwiGLU MLP
# pair runs the up layer's forward+backward and then the down layer's, and its
# time is their sum.
STEPS = {
    "mlp": ("mlp_up", "mlp_down"),
}
STEP_NOTES = {
    "mlp": "SwiGLU MLP pair: up 4096->12288 and down 12288->4096, both r=1024, M=16384 (8 windows x 2048); "
           "one step = both layers' forward+backward on their own inputs",
}


def step_layers(name: str, M: int = 0) -> list:
    """The layers one step of workload ``name`` runs (at ``M`` tokens when given)."""
    names = STEPS.get(name, (name,))
    out = []
    for n in names:
        w = WORKLOADS[n]
        out.append(w.with_shape(M=M) if M else w)
    return out


def step_note(name: str) -> str:
    return STEP_NOTES.get(name, WORKLOADS[name].note if name in WORKLOADS else name)


def _l_vector(kind: str, r: int, rng: np.random.Generator) -> np.ndarray:
    i = np.arange(r, dtype=np.float64)
    if kind == "exp1":
        return (0.05 * np.exp(-i / r)).astype(np.float32)
    if kind == "exp2":
        return (0.02 * np.exp(-2.0 * i / r)).astype(np.float32)
    if kind == "unif":
        return rng.uniform(1e-3, 1e-1, size=r).astype(np.float32)
    raise ValueError(kind)


def _signs(rng: np.random.Generator, rows: int, r: int, p_plus: float) -> np.ndarray:
    return np.where(rng.random((rows, r)) < p_plus, 1.0, -1.0).astype(np.float32)


def make_inputs(w: Workload, with_priors: bool = False) -> dict:
    """All host inputs of workload ``w`` as f32 numpy arrays (signs as +-1 f32).

    Keys: x [M][d_in], dy [M][d_out], su [d_out][r], sv [d_in][r], g [d_in],
    h [d_out], l [r]; with ``with_priors`` also y_prior [M][d_out] and
    dx_prior [M][d_in] (values already in the outputs for accumulate mode).
    """
    base = 1000 * w.wid

    def rng(t):
        return np.random.default_rng(base + t)

    out = {
        "x": rng(_T_X).standard_normal((w.M, w.d_in), dtype=np.float32),
        "dy": (rng(_T_DY).standard_normal((w.M, w.d_out), dtype=np.float32)
               * np.float32(w.dy_scale)),
        "su": _signs(rng(_T_SU), w.d_out, w.r, w.p_plus),
        "sv": _signs(rng(_T_SV), w.d_in, w.r, w.p_plus),
        "g": (1.0 + w.gh_sigma * rng(_T_G).standard_normal(w.d_in)).astype(np.float32),
        "h": (1.0 + w.gh_sigma * rng(_T_H).standard_normal(w.d_out)).astype(np.float32),
        "l": _l_vector(w.l_kind, w.r, rng(_T_L)),
    }
    if with_priors:
        out["y_prior"] = rng(_T_YP).standard_normal((w.M, w.d_out), dtype=np.float32)
        out["dx_prior"] = rng(_T_DXP).standard_normal((w.M, w.d_in), dtype=np.float32)
    return out


def _uniform(n: int, seed: int, scale: float) -> np.ndarray:
    """n seeded draws from U(-scale, scale) as f32 (PCG64 stream ``seed``)."""
    return np.random.default_rng(seed).uniform(-scale, scale, size=n).astype(np.float32)


def pages_case(path: int, ntok: int = 70, d_out: int = 256, d_in: int = 384, r: int = 128) -> dict:
    """Inputs shaped and distributed like the page's own two-path layer test.

    train_mm.rs, test ``blr_layer_matches_host``: d_out=256, d_in=384, r=128,
    70 tokens; signs from uniform draws (>= 0 gives +1); h = 0.02 + 0.05|u|,
    l = 0.5 + |u|, g = 0.1 + 0.2|u| with u ~ U(-0.5, 0.5); x ~ U(-2, 2);
    dy ~ U(-1e-3, 1e-3); the gradients are staged under gscale = 1024.
    ``path`` selects the path's seeds (0 or 1); x and dy are shared. Only the
    shapes and distributions are mirrored; the draws are this module's own.
    """
    base = 6000
    sgn = lambda v: np.where(v >= 0.0, 1.0, -1.0).astype(np.float32)  # noqa: E731
    return {
        "su": sgn(_uniform(d_out * r, base + 10 + path, 1.0)).reshape(d_out, r),
        "sv": sgn(_uniform(d_in * r, base + 20 + path, 1.0)).reshape(d_in, r),
        "h": (0.02 + np.abs(_uniform(d_out, base + 30 + path, 0.5)) * 0.05).astype(np.float32),
        "l": (0.5 + np.abs(_uniform(r, base + 40 + path, 0.5))).astype(np.float32),
        "g": (0.1 + np.abs(_uniform(d_in, base + 50 + path, 0.5)) * 0.2).astype(np.float32),
        "x": _uniform(ntok * d_in, base + 60, 2.0).reshape(ntok, d_in),
        "dy": _uniform(ntok * d_out, base + 61, 1e-3).reshape(ntok, d_out),
    }
