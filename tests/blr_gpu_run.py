"""Runs one blr forward+backward through the C ABI on the GPU (test helper).

Inputs come from ``binary_rank_linear_gb300.workloads`` as host arrays; signs are
packed on the device with ``blr_pack_signs``. Results come back as numpy.
"""
import numpy as np
import torch

import binary_rank_linear_gb300 as blr


def to_dev(a, dtype=torch.float32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(device="cuda", dtype=dtype)


def run_layer(t, gscale=0.0, y_prior=None, dx_prior=None, grad_prior=None, ws=None, backward=True, sign=False,
              sign_prior=None):
    """Forward (+ backward, + sign gradients) of one path. Priors given = accumulate mode."""
    x, dy = to_dev(t["x"]), to_dev(t["dy"]) if backward else None
    M, d_in = t["x"].shape
    d_out, r = t["su"].shape
    g, l, h = to_dev(t["g"]), to_dev(t["l"]), to_dev(t["h"])
    bu = blr.pack_signs(to_dev(t["su"]))
    bv = blr.pack_signs(to_dev(t["sv"]))
    if ws is None:
        ws = blr.alloc_workspace(M, d_in, d_out, r)
    y = to_dev(y_prior) if y_prior is not None else torch.full((M, d_out), float("nan"), device="cuda")
    blr.forward(x, bu, bv, g, l, h, y, ws, accumulate=y_prior is not None)
    out = {"y": y, "bu": bu, "bv": bv, "ws": ws}
    if backward:
        dx = to_dev(dx_prior) if dx_prior is not None else torch.full((M, d_in), float("nan"), device="cuda")
        if grad_prior is not None:
            dg, dl, dh = (to_dev(grad_prior[k]) for k in ("dg", "dl", "dh"))
        else:
            dg = torch.zeros(d_in, device="cuda")
            dl = torch.zeros(r, device="cuda")
            dh = torch.zeros(d_out, device="cuda")
        blr.backward(x, dy, bu, bv, g, l, h, dx, dg, dl, dh, ws, gscale=gscale, accumulate=dx_prior is not None)
        out.update(dx=dx, dg=dg, dl=dl, dh=dh)
        if sign:
            sws = blr.alloc_sign_workspace(M, d_in, d_out, r)
            if sign_prior is not None:
                gu, gv = to_dev(sign_prior["gu"]), to_dev(sign_prior["gv"])
            else:
                gu = torch.full((d_out, r), float("nan"), device="cuda")
                gv = torch.full((d_in, r), float("nan"), device="cuda")
            blr.sign_grads(x, g, l, gu, gv, ws, sws, accumulate=sign_prior is not None)
            out.update(gu=gu, gv=gv)
    out["status"] = blr.check_status(ws)
    host = {}
    for k, v in out.items():
        if isinstance(v, torch.Tensor) and k != "ws":
            host[k] = v.cpu().numpy()
        else:
            host[k] = v
    host["bu"] = host["bu"].view(np.uint32)
    host["bv"] = host["bv"].view(np.uint32)
    return host
