"""The C ABI without a GPU: the library loads, exports every symbol that
include/blr.h declares, and rejects bad arguments before touching the device.

The pointers passed here are never dereferenced: every call below fails its
host-side checks (or is pure host arithmetic) before any CUDA call.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from binary_rank_linear_gb300 import _build
    _build.build()
    import binary_rank_linear_gb300 as blr
    return blr.load()


def _declared_symbols():
    src = open(os.path.join(ROOT, "include", "blr.h")).read()
    return sorted(set(re.findall(r"BLR_API\s+[\w\s\*]+?\b(blr_\w+)\s*\(", src)))


def test_header_declares_entry_points():
    names = _declared_symbols()
    for n in ("blr_forward", "blr_backward", "blr_pack_signs", "blr_workspace_bytes"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_symbols()
    assert len(names) >= 8
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(0, -9, -1):
        s = lib.blr_status_string(code)
        assert s and s != b"unknown status"
    assert lib.blr_status_string(-100) == b"unknown status"


def test_workspace_bytes_shape_rule(lib):
    assert lib.blr_workspace_bytes(128, 256, 256, 64) > 0
    assert lib.blr_workspace_bytes(0, 256, 256, 64) == 0       # M >= 1
    assert lib.blr_workspace_bytes(128, 48, 256, 64) == 0      # d_in >= 64
    assert lib.blr_workspace_bytes(128, 256, 100, 64) == 0     # multiple of 32
    assert lib.blr_workspace_bytes(128, 256, 256, 65568) == 0  # r <= 65536
    assert lib.blr_workspace_bytes(128, 256, 32800, 64) == 0   # d_out <= 32768
    assert lib.blr_workspace_bytes(128, 65536, 32768, 64) > 0
    small = lib.blr_workspace_bytes(2048, 1024, 1024, 256)
    assert lib.blr_workspace_bytes(2049, 1024, 1024, 256) > small
    # tape alone: a f32 [M][r] + c f16 [M][d_out], and the four f16 stagings
    # x.g, dy.h, a.l, db.l kept side by side
    assert small > 2048 * 256 * 4 + 2048 * 1024 * 2 + 2048 * (1024 + 1024 + 256 + 256) * 2


FAKE = 1 << 20  # 16-byte aligned, never dereferenced


def _fwd(lib, **over):
    a = dict(x=FAKE, bu=FAKE, bv=FAKE, g=FAKE, l=FAKE, h=FAKE, y=FAKE, acc=0, M=64, di=128, do=128, r=64,
             ws=FAKE, wsb=1 << 40, s=None)
    a.update(over)
    return lib.blr_forward(a["x"], a["bu"], a["bv"], a["g"], a["l"], a["h"], a["y"], a["acc"], a["M"], a["di"],
                           a["do"], a["r"], a["ws"], a["wsb"], a["s"])


def _bwd(lib, **over):
    a = dict(x=FAKE, dy=FAKE, bu=FAKE, bv=FAKE, g=FAKE, l=FAKE, h=FAKE, dx=FAKE, acc=0, dg=FAKE, dl=FAKE,
             dh=FAKE, gs=0.0, M=64, di=128, do=128, r=64, ws=FAKE + 4096, wsb=1 << 40, s=None)
    a.update(over)
    return lib.blr_backward(a["x"], a["dy"], a["bu"], a["bv"], a["g"], a["l"], a["h"], a["dx"], a["acc"],
                            a["dg"], a["dl"], a["dh"], a["gs"], a["M"], a["di"], a["do"], a["r"], a["ws"],
                            a["wsb"], a["s"])


def test_workspace_reserves_the_staged_dh_rows(lib):
    """A db-product that stages dy writes four dh partial rows per CTA (up to
    160 CTAs) into the workspace, however few tokens the layer has."""
    for d_out in (256, 4096, 32768):
        assert lib.blr_workspace_bytes(64, 128, d_out, 64) >= 4 * 160 * d_out * 4


def test_forward_argument_errors(lib):
    import binary_rank_linear_gb300 as blr
    assert _fwd(lib, x=None) == blr.BLR_ERR_ARG
    assert _fwd(lib, acc=2) == blr.BLR_ERR_ARG
    assert _fwd(lib, M=0) == blr.BLR_ERR_SHAPE
    assert _fwd(lib, r=40) == blr.BLR_ERR_SHAPE
    assert _fwd(lib, y=FAKE + 4) == blr.BLR_ERR_ALIGN
    assert _fwd(lib, wsb=1000) == blr.BLR_ERR_WORKSPACE


def test_backward_argument_errors(lib):
    import binary_rank_linear_gb300 as blr
    assert _bwd(lib, dh=None) == blr.BLR_ERR_ARG
    assert _bwd(lib, gs=3.0) == blr.BLR_ERR_ARG          # not a power of two
    assert _bwd(lib, gs=float("nan")) == blr.BLR_ERR_ARG
    assert _bwd(lib, acc=-1) == blr.BLR_ERR_ARG
    assert _bwd(lib, do=70) == blr.BLR_ERR_SHAPE
    assert _bwd(lib, dx=FAKE + 8) == blr.BLR_ERR_ALIGN
    assert _bwd(lib, wsb=64) == blr.BLR_ERR_WORKSPACE
    # no forward ever ran on this workspace
    assert _bwd(lib) == blr.BLR_ERR_STATE
    assert _bwd(lib, gs=1024.0) == blr.BLR_ERR_STATE


def _sign(lib, **over):
    a = dict(x=FAKE, g=FAKE, l=FAKE, gu=FAKE, gv=FAKE, acc=0, M=64, di=128, do=128, r=64, ws=FAKE + 8192,
             wsb=1 << 40, sws=FAKE, swsb=1 << 40, s=None)
    a.update(over)
    return lib.blr_sign_grads(a["x"], a["g"], a["l"], a["gu"], a["gv"], a["acc"], a["M"], a["di"], a["do"], a["r"],
                              a["ws"], a["wsb"], a["sws"], a["swsb"], a["s"])


def test_sign_workspace_bytes(lib):
    assert lib.blr_sign_workspace_bytes(0, 256, 256, 64) == 0
    assert lib.blr_sign_workspace_bytes(128, 256, 100, 64) == 0
    # two rescaled rank-side f16 operands [M][r] plus a header
    n = lib.blr_sign_workspace_bytes(70, 384, 256, 128)
    assert 2 * 70 * 128 * 2 <= n < 2 * 70 * 128 * 2 + 2048
    assert lib.blr_sign_workspace_bytes(71, 384, 256, 128) > n
    assert lib.blr_sign_workspace_bytes(70, 4096, 4096, 128) == n


def test_sign_grads_argument_errors(lib):
    import binary_rank_linear_gb300 as blr
    assert _sign(lib, gu=None) == blr.BLR_ERR_ARG
    assert _sign(lib, sws=None) == blr.BLR_ERR_ARG
    assert _sign(lib, acc=3) == blr.BLR_ERR_ARG
    assert _sign(lib, r=48) == blr.BLR_ERR_SHAPE
    assert _sign(lib, gv=FAKE + 4) == blr.BLR_ERR_ALIGN
    assert _sign(lib, sws=FAKE + 2) == blr.BLR_ERR_ALIGN
    assert _sign(lib, wsb=64) == blr.BLR_ERR_WORKSPACE
    assert _sign(lib, swsb=64) == blr.BLR_ERR_WORKSPACE
    # no forward/backward ever ran on this workspace
    assert _sign(lib) == blr.BLR_ERR_STATE


def _adam(lib, **over):
    a = dict(w=FAKE, g=FAKE, m1=FAKE, m2=FAKE, mask=None, n=16, step=1, lr=1e-3, b1=0.9, b2=0.999, eps=1e-8,
             gmul=1.0, rel=0.0, s=None)
    a.update(over)
    return lib.blr_adam(a["w"], a["g"], a["m1"], a["m2"], a["mask"], a["n"], a["step"], a["lr"], a["b1"], a["b2"],
                        a["eps"], a["gmul"], a["rel"], a["s"])


def test_adam_argument_errors(lib):
    import binary_rank_linear_gb300 as blr
    assert _adam(lib, m2=None) == blr.BLR_ERR_ARG
    assert _adam(lib, step=0) == blr.BLR_ERR_ARG
    assert _adam(lib, b1=1.0) == blr.BLR_ERR_ARG
    assert _adam(lib, b2=-0.1) == blr.BLR_ERR_ARG
    assert _adam(lib, eps=-1e-8) == blr.BLR_ERR_ARG
    assert _adam(lib, lr=float("inf")) == blr.BLR_ERR_ARG
    assert _adam(lib, rel=float("nan")) == blr.BLR_ERR_ARG
    assert _adam(lib, n=-1) == blr.BLR_ERR_SHAPE
    assert _adam(lib, w=FAKE + 2) == blr.BLR_ERR_ALIGN
    assert _adam(lib, mask=FAKE + 1) == blr.BLR_ERR_ALIGN
    assert _adam(lib, n=0) == blr.BLR_OK  # nothing to do, nothing queued


def _plane(lib, **over):
    a = dict(x=FAKE, p=FAKE, y=FAKE, tr=0, acc=0, scale=1.0, ntok=64, n=128, k=96, ws=FAKE, wsb=1 << 40, s=None)
    a.update(over)
    return lib.blr_plane_linear(a["x"], a["p"], a["y"], a["tr"], a["acc"], a["scale"], a["ntok"], a["n"], a["k"],
                                a["ws"], a["wsb"], a["s"])


def test_plane_linear_argument_errors(lib):
    import binary_rank_linear_gb300 as blr
    assert lib.blr_plane_workspace_bytes(70, 128, 96) == 256 + ((70 * 128 * 2 + 255) // 256) * 256
    assert lib.blr_plane_workspace_bytes(0, 128, 96) == 0
    assert lib.blr_plane_workspace_bytes(8, 100, 96) == 0
    assert _plane(lib, p=None) == blr.BLR_ERR_ARG
    assert _plane(lib, tr=2) == blr.BLR_ERR_ARG
    assert _plane(lib, scale=3.0) == blr.BLR_ERR_ARG
    assert _plane(lib, scale=0.0) == blr.BLR_ERR_ARG
    assert _plane(lib, k=48) == blr.BLR_ERR_SHAPE
    assert _plane(lib, ntok=0) == blr.BLR_ERR_SHAPE
    assert _plane(lib, y=FAKE + 8) == blr.BLR_ERR_ALIGN
    assert _plane(lib, wsb=512) == blr.BLR_ERR_WORKSPACE


def test_paths_argument_errors(lib):
    import ctypes as C
    import binary_rank_linear_gb300 as blr
    one = lib.blr_workspace_bytes(64, 128, 128, 64)
    assert lib.blr_paths_workspace_bytes(3, 64, 128, 128, 64) == 3 * one
    assert lib.blr_paths_workspace_bytes(0, 64, 128, 128, 64) == 0
    assert lib.blr_paths_workspace_bytes(65, 64, 128, 128, 64) == 0
    arr = lambda *v: (C.c_void_p * len(v))(*v)  # noqa: E731
    good = arr(FAKE, FAKE)

    def fwd(P=2, bu=good, y=FAKE, wsb=1 << 40, r=64):
        return lib.blr_forward_paths(FAKE, P, bu, good, good, good, good, y, 0, 64, 128, 128, r, FAKE + 16384, wsb,
                                     None)

    assert fwd(P=0) == blr.BLR_ERR_ARG
    assert fwd(bu=None) == blr.BLR_ERR_ARG
    assert fwd(bu=arr(FAKE, None)) == blr.BLR_ERR_ARG
    assert fwd(bu=arr(FAKE, FAKE + 4)) == blr.BLR_ERR_ALIGN
    assert fwd(r=40) == blr.BLR_ERR_SHAPE
    assert fwd(wsb=one) == blr.BLR_ERR_WORKSPACE

    def bwd(dl=good, gs=0.0):
        return lib.blr_backward_paths(FAKE, FAKE, 2, good, good, good, good, good, FAKE, 0, good, dl, good, gs, 64,
                                      128, 128, 64, FAKE + 32768, 1 << 40, None)

    assert bwd(dl=arr(None, FAKE)) == blr.BLR_ERR_ARG
    assert bwd(gs=3.0) == blr.BLR_ERR_ARG
    assert bwd() == blr.BLR_ERR_STATE  # no forward ran on these workspace slices


def test_pack_argument_errors(lib):
    import binary_rank_linear_gb300 as blr
    assert lib.blr_pack_signs(None, FAKE, 4, 64, None) == blr.BLR_ERR_ARG
    assert lib.blr_pack_signs(FAKE, FAKE, 0, 64, None) == blr.BLR_ERR_SHAPE
    assert lib.blr_pack_signs(FAKE + 4, FAKE, 4, 64, None) == blr.BLR_ERR_ALIGN
    assert lib.blr_unpack_signs(FAKE, None, 4, 64, None) == blr.BLR_ERR_ARG
    assert lib.blr_unpack_signs(FAKE, FAKE, 4, 0, None) == blr.BLR_ERR_SHAPE


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    """No silent fallback: a missing library is an error, not another code path."""
    from binary_rank_linear_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _binding.load()


def test_workspace_release_host_only(lib):
    assert lib.blr_workspace_release(None) == -1  # BLR_ERR_ARG
    assert lib.blr_workspace_release(ctypes.c_void_p(FAKE)) == 0  # no record: nothing to drop, no GPU touched


def test_noalloc_argument_errors(lib):
    fn = lib.blr_forward_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P]
    fn.restype = I
    f = FAKE
    assert fn(None, f, f, f, f, f, f, 0, 64, 128, 128, 64, None) == -1      # null pointer
    assert fn(f, f, f, f, f, f, f, 2, 64, 128, 128, 64, None) == -1         # flag not 0/1
    assert fn(f, f, f, f, f, f, f, 0, 64, 100, 128, 64, None) == -2         # shape rule
    assert fn(f + 4, f, f, f, f, f, f, 0, 64, 128, 128, 64, None) == -3     # alignment
    assert fn(f, f, f, f, f, f, f, 0, 65536, 4096, 4096, 1024, None) == -4  # beyond the fixed scratch
