"""ctypes binding of libblr.so: the C ABI of include/blr.h with the same names.

Argument marshalling only: torch tensors are checked for device, dtype, shape
and contiguity, their data pointers and the current CUDA stream are passed to
the library, and negative status codes become ``BlrError``. Every step of the
layer runs in the library's CUDA kernels; if the library is missing this module
raises instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB

BLR_OK = 0
BLR_ERR_ARG = -1
BLR_ERR_SHAPE = -2
BLR_ERR_ALIGN = -3
BLR_ERR_WORKSPACE = -4
BLR_ERR_STATE = -5
BLR_ERR_CUDA = -6
BLR_ERR_DEVICE_CHECK = -7
BLR_ERR_UNSUPPORTED_DEVICE = -8

_lib = None


class BlrError(RuntimeError):
    """A negative status returned by the blr library."""

    def __init__(self, code: int, where: str):
        self.code = code
        msg = load().blr_status_string(code).decode()
        super().__init__(f"{where}: {msg} (status {code})")


def load() -> ctypes.CDLL:
    """Load libblr.so from the package tree (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise RuntimeError(
            f"{LIB} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(LIB)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.blr_workspace_bytes.argtypes = [I, I, I, I]
    lib.blr_workspace_bytes.restype = Z
    lib.blr_pack_signs.argtypes = [P, P, I, I, P]
    lib.blr_unpack_signs.argtypes = [P, P, I, I, P]
    lib.blr_forward.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P, Z, P]
    lib.blr_backward.argtypes = [P, P, P, P, P, P, P, P, I, P, P, P, F, I, I, I, I, P, Z, P]
    lib.blr_sign_workspace_bytes.argtypes = [I, I, I, I]
    lib.blr_sign_workspace_bytes.restype = Z
    lib.blr_sign_grads.argtypes = [P, P, P, P, P, I, I, I, I, I, P, Z, P, Z, P]
    lib.blr_adam.argtypes = [P, P, P, P, P, I, I, F, F, F, F, F, F, P]
    PP = ctypes.POINTER(ctypes.c_void_p)
    lib.blr_paths_workspace_bytes.argtypes = [I, I, I, I, I]
    lib.blr_paths_workspace_bytes.restype = Z
    lib.blr_forward_paths.argtypes = [P, I, PP, PP, PP, PP, PP, P, I, I, I, I, I, P, Z, P]
    lib.blr_backward_paths.argtypes = [P, P, I, PP, PP, PP, PP, PP, P, I, PP, PP, PP, F, I, I, I, I, P, Z, P]
    lib.blr_plane_workspace_bytes.argtypes = [I, I, I]
    lib.blr_plane_workspace_bytes.restype = Z
    lib.blr_plane_linear.argtypes = [P, P, P, I, I, F, I, I, I, P, Z, P]
    lib.blr_check_status.argtypes = [P, Z, P, ctypes.POINTER(ctypes.c_uint32)]
    lib.blr_noalloc_check_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32)]
    lib.blr_workspace_release.argtypes = [P]
    lib.blr_status_string.argtypes = [I]
    lib.blr_status_string.restype = ctypes.c_char_p
    lib.blr_trace_begin.argtypes = [I]
    lib.blr_trace_read.argtypes = [I, ctypes.POINTER(ctypes.c_float)]
    lib.blr_trace_read.restype = ctypes.c_char_p
    for f in ("blr_pack_signs", "blr_unpack_signs", "blr_forward", "blr_backward", "blr_sign_grads", "blr_adam", "blr_plane_linear", "blr_forward_paths", "blr_backward_paths",
              "blr_check_status", "blr_noalloc_check_status", "blr_workspace_release",
              "blr_trace_begin", "blr_trace_end", "blr_trace_count"):
        getattr(lib, f).restype = I
    _lib = lib
    return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor, name: str, dtype, shape=None) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t.data_ptr()


def _check(code: int, where: str) -> None:
    if code != BLR_OK:
        raise BlrError(code, where)


def words_per_row(r: int) -> int:
    return (r + 31) // 32


def workspace_bytes(M: int, d_in: int, d_out: int, r: int) -> int:
    return int(load().blr_workspace_bytes(M, d_in, d_out, r))


def alloc_workspace(M: int, d_in: int, d_out: int, r: int, device=None) -> torch.Tensor:
    """A caller-owned workspace for one layer instance (torch owns the memory)."""
    n = workspace_bytes(M, d_in, d_out, r)
    if n == 0:
        raise BlrError(BLR_ERR_SHAPE, "workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def pack_signs(src: torch.Tensor, bits: torch.Tensor = None, stream=None) -> torch.Tensor:
    """bits[rows][ceil(r/32)] (int32 storage of u32 words) from src[rows][r] f32."""
    rows, r = src.shape
    if bits is None:
        bits = torch.empty(rows, words_per_row(r), dtype=torch.int32, device=src.device)
    _check(load().blr_pack_signs(_ptr(src, "src", torch.float32), _ptr(bits, "bits", torch.int32,
                                 (rows, words_per_row(r))), rows, r, _stream(stream)), "blr_pack_signs")
    return bits


def unpack_signs(bits: torch.Tensor, r: int, dst: torch.Tensor = None, stream=None) -> torch.Tensor:
    """+-1 f16 [rows][r] from a bitmap, through the GEMMs' expansion code."""
    rows = bits.shape[0]
    if dst is None:
        dst = torch.empty(rows, r, dtype=torch.float16, device=bits.device)
    _check(load().blr_unpack_signs(_ptr(bits, "bits", torch.int32, (rows, words_per_row(r))),
                                   _ptr(dst, "dst", torch.float16, (rows, r)), rows, r, _stream(stream)),
           "blr_unpack_signs")
    return dst


def forward(x, bits_u, bits_v, g, l, h, y, ws, accumulate: bool = False, stream=None) -> torch.Tensor:
    """y (+)= h.c with a = (x.g) S_V, c = (a.l) S_U^T; the tape goes to ``ws``."""
    M, d_in = x.shape
    d_out, r = h.shape[0], l.shape[0]
    w = words_per_row(r)
    code = load().blr_forward(
        _ptr(x, "x", torch.float32, (M, d_in)), _ptr(bits_u, "bits_u", torch.int32, (d_out, w)),
        _ptr(bits_v, "bits_v", torch.int32, (d_in, w)), _ptr(g, "g", torch.float32, (d_in,)),
        _ptr(l, "l", torch.float32, (r,)), _ptr(h, "h", torch.float32, (d_out,)),
        _ptr(y, "y", torch.float32, (M, d_out)), int(bool(accumulate)), M, d_in, d_out, r,
        _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check(code, "blr_forward")
    return y


def backward(x, dy, bits_u, bits_v, g, l, h, dx, dg, dl, dh, ws, gscale: float = 0.0,
             accumulate: bool = False, stream=None) -> torch.Tensor:
    """dx (+)= g.dx'; dg, dl, dh += their token sums (the last forward's tape in ``ws``)."""
    M, d_in = x.shape
    d_out, r = h.shape[0], l.shape[0]
    w = words_per_row(r)
    code = load().blr_backward(
        _ptr(x, "x", torch.float32, (M, d_in)), _ptr(dy, "dy", torch.float32, (M, d_out)),
        _ptr(bits_u, "bits_u", torch.int32, (d_out, w)), _ptr(bits_v, "bits_v", torch.int32, (d_in, w)),
        _ptr(g, "g", torch.float32, (d_in,)), _ptr(l, "l", torch.float32, (r,)),
        _ptr(h, "h", torch.float32, (d_out,)), _ptr(dx, "dx", torch.float32, (M, d_in)),
        int(bool(accumulate)), _ptr(dg, "dg", torch.float32, (d_in,)), _ptr(dl, "dl", torch.float32, (r,)),
        _ptr(dh, "dh", torch.float32, (d_out,)), float(gscale), M, d_in, d_out, r,
        _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check(code, "blr_backward")
    return dx


def paths_workspace_bytes(P: int, M: int, d_in: int, d_out: int, r: int) -> int:
    return int(load().blr_paths_workspace_bytes(P, M, d_in, d_out, r))


def alloc_paths_workspace(P: int, M: int, d_in: int, d_out: int, r: int, device=None) -> torch.Tensor:
    n = paths_workspace_bytes(P, M, d_in, d_out, r)
    if n == 0:
        raise BlrError(BLR_ERR_SHAPE, "paths_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def path_workspace(ws: torch.Tensor, p: int, M: int, d_in: int, d_out: int, r: int) -> torch.Tensor:
    """Path p's slice of a multi-path workspace (its tape, e.g. for sign_grads)."""
    one = workspace_bytes(M, d_in, d_out, r)
    return ws[p * one:(p + 1) * one]


def _ptr_array(tensors, name, dtype, shape):
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = _ptr(t, f"{name}[{i}]", dtype, shape)
    return arr


def forward_paths(x, paths, y, ws, accumulate: bool = False, stream=None) -> torch.Tensor:
    """y (+)= sum_p W_hat_p x; ``paths`` is a list of dicts with bu, bv, g, l, h."""
    M, d_in = x.shape
    d_out, r = paths[0]["h"].shape[0], paths[0]["l"].shape[0]
    w, P = words_per_row(r), len(paths)
    code = load().blr_forward_paths(
        _ptr(x, "x", torch.float32, (M, d_in)), P,
        _ptr_array([p["bu"] for p in paths], "bu", torch.int32, (d_out, w)),
        _ptr_array([p["bv"] for p in paths], "bv", torch.int32, (d_in, w)),
        _ptr_array([p["g"] for p in paths], "g", torch.float32, (d_in,)),
        _ptr_array([p["l"] for p in paths], "l", torch.float32, (r,)),
        _ptr_array([p["h"] for p in paths], "h", torch.float32, (d_out,)),
        _ptr(y, "y", torch.float32, (M, d_out)), int(bool(accumulate)), M, d_in, d_out, r,
        _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check(code, "blr_forward_paths")
    return y


def backward_paths(x, dy, paths, dx, grads, ws, gscale: float = 0.0, accumulate: bool = False,
                   stream=None) -> torch.Tensor:
    """dx (+)= sum_p dx_p; ``grads`` is a list of dicts with dg, dl, dh per path (always +=)."""
    M, d_in = x.shape
    d_out, r = paths[0]["h"].shape[0], paths[0]["l"].shape[0]
    w, P = words_per_row(r), len(paths)
    code = load().blr_backward_paths(
        _ptr(x, "x", torch.float32, (M, d_in)), _ptr(dy, "dy", torch.float32, (M, d_out)), P,
        _ptr_array([p["bu"] for p in paths], "bu", torch.int32, (d_out, w)),
        _ptr_array([p["bv"] for p in paths], "bv", torch.int32, (d_in, w)),
        _ptr_array([p["g"] for p in paths], "g", torch.float32, (d_in,)),
        _ptr_array([p["l"] for p in paths], "l", torch.float32, (r,)),
        _ptr_array([p["h"] for p in paths], "h", torch.float32, (d_out,)),
        _ptr(dx, "dx", torch.float32, (M, d_in)), int(bool(accumulate)),
        _ptr_array([q["dg"] for q in grads], "dg", torch.float32, (d_in,)),
        _ptr_array([q["dl"] for q in grads], "dl", torch.float32, (r,)),
        _ptr_array([q["dh"] for q in grads], "dh", torch.float32, (d_out,)),
        float(gscale), M, d_in, d_out, r, _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check(code, "blr_backward_paths")
    return dx


def sign_workspace_bytes(M: int, d_in: int, d_out: int, r: int) -> int:
    return int(load().blr_sign_workspace_bytes(M, d_in, d_out, r))


def alloc_sign_workspace(M: int, d_in: int, d_out: int, r: int, device=None) -> torch.Tensor:
    """The second, caller-owned workspace of ``sign_grads`` (transposed f16 operands)."""
    n = sign_workspace_bytes(M, d_in, d_out, r)
    if n == 0:
        raise BlrError(BLR_ERR_SHAPE, "sign_workspace_bytes")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def sign_grads(x, g, l, gu, gv, ws, sws, accumulate: bool = False, stream=None):
    """G_U = diag(h) dy^T a diag(l) -> gu [d_out][r], G_V = diag(g) x^T db diag(l) -> gv [d_in][r],
    from the tape of the last forward/backward pair on ``ws``."""
    M, d_in = x.shape
    d_out, r = gu.shape
    code = load().blr_sign_grads(
        _ptr(x, "x", torch.float32, (M, d_in)), _ptr(g, "g", torch.float32, (d_in,)),
        _ptr(l, "l", torch.float32, (r,)), _ptr(gu, "gu", torch.float32, (d_out, r)),
        _ptr(gv, "gv", torch.float32, (d_in, r)), int(bool(accumulate)), M, d_in, d_out, r,
        _ptr(ws, "ws", torch.uint8), ws.numel(), _ptr(sws, "sws", torch.uint8), sws.numel(), _stream(stream))
    _check(code, "blr_sign_grads")
    return gu, gv


def plane_workspace_bytes(ntok: int, n: int, k: int) -> int:
    return int(load().blr_plane_workspace_bytes(ntok, n, k))


def alloc_plane_workspace(ntok: int, n: int, k: int, device=None) -> torch.Tensor:
    nb = plane_workspace_bytes(ntok, n, k)
    if nb == 0:
        raise BlrError(BLR_ERR_SHAPE, "plane_workspace_bytes")
    return torch.empty(nb, dtype=torch.uint8, device=device or "cuda")


def plane_linear(x, plane, y, ws, transpose: bool = False, accumulate: bool = False, scale: float = 1.0,
                 stream=None) -> torch.Tensor:
    """y (+)= x plane^T (x [ntok][k]) or, with transpose, y (+)= x plane (x [ntok][n]); plane [n][k] f16."""
    n, k = plane.shape
    ntok = x.shape[0]
    kin, nout = (n, k) if transpose else (k, n)
    code = load().blr_plane_linear(
        _ptr(x, "x", torch.float32, (ntok, kin)), _ptr(plane, "plane", torch.float16, (n, k)),
        _ptr(y, "y", torch.float32, (ntok, nout)), int(bool(transpose)), int(bool(accumulate)), float(scale),
        ntok, n, k, _ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream))
    _check(code, "blr_plane_linear")
    return y


def adam(w, grad, m1, m2, step: int, lr: float, b1: float = 0.9, b2: float = 0.999, eps: float = 1e-8,
         mask=None, gmul: float = 1.0, rel: float = 0.0, stream=None):
    """One Adam step in place on w, m1, m2 (f32 [n] CUDA tensors); mask 0 freezes an entry."""
    n = w.numel()
    shape = tuple(w.shape)
    code = load().blr_adam(
        _ptr(w, "w", torch.float32), _ptr(grad, "grad", torch.float32, shape), _ptr(m1, "m1", torch.float32, shape),
        _ptr(m2, "m2", torch.float32, shape), _ptr(mask, "mask", torch.float32, shape) if mask is not None else None,
        n, int(step), float(lr), float(b1), float(b2), float(eps), float(gmul), float(rel), _stream(stream))
    _check(code, "blr_adam")
    return w


def check_status(ws: torch.Tensor, stream=None) -> int:
    """Synchronise and return the workspace's device status word (0 = no failure)."""
    code = ctypes.c_uint32(0)
    rc = load().blr_check_status(_ptr(ws, "ws", torch.uint8), ws.numel(), _stream(stream), ctypes.byref(code))
    if rc not in (BLR_OK, BLR_ERR_DEVICE_CHECK):
        raise BlrError(rc, "blr_check_status")
    return int(code.value)


def workspace_release(ws: torch.Tensor) -> None:
    """Forget the tape record of ``ws`` (call before freeing a workspace whose
    address may be handed out again)."""
    _check(load().blr_workspace_release(_ptr(ws, "ws", torch.uint8)), "blr_workspace_release")


def noalloc_check_status(stream=None) -> int:
    """Synchronise and return the status word of the current device's
    blr_forward_noalloc scratch array (0 = no failure)."""
    code = ctypes.c_uint32(0)
    rc = load().blr_noalloc_check_status(_stream(stream), ctypes.byref(code))
    if rc not in (BLR_OK, BLR_ERR_DEVICE_CHECK):
        raise BlrError(rc, "blr_noalloc_check_status")
    return int(code.value)


def trace_begin(capacity: int = 64) -> None:
    _check(load().blr_trace_begin(capacity), "blr_trace_begin")


def trace_end(read: bool = True) -> list:
    """Stop tracing; return [(kernel name, ms), ...] for the kernels recorded
    (nothing with read=False, e.g. when the calls were captured into a graph
    that has not run yet: ``trace_read`` then reads each replay)."""
    lib = load()
    lib.blr_trace_end()
    return trace_read() if read else []


def trace_count() -> int:
    return int(load().blr_trace_count())


def trace_read(first: int = 0, last: int = None) -> list:
    """[(kernel name, ms), ...] of trace entries first .. last-1 (synchronises)."""
    lib = load()
    last = lib.blr_trace_count() if last is None else last
    out = []
    for i in range(first, last):
        ms = ctypes.c_float(0.0)
        name = lib.blr_trace_read(i, ctypes.byref(ms))
        if name is None:
            raise BlrError(BLR_ERR_CUDA, "blr_trace_read")
        out.append((name.decode(), float(ms.value)))
    return out


def forward_noalloc(x, bits_u, bits_v, g, l, h, y, accumulate: bool = False, stream=None) -> torch.Tensor:
    """blr_forward_noalloc: the forward pass for callers that cannot allocate device memory.

    Same inputs and output as ``forward`` but no workspace: the library uses a
    fixed scratch array in its own device memory (BLR_NOALLOC_SCRATCH_BYTES =
    16 MiB, held by every GPU that loads the library). The first call on a
    device looks up that array's address, so make it before any stream
    capture. Calls share the array: calls that overlap on the GPU race.
    """
    lib = load()
    fn = lib.blr_forward_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    fn.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P]
    fn.restype = I
    M, d_in = x.shape
    d_out, r = h.shape[0], l.shape[0]
    w = words_per_row(r)
    code = fn(_ptr(x, "x", torch.float32, (M, d_in)), _ptr(bits_u, "bits_u", torch.int32, (d_out, w)),
              _ptr(bits_v, "bits_v", torch.int32, (d_in, w)), _ptr(g, "g", torch.float32, (d_in,)),
              _ptr(l, "l", torch.float32, (r,)), _ptr(h, "h", torch.float32, (d_out,)),
              _ptr(y, "y", torch.float32, (M, d_out)), int(bool(accumulate)), M, d_in, d_out, r, _stream(stream))
    _check(code, "blr_forward_noalloc")
    return y
