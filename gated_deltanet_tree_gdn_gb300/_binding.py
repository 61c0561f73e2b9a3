"""ctypes binding of libgdntree's C ABI (include/gdn_tree.h).

Argument marshalling only: dtype/shape/contiguity checks on torch tensors,
then device pointers and the current CUDA stream go straight to the C entry
points; every step of the computation runs in the library's kernels.  There
is no fallback: if the library is not built, every call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

BF16, F32 = 0, 1
OK, EINVAL, EUNSUPPORTED, ECUDA = 0, -1, -2, -3
STATUS_OK, STATUS_BAD_TREE, STATUS_BAD_PATH, STATUS_TIMEOUT = 0, 1, 2, 3

SYMBOLS = ("gdn_tree_verify", "gdn_tree_commit", "gdn_tree_commit_verify",
           "gdn_tree_verify_recurrent", "gdn_tree_strerror", "gdn_tree_version")


class Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "N", "Hqk", "Hv", "dk", "dv", "dtype")]


class GdnTreeError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {strerror(code)} (code {code})")
        self.code = code


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libgdntree (built by ``build.build_library``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(
            f"libgdntree is not built ({p} missing): run "
            "`python -m gated_deltanet_tree_gdn_gb300.build` first")
    lib = ctypes.CDLL(p)
    vp, fp, ip = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    lib.gdn_tree_verify.argtypes = [vp, vp, vp, fp, fp, ip, fp, vp, fp, Dims, ip, vp]
    lib.gdn_tree_verify.restype = ctypes.c_int
    lib.gdn_tree_verify_recurrent.argtypes = [vp, vp, vp, fp, fp, ip, fp, vp, fp, Dims, ip, vp]
    lib.gdn_tree_verify_recurrent.restype = ctypes.c_int
    lib.gdn_tree_commit.argtypes = [ip, ip, ip, fp, vp, fp, fp, fp, Dims, ctypes.c_int32, ip, vp]
    lib.gdn_tree_commit.restype = ctypes.c_int
    lib.gdn_tree_commit_verify.argtypes = [ip, ip, ip, fp, vp, fp, ctypes.c_int32, ctypes.c_int32,
                                           fp, fp, vp, vp, vp, fp, fp, ip, vp, fp, Dims, ip, ip,
                                           vp]
    lib.gdn_tree_commit_verify.restype = ctypes.c_int
    lib.gdn_tree_strerror.argtypes = [ctypes.c_int]
    lib.gdn_tree_strerror.restype = ctypes.c_char_p
    lib.gdn_tree_version.argtypes = []
    lib.gdn_tree_version.restype = ctypes.c_int
    if path is None:
        _lib = lib
    return lib


def strerror(code: int) -> str:
    try:
        return load().gdn_tree_strerror(int(code)).decode()
    except RuntimeError:
        return f"code {code}"


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"q/k/v must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def dims_of(q: torch.Tensor, v: torch.Tensor) -> Dims:
    B, N, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    return Dims(B, N, Hqk, Hv, dk, dv, _dtype_code(q))


def verify(q, k, v, log_alpha, beta, parent, S0, *, o=None, U=None, dev_status=None,
           stream=None):
    """Tree verification (C ABI gdn_tree_verify).  Returns (o, U).

    q, k [B,N,Hqk,dk] and v [B,N,Hv,dv] in bf16 or fp32; log_alpha, beta
    [B,N,Hv] fp32; parent [B,N] int32; S0 [B,Hv,dk,dv] fp32.  o [B,N,Hv,dv]
    (q's dtype) and U [B,Hv,N,dv] fp32 are allocated when not given.
    dev_status, if given, is an int32 [B] CUDA tensor filled per sequence.
    """
    return _verify("gdn_tree_verify", q, k, v, log_alpha, beta, parent, S0, o, U, dev_status,
                   stream)


def verify_recurrent(q, k, v, log_alpha, beta, parent, S0, *, o=None, U=None, dev_status=None,
                     stream=None):
    """Single-branch recurrent verification (C ABI gdn_tree_verify_recurrent), the
    baseline the tree verification is measured against: same arguments and
    outputs as ``verify``.  Returns (o, U)."""
    return _verify("gdn_tree_verify_recurrent", q, k, v, log_alpha, beta, parent, S0, o, U,
                   dev_status, stream)


def _verify(symbol, q, k, v, log_alpha, beta, parent, S0, o, U, dev_status, stream):
    B, N, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    dt = q.dtype
    _check(q, "q", dt)
    _check(k, "k", dt, (B, N, Hqk, dk))
    _check(v, "v", dt, (B, N, Hv, dv))
    _check(log_alpha, "log_alpha", torch.float32, (B, N, Hv))
    _check(beta, "beta", torch.float32, (B, N, Hv))
    _check(parent, "parent", torch.int32, (B, N))
    _check(S0, "S0", torch.float32, (B, Hv, dk, dv))
    if o is None:
        o = torch.empty((B, N, Hv, dv), dtype=dt, device=q.device)
    if U is None:
        U = torch.empty((B, Hv, N, dv), dtype=torch.float32, device=q.device)
    _check(o, "o", dt, (B, N, Hv, dv))
    _check(U, "U", torch.float32, (B, Hv, N, dv))
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (B,))
    rc = getattr(load(), symbol)(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                 _ptr(parent), _ptr(S0), _ptr(o), _ptr(U), dims_of(q, v),
                                 _ptr(dev_status), _stream(stream))
    if rc != OK:
        raise GdnTreeError(rc, symbol)
    return o, U


def commit(path, path_len, U, k, log_alpha, S0, *, S1=None, parent=None, dev_status=None,
           stream=None, dv: int | None = None):
    """Delayed state commitment (C ABI gdn_tree_commit).  Returns S1.

    path [B,Lmax] int32 (-1 padded), path_len [B] int32, U [B,Hv,N,dv] fp32
    from verify, k [B,N,Hqk,dk], log_alpha [B,N,Hv], S0 [B,Hv,dk,dv].  S1 is
    allocated when not given; pass S1=S0 for an in-place commit.  parent
    (optional) enables the chain check of the path.
    """
    B, N, Hqk, dk = k.shape
    Hv, dv = S0.shape[1], S0.shape[3]
    _check(path, "path", torch.int32)
    Lmax = path.shape[1]
    _check(path_len, "path_len", torch.int32, (B,))
    _check(U, "U", torch.float32, (B, Hv, N, dv))
    _check(k, "k")
    _check(log_alpha, "log_alpha", torch.float32, (B, N, Hv))
    _check(S0, "S0", torch.float32, (B, Hv, dk, dv))
    if S1 is None:
        S1 = torch.empty_like(S0)
    _check(S1, "S1", torch.float32, (B, Hv, dk, dv))
    if parent is not None:
        _check(parent, "parent", torch.int32, (B, N))
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (B,))
    d = Dims(B, N, Hqk, Hv, dk, dv, _dtype_code(k))
    rc = load().gdn_tree_commit(_ptr(path), _ptr(path_len), _ptr(parent), _ptr(U), _ptr(k),
                                _ptr(log_alpha), _ptr(S0), _ptr(S1), d, Lmax,
                                _ptr(dev_status), _stream(stream))
    if rc != OK:
        raise GdnTreeError(rc, "gdn_tree_commit")
    return S1


def commit_verify(prev_path, prev_path_len, prev_U, prev_k, prev_log_alpha, S_prev, q, k, v,
                  log_alpha, beta, parent, *, S1=None, prev_parent=None, o=None, U=None,
                  commit_status=None, verify_status=None, stream=None):
    """One decoding iteration (C ABI gdn_tree_commit_verify): commit the previous
    tree's accepted path into S1, then verify the next tree from S1.
    Returns (S1, o, U).  S1=S_prev commits in place; U=prev_U reuses the buffer."""
    B, N, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    dt = q.dtype
    Np = prev_k.shape[1]
    _check(prev_path, "prev_path", torch.int32)
    Lmax = prev_path.shape[1]
    _check(prev_path_len, "prev_path_len", torch.int32, (B,))
    _check(prev_U, "prev_U", torch.float32, (B, Hv, Np, dv))
    _check(prev_k, "prev_k", dt, (B, Np, Hqk, dk))
    _check(prev_log_alpha, "prev_log_alpha", torch.float32, (B, Np, Hv))
    _check(S_prev, "S_prev", torch.float32, (B, Hv, dk, dv))
    _check(q, "q", dt)
    _check(k, "k", dt, (B, N, Hqk, dk))
    _check(v, "v", dt, (B, N, Hv, dv))
    _check(log_alpha, "log_alpha", torch.float32, (B, N, Hv))
    _check(beta, "beta", torch.float32, (B, N, Hv))
    _check(parent, "parent", torch.int32, (B, N))
    if S1 is None:
        S1 = torch.empty_like(S_prev)
    if o is None:
        o = torch.empty((B, N, Hv, dv), dtype=dt, device=q.device)
    if U is None:
        U = torch.empty((B, Hv, N, dv), dtype=torch.float32, device=q.device)
    _check(S1, "S1", torch.float32, (B, Hv, dk, dv))
    _check(o, "o", dt, (B, N, Hv, dv))
    _check(U, "U", torch.float32, (B, Hv, N, dv))
    if prev_parent is not None:
        _check(prev_parent, "prev_parent", torch.int32, (B, Np))
    for name, st in (("commit_status", commit_status), ("verify_status", verify_status)):
        if st is not None:
            _check(st, name, torch.int32, (B,))
    rc = load().gdn_tree_commit_verify(
        _ptr(prev_path), _ptr(prev_path_len), _ptr(prev_parent), _ptr(prev_U), _ptr(prev_k),
        _ptr(prev_log_alpha), Np, Lmax, _ptr(S_prev), _ptr(S1), _ptr(q), _ptr(k), _ptr(v),
        _ptr(log_alpha), _ptr(beta), _ptr(parent), _ptr(o), _ptr(U), dims_of(q, v),
        _ptr(commit_status), _ptr(verify_status), _stream(stream))
    if rc != OK:
        raise GdnTreeError(rc, "gdn_tree_commit_verify")
    return S1, o, U
