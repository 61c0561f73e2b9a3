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
STATUS_OK, STATUS_BAD_TREE, STATUS_BAD_PATH, STATUS_TIMEOUT, STATUS_BAD_LAYOUT = 0, 1, 2, 3, 4

SYMBOLS = ("gdn_tree_verify", "gdn_tree_commit", "gdn_tree_commit_verify",
           "gdn_tree_verify_recurrent", "gdn_tree_verify_packed", "gdn_tree_commit_packed",
           "gdn_tree_commit_verify_packed", "gdn_tree_build_topw", "gdn_tree_strerror",
           "gdn_tree_version")


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
    i32 = ctypes.c_int32
    lib.gdn_tree_verify_packed.argtypes = [vp, vp, vp, fp, fp, ip, ip, i32, fp, ip, i32, vp, fp,
                                           Dims, ip, vp]
    lib.gdn_tree_verify_packed.restype = ctypes.c_int
    lib.gdn_tree_commit_packed.argtypes = [ip, ip, ip, ip, i32, fp, vp, fp, fp, fp, ip, i32, Dims,
                                           i32, ip, vp]
    lib.gdn_tree_commit_packed.restype = ctypes.c_int
    lib.gdn_tree_commit_verify_packed.argtypes = [ip, ip, ip, ip, i32, fp, vp, fp, i32, i32, fp,
                                                  fp, ip, i32, vp, vp, vp, fp, fp, ip, ip, i32,
                                                  vp, fp, Dims, ip, ip, vp]
    lib.gdn_tree_commit_verify_packed.restype = ctypes.c_int
    lib.gdn_tree_build_topw.argtypes = [fp, i32, i32, i32, i32, i32, ip, ip, fp, ip, vp]
    lib.gdn_tree_build_topw.restype = ctypes.c_int
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


# The marshalling below runs on every call, ahead of a launch that can take only a few
# microseconds (a decoding step of one sequence), so it is kept lean: pointers go to
# ctypes as plain integers, shapes are compared as they are, and the stream is read as
# its raw handle.

def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and t.shape != shape:
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


# the current stream's handle without building a Stream object (the public call is the
# fallback where the accessor is absent)
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        return _raw_stream(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


_dims_cache: dict = {}


def dims_of(q: torch.Tensor, v: torch.Tensor) -> Dims:
    key = (q.shape, v.shape, q.dtype)
    d = _dims_cache.get(key)
    if d is None:
        B, N, Hqk, dk = q.shape
        Hv, dv = v.shape[2], v.shape[3]
        d = Dims(B, N, Hqk, Hv, dk, dv, _dtype_code(q))
        if len(_dims_cache) < 256:
            _dims_cache[key] = d
    return d


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


# ---------------------------------------------------------------------------
# packed (ragged) batches with a state pool
# ---------------------------------------------------------------------------

def _packed_rows(cu_nodes, B):
    _check(cu_nodes, "cu_nodes", torch.int32, (B + 1,))


def _slots(state_slot, B, pool):
    if state_slot is not None:
        _check(state_slot, "state_slot", torch.int32, (B,))
    return pool.shape[0]


def verify_packed(q, k, v, log_alpha, beta, parent, cu_nodes, state_pool, *, state_slot=None,
                  N_max=None, o=None, U=None, dev_status=None, stream=None):
    """Tree verification of a packed (ragged) batch (C ABI gdn_tree_verify_packed).
    Returns (o, U).

    q, k [T,Hqk,dk], v [T,Hv,dv] (bf16 or fp32); log_alpha, beta [T,Hv]; parent
    [T] (indices within each sequence); cu_nodes [B+1] int32 row offsets;
    state_pool [n_slots,Hv,dk,dv] fp32 with state_slot [B] (None: slot b).
    N_max is the largest tree (computed from cu_nodes on the host if None).
    o [T,Hv,dv] and U [Hv,T,dv] are allocated when not given."""
    T, Hqk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    B = cu_nodes.shape[0] - 1
    dt = q.dtype
    _packed_rows(cu_nodes, B)
    _check(q, "q", dt)
    _check(k, "k", dt, (T, Hqk, dk))
    _check(v, "v", dt, (T, Hv, dv))
    _check(log_alpha, "log_alpha", torch.float32, (T, Hv))
    _check(beta, "beta", torch.float32, (T, Hv))
    _check(parent, "parent", torch.int32, (T,))
    _check(state_pool, "state_pool", torch.float32, (state_pool.shape[0], Hv, dk, dv))
    n_slots = _slots(state_slot, B, state_pool)
    if N_max is None:
        N_max = int((cu_nodes[1:] - cu_nodes[:-1]).max().item()) if B > 0 else 0
    if o is None:
        o = torch.empty((T, Hv, dv), dtype=dt, device=q.device)
    if U is None:
        U = torch.empty((Hv, T, dv), dtype=torch.float32, device=q.device)
    _check(o, "o", dt, (T, Hv, dv))
    _check(U, "U", torch.float32, (Hv, T, dv))
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (B,))
    d = Dims(B, N_max, Hqk, Hv, dk, dv, _dtype_code(q))
    rc = load().gdn_tree_verify_packed(_ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha), _ptr(beta),
                                       _ptr(parent), _ptr(cu_nodes), T, _ptr(state_pool),
                                       _ptr(state_slot), n_slots, _ptr(o), _ptr(U), d,
                                       _ptr(dev_status), _stream(stream))
    if rc != OK:
        raise GdnTreeError(rc, "gdn_tree_verify_packed")
    return o, U


def commit_packed(path, path_len, U, k, log_alpha, cu_nodes, pool_in, *, pool_out=None,
                  state_slot=None, parent=None, N_max=None, dev_status=None, stream=None):
    """Delayed commitment of a packed batch (C ABI gdn_tree_commit_packed):
    pool_out[state_slot[b]] = the state after sequence b's accepted path.  Returns
    pool_out (pool_out=pool_in commits in place; a new pool starts as a copy of
    pool_in, so that untouched slots keep their states)."""
    T, Hqk, dk = k.shape
    Hv, dv = pool_in.shape[1], pool_in.shape[3]
    B = cu_nodes.shape[0] - 1
    _packed_rows(cu_nodes, B)
    _check(path, "path", torch.int32)
    Lmax = path.shape[1]
    _check(path_len, "path_len", torch.int32, (B,))
    _check(U, "U", torch.float32, (Hv, T, dv))
    _check(k, "k")
    _check(log_alpha, "log_alpha", torch.float32, (T, Hv))
    _check(pool_in, "pool_in", torch.float32)
    n_slots = _slots(state_slot, B, pool_in)
    if pool_out is None:
        pool_out = pool_in.clone()
    _check(pool_out, "pool_out", torch.float32, tuple(pool_in.shape))
    if parent is not None:
        _check(parent, "parent", torch.int32, (T,))
    if dev_status is not None:
        _check(dev_status, "dev_status", torch.int32, (B,))
    if N_max is None:
        N_max = int((cu_nodes[1:] - cu_nodes[:-1]).max().item()) if B > 0 else 0
    d = Dims(B, N_max, Hqk, Hv, dk, dv, _dtype_code(k))
    rc = load().gdn_tree_commit_packed(_ptr(path), _ptr(path_len), _ptr(parent), _ptr(cu_nodes),
                                       T, _ptr(U), _ptr(k), _ptr(log_alpha), _ptr(pool_in),
                                       _ptr(pool_out), _ptr(state_slot), n_slots, d, Lmax,
                                       _ptr(dev_status), _stream(stream))
    if rc != OK:
        raise GdnTreeError(rc, "gdn_tree_commit_packed")
    return pool_out


def commit_verify_packed(prev_path, prev_path_len, prev_U, prev_k, prev_log_alpha, prev_cu_nodes,
                         pool_in, q, k, v, log_alpha, beta, parent, cu_nodes, *, pool_out=None,
                         state_slot=None, prev_parent=None, prev_N_max=None, N_max=None, o=None,
                         U=None, commit_status=None, verify_status=None, stream=None):
    """One decoding iteration of a packed batch (C ABI gdn_tree_commit_verify_packed).
    Returns (pool_out, o, U); pool_out=pool_in commits in place."""
    T, Hqk, dk = q.shape
    Hv, dv = v.shape[1], v.shape[2]
    Tp = prev_k.shape[0]
    B = cu_nodes.shape[0] - 1
    dt = q.dtype
    _packed_rows(cu_nodes, B)
    _packed_rows(prev_cu_nodes, B)
    _check(prev_path, "prev_path", torch.int32)
    Lmax = prev_path.shape[1]
    _check(prev_path_len, "prev_path_len", torch.int32, (B,))
    _check(prev_U, "prev_U", torch.float32, (Hv, Tp, dv))
    _check(prev_k, "prev_k", dt, (Tp, Hqk, dk))
    _check(prev_log_alpha, "prev_log_alpha", torch.float32, (Tp, Hv))
    _check(pool_in, "pool_in", torch.float32)
    n_slots = _slots(state_slot, B, pool_in)
    _check(q, "q", dt)
    _check(k, "k", dt, (T, Hqk, dk))
    _check(v, "v", dt, (T, Hv, dv))
    _check(log_alpha, "log_alpha", torch.float32, (T, Hv))
    _check(beta, "beta", torch.float32, (T, Hv))
    _check(parent, "parent", torch.int32, (T,))
    if pool_out is None:
        pool_out = pool_in.clone()
    if o is None:
        o = torch.empty((T, Hv, dv), dtype=dt, device=q.device)
    if U is None:
        U = torch.empty((Hv, T, dv), dtype=torch.float32, device=q.device)
    _check(pool_out, "pool_out", torch.float32, tuple(pool_in.shape))
    _check(o, "o", dt, (T, Hv, dv))
    _check(U, "U", torch.float32, (Hv, T, dv))
    if prev_parent is not None:
        _check(prev_parent, "prev_parent", torch.int32, (Tp,))
    for name, st in (("commit_status", commit_status), ("verify_status", verify_status)):
        if st is not None:
            _check(st, name, torch.int32, (B,))
    if N_max is None:
        N_max = int((cu_nodes[1:] - cu_nodes[:-1]).max().item()) if B > 0 else 0
    if prev_N_max is None:
        prev_N_max = int((prev_cu_nodes[1:] - prev_cu_nodes[:-1]).max().item()) if B > 0 else 0
    d = Dims(B, N_max, Hqk, Hv, dk, dv, _dtype_code(q))
    rc = load().gdn_tree_commit_verify_packed(
        _ptr(prev_path), _ptr(prev_path_len), _ptr(prev_parent), _ptr(prev_cu_nodes), Tp,
        _ptr(prev_U), _ptr(prev_k), _ptr(prev_log_alpha), prev_N_max, Lmax, _ptr(pool_in),
        _ptr(pool_out), _ptr(state_slot), n_slots, _ptr(q), _ptr(k), _ptr(v), _ptr(log_alpha),
        _ptr(beta), _ptr(parent), _ptr(cu_nodes), T, _ptr(o), _ptr(U), d, _ptr(commit_status),
        _ptr(verify_status), _stream(stream))
    if rc != OK:
        raise GdnTreeError(rc, "gdn_tree_commit_verify_packed")
    return pool_out, o, U


# ---------------------------------------------------------------------------
# draft-tree construction
# ---------------------------------------------------------------------------

def build_topw(cand_logp, w: int, max_depth: int, *, parent=None, cand_index=None, score=None,
               n_built=None, stream=None):
    """Top-w best-first draft-tree construction (C ABI gdn_tree_build_topw).

    cand_logp [B, N, c] fp32: the log-probabilities of each node's c candidate
    children.  Returns (parent [B, N] int32, cand_index [B, N] int32, score [B, N]
    fp32, n_built [B] int32); outputs are allocated when not given."""
    _check(cand_logp, "cand_logp", torch.float32)
    B, N, c = cand_logp.shape
    dev = cand_logp.device
    if parent is None:
        parent = torch.empty((B, N), dtype=torch.int32, device=dev)
    if cand_index is None:
        cand_index = torch.empty((B, N), dtype=torch.int32, device=dev)
    if score is None:
        score = torch.empty((B, N), dtype=torch.float32, device=dev)
    if n_built is None:
        n_built = torch.empty((B,), dtype=torch.int32, device=dev)
    _check(parent, "parent", torch.int32, (B, N))
    _check(cand_index, "cand_index", torch.int32, (B, N))
    _check(score, "score", torch.float32, (B, N))
    _check(n_built, "n_built", torch.int32, (B,))
    rc = load().gdn_tree_build_topw(_ptr(cand_logp), B, N, c, w, max_depth, _ptr(parent),
                                    _ptr(cand_index), _ptr(score), _ptr(n_built),
                                    _stream(stream))
    if rc != OK:
        raise GdnTreeError(rc, "gdn_tree_build_topw")
    return parent, cand_index, score, n_built
