"""fp64 CPU oracle for rollback-free GDN tree verification.

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product package.  It shares no code
with the CUDA library.

Two independent implementations live here:

* ``gdn_oracle.c`` (wrapped below): the GDN recurrence of the DFlash-TfM page
  (gist.science/it/paper/2607.06763, section 3, "Sfida") run literally along
  every root-to-node path (``mode="path"``) or memoised per parent
  (``mode="memo"``; same operations in the same order, so bitwise equal), and
  the delayed commitment of section 3 as the recurrence run along the
  accepted path.
* ``chunked.py``: the chunked, masked-triangular-solve form of section 3
  ("Soluzione": interaction matrices X and Y, the system (I+X)U = ...), written
  with dense numpy/scipy for one (sequence, head) unit.  It pins the algebra
  the GPU follows against the recurrence.

Parity status: pinned (see tests/test_oracle_pins.py); no function here is
unpinned.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libgdnoracle.so")
_lock = threading.Lock()
_lib = None


class _Dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("B", "N", "Hqk", "Hv", "dk", "dv")]


def compile_library(out_path: str = _LIB_PATH, defines: tuple[str, ...] = ()) -> str:
    """Compile the C oracle with gcc (also used to build planted-mistake
    variants for the tests that check the pins bite)."""
    os.makedirs(os.path.dirname(out_path), exist_ok=True)
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           "-pthread", _SRC, "-o", tmp, "-lm"] + [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_library(_LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    lib = ctypes.CDLL(path)
    dp = ctypes.POINTER(ctypes.c_double)
    ip = ctypes.POINTER(ctypes.c_int32)
    lib.gdn_oracle_verify.argtypes = [dp, dp, dp, dp, dp, ip, dp, dp, dp, _Dims,
                                      ctypes.c_int, ip, ctypes.c_int, ctypes.c_int]
    lib.gdn_oracle_verify.restype = ctypes.c_int
    lib.gdn_oracle_commit.argtypes = [ip, ip, ip, dp, dp, dp, dp, dp, dp, _Dims,
                                      ctypes.c_int, ip, ctypes.c_int, ctypes.c_int]
    lib.gdn_oracle_commit.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """The oracle library (built on first use) or a given variant of it."""
    global _lib
    if path is not None:
        return _bind(path)
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a, t):
    return a.ctypes.data_as(ctypes.POINTER(t))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class OracleError(RuntimeError):
    pass


def verify(q, k, v, log_alpha, beta, parent, S0, *, mode: str = "memo",
           units=None, threads: int | None = None, lib=None):
    """Run the oracle's verification.

    Shapes: q, k [B,N,Hqk,dk]; v [B,N,Hv,dv]; log_alpha, beta [B,N,Hv];
    parent [B,N]; S0 [B,Hv,dk,dv].  Returns (o [B,N,Hv,dv], U [B,Hv,N,dv]) in
    fp64; entries of units not listed in ``units`` (flat b*Hv+h) are NaN.
    """
    lib = lib or load()
    q, k, v, la, be, S0 = map(_f64, (q, k, v, log_alpha, beta, S0))
    parent = _i32(parent)
    B, N, Hqk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    d = _Dims(B, N, Hqk, Hv, dk, dv)
    o = np.full((B, N, Hv, dv), np.nan)
    U = np.full((B, Hv, N, dv), np.nan)
    if units is None:
        up, nu = None, 0
    else:
        ua = _i32(units)
        up, nu = _ptr(ua, ctypes.c_int32), len(ua)
    m = {"path": 0, "memo": 1}[mode]
    rc = lib.gdn_oracle_verify(_ptr(q, ctypes.c_double), _ptr(k, ctypes.c_double),
                               _ptr(v, ctypes.c_double), _ptr(la, ctypes.c_double),
                               _ptr(be, ctypes.c_double), _ptr(parent, ctypes.c_int32),
                               _ptr(S0, ctypes.c_double), _ptr(o, ctypes.c_double),
                               _ptr(U, ctypes.c_double), d, m, up, nu,
                               threads or default_threads())
    if rc != 0:
        raise OracleError(f"gdn_oracle_verify returned {rc}")
    return o, U


def commit(path, path_len, k, v, log_alpha, beta, S0, *, parent=None, units=None,
           threads: int | None = None, lib=None):
    """Delayed commitment: S1 [B,Hv,dk,dv] (fp64) after running the recurrence
    along path[b, :path_len[b]] from S0.  ``parent`` (optional) makes the
    oracle reject paths that are not root-to-node chains."""
    lib = lib or load()
    k, v, la, be, S0 = map(_f64, (k, v, log_alpha, beta, S0))
    path, path_len = _i32(path), _i32(path_len)
    B, N, Hqk, dk = k.shape
    Hv, dv = v.shape[2], v.shape[3]
    d = _Dims(B, N, Hqk, Hv, dk, dv)
    S1 = np.full((B, Hv, dk, dv), np.nan)
    pp = None
    if parent is not None:
        parent_arr = _i32(parent)  # kept alive for the call
        pp = _ptr(parent_arr, ctypes.c_int32)
    if units is None:
        up, nu = None, 0
    else:
        ua = _i32(units)
        up, nu = _ptr(ua, ctypes.c_int32), len(ua)
    rc = lib.gdn_oracle_commit(_ptr(path, ctypes.c_int32), _ptr(path_len, ctypes.c_int32),
                               pp, _ptr(k, ctypes.c_double), _ptr(v, ctypes.c_double),
                               _ptr(la, ctypes.c_double), _ptr(be, ctypes.c_double),
                               _ptr(S0, ctypes.c_double), _ptr(S1, ctypes.c_double), d,
                               path.shape[1], up, nu, threads or default_threads())
    if rc != 0:
        raise OracleError(f"gdn_oracle_commit returned {rc}")
    return S1


def warmup_state(k, v, log_alpha, beta, Hv: int, dk: int, dv: int,
                 threads: int | None = None) -> np.ndarray:
    """State reached from S = 0 by running the recurrence over a plain token
    sequence (a chain): the fp64 result rounded to fp32 (round to nearest).
    k [B,T,Hqk,dk], v [B,T,Hv,dv], gates [B,T,Hv]."""
    B, T = k.shape[0], k.shape[1]
    path = np.tile(np.arange(T, dtype=np.int32), (B, 1))
    plen = np.full(B, T, dtype=np.int32)
    S = commit(path, plen, k, v, log_alpha, beta, np.zeros((B, Hv, dk, dv)),
               threads=threads)
    return S.astype(np.float32)


def verify_workload(w, **kw):
    return verify(w.q, w.k, w.v, w.log_alpha, w.beta, w.parent, w.S0, **kw)


def commit_workload(w, **kw):
    return commit(w.path, w.path_len, w.k, w.v, w.log_alpha, w.beta, w.S0,
                  parent=w.parent, **kw)
