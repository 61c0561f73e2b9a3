"""The C-ABI library builds, loads and exports every entry point declared in
include/*.h; host-side argument checks answer before any CUDA call (these
tests make no compute call and need no GPU)."""

import ctypes
import glob
import os
import re

import pytest

import gated_deltanet_tree_gdn_gb300 as gt
from gated_deltanet_tree_gdn_gb300 import _binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(gdn_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return _binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("gdn_tree_verify", "gdn_tree_commit", "gdn_tree_strerror", "gdn_tree_version"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_version_and_strerror(lib):
    assert lib.gdn_tree_version() >= 100
    assert b"invalid" in lib.gdn_tree_strerror(gt.EINVAL)
    assert b"path" in lib.gdn_tree_strerror(gt.STATUS_BAD_PATH)


def _dims(**kw):
    d = dict(B=2, N=16, Hqk=2, Hv=4, dk=64, dv=64, dtype=gt.BF16)
    d.update(kw)
    return gt.Dims(**d)


def _verify(lib, dims, ptr=16):
    p = ctypes.c_void_p(ptr) if ptr else None
    return lib.gdn_tree_verify(p, p, p, p, p, p, p, p, p, dims, None, None)


def _commit(lib, dims, ptr=16, Lmax=4):
    p = ctypes.c_void_p(ptr) if ptr else None
    return lib.gdn_tree_commit(p, p, None, p, p, p, p, ctypes.c_void_p(1 << 40), dims, Lmax,
                               None, None)


@pytest.mark.parametrize("kw,code", [
    (dict(N=1025), gt.EUNSUPPORTED),
    (dict(dk=24), gt.EUNSUPPORTED),
    (dict(dv=256), gt.EUNSUPPORTED),
    (dict(dtype=7), gt.EUNSUPPORTED),
    (dict(Hv=3), gt.EINVAL),
    (dict(Hqk=0), gt.EINVAL),
    (dict(B=-1), gt.EINVAL),
])
def test_bad_dims_rejected_before_launch(lib, kw, code):
    assert _verify(lib, _dims(**kw)) == code
    assert _commit(lib, _dims(**kw)) == code


def test_null_or_misaligned_pointers_rejected(lib):
    assert _verify(lib, _dims(), ptr=0) == gt.EINVAL
    assert _verify(lib, _dims(), ptr=24) == gt.EINVAL  # 8-byte aligned only
    assert _commit(lib, _dims(), ptr=0) == gt.EINVAL
    assert _commit(lib, _dims(), Lmax=-1) == gt.EINVAL
    assert _commit(lib, _dims(), Lmax=1025) == gt.EUNSUPPORTED


def test_recurrent_baseline_keeps_the_on_chip_limit(lib):
    # trees past 256 nodes verify through the chunked kernel; the single-branch
    # baseline keeps its path in shared memory and refuses them before launch
    p = ctypes.c_void_p(16)
    assert lib.gdn_tree_verify_recurrent(*(p,) * 9, _dims(N=257), None, None) == gt.EUNSUPPORTED
    # at 256 nodes the shape passes and the NULL pointers are what is refused
    assert lib.gdn_tree_verify_recurrent(*(None,) * 9, _dims(N=256), None, None) == gt.EINVAL
    assert _verify(lib, _dims(N=1024), ptr=0) == gt.EINVAL


def test_partial_overlap_of_S0_and_S1_rejected(lib):
    d = _dims()
    p = ctypes.c_void_p(1 << 20)
    q = ctypes.c_void_p((1 << 20) + 256)  # overlaps S0 but is not S0
    assert lib.gdn_tree_commit(p, p, None, p, p, p, p, q, d, 4, None, None) == gt.EINVAL


def test_empty_calls_are_noops(lib):
    assert _verify(lib, _dims(B=0), ptr=0) == gt.OK
    assert _verify(lib, _dims(N=0), ptr=0) == gt.OK
    assert _commit(lib, _dims(B=0), ptr=0) == gt.OK


def _commit_verify(lib, dims, prev_N, U, prev_U):
    """gdn_tree_commit_verify with distinct, aligned placeholder pointers except
    for U and prev_U (no call here gets past the host checks)."""
    P = [ctypes.c_void_p((1 << 36) + (i << 28)) for i in range(16)]
    return lib.gdn_tree_commit_verify(
        P[0], P[1], None, ctypes.c_void_p(prev_U), P[2], P[3], prev_N, 4, P[4], P[5],
        P[6], P[7], P[8], P[9], P[10], P[11], P[12], ctypes.c_void_p(U), dims, None, None,
        None)


def test_commit_verify_refuses_U_overlapping_prev_U(lib):
    d = _dims(N=16)
    base = 1 << 44
    unit_bytes = d.Hv * 16 * d.dv * 4
    # the same buffer but trees of different sizes: units would overwrite each
    # other's previous rows before reading them
    assert _commit_verify(lib, d, 12, base, base) == gt.EINVAL
    # a partial overlap
    assert _commit_verify(lib, d, 16, base + unit_bytes, base) == gt.EINVAL
    assert _commit_verify(lib, d, 16, base, base + 256) == gt.EINVAL


def test_binding_marshalling_helpers():
    """The binding's per-call marshalling: pointers pass as plain integers (NULL as
    None), the dims struct matches the tensors and is reused for equal shapes, and a
    shape or dtype mismatch is refused before any call."""
    import torch
    from gated_deltanet_tree_gdn_gb300 import _binding as bd
    q = torch.zeros((2, 8, 4, 32), dtype=torch.bfloat16)
    v = torch.zeros((2, 8, 8, 32), dtype=torch.bfloat16)
    d = bd.dims_of(q, v)
    assert (d.B, d.N, d.Hqk, d.Hv, d.dk, d.dv, d.dtype) == (2, 8, 4, 8, 32, 32, bd.BF16)
    assert bd.dims_of(q.clone(), v.clone()) is d
    d2 = bd.dims_of(q.float(), v.float())
    assert d2 is not d and d2.dtype == bd.F32
    assert bd._ptr(None) is None and bd._ptr(q) == q.data_ptr()
    with pytest.raises(ValueError):  # not a CUDA tensor
        bd._check(q, "q", torch.bfloat16, (2, 8, 4, 32))
