"""GPU parity of the single-branch recurrent verification (gdn_tree_verify_recurrent,
the measurement baseline of the DFlash-TfM page's results section) against the
fp64 oracle and against the tree verification, through the C ABI."""

import numpy as np
import pytest

import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    import gated_deltanet_tree_gdn_gb300 as gt
    gt.build_library()
    gt.load()


def run_recurrent(w, o_fill=None):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    x = H.to_device(w)
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o = None
    if o_fill is not None:
        dt = torch.bfloat16 if w.dtype == W.BF16 else torch.float32
        o = torch.full((w.B, w.N, w.Hv, w.dv), o_fill, dtype=dt, device="cuda")
    o, U = gt.verify_recurrent(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                               x["S0"], o=o, dev_status=st)
    torch.cuda.synchronize()
    return o.float().cpu().numpy(), U.cpu().numpy(), st.cpu().numpy()


def check(w, units=None):
    o, U, st = run_recurrent(w)
    assert (st == 0).all()
    ref_o, ref_U = __import__("oracle").verify_workload(w, mode="memo", units=units)
    if units is not None:
        sel = H.unit_mask(w, units)
        o, ref_o = o.transpose(0, 2, 1, 3)[sel], ref_o.transpose(0, 2, 1, 3)[sel]
        U, ref_U = U[sel], ref_U[sel]
    eo, eu = H.rel_err(o, ref_o), H.rel_err(U, ref_U)
    H.report(w, dict(o=eo, U=eu, S1=0.0), tag="recurrent")
    assert eo <= H.TOL_O[w.dtype], f"{w.name}: o rel err {eo:.3e}"
    assert eu <= H.TOL_U, f"{w.name}: U rel err {eu:.3e}"


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_recurrent_configs(cfg):
    check(H.ensure_state(W.make_config(cfg)))


def test_recurrent_config4_sampled_units():
    w = W.make_config(4)
    rng = np.random.default_rng(44)
    units = sorted(set(int(b) * w.Hv + int(h) for b in rng.choice(w.B, 10, replace=False)
                       for h in rng.choice(w.Hv, 3, replace=False))
                   | {(w.B - 1) * w.Hv, 0})
    check(w, units=units)


@pytest.mark.parametrize("shape", [
    (2, 37, 1, 2, 32, 32, W.F32, "uniform"),
    (1, 256, 1, 2, 128, 128, W.BF16, "chain"),
    (2, 256, 1, 2, 64, 128, W.BF16, "flatstar"),
    (1, 5, 1, 1, 16, 48, W.F32, "uniform"),
    (1, 1, 1, 1, 128, 128, W.BF16, "chain"),
    (3, 61, 2, 8, 128, 128, W.BF16, "mixed"),
], ids=lambda s: "x".join(map(str, s)))
def test_recurrent_shapes(shape):
    B, N, Hqk, Hv, dk, dv, dt, tree = shape
    check(W.make_custom(seed=300 + N, B=B, N=N, Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, dtype=dt,
                        tree=tree, max_depth=256))


def test_recurrent_matches_tree_verification():
    """Both verifications of the serving workload agree within the output tolerance."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    w = W.make_config(3)
    x = H.to_device(w)
    o1, U1 = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"])
    o2, U2 = gt.verify_recurrent(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                 x["parent"], x["S0"])
    torch.cuda.synchronize()
    assert H.rel_err(o2.float().cpu().numpy(), o1.float().cpu().numpy()) <= H.TOL_O[W.BF16]
    assert H.rel_err(U2.cpu().numpy(), U1.cpu().numpy()) <= H.TOL_U


def test_recurrent_invalid_tree_left_unwritten():
    w = W.make_custom(seed=9, B=3, N=16, Hqk=1, Hv=2, dk=32, dv=32, dtype=W.BF16)
    ref_o, _ = __import__("oracle").verify_workload(w, mode="memo", units=[0, 1, 4, 5])
    w.parent[1, 7] = 12  # not topologically ordered
    o, U, st = run_recurrent(w, o_fill=123.0)
    assert st.tolist() == [0, 1, 0]
    assert (o[1] == 123.0).all()
    assert H.rel_err(o[[0, 2]], ref_o[[0, 2]]) <= H.TOL_O[W.BF16]
