"""The bounded on-device waits of the tensor-core verification, the 256-node
kernel, the tensor-core chunk pass and the tensor-core commit, made to run out
on purpose (no fault, no trap, nothing left in flight): a short wait limit and a
solve-barrier arrival that is withheld (test-only controls read from the
environment).  The kernel must report GDN_TREE_STATUS_TIMEOUT for the
sequences it could not finish, leave the other sequences correct, free its
resources, and leave the context usable: the next normal call on the same
stream matches the oracle.  The tensor-core commit's state-copy wait is made to
run out the same way (a copy that is expected but never issued)."""

import numpy as np
import pytest

import oracle
import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu

LIMIT_NS = "1000000"  # 1 ms


@pytest.fixture(scope="module", autouse=True)
def built_library():
    import gated_deltanet_tree_gdn_gb300 as gt
    gt.build_library()
    gt.load()


def _workload():
    # 8 x 4 units: fewer than the SMs, so every unit has a CTA of its own
    return W.make_custom(seed=901, B=8, N=96, Hqk=2, Hv=4, dk=128, dv=128, dtype=W.BF16,
                         tree="random", max_depth=24)


def _withheld(w, b):
    """A node of sequence b with a child (its children's waits run out)."""
    node = int(w.parent[b, w.N - 1])
    assert node >= 0
    return node


def test_solve_barrier_wait_runs_out(monkeypatch):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = _workload()
    b, h = 3, 1
    monkeypatch.setenv("GDN_TREE_TEST_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("GDN_TREE_TEST_WITHHOLD_NODE", f"{b * w.Hv + h}:{_withheld(w, b)}")
    x = H.to_device(w)
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                     dev_status=st)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert s[b] == gt.STATUS_TIMEOUT
    assert (np.delete(s, b) == gt.STATUS_OK).all()
    ok = np.arange(w.B) != b
    o_ref, U_ref = oracle.verify_workload(w)
    assert H.rel_err(o.float().cpu().numpy()[ok], o_ref[ok]) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy()[ok], U_ref[ok]) <= H.TOL_U
    # the context is still usable: a normal call on the same stream is exact
    monkeypatch.delenv("GDN_TREE_TEST_WAIT_LIMIT_NS")
    monkeypatch.delenv("GDN_TREE_TEST_WITHHOLD_NODE")
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))


def test_fused_iteration_reports_timeout_for_both_calls(monkeypatch):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = _workload()
    x = H.to_device(w)
    _, U_prev = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                          x["S0"])
    b = 5
    monkeypatch.setenv("GDN_TREE_TEST_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("GDN_TREE_TEST_WITHHOLD_NODE", f"{b * w.Hv}:{_withheld(w, b)}")
    cs = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    vs = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    S1, o, U = gt.commit_verify(x["path"], x["path_len"], U_prev, x["k"], x["log_alpha"],
                                x["S0"], x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                                x["parent"], prev_parent=x["parent"], commit_status=cs,
                                verify_status=vs)
    torch.cuda.synchronize()
    c, v = cs.cpu().numpy(), vs.cpu().numpy()
    assert c[b] == gt.STATUS_TIMEOUT and v[b] == gt.STATUS_TIMEOUT
    assert (np.delete(c, b) == 0).all() and (np.delete(v, b) == 0).all()
    ok = np.arange(w.B) != b
    S1_ref = oracle.commit_workload(w)
    assert H.rel_err(S1.cpu().numpy()[ok], S1_ref[ok]) <= H.TOL_S1


def test_mid_kernel_solve_wait_runs_out(monkeypatch):
    """The same on the 256-node kernel: a withheld solve-barrier arrival of one
    (sequence, head) unit makes its descendants' bounded waits run out."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=903, B=6, N=160, Hqk=2, Hv=4, dk=128, dv=128, dtype=W.BF16,
                      tree="random", max_depth=24)
    b, h = 4, 2
    monkeypatch.setenv("GDN_TREE_TEST_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("GDN_TREE_TEST_WITHHOLD_NODE", f"{b * w.Hv + h}:{_withheld(w, b)}")
    x = H.to_device(w)
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                     dev_status=st)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert s[b] == gt.STATUS_TIMEOUT
    assert (np.delete(s, b) == gt.STATUS_OK).all()
    ok = np.arange(w.B) != b
    o_ref, U_ref = oracle.verify_workload(w)
    assert H.rel_err(o.float().cpu().numpy()[ok], o_ref[ok]) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy()[ok], U_ref[ok]) <= H.TOL_U
    monkeypatch.delenv("GDN_TREE_TEST_WAIT_LIMIT_NS")
    monkeypatch.delenv("GDN_TREE_TEST_WITHHOLD_NODE")
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))


def test_long_kernel_parent_wait_runs_out(monkeypatch):
    """The chunk pass with R on the tensor cores (trees past 256 nodes): a withheld
    arrival of a node whose child sits in the same chunk makes that child's bounded
    wait run out."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=905, B=3, N=300, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="random", max_depth=24)
    b, h = 1, 1
    kids = [t for t in range(w.N) if w.parent[b, t] >= 128 * (t // 128)]
    node = int(w.parent[b, kids[-1]])
    monkeypatch.setenv("GDN_TREE_TEST_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("GDN_TREE_TEST_WITHHOLD_NODE", f"{b * w.Hv + h}:{node}")
    x = H.to_device(w)
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                     dev_status=st)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert s[b] == gt.STATUS_TIMEOUT
    assert (np.delete(s, b) == gt.STATUS_OK).all()
    ok = np.arange(w.B) != b
    o_ref, U_ref = oracle.verify_workload(w)
    assert H.rel_err(o.float().cpu().numpy()[ok], o_ref[ok]) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy()[ok], U_ref[ok]) <= H.TOL_U


def test_commit_state_copy_wait_runs_out(monkeypatch):
    """The tensor-core commit (paths of more than 32 entries): one sequence's
    state copy is expected but never issued, so its bounded wait runs out."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=905, B=8, N=96, Hqk=2, Hv=4, dk=128, dv=128, dtype=W.BF16,
                      tree="random", max_depth=24, lmax=48)
    x = H.to_device(w)
    _, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"])
    b = 2
    monkeypatch.setenv("GDN_TREE_TEST_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("GDN_TREE_TEST_WITHHOLD_COPY", str(b))
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    S1 = torch.full_like(x["S0"], 5.0)
    gt.commit(x["path"], x["path_len"], U, x["k"], x["log_alpha"], x["S0"], S1=S1,
              parent=x["parent"], dev_status=st)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert s[b] == gt.STATUS_TIMEOUT and (np.delete(s, b) == 0).all()
    got = S1.cpu().numpy()
    assert (got[b] == 5.0).all()  # left unwritten
    ok = np.arange(w.B) != b
    S1_ref = oracle.commit_workload(w)
    assert H.rel_err(got[ok], S1_ref[ok]) <= H.TOL_S1
    monkeypatch.delenv("GDN_TREE_TEST_WITHHOLD_COPY")
    monkeypatch.delenv("GDN_TREE_TEST_WAIT_LIMIT_NS")
    S1b = gt.commit(x["path"], x["path_len"], U, x["k"], x["log_alpha"], x["S0"],
                    parent=x["parent"], dev_status=st)
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    assert H.rel_err(S1b.cpu().numpy(), S1_ref) <= H.TOL_S1


def test_timeout_with_units_taken_over(monkeypatch):
    """More units than SMs (256 on 152), so running CTAs take over the units of CTAs not
    launched yet.  A withheld solve-barrier arrival makes one unit's wait run out: its
    CTA reports TIMEOUT for the units it owns (that unit, and at most the next one and
    the one a request in flight took over, which may be other sequences') and leaves
    them unwritten; every other sequence is exact and the next call is clean."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=907, B=64, N=96, Hqk=2, Hv=4, dk=128, dv=128, dtype=W.BF16,
                      tree="random", max_depth=24)
    b, h = 37, 2
    monkeypatch.setenv("GDN_TREE_TEST_WAIT_LIMIT_NS", LIMIT_NS)
    monkeypatch.setenv("GDN_TREE_TEST_WITHHOLD_NODE", f"{b * w.Hv + h}:{_withheld(w, b)}")
    x = H.to_device(w)
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                     dev_status=st)
    torch.cuda.synchronize()
    s = st.cpu().numpy()
    assert s[b] == gt.STATUS_TIMEOUT
    others = np.flatnonzero((s != gt.STATUS_OK) & (np.arange(w.B) != b))
    assert len(others) <= 2 and (s[others] == gt.STATUS_TIMEOUT).all()
    ok = s == gt.STATUS_OK
    o_ref, U_ref = oracle.verify_workload(w)
    assert H.rel_err(o.float().cpu().numpy()[ok], o_ref[ok]) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy()[ok], U_ref[ok]) <= H.TOL_U
    monkeypatch.delenv("GDN_TREE_TEST_WAIT_LIMIT_NS")
    monkeypatch.delenv("GDN_TREE_TEST_WITHHOLD_NODE")
    st2 = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o2, U2 = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                       dev_status=st2)
    torch.cuda.synchronize()
    assert (st2.cpu().numpy() == gt.STATUS_OK).all()
    assert H.rel_err(o2.float().cpu().numpy(), o_ref) <= H.TOL_O[W.BF16]
    assert H.rel_err(U2.cpu().numpy(), U_ref) <= H.TOL_U
