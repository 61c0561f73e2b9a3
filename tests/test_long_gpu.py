"""GPU parity of trees longer than the on-chip kernels take (N up to 1024): the
two-level chunk pass of the verification and commit paths longer than 256
entries, through the C ABI, against the fp64 oracle.  The chunked kernel is
also forced onto small shapes (GDN_TREE_KERNEL=long: its tensor-core form for
bf16 with dk = dv = 128; =long_cuda: the CUDA-core form), where its chunk
boundary (128 nodes) and ragged tails meet every tree family."""

import numpy as np
import pytest

import oracle
import workloads as W
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    import gated_deltanet_tree_gdn_gb300 as gt
    gt.build_library()
    gt.load()


LONG = [
    # (B, N, Hqk, Hv, dk, dv, dtype, tree, max_depth)
    (2, 300, 1, 2, 128, 128, W.BF16, "mixed", 300),     # three chunks, ragged tail
    (1, 1024, 1, 2, 128, 128, W.BF16, "chain", 1024),   # the longest tree and path
    (2, 700, 2, 4, 64, 64, W.F32, "random", 60),
    (1, 513, 1, 1, 32, 48, W.F32, "uniform", 513),
    (2, 1024, 1, 2, 128, 128, W.BF16, "flatstar", 2),   # a forest of 1024 roots
    (6, 400, 1, 2, 128, 128, W.BF16, "mixed", 400),     # every tree family
]


_ORACLE = {}  # the oracle's results by case, shared by the kernels' runs


def _long_case(idx):
    B, N, Hqk, Hv, dk, dv, dt, tree, depth = LONG[idx]
    w = W.make_custom(seed=700 + idx, B=B, N=N, Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, dtype=dt,
                      tree=tree, max_depth=depth)
    if idx not in _ORACLE:
        _ORACLE[idx] = H.run_oracle(w)
    return w, _ORACLE[idx]


@pytest.mark.parametrize("kernel", ["auto", "long_cuda"])
@pytest.mark.parametrize("idx", range(len(LONG)), ids=["x".join(map(str, c[:8])) for c in LONG])
def test_long_trees_match_oracle(idx, kernel, monkeypatch):
    """The default dispatch (bf16 with dk = dv = 128: the chunk pass with R and the
    seeds on the tensor cores) and the chunk pass on CUDA cores."""
    if kernel == "auto":
        monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    else:
        monkeypatch.setenv("GDN_TREE_KERNEL", kernel)
    w, ref = _long_case(idx)
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, ref))


def test_commit_path_longer_than_256():
    """A chain of 1024 with its whole path accepted (the commit's blocked scan)."""
    w = W.make_custom(seed=731, B=2, N=1024, Hqk=1, Hv=2, dk=64, dv=64, dtype=W.F32,
                      tree="chain", max_depth=1024, lmax=1024)
    w.path[:] = np.arange(1024, dtype=np.int32)
    w.path_len[:] = [1024, 777]
    gpu = H.run_gpu(w)
    assert (gpu["status_commit"] == 0).all()
    ref = oracle.commit_workload(w)
    assert H.rel_err(gpu["S1"], ref) <= H.TOL_S1


SMALL = [
    # (B, N, Hqk, Hv, dk, dv, dtype, tree): the chunked kernel forced
    (2, 37, 1, 2, 32, 32, W.F32, "uniform"),
    (3, 129, 1, 1, 128, 128, W.BF16, "mixed"),
    (2, 256, 1, 4, 128, 128, W.BF16, "chain"),
    (6, 200, 2, 4, 64, 128, W.BF16, "mixed"),
    (1, 5, 1, 1, 16, 48, W.F32, "uniform"),
    (1, 1, 1, 1, 128, 128, W.BF16, "chain"),
    (5, 33, 4, 8, 128, 128, W.BF16, "flatstar"),
]


@pytest.mark.parametrize("kernel", ["long", "long_cuda"])
@pytest.mark.parametrize("idx", range(len(SMALL)), ids=["x".join(map(str, c)) for c in SMALL])
def test_chunked_kernel_forced_on_small_shapes(idx, kernel, monkeypatch):
    monkeypatch.setenv("GDN_TREE_KERNEL", kernel)
    B, N, Hqk, Hv, dk, dv, dt, tree = SMALL[idx]
    w = W.make_custom(seed=760 + idx, B=B, N=N, Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, dtype=dt,
                      tree=tree, max_depth=N)
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))


def test_long_strong_decay_and_high_beta(monkeypatch):
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=780, B=6, N=600, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="mixed", max_depth=600, la_range=(0.01, 4.0), beta_kind="uniform")
    w.beta[:] = np.float32(0.99)
    gpu = H.run_gpu(w)
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))
    assert np.isfinite(gpu["o"]).all() and np.isfinite(gpu["U"]).all()


def test_long_invalid_tree_reported_and_left_unwritten(monkeypatch):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=790, B=3, N=300, Hqk=1, Hv=2, dk=64, dv=64, dtype=W.BF16,
                      tree="random", max_depth=40)
    w.parent[1, 290] = 295  # not topologically ordered
    x = H.to_device(w)
    st = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    o = torch.full((3, 300, 2, 64), 123.0, dtype=torch.bfloat16, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"],
                     o=o, dev_status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [gt.STATUS_OK, gt.STATUS_BAD_TREE, gt.STATUS_OK]
    on = o.float().cpu().numpy()
    assert (on[1] == 123.0).all()
    ok = [0, 2]
    ref_o, ref_U = oracle.verify(w.q[ok], w.k[ok], w.v[ok], w.log_alpha[ok], w.beta[ok],
                                 w.parent[ok], w.S0[ok])
    assert H.rel_err(on[ok], ref_o) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy()[ok], ref_U) <= H.TOL_U


def test_long_packed_pool_verify_and_commit(monkeypatch):
    """Ragged batch whose longest tree takes the chunked kernel, with a state pool."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    from tests.test_packed_gpu import Packed, check_verify
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    P = Packed(801, [300, 5, 0, 640, 129], 1, 2, 128, 128, W.BF16, n_slots=8)
    x = P.device()
    st = torch.full((P.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify_packed(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                            x["cu"], x["pool"], state_slot=x["slot"], dev_status=st)
    torch.cuda.synchronize()
    check_verify(P, o.float().cpu().numpy(), U.cpu().numpy(), st.cpu().numpy())
    pool = x["pool"]
    cs = torch.full((P.B,), -7, dtype=torch.int32, device="cuda")
    gt.commit_packed(x["path"], x["path_len"], U, x["k"], x["log_alpha"], x["cu"], pool,
                     pool_out=pool, state_slot=x["slot"], parent=x["parent"], dev_status=cs)
    torch.cuda.synchronize()
    assert (cs.cpu().numpy() == 0).all()
    got, ref = pool.cpu().numpy(), P.oracle_commit()
    used = np.zeros(len(ref), bool)
    used[P.slot] = True
    assert H.rel_err(got[used], ref[used]) <= H.TOL_S1
    assert np.array_equal(got[~used], P.pool[~used])


def test_commit_verify_with_a_long_previous_tree(monkeypatch):
    """One decoding iteration whose previous tree (and accepted path) is longer
    than the fused kernel takes: commit then verify, on the same stream."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    prev = W.make_custom(seed=811, B=2, N=500, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                         tree="chain", max_depth=500)
    nxt = W.make_custom(seed=812, B=2, N=128, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                        tree="mixed", max_depth=24)
    xp, xn = H.to_device(prev), H.to_device(nxt)
    _, U_prev = gt.verify(xp["q"], xp["k"], xp["v"], xp["log_alpha"], xp["beta"], xp["parent"],
                          xp["S0"])
    cs = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    vs = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    S1, o, U = gt.commit_verify(xp["path"], xp["path_len"], U_prev, xp["k"], xp["log_alpha"],
                                xp["S0"], xn["q"], xn["k"], xn["v"], xn["log_alpha"],
                                xn["beta"], xn["parent"], prev_parent=xp["parent"],
                                commit_status=cs, verify_status=vs)
    torch.cuda.synchronize()
    assert (cs.cpu().numpy() == 0).all() and (vs.cpu().numpy() == 0).all()
    S1_ref = oracle.commit_workload(prev)
    o_ref, U_ref = oracle.verify(nxt.q, nxt.k, nxt.v, nxt.log_alpha, nxt.beta, nxt.parent,
                                 S1_ref.astype(np.float32))
    assert H.rel_err(S1.cpu().numpy(), S1_ref) <= H.TOL_S1
    assert H.rel_err(o.float().cpu().numpy(), o_ref) <= H.TOL_O[W.BF16]
    # U against the oracle run from the state the GPU committed (U is linear in it)
    _, U_own = oracle.verify(nxt.q, nxt.k, nxt.v, nxt.log_alpha, nxt.beta, nxt.parent,
                             S1.cpu().numpy())
    assert H.rel_err(U.cpu().numpy(), U_own) <= H.TOL_U


def test_stress_workload_on_the_chunked_kernel(monkeypatch):
    """The stress workload (64 x 32 units of 256-node chains, stars and random trees,
    log alpha down to -4, a beta = 0.99 sequence) through the chunked kernel,
    compared over the whole tensor."""
    monkeypatch.setenv("GDN_TREE_KERNEL", "long")
    w = W.make_config(4)
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    errs = H.compare(w, gpu, H.run_oracle(w))
    H.assert_parity(w, errs)
    assert np.isfinite(gpu["o"]).all() and np.isfinite(gpu["U"]).all()
