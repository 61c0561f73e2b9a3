"""GPU parity of the chunkwise path for trees that are one branch (parent of t =
t - 1, past 128 nodes, bf16 with dk = dv = 128), which the 256-node kernel and the
chunk pass run for such units: the state passed between 64-node chunks, through
the C ABI, against the fp64 oracle.  Chains sit beside other tree families in one
call too (the same launch takes both paths)."""

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


CHAINS = [
    # (B, N, Hqk, Hv): chunk tails of every size, one and several chunks
    (2, 129, 1, 2),
    (2, 200, 2, 4),
    (1, 256, 1, 2),
    (2, 257, 1, 2),
    (1, 513, 1, 2),
    (1, 1024, 1, 2),
]


@pytest.mark.parametrize("idx", range(len(CHAINS)), ids=["x".join(map(str, c)) for c in CHAINS])
def test_chains_match_oracle(idx, monkeypatch):
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    B, N, Hqk, Hv = CHAINS[idx]
    w = W.make_custom(seed=1100 + idx, B=B, N=N, Hqk=Hqk, Hv=Hv, dk=128, dv=128,
                      dtype=W.BF16, tree="chain", max_depth=N)
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))


def test_chain_strong_decay_and_high_beta(monkeypatch):
    """log alpha down to -4 a node and beta = 0.99: the state's decay between chunks
    spans e^-256, and the terms inside a chunk are large."""
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=1120, B=2, N=256, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="chain", max_depth=256, la_range=(0.01, 4.0), beta_kind="uniform")
    w.beta[:] = np.float32(0.99)
    gpu = H.run_gpu(w)
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))
    assert np.isfinite(gpu["o"]).all() and np.isfinite(gpu["U"]).all()


@pytest.mark.parametrize("N", [256, 400])
def test_chains_beside_other_trees(N, monkeypatch):
    """Every tree family in one call: the chain takes the chunkwise path, the others
    the 256-node kernel's (N = 256) or the chunk pass's (N = 400) tree path."""
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    w = W.make_custom(seed=1130 + N, B=6, N=N, Hqk=2, Hv=4, dk=128, dv=128, dtype=W.BF16,
                      tree="mixed", max_depth=N)
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))


@pytest.mark.parametrize("kernel", ["mid", "long"])
def test_tree_kernels_still_take_chains_when_forced(kernel, monkeypatch):
    """With a kernel forced the chunkwise path stays out: the tree kernels' own
    chain handling is covered on the same shape."""
    monkeypatch.setenv("GDN_TREE_KERNEL", kernel)
    w = W.make_custom(seed=1140, B=2, N=200, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="chain", max_depth=200)
    gpu = H.run_gpu(w)
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))


@pytest.mark.parametrize("Ns", [[129, 200, 0, 256, 64, 5], [300, 700, 1, 0, 257]],
                         ids=["256-node-kernel", "chunk-pass"])
def test_ragged_chains_with_a_state_pool(Ns, monkeypatch):
    """Ragged batches of chains (short ones too: a chain of 5 takes one partial
    chunk) through the packed entry points, states from a pool; then the commit of
    each accepted path into the pool."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    from tests.test_packed_gpu import Packed, check_verify
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    P = Packed(1150 + len(Ns), Ns, 1, 2, 128, 128, W.BF16, n_slots=9, tree="chain")
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


def test_decoding_iteration_into_chains(monkeypatch):
    """One decoding iteration (commit of the previous path, then the verification of
    the next tree from S1) whose next trees are 200-node chains and mixed families:
    the verification's chains take the chunkwise path."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    import oracle
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    prev = W.make_custom(seed=1160, B=3, N=128, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                         tree="random", max_depth=24)
    nxt = W.make_custom(seed=1161, B=3, N=200, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                        tree="mixed", max_depth=200)
    xp, xn = H.to_device(prev), H.to_device(nxt)
    _, U_prev = gt.verify(xp["q"], xp["k"], xp["v"], xp["log_alpha"], xp["beta"], xp["parent"],
                          xp["S0"])
    cs = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    vs = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    S1, o, U = gt.commit_verify(xp["path"], xp["path_len"], U_prev, xp["k"], xp["log_alpha"],
                                xp["S0"], xn["q"], xn["k"], xn["v"], xn["log_alpha"],
                                xn["beta"], xn["parent"], prev_parent=xp["parent"],
                                commit_status=cs, verify_status=vs)
    torch.cuda.synchronize()
    assert (cs.cpu().numpy() == 0).all() and (vs.cpu().numpy() == 0).all()
    S1_ref = oracle.commit_workload(prev)
    assert H.rel_err(S1.cpu().numpy(), S1_ref) <= H.TOL_S1
    # the next tree against the oracle run from the state the GPU committed
    o_ref, U_ref = oracle.verify(nxt.q, nxt.k, nxt.v, nxt.log_alpha, nxt.beta, nxt.parent,
                                 S1.cpu().numpy())
    assert H.rel_err(o.float().cpu().numpy(), o_ref) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy(), U_ref) <= H.TOL_U
