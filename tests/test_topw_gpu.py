"""GPU parity of the top-w best-first draft-tree construction (gdn_tree_build_topw,
DFlash-TfM section 2) against the oracle, through the C ABI: every output exact
(parent, candidate index and n_built are integers decided by fp32 comparisons
that both sides make in fp32; scores are the same fp32 sums)."""

import numpy as np
import pytest

from oracle.topw import build_topw as oracle_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built_library():
    import gated_deltanet_tree_gdn_gb300 as gt
    gt.build_library()
    gt.load()


def run(logp, w, max_depth):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    x = torch.from_numpy(np.ascontiguousarray(logp, np.float32)).cuda()
    p, j, s, n = gt.build_topw(x, w, max_depth)
    torch.cuda.synchronize()
    return p.cpu().numpy(), j.cpu().numpy(), s.cpu().numpy(), n.cpu().numpy()


def check(logp, w, max_depth):
    p, j, s, n = run(logp, w, max_depth)
    rp, rj, rs, rd, rn, _ = oracle_build(logp, w, max_depth)
    np.testing.assert_array_equal(n, rn)
    np.testing.assert_array_equal(p, rp)
    np.testing.assert_array_equal(j, rj)
    np.testing.assert_array_equal(s, rs)  # NaN past n_built on both sides
    return p, n


@pytest.mark.parametrize("B,N,c,w,max_depth", [
    (8, 64, 4, 4, 16),      # the top-4 best-first trees of the dense-prefill workload
    (32, 128, 4, 4, 24),
    (5, 256, 8, 8, 12),
    (3, 40, 3, 1, 40),      # sequential best-first
    (7, 31, 2, 5, 6),
    (4, 100, 32, 17, 9),
    (2, 1, 4, 1, 5),        # the root alone
])
def test_topw_matches_oracle(B, N, c, w, max_depth):
    rng = np.random.default_rng(B * 1000 + N + c)
    logp = np.log(rng.uniform(1e-6, 1.0, size=(B, N, c))).astype(np.float32)
    check(logp, w, max_depth)


@pytest.mark.parametrize("B,N,c,w,max_depth", [
    (6, 128, 8, 4, 30),     # 32 offers a round, the 128-node list
    (6, 129, 4, 4, 30),     # the 256-node list from 129 nodes
    (4, 256, 4, 8, 40),     # 256 nodes, 32 offers
    (4, 256, 2, 3, 300),    # deep trees, few offers
    (3, 200, 1, 32, 300),   # one offer per take, 32 takes a round
    (2, 256, 32, 1, 300),   # the list kernel's largest shared memory (32 K log-probabilities)
])
def test_topw_list_shapes_with_positive_scores(B, N, c, w, max_depth):
    """The sorted-list kernel at its size boundaries, with log-probabilities of both
    signs (a new candidate can then outrank the nodes just taken) and rounded values
    (many equal scores: creation order decides)."""
    rng = np.random.default_rng(N * 31 + c * 7 + w)
    logp = rng.normal(0.0, 1.0, size=(B, N, c)).astype(np.float32)
    logp[B // 2:] = np.round(logp[B // 2:])
    check(logp, w, max_depth)


def test_topw_ties_infinities_and_exhaustion():
    rng = np.random.default_rng(9)
    logp = np.round(np.log(rng.uniform(0.05, 1.0, size=(6, 50, 4))), 1).astype(np.float32)
    logp[1] = -1.0                      # all ties: creation order decides
    logp[2, :, 1:] = -np.inf            # one live candidate per node: a chain
    logp[3, 0, :] = -np.inf             # the root offers nothing
    _, n = check(logp, 3, 8)
    assert n[3] == 1 and n[2] == 8      # chain stops at max_depth


def test_built_trees_verify():
    """A tree built on the GPU goes straight into the verification."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    import workloads as W
    from tests import harness as H
    w = W.make_config(2)
    rng = np.random.default_rng(2)
    logp = np.log(rng.uniform(1e-6, 1.0, size=(w.B, w.N, 4))).astype(np.float32)
    p, n = check(logp, 4, 16)
    assert (n == w.N).all()
    w.parent = p.astype(np.int32)
    x = H.to_device(w)
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"])
    torch.cuda.synchronize()
    ref_o, ref_U = __import__("oracle").verify_workload(w, mode="memo")
    assert H.rel_err(o.float().cpu().numpy(), ref_o) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy(), ref_U) <= H.TOL_U
