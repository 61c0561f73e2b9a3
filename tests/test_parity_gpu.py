"""GPU parity: the CUDA path through the C ABI against the fp64 oracle on
the same seeded inputs, element by element.

The five workloads of the tree-verification setting run at full size and are
compared over the whole tensor; smaller shapes span several tiles
and ragged tails; edge cases cover single nodes, forests, stars, chains,
invalid trees/paths, empty paths and in-place commits."""

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


@pytest.fixture(params=["auto", "generic", "mid"])
def kernel(request, monkeypatch):
    """Runs a test with the default kernel choice (the tensor-core kernel where
    it takes the shape), again with the general CUDA-core kernel forced, and
    again with the 256-node bf16 kernel forced (shapes it does not take fall
    back to the general kernel)."""
    if request.param in ("generic", "mid"):
        monkeypatch.setenv("GDN_TREE_KERNEL", request.param)
    else:
        monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    return request.param


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_config_full(cfg, kernel):
    w = H.ensure_state(W.make_config(cfg))
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    errs = H.compare(w, gpu, H.run_oracle(w))
    H.assert_parity(w, errs)


_CONFIG4_REF = {}


def _config4_reference(w):
    """The oracle over the whole stress workload (computed once per session)."""
    if "ref" not in _CONFIG4_REF:
        _CONFIG4_REF["ref"] = H.run_oracle(w)
    return _CONFIG4_REF["ref"]


def test_config4_whole_tensor(kernel):
    """The stress workload (64 x 32 units, 256-node chains, stars and random
    trees, log alpha down to -4, a beta = 0.99 sequence), every element of o, U
    and S1 against the oracle, on every kernel the dispatcher can choose for it."""
    w = W.make_config(4)
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, _config4_reference(w)))
    assert np.isfinite(gpu["o"]).all() and np.isfinite(gpu["S1"]).all()


SHAPES = [
    # (B, N, Hqk, Hv, dk, dv, dtype, tree)
    (2, 37, 1, 2, 32, 32, W.F32, "uniform"),
    (2, 100, 2, 4, 64, 64, W.BF16, "mixed"),
    (3, 129, 1, 1, 128, 128, W.BF16, "mixed"),
    (1, 200, 2, 2, 128, 64, W.F32, "random"),
    (2, 256, 1, 4, 128, 128, W.BF16, "chain"),
    (2, 256, 1, 2, 64, 128, W.BF16, "flatstar"),
    (6, 61, 2, 8, 128, 128, W.BF16, "mixed"),
    (1, 5, 1, 1, 16, 48, W.F32, "uniform"),
    (1, 1, 1, 1, 128, 128, W.BF16, "chain"),
    (4, 128, 2, 4, 128, 128, W.BF16, "mixed"),
    (3, 97, 1, 3, 128, 128, W.BF16, "chain"),
    (5, 33, 4, 8, 128, 128, W.BF16, "flatstar"),
    (2, 128, 1, 2, 128, 128, W.BF16, "chain"),
]


@pytest.mark.parametrize("idx", range(len(SHAPES)), ids=["x".join(map(str, s)) for s in SHAPES])
def test_shapes_elementwise(idx, kernel):
    B, N, Hqk, Hv, dk, dv, dt, tree = SHAPES[idx]
    w = W.make_custom(seed=100 + idx, B=B, N=N, Hqk=Hqk, Hv=Hv, dk=dk, dv=dv,
                      dtype=dt, tree=tree, max_depth=40)
    H.assert_parity(w, H.compare(w, H.run_gpu(w), H.run_oracle(w)))


@pytest.mark.parametrize("N", [128, 160])
def test_strong_decay_and_high_beta(kernel, N):
    w = W.make_custom(seed=5, B=6, N=N, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="mixed", max_depth=160, la_range=(0.01, 4.0), beta_kind="uniform")
    w.beta[:] = np.float32(0.99)
    H.assert_parity(w, H.compare(w, H.run_gpu(w), H.run_oracle(w)))


def test_inplace_commit_and_no_parent_check(kernel):
    w = W.make_custom(seed=6, B=3, N=48, Hqk=2, Hv=4, dk=64, dv=64, dtype=W.BF16)
    ref = H.run_oracle(w)
    gpu = H.run_gpu(w, inplace=True, with_parent=False)
    H.assert_parity(w, H.compare(w, gpu, ref))


def test_empty_path_commits_S0():
    w = W.make_custom(seed=7, B=2, N=20, Hqk=1, Hv=2, dk=32, dv=32, dtype=W.F32)
    w.path[:] = -1
    w.path_len[:] = 0
    gpu = H.run_gpu(w)
    assert np.array_equal(gpu["S1"], w.S0)


def test_invalid_tree_and_path_reported_per_sequence(kernel):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    w = W.make_custom(seed=8, B=3, N=16, Hqk=1, Hv=2, dk=32, dv=32, dtype=W.BF16, lmax=16)
    w.parent[1, 5] = 9          # not topologically ordered
    w.path[2, :] = -1           # sequence 2: path 0 -> 2 where 2's parent may differ
    w.path[2, 0], w.path[2, 1] = 0, 3
    w.path_len[2] = 2
    ok_chain = w.parent[2, 3] == 0
    x = H.to_device(w)
    st = torch.full((3,), -7, dtype=torch.int32, device="cuda")
    o = torch.full((3, 16, 2, 32), 123.0, dtype=torch.bfloat16, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                     x["S0"], o=o, dev_status=st)
    torch.cuda.synchronize()
    assert st.cpu().tolist() == [gt.STATUS_OK, gt.STATUS_BAD_TREE, gt.STATUS_OK]
    assert (o[1].float() == 123.0).all()  # invalid sequence left unwritten
    w.parent[1, 5] = 4
    x = H.to_device(w)
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"])
    x["path_len"][1] = 99       # longer than the tree
    S1 = torch.full_like(x["S0"], 5.0)
    gt.commit(x["path"], x["path_len"], U, x["k"], x["log_alpha"], x["S0"], S1=S1,
              parent=x["parent"], dev_status=st)
    torch.cuda.synchronize()
    want2 = gt.STATUS_OK if ok_chain else gt.STATUS_BAD_PATH
    assert st.cpu().tolist() == [gt.STATUS_OK, gt.STATUS_BAD_PATH, want2]
    assert (S1[1] == 5.0).all()


def test_sibling_permutation_on_gpu(kernel):
    from tests.pins import random_topological_relabel
    w = W.make_custom(seed=9, B=1, N=90, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="random", max_depth=12)
    a = H.run_gpu(w)
    perm, newp = random_topological_relabel(np.random.default_rng(1), w.parent[0])
    for name in ("q", "k", "v", "log_alpha", "beta"):
        setattr(w, name, np.ascontiguousarray(getattr(w, name)[:, perm]))
    w.parent = newp[None].astype(np.int32)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    w.path[0, : w.path_len[0]] = inv[w.path[0, : w.path_len[0]]]
    b = H.run_gpu(w)
    assert H.rel_err(b["o"][0], a["o"][0, perm]) <= 1e-2
    assert H.rel_err(b["U"][0], a["U"][0][:, perm]) <= 1e-4
    assert H.rel_err(b["S1"], a["S1"]) <= 1e-4


def test_invalid_tree_among_many_units(kernel):
    """More units than SMs: every v-head of a sequence with an invalid tree is left
    unwritten and reported, whichever CTA walks it and whatever it walked before."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    w = W.make_custom(seed=9, B=20, N=64, Hqk=8, Hv=16, dk=128, dv=128, dtype=W.BF16,
                      tree="mixed", max_depth=24)
    w.parent[5, 40] = 50   # not topologically ordered
    w.parent[6, 3] = -5    # out of range
    x = H.to_device(w)
    st = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
    o = torch.full((w.B, w.N, w.Hv, w.dv), 123.0, dtype=torch.bfloat16, device="cuda")
    o, U = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                     x["S0"], o=o, dev_status=st)
    torch.cuda.synchronize()
    want = [gt.STATUS_OK] * w.B
    want[5] = want[6] = gt.STATUS_BAD_TREE
    assert st.cpu().tolist() == want
    on = o.float().cpu().numpy()
    assert (on[5] == 123.0).all() and (on[6] == 123.0).all()
    ok = [b for b in range(w.B) if b not in (5, 6)]
    ref_o, ref_U = oracle.verify(w.q[ok], w.k[ok], w.v[ok], w.log_alpha[ok], w.beta[ok],
                                 w.parent[ok], w.S0[ok])
    assert H.rel_err(on[ok], ref_o) <= H.TOL_O[W.BF16]
    assert H.rel_err(U.cpu().numpy()[ok], ref_U) <= H.TOL_U


def test_linearity_on_gpu(kernel):
    """Invariant I5 on the GPU path, without the oracle: o and U are linear in (V, S0)
    jointly, so scaling both by 2 (exact in binary floating point) scales o and U by 2."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    w = W.make_custom(seed=12, B=3, N=100, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="mixed", max_depth=24)
    x = H.to_device(w)
    o1, U1 = gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], x["S0"])
    o2, U2 = gt.verify(x["q"], x["k"], 2 * x["v"], x["log_alpha"], x["beta"], x["parent"],
                       2 * x["S0"])
    torch.cuda.synchronize()
    assert H.rel_err(o2.float().cpu().numpy(), 2 * o1.float().cpu().numpy()) <= 1e-2
    assert H.rel_err(U2.cpu().numpy(), 2 * U1.cpu().numpy()) <= 1e-6


def test_graft_on_gpu(kernel):
    """Invariant I4 on the GPU path, without the oracle: committing an accepted path
    and verifying the next tree from S1 gives that tree's outputs of verifying, from
    S0, the path as a chain with the next tree grafted below its last node."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    A = W.make_custom(seed=13, B=2, N=40, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="chain", max_depth=40)  # accepted paths of 24 and 23 nodes
    T = W.make_custom(seed=14, B=2, N=50, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                      tree="mixed", max_depth=10)
    L = int(A.path_len.min())
    A.path_len[:] = L
    xa, xt = H.to_device(A), H.to_device(T)
    _, Ua = gt.verify(xa["q"], xa["k"], xa["v"], xa["log_alpha"], xa["beta"], xa["parent"],
                      xa["S0"])
    S1 = gt.commit(xa["path"], xa["path_len"], Ua, xa["k"], xa["log_alpha"], xa["S0"],
                   parent=xa["parent"])
    o_t, U_t = gt.verify(xt["q"], xt["k"], xt["v"], xt["log_alpha"], xt["beta"], xt["parent"],
                         S1)
    # the grafted tree: the path's L nodes as a chain, then T's nodes below it
    B, Ng = A.B, L + T.N
    par = np.empty((B, Ng), np.int32)
    par[:, :L] = np.arange(-1, L - 1)
    par[:, L:] = np.where(T.parent >= 0, T.parent + L, L - 1)
    rows = [np.concatenate([A.path[b, :L], A.N + np.arange(T.N)]) for b in range(B)]

    def cat(name):
        a, t = getattr(A, name), getattr(T, name)
        both = np.concatenate([a, t], axis=1)
        return np.stack([both[b][rows[b]] for b in range(B)])

    G = W.Workload(name="graft", B=B, N=Ng, Hqk=1, Hv=2, dk=128, dv=128, dtype=W.BF16,
                   q=cat("q"), k=cat("k"), v=cat("v"), log_alpha=cat("log_alpha"),
                   beta=cat("beta"), parent=par, S0=A.S0, path=A.path, path_len=A.path_len)
    xg = H.to_device(G)
    o_g, U_g = gt.verify(xg["q"], xg["k"], xg["v"], xg["log_alpha"], xg["beta"], xg["parent"],
                         xg["S0"])
    torch.cuda.synchronize()
    assert H.rel_err(o_t.float().cpu().numpy(), o_g[:, L:].float().cpu().numpy()) <= 1e-2
    assert H.rel_err(U_t.cpu().numpy(), U_g[:, :, L:].cpu().numpy()) <= 1e-4


@pytest.mark.parametrize("inplace,with_parent", [(False, True), (True, True), (False, False)])
def test_commit_paths_past_32_entries(inplace, with_parent, kernel):
    """Paths of up to 64 entries (Lmax > 32: the tensor-core commit for bf16,
    d = 128; the CUDA-core commit when the generic kernels are forced) on
    chains, stars and random trees, one sequence with an empty path (S1 = S0),
    in place or not, with and without the parent-link check."""
    w = W.make_custom(seed=31, B=6, N=80, Hqk=2, Hv=4, dk=128, dv=128, dtype=W.BF16,
                      tree="mixed", max_depth=80, lmax=64)
    w.path_len[3] = 0
    ref = H.run_oracle(w)
    gpu = H.run_gpu(w, inplace=inplace, with_parent=with_parent)
    assert (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, ref))
    assert np.array_equal(gpu["S1"][3], w.S0[3])
