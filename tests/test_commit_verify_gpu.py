"""GPU parity of one decoding iteration, gdn_tree_commit_verify: the delayed
commitment of the previous tree's accepted path fused with the verification
of the next tree.  Checked against the oracle (commit of the previous path by
the recurrence, then verification of the next tree from that state) and
against the two separate calls, on the tensor-core path and the two-launch
fallback."""

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


def _pair(seed, B, Np, N, Hqk, Hv, d, dtype, tree="random"):
    prev = W.make_custom(seed=seed, B=B, N=Np, Hqk=Hqk, Hv=Hv, dk=d, dv=d, dtype=dtype,
                         tree=tree, max_depth=24)
    nxt = W.make_custom(seed=seed + 1, B=B, N=N, Hqk=Hqk, Hv=Hv, dk=d, dv=d, dtype=dtype,
                        tree="mixed", max_depth=24)
    return prev, nxt


def _run(prev, nxt, inplace=False):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    xp, xn = H.to_device(prev), H.to_device(nxt)
    _, U_prev = gt.verify(xp["q"], xp["k"], xp["v"], xp["log_alpha"], xp["beta"], xp["parent"],
                          xp["S0"])
    # separate calls
    S1_sep = gt.commit(xp["path"], xp["path_len"], U_prev, xp["k"], xp["log_alpha"], xp["S0"],
                       parent=xp["parent"])
    o_sep, U_sep = gt.verify(xn["q"], xn["k"], xn["v"], xn["log_alpha"], xn["beta"],
                             xn["parent"], S1_sep)
    # fused
    cs = torch.full((prev.B,), -7, dtype=torch.int32, device="cuda")
    vs = torch.full((prev.B,), -7, dtype=torch.int32, device="cuda")
    S_prev = xp["S0"].clone()
    U_buf = U_prev.clone() if inplace and prev.N == nxt.N else None
    S1, o, U = gt.commit_verify(xp["path"], xp["path_len"], U_prev if U_buf is None else U_buf,
                                xp["k"], xp["log_alpha"], S_prev, xn["q"], xn["k"], xn["v"],
                                xn["log_alpha"], xn["beta"], xn["parent"],
                                S1=S_prev if inplace else None, prev_parent=xp["parent"],
                                U=U_buf, commit_status=cs, verify_status=vs)
    torch.cuda.synchronize()
    return dict(S1=S1.cpu().numpy(), o=o.float().cpu().numpy(), U=U.cpu().numpy(),
                cs=cs.cpu().numpy(), vs=vs.cpu().numpy(), S1_sep=S1_sep.cpu().numpy(),
                o_sep=o_sep.float().cpu().numpy(), U_sep=U_sep.cpu().numpy())


def _oracle(prev, nxt):
    S1 = oracle.commit_workload(prev)
    o, U = oracle.verify(nxt.q, nxt.k, nxt.v, nxt.log_alpha, nxt.beta, nxt.parent, S1)
    return S1, o, U


CASES = [
    # (B, prev N, next N, Hqk, Hv, d, dtype, prev tree)
    (4, 128, 128, 2, 4, 128, W.BF16, "random"),   # tensor-core fused path
    (3, 100, 64, 1, 2, 128, W.BF16, "chain"),     # long paths (> one staging chunk)
    (2, 200, 90, 1, 2, 128, W.BF16, "random"),    # previous tree larger than a tile
    (2, 48, 40, 1, 2, 64, W.BF16, "mixed"),       # fallback: two launches
    (2, 20, 24, 1, 1, 32, W.F32, "uniform"),      # fallback, fp32
]


@pytest.mark.parametrize("idx", range(len(CASES)), ids=["x".join(map(str, c)) for c in CASES])
def test_commit_verify_matches_oracle_and_separate_calls(idx):
    B, Np, N, Hqk, Hv, d, dt, tree = CASES[idx]
    prev, nxt = _pair(300 + idx, B, Np, N, Hqk, Hv, d, dt, tree)
    g = _run(prev, nxt)
    assert (g["cs"] == 0).all() and (g["vs"] == 0).all()
    S1_ref, o_ref, U_ref = _oracle(prev, nxt)
    assert H.rel_err(g["S1"], S1_ref) <= H.TOL_S1
    assert H.rel_err(g["U"], U_ref) <= H.TOL_U
    assert H.rel_err(g["o"], o_ref) <= H.TOL_O[dt]
    # and it is the same computation as the two calls: the fused commit runs on
    # the tensor cores with w U split into bf16 hi + lo (each product to about
    # 2^-17 relative), the separate one in fp32 FMAs, so the two states agree to
    # a few 2^-17 of the state's scale (and U, from them, likewise)
    assert H.rel_err(g["S1"], g["S1_sep"]) <= 2e-5
    assert H.rel_err(g["U"], g["U_sep"]) <= 2e-5
    assert H.rel_err(g["o"], g["o_sep"]) <= 1e-2


def test_commit_verify_in_place_buffers():
    prev, nxt = _pair(400, 3, 96, 96, 1, 2, 128, W.BF16)
    g = _run(prev, nxt, inplace=True)
    S1_ref, o_ref, U_ref = _oracle(prev, nxt)
    assert H.rel_err(g["S1"], S1_ref) <= H.TOL_S1
    assert H.rel_err(g["U"], U_ref) <= H.TOL_U


def test_commit_verify_empty_and_invalid_paths():
    prev, nxt = _pair(500, 3, 64, 64, 1, 2, 128, W.BF16)
    prev.path_len[0] = 0                      # empty: S1 = S_prev
    prev.path[1, :] = -1                      # invalid: not a root chain
    prev.path[1, 0], prev.path[1, 1] = 5, 3
    prev.path_len[1] = 2
    g = _run(prev, nxt)
    assert g["cs"].tolist()[0] == 0 and g["cs"].tolist()[1] == 2 and g["cs"].tolist()[2] == 0
    assert g["vs"].tolist()[1] == 2
    assert np.array_equal(g["S1"][0], prev.S0[0])
    S1_ref = oracle.commit(prev.path[[0, 2]], prev.path_len[[0, 2]], prev.k[[0, 2]],
                           prev.v[[0, 2]], prev.log_alpha[[0, 2]], prev.beta[[0, 2]],
                           prev.S0[[0, 2]])
    assert H.rel_err(g["S1"][[0, 2]], S1_ref) <= H.TOL_S1


def test_bench_step_two_iterations_match_oracle():
    """Exactly the benchmark's timed step: the serving workload (32 sequences x 32
    v-heads, 128-node trees) on the fixed layout, gdn_tree_commit_verify over two
    consecutive decoding iterations with ping-pong state and U buffers, each
    iteration committing the accepted path of the tree verified before it and
    verifying the next tree from the committed state.  Checked against the
    oracle's commit (the recurrence along the path) then verification, chained
    the same way.  U is held to its bound against the oracle run from the state
    the GPU committed, and against the oracle's own chain with the state's
    bound carried through (U is linear in the state)."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    w = W.make_config(3)
    x = H.to_device(w)
    o = torch.empty((w.B, w.N, w.Hv, w.dv), dtype=torch.bfloat16, device="cuda")
    Sb = [x["S0"].clone(), torch.empty_like(x["S0"])]
    Ub = [torch.empty((w.B, w.Hv, w.N, w.dv), dtype=torch.float32, device="cuda")
          for _ in range(2)]
    gt.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"], Sb[0], o=o,
              U=Ub[0])
    S_ref = w.S0.astype(np.float64)
    for i in range(2):
        cur, nxt = i & 1, (i + 1) & 1
        cs = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
        vs = torch.full((w.B,), -7, dtype=torch.int32, device="cuda")
        gt.commit_verify(x["path"], x["path_len"], Ub[cur], x["k"], x["log_alpha"], Sb[cur],
                         x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                         S1=Sb[nxt], o=o, U=Ub[nxt], prev_parent=x["parent"],
                         commit_status=cs, verify_status=vs)
        torch.cuda.synchronize()
        assert (cs.cpu().numpy() == 0).all() and (vs.cpu().numpy() == 0).all()
        S_gpu, U_gpu = Sb[nxt].cpu().numpy(), Ub[nxt].cpu().numpy()
        o_gpu = o.float().cpu().numpy()
        S_ref = oracle.commit(w.path, w.path_len, w.k, w.v, w.log_alpha, w.beta, S_ref,
                              parent=w.parent)
        o_ref, U_ref = oracle.verify(w.q, w.k, w.v, w.log_alpha, w.beta, w.parent, S_ref)
        _, U_own = oracle.verify(w.q, w.k, w.v, w.log_alpha, w.beta, w.parent, S_gpu)
        errs = dict(o=H.rel_err(o_gpu, o_ref), U=H.rel_err(U_gpu, U_own),
                    S1=H.rel_err(S_gpu, S_ref))
        H.report(w, errs, tag=f"bench-step iteration {i}")
        assert errs["S1"] <= H.TOL_S1, errs
        assert errs["o"] <= H.TOL_O[W.BF16], errs
        assert errs["U"] <= H.TOL_U, errs
        assert H.rel_err(U_gpu, U_ref) <= H.TOL_U + (i + 1) * H.TOL_S1


def test_commit_verify_invalid_paths_among_many_units():
    """More units than SMs (384 on 152, so CTAs take over the units of CTAs not launched
    yet): sequences whose accepted path is invalid are reported by both calls and left
    unwritten, an empty path commits S_prev, and every other sequence matches the oracle
    in S1, o and U."""
    prev, nxt = _pair(520, 24, 96, 96, 8, 16, 128, W.BF16)
    prev.path_len[2] = 0                       # empty: S1 = S_prev
    prev.path[7, :] = -1                       # not a root chain
    prev.path[7, 0], prev.path[7, 1] = 5, 3
    prev.path_len[7] = 2
    prev.path_len[19] = 200                    # longer than the tree
    g = _run(prev, nxt)
    bad = [7, 19]
    cs, vs = g["cs"].tolist(), g["vs"].tolist()
    for b in range(prev.B):
        want = 2 if b in bad else 0            # GDN_TREE_STATUS_BAD_PATH
        assert cs[b] == want and vs[b] == want, (b, cs[b], vs[b])
    assert np.array_equal(g["S1"][2], prev.S0[2])
    ok = [b for b in range(prev.B) if b not in bad]
    S1_ref = oracle.commit(prev.path[ok], prev.path_len[ok], prev.k[ok], prev.v[ok],
                           prev.log_alpha[ok], prev.beta[ok], prev.S0[ok])
    o_ref, _ = oracle.verify(nxt.q[ok], nxt.k[ok], nxt.v[ok], nxt.log_alpha[ok],
                             nxt.beta[ok], nxt.parent[ok], S1_ref)
    assert H.rel_err(g["S1"][ok], S1_ref) <= H.TOL_S1
    assert H.rel_err(g["o"][ok], o_ref) <= H.TOL_O[W.BF16]
    # U against the oracle run from the GPU's own S1 (the state it verified from)
    _, U_own = oracle.verify(nxt.q[ok], nxt.k[ok], nxt.v[ok], nxt.log_alpha[ok],
                             nxt.beta[ok], nxt.parent[ok], g["S1"][ok])
    assert H.rel_err(g["U"][ok], U_own) <= H.TOL_U
