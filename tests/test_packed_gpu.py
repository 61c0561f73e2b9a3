"""GPU parity of the packed (ragged) layout with a state pool: gdn_tree_verify_packed,
gdn_tree_commit_packed and gdn_tree_commit_verify_packed through the C ABI, against
the fp64 oracle run sequence by sequence on each sequence's own tree."""

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
    if request.param in ("generic", "mid"):
        monkeypatch.setenv("GDN_TREE_KERNEL", request.param)
    else:
        monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    return request.param


class Packed:
    """A ragged batch: one workload per sequence (its own tree size), packed rows,
    and a state pool whose slot state_slot[b] holds sequence b's state."""

    def __init__(self, seed, Ns, Hqk, Hv, dk, dv, dtype, n_slots, tree="mixed"):
        rng = np.random.default_rng(seed)
        self.Ns, self.Hqk, self.Hv, self.dk, self.dv, self.dtype = Ns, Hqk, Hv, dk, dv, dtype
        self.B = len(Ns)
        self.cu = np.concatenate([[0], np.cumsum(Ns)]).astype(np.int32)
        self.T = int(self.cu[-1])
        self.slot = rng.permutation(n_slots)[:self.B].astype(np.int32)
        self.pool = (rng.standard_normal((n_slots, Hv, dk, dv)) * 0.1).astype(np.float32)
        self.ws = []
        for b, n in enumerate(Ns):
            if n == 0:
                self.ws.append(None)
                continue
            w = W.make_custom(seed=seed * 100 + b, B=1, N=n, Hqk=Hqk, Hv=Hv, dk=dk, dv=dv,
                              dtype=dtype, tree=tree, max_depth=64, lmax=n)
            w.S0 = self.pool[self.slot[b]][None].copy()
            self.ws.append(w)
        self.Lmax = max([w.path.shape[1] for w in self.ws if w is not None] + [1])

    def cat(self, name, shape_tail, dtype):
        parts = [getattr(w, name)[0] for w in self.ws if w is not None]
        if not parts:
            return np.zeros((0,) + shape_tail, dtype=dtype)
        return np.concatenate(parts, axis=0).astype(dtype)

    def device(self):
        import torch
        dt = torch.bfloat16 if self.dtype == W.BF16 else torch.float32
        t = lambda x, d=None: torch.from_numpy(np.ascontiguousarray(x)).to("cuda", dtype=d)
        np_dt = np.float32
        path = np.full((self.B, self.Lmax), -1, np.int32)
        plen = np.zeros(self.B, np.int32)
        for b, w in enumerate(self.ws):
            if w is not None:
                path[b, :w.path.shape[1]] = w.path[0]
                plen[b] = w.path_len[0]
        return dict(
            q=t(self.cat("q", (self.Hqk, self.dk), np_dt), dt),
            k=t(self.cat("k", (self.Hqk, self.dk), np_dt), dt),
            v=t(self.cat("v", (self.Hv, self.dv), np_dt), dt),
            log_alpha=t(self.cat("log_alpha", (self.Hv,), np_dt)),
            beta=t(self.cat("beta", (self.Hv,), np_dt)),
            parent=t(self.cat("parent", (), np.int32)),
            cu=t(self.cu), slot=t(self.slot), pool=t(self.pool), path=t(path),
            path_len=t(plen))

    def oracle_verify(self):
        o = np.full((self.T, self.Hv, self.dv), np.nan)
        U = np.full((self.Hv, self.T, self.dv), np.nan)
        for b, w in enumerate(self.ws):
            if w is None:
                continue
            ob, Ub = oracle.verify_workload(w, mode="memo")
            a, e = self.cu[b], self.cu[b + 1]
            o[a:e] = ob[0]
            U[:, a:e] = Ub[0]
        return o, U

    def oracle_commit(self):
        pool = self.pool.astype(np.float64).copy()
        for b, w in enumerate(self.ws):
            if w is not None:
                pool[self.slot[b]] = oracle.commit_workload(w)[0]
        return pool


def check_verify(P, o, U, st):
    assert (st == 0).all(), st
    ref_o, ref_U = P.oracle_verify()
    eo, eu = H.rel_err(o, ref_o), H.rel_err(U, ref_U)
    assert eo <= H.TOL_O[P.dtype], f"o rel err {eo:.3e}"
    assert eu <= H.TOL_U, f"U rel err {eu:.3e}"


CASES = [
    # (Ns, Hqk, Hv, dk, dv, dtype): the tensor-core kernel takes the first two
    ([37, 128, 1, 0, 64, 100, 5], 2, 4, 128, 128, W.BF16),
    ([128, 17, 96], 1, 2, 128, 128, W.BF16),
    ([200, 3, 0, 77], 1, 2, 64, 64, W.BF16),
    ([9, 31, 1, 50], 1, 1, 32, 32, W.F32),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_verify_packed(case, kernel):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    Ns, Hqk, Hv, dk, dv, dt = CASES[case]
    P = Packed(11 + case, Ns, Hqk, Hv, dk, dv, dt, n_slots=len(Ns) + 3)
    x = P.device()
    st = torch.full((P.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify_packed(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                            x["cu"], x["pool"], state_slot=x["slot"], dev_status=st)
    torch.cuda.synchronize()
    check_verify(P, o.float().cpu().numpy(), U.cpu().numpy(), st.cpu().numpy())


@pytest.mark.parametrize("case", [0, 3])
def test_commit_packed_in_place(case, kernel):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    Ns, Hqk, Hv, dk, dv, dt = CASES[case]
    P = Packed(21 + case, Ns, Hqk, Hv, dk, dv, dt, n_slots=len(Ns) + 3)
    x = P.device()
    o, U = gt.verify_packed(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                            x["cu"], x["pool"], state_slot=x["slot"])
    st = torch.full((P.B,), -7, dtype=torch.int32, device="cuda")
    pool = x["pool"]
    gt.commit_packed(x["path"], x["path_len"], U, x["k"], x["log_alpha"], x["cu"], pool,
                     pool_out=pool, state_slot=x["slot"], parent=x["parent"], dev_status=st)
    torch.cuda.synchronize()
    assert (st.cpu().numpy() == 0).all()
    got, ref = pool.cpu().numpy(), P.oracle_commit()
    used = np.zeros(len(ref), bool)
    used[P.slot] = True
    assert H.rel_err(got[used], ref[used]) <= H.TOL_S1
    assert np.array_equal(got[~used], P.pool[~used])  # other slots untouched


def test_commit_verify_packed_matches_separate_calls(kernel):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    prev = Packed(31, [50, 128, 7, 0, 90], 2, 4, 128, 128, W.BF16, n_slots=8)
    nxt = Packed(32, [128, 3, 64, 31, 100], 2, 4, 128, 128, W.BF16, n_slots=8)
    nxt.slot, nxt.pool = prev.slot, prev.pool  # one pool, one slot per sequence
    xp, xn = prev.device(), nxt.device()
    _, Up = gt.verify_packed(xp["q"], xp["k"], xp["v"], xp["log_alpha"], xp["beta"],
                             xp["parent"], xp["cu"], xp["pool"], state_slot=xp["slot"])
    # separate calls: commit into a copy, then verify from it
    pool_a = gt.commit_packed(xp["path"], xp["path_len"], Up, xp["k"], xp["log_alpha"],
                              xp["cu"], xp["pool"], state_slot=xp["slot"], parent=xp["parent"])
    o_a, U_a = gt.verify_packed(xn["q"], xn["k"], xn["v"], xn["log_alpha"], xn["beta"],
                                xn["parent"], xn["cu"], pool_a, state_slot=xp["slot"])
    cs = torch.full((5,), -7, dtype=torch.int32, device="cuda")
    vs = torch.full((5,), -7, dtype=torch.int32, device="cuda")
    pool_b, o_b, U_b = gt.commit_verify_packed(
        xp["path"], xp["path_len"], Up, xp["k"], xp["log_alpha"], xp["cu"], xp["pool"],
        xn["q"], xn["k"], xn["v"], xn["log_alpha"], xn["beta"], xn["parent"], xn["cu"],
        state_slot=xp["slot"], prev_parent=xp["parent"], commit_status=cs, verify_status=vs)
    torch.cuda.synchronize()
    assert (cs.cpu().numpy() == 0).all() and (vs.cpu().numpy() == 0).all()
    assert H.rel_err(pool_b.cpu().numpy(), pool_a.cpu().numpy()) <= H.TOL_S1
    assert H.rel_err(o_b.float().cpu().numpy(), o_a.float().cpu().numpy()) <= H.TOL_O[W.BF16]
    assert H.rel_err(U_b.cpu().numpy(), U_a.cpu().numpy()) <= H.TOL_U
    # and against the oracle: commit the previous trees, verify the next ones
    ref_pool = prev.oracle_commit()
    for b, w in enumerate(nxt.ws):
        if w is not None:
            w.S0 = ref_pool[prev.slot[b]][None].astype(np.float32)
    ref_o, _ = nxt.oracle_verify()
    assert H.rel_err(o_b.float().cpu().numpy(), ref_o) <= H.TOL_O[W.BF16]
    # U against the oracle run from the state the GPU committed (U is linear in
    # the state, so this separates the verification's error from the commit's)
    got_pool = pool_b.cpu().numpy()
    for b, w in enumerate(nxt.ws):
        if w is not None:
            w.S0 = got_pool[prev.slot[b]][None]
    _, own_U = nxt.oracle_verify()
    assert H.rel_err(U_b.cpu().numpy(), own_U) <= H.TOL_U


def test_bad_layout_reported_and_left_unwritten(kernel):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    P = Packed(41, [20, 30, 40, 10], 1, 2, 128, 128, W.BF16, n_slots=6)
    x = P.device()
    cu = x["cu"].clone()
    cu[2] = cu[3] + 1          # sequence 2: end before start; sequence 1 ends past its start + N
    slot = x["slot"].clone()
    slot[3] = 99               # sequence 3: slot out of range
    st = torch.full((P.B,), -7, dtype=torch.int32, device="cuda")
    o = torch.full((P.T, 2, 128), 123.0, dtype=torch.bfloat16, device="cuda")
    o, U = gt.verify_packed(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                            cu, x["pool"], state_slot=slot, N_max=40, o=o, dev_status=st)
    torch.cuda.synchronize()
    s = st.cpu().tolist()
    assert s[0] == gt.STATUS_OK and s[2] == gt.STATUS_BAD_LAYOUT and s[3] == gt.STATUS_BAD_LAYOUT
    on = o.float().cpu().numpy()
    assert (on[P.cu[3]:P.cu[4]] == 123.0).all()   # the bad-slot sequence's rows unwritten
    ref_o, _ = P.oracle_verify()
    assert H.rel_err(on[:P.cu[1]], ref_o[:P.cu[1]]) <= H.TOL_O[W.BF16]


def test_many_units_of_varying_size(kernel):
    """More (sequence, head) units than SMs, so the persistent tensor-core kernel
    walks several units of different tree sizes (and empty sequences) per CTA."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    rng = np.random.default_rng(51)
    Ns = [int(n) for n in rng.integers(0, 129, size=40)]
    Ns[3], Ns[17] = 0, 128
    P = Packed(51, Ns, 4, 8, 128, 128, W.BF16, n_slots=44)
    x = P.device()
    st = torch.full((P.B,), -7, dtype=torch.int32, device="cuda")
    o, U = gt.verify_packed(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], x["parent"],
                            x["cu"], x["pool"], state_slot=x["slot"], dev_status=st)
    torch.cuda.synchronize()
    check_verify(P, o.float().cpu().numpy(), U.cpu().numpy(), st.cpu().numpy())


def test_commit_verify_many_units_of_varying_size(kernel):
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    rng = np.random.default_rng(52)
    n_prev = [int(n) for n in rng.integers(1, 129, size=24)]
    n_next = [int(n) for n in rng.integers(0, 129, size=24)]
    prev = Packed(52, n_prev, 4, 8, 128, 128, W.BF16, n_slots=30)
    nxt = Packed(53, n_next, 4, 8, 128, 128, W.BF16, n_slots=30)
    nxt.slot, nxt.pool = prev.slot, prev.pool
    xp, xn = prev.device(), nxt.device()
    _, Up = gt.verify_packed(xp["q"], xp["k"], xp["v"], xp["log_alpha"], xp["beta"],
                             xp["parent"], xp["cu"], xp["pool"], state_slot=xp["slot"])
    cs = torch.full((24,), -7, dtype=torch.int32, device="cuda")
    vs = torch.full((24,), -7, dtype=torch.int32, device="cuda")
    pool_b, o_b, U_b = gt.commit_verify_packed(
        xp["path"], xp["path_len"], Up, xp["k"], xp["log_alpha"], xp["cu"], xp["pool"],
        xn["q"], xn["k"], xn["v"], xn["log_alpha"], xn["beta"], xn["parent"], xn["cu"],
        state_slot=xp["slot"], prev_parent=xp["parent"], commit_status=cs, verify_status=vs)
    torch.cuda.synchronize()
    assert (cs.cpu().numpy() == 0).all() and (vs.cpu().numpy() == 0).all()
    ref_pool = prev.oracle_commit()
    used = np.zeros(len(ref_pool), bool)
    used[prev.slot] = True
    assert H.rel_err(pool_b.cpu().numpy()[used], ref_pool[used]) <= H.TOL_S1
    for b, w in enumerate(nxt.ws):
        if w is not None:
            w.S0 = ref_pool[prev.slot[b]][None].astype(np.float32)
    ref_o, _ = nxt.oracle_verify()
    assert H.rel_err(o_b.float().cpu().numpy(), ref_o) <= H.TOL_O[W.BF16]
    # U against the oracle run from the state the GPU committed (U is linear in
    # the state, so this separates the verification's error from the commit's)
    got_pool = pool_b.cpu().numpy()
    for b, w in enumerate(nxt.ws):
        if w is not None:
            w.S0 = got_pool[prev.slot[b]][None]
    _, own_U = nxt.oracle_verify()
    assert H.rel_err(U_b.cpu().numpy(), own_U) <= H.TOL_U
