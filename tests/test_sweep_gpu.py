"""A seeded sweep of shapes through the C ABI against the fp64 oracle: tree sizes
on both sides of every kernel boundary (128, 256 and the 128-node chunks of the
chunk pass, the 64-node chunks of the chain path), every tree family, both
dtypes, several head sizes and GQA ratios, mild and strong decay.  The default
dispatch picks the kernel; the cases are drawn once from a fixed seed."""

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


def _cases(n=32, seed=2026):
    rng = np.random.default_rng(seed)
    sizes = [1, 2, 31, 63, 64, 65, 127, 128, 129, 191, 192, 255, 256, 257, 300, 383, 511, 640, 1024]
    trees = ["random", "chain", "star", "flatstar", "uniform", "topw", "mixed"]
    heads = [(1, 1), (1, 2), (2, 4), (4, 8)]
    out = []
    for i in range(n):
        N = int(rng.choice(sizes))
        tree = str(rng.choice(trees))
        if tree == "topw" and N < 2:
            tree = "random"
        bf16 = rng.random() < 0.7
        d = 128 if (bf16 and rng.random() < 0.8) else int(rng.choice([32, 64, 128]))
        Hqk, Hv = heads[int(rng.integers(len(heads)))]
        # bounded work: the oracle's memoised walk is O(units N d^2)
        B = int(rng.integers(1, 4)) if N <= 300 else 1
        if Hv * B * N * d * d > 2_000_000_000:
            Hqk, Hv = 1, 1
        strong = rng.random() < 0.3
        depth = int(rng.choice([8, 24, N])) if tree in ("random", "topw") else N
        out.append(dict(N=N, tree=tree, dtype=W.BF16 if bf16 else W.F32, d=d, Hqk=Hqk, Hv=Hv,
                        B=B, strong=strong, depth=max(2, depth), seed=3000 + i))
    return out


CASES = _cases()


@pytest.mark.parametrize("case", CASES, ids=[
    f"{c['tree']}-N{c['N']}-{c['dtype']}-d{c['d']}-h{c['Hqk']}x{c['Hv']}-B{c['B']}"
    + ("-strong" if c["strong"] else "") for c in CASES])
def test_sweep_matches_oracle(case, monkeypatch):
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    c = case
    kw = dict(la_range=(0.01, 4.0), beta_kind="uniform") if c["strong"] else {}
    w = W.make_custom(seed=c["seed"], B=c["B"], N=c["N"], Hqk=c["Hqk"], Hv=c["Hv"], dk=c["d"],
                      dv=c["d"], dtype=c["dtype"], tree=c["tree"], max_depth=c["depth"], **kw)
    gpu = H.run_gpu(w)
    assert (gpu["status_verify"] == 0).all() and (gpu["status_commit"] == 0).all()
    H.assert_parity(w, H.compare(w, gpu, H.run_oracle(w)))


def _packed_cases(n=12, seed=2027):
    rng = np.random.default_rng(seed)
    trees = ["random", "chain", "star", "uniform", "topw", "mixed"]
    out = []
    for i in range(n):
        top = int(rng.choice([64, 128, 256, 640, 1024]))
        Ns = [int(x) for x in rng.integers(0, top + 1, size=int(rng.integers(2, 6)))]
        Ns[int(rng.integers(len(Ns)))] = top  # the longest tree sets the kernel
        out.append(dict(Ns=Ns, tree=str(rng.choice(trees)), seed=4000 + i))
    return out


PACKED = _packed_cases()


@pytest.mark.parametrize("case", PACKED, ids=[f"{c['tree']}-{'-'.join(map(str, c['Ns']))}"
                                              for c in PACKED])
def test_sweep_packed_matches_oracle(case, monkeypatch):
    """Ragged batches (bf16, d = 128, states from a pool) through the packed entry
    points: verify, then the commit of each accepted path into the pool."""
    import torch
    import gated_deltanet_tree_gdn_gb300 as gt
    from tests.test_packed_gpu import Packed, check_verify
    monkeypatch.delenv("GDN_TREE_KERNEL", raising=False)
    P = Packed(case["seed"], case["Ns"], 2, 4, 128, 128, W.BF16, n_slots=len(case["Ns"]) + 2,
               tree=case["tree"])
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
