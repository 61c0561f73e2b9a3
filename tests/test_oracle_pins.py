"""The fp64 oracle against closed forms, special cases and invariants of the
GDN recurrence (DFlash-TfM page, section 3).  See tests/pins.py."""

import numpy as np
import pytest

import oracle
import workloads as W
from tests import pins


@pytest.fixture(scope="module")
def lib():
    return oracle.load()


@pytest.mark.parametrize("pin", pins.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(lib, pin):
    err = pin(lib)
    assert err <= pins.PIN_TOL, f"{pin.__name__}: {err:.3e}"


def test_invalid_tree_rejected(lib):
    x = pins._inputs(np.random.default_rng(0), 1, 4, 1, 1, 2, 2, [np.array([-1, 0, 2, 1])])
    with pytest.raises(oracle.OracleError):
        pins._verify(lib, x)


def test_non_chain_path_rejected(lib):
    rng = np.random.default_rng(1)
    parent = np.array([-1, 0, 0, 1], dtype=np.int32)
    x = pins._inputs(rng, 1, 4, 1, 1, 2, 2, [parent])
    path, plen = W.pack_paths([[0, 2, 3]], 4)  # 3's parent is 1, not 2
    with pytest.raises(oracle.OracleError):
        oracle.commit(path, plen, x["k"], x["v"], x["log_alpha"], x["beta"], x["S0"],
                      parent=x["parent"], lib=lib)


def test_config0_oracle_matches_chunked_form():
    w = W.make_config(0)
    o, U = oracle.verify_workload(w, mode="path")
    from oracle import chunked
    O, Uc = chunked.verify_workload_unit(w, 0, 0)
    assert np.abs(O - o[0, :, 0]).max() <= 1e-13 * np.abs(o).max()
    assert np.abs(Uc - U[0, 0]).max() <= 1e-13 * np.abs(U).max()


def test_golden_config0_regression():
    import os
    g = np.load(os.path.join(os.path.dirname(__file__), "golden", "config0_oracle.npz"))
    w = W.make_config(0)
    assert np.array_equal(g["parent"], w.parent) and np.array_equal(g["path"], w.path)
    o, U = oracle.verify_workload(w, mode="memo")
    S1 = oracle.commit_workload(w)
    assert np.array_equal(o, g["o"]) and np.array_equal(U, g["U"])
    assert np.array_equal(S1, g["S1"])


@pytest.mark.parametrize("tree", ["chain", "uniform"])
def test_oracle_past_256_nodes(tree):
    """At the tree sizes the chunked GPU kernel is held to (N > 256): the memoised
    oracle equals the literal path walk bitwise and the dense chunked form to
    fp64 rounding, and its commit of a path longer than 256 entries equals the
    closed form S1 = gamma_L S0 + sum_j e^{g_L - g_j} k_j u_j^T."""
    from oracle import chunked
    N = 300
    w = W.make_custom(seed=31, B=1, N=N, Hqk=1, Hv=1, dk=16, dv=16, dtype=W.F32, tree=tree,
                      max_depth=N, lmax=N)
    if tree == "chain":
        w.path[0, :] = np.arange(N, dtype=np.int32)
        w.path_len[0] = N
    o_m, U_m = oracle.verify_workload(w, mode="memo")
    o_p, U_p = oracle.verify_workload(w, mode="path")
    assert np.array_equal(o_m, o_p) and np.array_equal(U_m, U_p)
    O, Uc = chunked.verify_workload_unit(w, 0, 0)
    assert np.abs(O - o_m[0, :, 0]).max() <= 1e-11 * np.abs(o_m).max()
    assert np.abs(Uc - U_m[0, 0]).max() <= 1e-11 * np.abs(U_m).max()
    S1 = oracle.commit_workload(w)
    path = w.path[0, :w.path_len[0]]
    S1c = chunked.commit_unit(path, U_m[0, 0], w.k[0, :, 0], w.log_alpha[0, :, 0], w.S0[0, 0])
    assert np.abs(S1[0, 0] - S1c).max() <= 1e-11 * np.abs(S1c).max()
