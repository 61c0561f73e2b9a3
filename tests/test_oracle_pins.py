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
