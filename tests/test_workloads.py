"""Seeded input generators: determinism, tree validity and the workload recipe."""

import numpy as np
import pytest

import workloads as W


def test_bf16_round_is_ties_to_even():
    x = np.array([1.0, 1.0 + 2**-8, 1.0 + 3 * 2**-8, -2.5, 1.0 + 2**-9], dtype=np.float32)
    r = W.bf16_round(x)
    assert r.tolist() == [1.0, 1.0, 1.0 + 4 * 2**-8, -2.5, 1.0]


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_config_shapes_and_trees(cfg):
    w = W.make_config(cfg)
    w2 = W.make_config(cfg)
    assert np.array_equal(w.q, w2.q) and np.array_equal(w.parent, w2.parent)
    assert w.q.shape == (w.B, w.N, w.Hqk, w.dk) and w.v.shape == (w.B, w.N, w.Hv, w.dv)
    for b in range(w.B):
        W.check_tree(w.parent[b])
        L = int(w.path_len[b])
        p = w.path[b, :L].tolist()
        assert 1 <= L <= w.Lmax
        assert p == W.root_path(w.parent[b], p[-1])
    if w.dtype == W.BF16:
        assert np.array_equal(W.bf16_round(w.q), w.q)
    assert (w.log_alpha < 0).all() and ((w.beta > 0) & (w.beta < 1)).all()


def test_depth_and_shape_limits():
    w = W.make_config(3)
    assert max(W.node_depths(p).max() for p in w.parent) <= 24
    assert w.path_len.max() <= 24
    w = W.make_config(2)
    assert max(W.node_depths(p).max() for p in w.parent) <= 16
    # different tree per sequence
    assert len({tuple(p) for p in w.parent}) == w.B


def test_top_w_tree_grows_by_rounds():
    rng = np.random.default_rng(3)
    p = W.tree_top_w(rng, 64, w=4, max_depth=16)
    W.check_tree(p)
    assert p[0] == -1 and (p[1:] >= 0).all()
