"""Pins of the draft-tree construction oracle (oracle/topw.py): checks against
what the page and the mathematics fix, not against a retyped copy of the loop."""

import itertools

import numpy as np
import pytest

from oracle.topw import build_topw, build_topw_one


def implicit_topn(m, N, max_depth):
    """Brute force: every node of the implicit candidate tree whose candidates at
    depth d score m[d][j] (a factorized drafter: the same marginal for every node
    of a depth), ranked by path score; the N best (ties impossible here)."""
    c = m.shape[1]
    scores = [0.0]
    for length in range(1, max_depth):
        for path in itertools.product(range(c), repeat=length):
            s = np.float32(0.0)
            for d, j in enumerate(path):
                s = np.float32(s + m[d + 1][j])
            scores.append(float(s))
    return sorted(scores, reverse=True)[:N]


@pytest.mark.parametrize("c,max_depth,N,seed", [(2, 4, 9, 0), (3, 3, 10, 1), (3, 4, 20, 2),
                                                (2, 5, 17, 3)])
def test_sequential_best_first_takes_the_global_top_n(c, max_depth, N, seed):
    """With w = 1 (sequential best-first) and log-probabilities <= 0, a child never
    outscores its parent, so the N nodes built are the N best of the whole
    implicit tree."""
    rng = np.random.default_rng(seed)
    m = np.log(rng.uniform(0.05, 1.0, size=(max_depth + 1, c))).astype(np.float32)
    parent, cidx, score, depth, n, rnd = build_topw_one(lambda p, d: m[d], N, 1, max_depth, c=c)
    assert n == N
    np.testing.assert_array_equal(np.sort(score)[::-1], np.array(implicit_topn(m, N, max_depth),
                                                                  np.float32))


def test_round_expands_only_after_all_pops():
    """w = 2: the root offers A (-1) and B (-2); A's child would score -1.1, but the
    new nodes offer their candidates only after the round, so B is taken."""
    logp = np.full((8, 2), -50.0, np.float32)
    logp[0] = [-1.0, -2.0]
    logp[1] = [-0.1, -30.0]
    parent, cidx, score, depth, n, rnd = build_topw_one(logp, 4, 2, 10)
    assert parent.tolist()[:3] == [-1, 0, 0] and cidx.tolist()[:3] == [-1, 0, 1]
    assert parent[3] == 1 and cidx[3] == 0  # round 2: A's first child (-1.1)


def test_star_and_depth_limit():
    rng = np.random.default_rng(5)
    logp = np.log(rng.uniform(size=(9, 6))).astype(np.float32)
    # max_depth 2: only the root offers; the tree is its c children, best first
    parent, cidx, score, depth, n, rnd = build_topw_one(logp, 9, 3, 2)
    assert n == 7 and (parent[1:7] == 0).all() and (depth[1:7] == 2).all()
    assert cidx[1:7].tolist() == list(np.argsort(-logp[0], kind="stable"))
    assert (parent[7:] == -2).all()  # ran out of candidates


def test_chain():
    logp = np.log(np.full((12, 1), 0.5)).astype(np.float32)
    parent, cidx, score, depth, n, rnd = build_topw_one(logp, 12, 1, 7)
    assert n == 7 and parent[:7].tolist() == [-1, 0, 1, 2, 3, 4, 5]
    np.testing.assert_array_equal(score[:7], np.cumsum(np.r_[0, logp[:6, 0]]).astype(np.float32))


def test_ties_go_to_creation_order():
    logp = np.zeros((6, 3), np.float32) - 1.0
    parent, cidx, score, depth, n, rnd = build_topw_one(logp, 6, 2, 5)
    # round 1: root's candidates 0, 1; round 2: root's candidate 2, then node 1's first
    assert list(zip(parent[1:5].tolist(), cidx[1:5].tolist())) == [(0, 0), (0, 1), (0, 2), (1, 0)]


@pytest.mark.parametrize("c,w,N,max_depth", [(4, 4, 64, 16), (4, 4, 128, 24), (8, 8, 256, 12),
                                              (3, 1, 40, 40), (2, 5, 31, 6)])
def test_invariants(c, w, N, max_depth):
    rng = np.random.default_rng(N + c)
    logp = np.log(rng.uniform(1e-6, 1.0, size=(3, N, c))).astype(np.float32)
    parent, cidx, score, depth, n, rnd = build_topw(logp, w, max_depth)
    for b in range(3):
        nb = n[b]
        p, j, s, d = parent[b, :nb], cidx[b, :nb], score[b, :nb], depth[b, :nb]
        assert p[0] == -1 and (p[1:] >= 0).all() and (p[1:] < np.arange(1, nb)).all()
        assert (d[1:] == d[p[1:]] + 1).all() and d.max() <= max_depth
        # every score is its parent's plus the chosen candidate's, in fp32
        want = (s[p[1:]] + logp[b, p[1:], j[1:]]).astype(np.float32)
        np.testing.assert_array_equal(s[1:], want)
        assert len(set(zip(p[1:].tolist(), j[1:].tolist()))) == nb - 1  # each candidate once
        # rounds take at most w nodes each, best first; ceil(n / w) rounds at least
        rb = rnd[b, 1:nb]
        assert (np.diff(rb) >= 0).all() and np.bincount(rb).max() <= w
        for r in np.unique(rb):
            assert (np.diff(s[1:][rb == r]) <= 0).all()
        if nb < N:  # ran out: no node could offer a live candidate any more
            offered = int(((d < max_depth) * c).sum())
            assert offered == nb - 1
