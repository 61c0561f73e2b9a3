"""Pins for the fp64 oracle: closed forms, special cases and invariants that
follow from the GDN recurrence of the DFlash-TfM page
(gist.science/it/paper/2607.06763, section 3, "Sfida") and from the
tree-verification statement of the same section ("Soluzione"), none of which
re-types the oracle's own loop.

Every pin takes an oracle library handle (so planted-mistake builds of the
oracle can be run through the same checks) and returns the largest relative
error it saw; the caller compares with PIN_TOL.
"""

from __future__ import annotations

import numpy as np

import oracle
from oracle import chunked
import workloads as W

PIN_TOL = 1e-12


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    den = max(np.abs(b).max(), 1e-300)
    return float(np.abs(a - b).max() / den)


def _unit(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _inputs(rng, B, N, Hqk, Hv, dk, dv, parents, la=(0.01, 0.5)):
    q = _unit(rng, (B, N, Hqk, dk))
    k = _unit(rng, (B, N, Hqk, dk))
    v = rng.standard_normal((B, N, Hv, dv))
    log_alpha = -rng.uniform(*la, size=(B, N, Hv))
    beta = 1 / (1 + np.exp(-rng.standard_normal((B, N, Hv))))
    S0 = 0.3 * rng.standard_normal((B, Hv, dk, dv))
    parent = np.stack(parents).astype(np.int32)
    return dict(q=q, k=k, v=v, log_alpha=log_alpha, beta=beta, parent=parent, S0=S0)


def _verify(lib, x, mode="memo"):
    return oracle.verify(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"],
                         x["parent"], x["S0"], mode=mode, lib=lib, threads=2)


# --------------------------------------------------------------------------
# C1: a single node has a closed form
# --------------------------------------------------------------------------

def pin_single_node_closed_form(lib) -> float:
    """One node off S0: S1 = a (I - b k k^T) S0 + b k v^T, so
    o = a S0^T q - a b (k.q) S0^T k + b (k.q) v and u = b (v - a S0^T k).
    Checked for dk != dv and for a square non-symmetric S0."""
    rng = np.random.default_rng(11)
    worst = 0.0
    for dk, dv in ((3, 5), (6, 6), (4, 2)):
        x = _inputs(rng, 1, 1, 1, 1, dk, dv, [np.array([-1])])
        x["k"] = rng.standard_normal(x["k"].shape)  # unnormalised is fine too
        o, U = _verify(lib, x)
        a = np.exp(x["log_alpha"][0, 0, 0])
        b = x["beta"][0, 0, 0]
        q, k, v, S0 = x["q"][0, 0, 0], x["k"][0, 0, 0], x["v"][0, 0, 0], x["S0"][0, 0]
        kq = k @ q
        o_ref = a * (S0.T @ q) - a * b * kq * (S0.T @ k) + b * kq * v
        u_ref = b * (v - a * (S0.T @ k))
        worst = max(worst, _rel(o[0, 0, 0], o_ref), _rel(U[0, 0, 0], u_ref))
        # with S0 = 0 the output is b (k.q) v
        x["S0"] = np.zeros_like(x["S0"])
        o, _ = _verify(lib, x)
        worst = max(worst, _rel(o[0, 0, 0], b * kq * v))
    return worst


# --------------------------------------------------------------------------
# C2: beta = 0 leaves only the decay
# --------------------------------------------------------------------------

def pin_pure_decay(lib) -> float:
    """beta = 0: S_t = gamma_t S0 with gamma_t the product of alpha over the
    root-to-t path, so o_t = gamma_t S0^T q_t, u_t = 0, S1 = gamma_L S0."""
    rng = np.random.default_rng(12)
    N = 9
    parents = [W.tree_uniform_parent(rng, N), W.tree_chain(N)]
    x = _inputs(rng, 2, N, 1, 2, 4, 3, parents)
    x["beta"][:] = 0.0
    o, U = _verify(lib, x)
    worst = float(np.abs(U).max())
    for b in range(2):
        for h in range(2):
            for t in range(N):
                path = W.root_path(parents[b], t)
                gam = np.prod(np.exp(x["log_alpha"][b, path, h]))
                ref = gam * (x["S0"][b, h].T @ x["q"][b, t, 0])
                worst = max(worst, _rel(o[b, t, h], ref))
    p = W.root_path(parents[0], N - 1)
    path, plen = W.pack_paths([p, [0, 1, 2]], N)
    S1 = oracle.commit(path, plen, x["k"], x["v"], x["log_alpha"], x["beta"], x["S0"],
                       parent=x["parent"], lib=lib)
    for b, pp in enumerate((p, [0, 1, 2])):
        for h in range(2):
            gam = np.prod(np.exp(x["log_alpha"][b, pp, h]))
            worst = max(worst, _rel(S1[b, h], gam * x["S0"][b, h]))
    return worst


# --------------------------------------------------------------------------
# C3: the delta rule writes v back along k
# --------------------------------------------------------------------------

def pin_delta_write_back(lib) -> float:
    """With |k_t| = 1: S_t^T k_t = a_t (1 - b_t) S_par^T k_t + b_t v_t.
    (a) a = b = 1 and q_t = k_t give o_t = v_t exactly;
    (b) in general, with q_t = k_t and u_t = b_t (v_t - a_t S_par^T k_t),
        o_t = v_t - (1 - b_t) / b_t * u_t."""
    rng = np.random.default_rng(13)
    N = 12
    parents = [W.tree_uniform_parent(rng, N), W.tree_random_capped(rng, N, 5)]
    x = _inputs(rng, 2, N, 2, 4, 5, 7, parents)
    x["q"] = x["k"].copy()
    o, U = _verify(lib, x)
    worst = 0.0
    for b in range(2):
        for h in range(4):
            be = x["beta"][b, :, h][:, None]
            ref = x["v"][b, :, h] - (1 - be) / be * U[b, h]
            worst = max(worst, _rel(o[b, :, h], ref))
    x["log_alpha"][:] = 0.0
    x["beta"][:] = 1.0
    o, _ = _verify(lib, x)
    worst = max(worst, _rel(o, x["v"]))
    return worst


# --------------------------------------------------------------------------
# C4: literal walk == memoised (bitwise) == dense chunked solve
# --------------------------------------------------------------------------

def pin_modes_and_chunked_form(lib) -> float:
    rng = np.random.default_rng(14)
    N = 10
    fams = [W.tree_uniform_parent(rng, N), W.tree_chain(N), W.tree_star(N),
            W.tree_star(N, rooted=False), W.tree_top_w(rng, N, 3, 4),
            W.tree_random_capped(rng, N, 4)]
    x = _inputs(rng, len(fams), N, 2, 4, 6, 6, fams)
    o_p, U_p = _verify(lib, x, "path")
    o_m, U_m = _verify(lib, x, "memo")
    worst = 0.0 if (np.array_equal(o_p, o_m) and np.array_equal(U_p, U_m)) else 1.0
    for b in range(len(fams)):
        for h in range(4):
            O, U = chunked.verify_unit(x["q"][b, :, h // 2], x["k"][b, :, h // 2],
                                       x["v"][b, :, h], x["log_alpha"][b, :, h],
                                       x["beta"][b, :, h], x["parent"][b], x["S0"][b, h])
            worst = max(worst, _rel(o_m[b, :, h], O), _rel(U_m[b, h], U))
    return worst


# --------------------------------------------------------------------------
# I1: a chain is the plain sequential recurrence, written with explicit
#     transition matrices A_t = a_t (I - b_t k_t k_t^T)
# --------------------------------------------------------------------------

def pin_chain_matrix_form(lib) -> float:
    rng = np.random.default_rng(15)
    N, dk, dv = 11, 5, 4
    x = _inputs(rng, 1, N, 1, 1, dk, dv, [W.tree_chain(N)])
    o, _ = _verify(lib, x)
    S = x["S0"][0, 0].copy()
    worst = 0.0
    for t in range(N):
        a = np.exp(x["log_alpha"][0, t, 0])
        b = x["beta"][0, t, 0]
        k = x["k"][0, t, 0]
        A = a * (np.eye(dk) - b * np.outer(k, k))
        S = A @ S + b * np.outer(k, x["v"][0, t, 0])
        worst = max(worst, _rel(o[0, t, 0], S.T @ x["q"][0, t, 0]))
    # prefix stability: the first M nodes of a chain do not see later nodes
    M = 6
    xs = {kk: (vv[:, :M] if kk in ("q", "k", "v", "log_alpha", "beta", "parent") else vv)
          for kk, vv in x.items()}
    o2, _ = _verify(lib, xs)
    worst = max(worst, _rel(o2[0], o[0, :M]))
    return worst


# --------------------------------------------------------------------------
# I2: every node equals its own path run alone as a chain
# --------------------------------------------------------------------------

def pin_path_isolation(lib) -> float:
    rng = np.random.default_rng(16)
    N = 14
    parents = [W.tree_uniform_parent(rng, N), W.tree_top_w(rng, N, 2, 6)]
    x = _inputs(rng, 2, N, 1, 2, 4, 5, parents)
    o, U = _verify(lib, x)
    worst = 0.0
    for b in range(2):
        for t in range(N):
            p = W.root_path(parents[b], t)
            L = len(p)
            xs = dict(q=x["q"][b:b + 1, p], k=x["k"][b:b + 1, p], v=x["v"][b:b + 1, p],
                      log_alpha=x["log_alpha"][b:b + 1, p], beta=x["beta"][b:b + 1, p],
                      parent=W.tree_chain(L)[None], S0=x["S0"][b:b + 1])
            oc, Uc = _verify(lib, xs)
            worst = max(worst, _rel(oc[0, L - 1], o[b, t]), _rel(Uc[0, :, L - 1], U[b, :, t]))
    return worst


# --------------------------------------------------------------------------
# I3: relabelling by another topological order only permutes the outputs
# --------------------------------------------------------------------------

def random_topological_relabel(rng, parent):
    """perm[new] = old, for a random order in which parents precede children."""
    N = len(parent)
    children = [[] for _ in range(N)]
    ready = []
    for i, p in enumerate(parent):
        (ready if p < 0 else children[p]).append(i)
    order = []
    while ready:
        j = ready.pop(int(rng.integers(len(ready))))
        order.append(j)
        ready.extend(children[j])
    perm = np.array(order)
    inv = np.empty(N, dtype=np.int64)
    inv[perm] = np.arange(N)
    new_parent = np.array([-1 if parent[o] < 0 else inv[parent[o]] for o in perm],
                          dtype=np.int32)
    return perm, new_parent


def pin_sibling_permutation(lib) -> float:
    rng = np.random.default_rng(17)
    N = 16
    parent = W.tree_random_capped(rng, N, 6)
    x = _inputs(rng, 1, N, 1, 2, 4, 4, [parent])
    o, U = _verify(lib, x)
    perm, new_parent = random_topological_relabel(rng, parent)
    assert not np.array_equal(perm, np.arange(N))
    xp = {kk: (vv[:, perm] if kk in ("q", "k", "v", "log_alpha", "beta") else vv)
          for kk, vv in x.items()}
    xp["parent"] = new_parent[None]
    op, Up = _verify(lib, xp)
    return max(_rel(op[0], o[0, perm]), _rel(Up[0][:, :], U[0][:, perm]))


# --------------------------------------------------------------------------
# I4: commit consistency and grafting
# --------------------------------------------------------------------------

def pin_commit_and_graft(lib) -> float:
    """Commit along p equals (a) the chunked commit formula fed by the verify's
    U rows, and (b) grafting: verifying a new tree T from S1 equals verifying
    p followed by T from S0, restricted to T's nodes.  An empty path commits
    S0 unchanged."""
    rng = np.random.default_rng(18)
    N = 12
    parent = W.tree_random_capped(rng, N, 6)
    x = _inputs(rng, 1, N, 1, 2, 5, 4, [parent])
    o, U = _verify(lib, x)
    p = W.random_leaf_path(rng, parent)
    path, plen = W.pack_paths([p], N)
    S1 = oracle.commit(path, plen, x["k"], x["v"], x["log_alpha"], x["beta"], x["S0"],
                       parent=x["parent"], lib=lib)
    worst = 0.0
    for h in range(2):
        ref = chunked.commit_unit(p, U[0, h], x["k"][0, :, 0], x["log_alpha"][0, :, h],
                                  x["S0"][0, h])
        worst = max(worst, _rel(S1[0, h], ref))
    # grafting
    M = 7
    T_parent = W.tree_uniform_parent(rng, M)
    y = _inputs(rng, 1, M, 1, 2, 5, 4, [T_parent])
    y["S0"] = S1
    oT, UT = _verify(lib, y)
    L = len(p)
    gp = np.concatenate([W.tree_chain(L), np.where(T_parent < 0, L - 1, T_parent + L)])
    z = {kk: np.concatenate([x[kk][:, p], y[kk]], axis=1)
         for kk in ("q", "k", "v", "log_alpha", "beta")}
    z["parent"] = gp[None].astype(np.int32)
    z["S0"] = x["S0"]
    oG, UG = _verify(lib, z)
    worst = max(worst, _rel(oG[0, L:], oT[0]), _rel(UG[0][:, L:], UT[0]))
    # empty path
    S1e = oracle.commit(np.full((1, 1), -1, np.int32), np.zeros(1, np.int32), x["k"],
                        x["v"], x["log_alpha"], x["beta"], x["S0"], lib=lib)
    worst = max(worst, _rel(S1e, x["S0"]))
    return worst


# --------------------------------------------------------------------------
# I5: outputs are linear in (V, S0) jointly
# --------------------------------------------------------------------------

def pin_linearity(lib) -> float:
    """The recurrence is linear in (S, v) for fixed k, alpha, beta: scaling v and
    S0 by 2 scales o and U by exactly 2, and sums superpose."""
    rng = np.random.default_rng(19)
    N = 10
    x = _inputs(rng, 1, N, 1, 1, 4, 6, [W.tree_uniform_parent(rng, N)])
    o, U = _verify(lib, x)
    x2 = dict(x, v=2 * x["v"], S0=2 * x["S0"])
    o2, U2 = _verify(lib, x2)
    worst = 0.0 if (np.array_equal(o2, 2 * o) and np.array_equal(U2, 2 * U)) else 1.0
    v_b = rng.standard_normal(x["v"].shape)
    S_b = rng.standard_normal(x["S0"].shape)
    ob, Ub = _verify(lib, dict(x, v=v_b, S0=S_b))
    os_, Us = _verify(lib, dict(x, v=x["v"] + v_b, S0=x["S0"] + S_b))
    worst = max(worst, _rel(os_, o + ob), _rel(Us, U + Ub))
    return worst


ALL_PINS = [
    pin_single_node_closed_form,
    pin_pure_decay,
    pin_delta_write_back,
    pin_modes_and_chunked_form,
    pin_chain_matrix_form,
    pin_path_isolation,
    pin_sibling_permutation,
    pin_commit_and_graft,
    pin_linearity,
]
