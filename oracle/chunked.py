"""Dense numpy form of the chunked, masked-triangular-solve verification.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Everything is fp64 and
works on ONE (sequence, v-head) unit.

Source: DFlash-TfM (gist.science/it/paper/2607.06763), section 3 "Soluzione":
the verification is a chunked form of the linear recurrence, posed as a masked
triangular solve over the topologically ordered tree, with interaction
matrices X and Y built from the ancestor relation and a linear system
(I + X) U = ... .  The page prints the right-hand side only as "beta V"; the
exact form used here follows from unrolling the recurrence along the path
(S0 = 0 gives the page's form):

    g_t      = sum of log alpha_s over the root-to-t path P(t), gamma_t = e^{g_t}
    X[t, s]  = beta_t e^{g_t - g_s} (k_t . k_s)     for s a strict ancestor of t
    Y[t, s]  =        e^{g_t - g_s} (q_t . k_s)     for s in P(t) (incl. t)
    (I + X) U = diag(beta) (V - diag(gamma) K S0)
    O         = diag(gamma) Q S0 + Y U
    commit:   S1 = gamma_{p_L} S0 + sum_j e^{g_{p_L} - g_{p_j}} k_{p_j} u_{p_j}^T
"""

from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def ancestors(parent: np.ndarray) -> list[list[int]]:
    """Strict ancestors of every node (root first)."""
    out = []
    for t in range(len(parent)):
        a = []
        s = int(parent[t])
        while s >= 0:
            a.append(s)
            s = int(parent[s])
        out.append(a[::-1])
    return out


def path_log_decay(parent: np.ndarray, log_alpha: np.ndarray) -> np.ndarray:
    """g_t = sum of log_alpha over the root-to-t path, fp64."""
    g = np.zeros(len(parent))
    for t in range(len(parent)):
        g[t] = log_alpha[t] + (g[parent[t]] if parent[t] >= 0 else 0.0)
    return g


def interaction_matrices(q, k, log_alpha, beta, parent):
    """X (strictly lower, ancestor-masked) and Y (ancestor-or-self masked)."""
    q, k = np.asarray(q, np.float64), np.asarray(k, np.float64)
    la, be = np.asarray(log_alpha, np.float64), np.asarray(beta, np.float64)
    N = len(parent)
    g = path_log_decay(parent, la)
    X = np.zeros((N, N))
    Y = np.zeros((N, N))
    for t, anc in enumerate(ancestors(parent)):
        for s in anc:
            X[t, s] = be[t] * np.exp(g[t] - g[s]) * (k[t] @ k[s])
            Y[t, s] = np.exp(g[t] - g[s]) * (q[t] @ k[s])
        Y[t, t] = q[t] @ k[t]
    return X, Y, g


def verify_unit(q, k, v, log_alpha, beta, parent, S0):
    """One unit: q, k [N, dk]; v [N, dv]; gates [N]; S0 [dk, dv].
    Returns (O [N, dv], U [N, dv])."""
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    S0 = np.asarray(S0, np.float64)
    be = np.asarray(beta, np.float64)
    X, Y, g = interaction_matrices(q, k, log_alpha, beta, parent)
    gam = np.exp(g)
    R = be[:, None] * (v - gam[:, None] * (k @ S0))
    N = len(parent)
    U = solve_triangular(np.eye(N) + X, R, lower=True, unit_diagonal=True)
    O = gam[:, None] * (q @ S0) + Y @ U
    return O, U


def commit_unit(path, U, k, log_alpha, S0):
    """S1 from the verify's U rows along the accepted path p_1..p_L."""
    k = np.asarray(k, np.float64)
    U = np.asarray(U, np.float64)
    S0 = np.asarray(S0, np.float64)
    la = np.asarray(log_alpha, np.float64)
    if len(path) == 0:
        return S0.copy()
    G = np.cumsum(la[list(path)])  # g along the path
    S1 = np.exp(G[-1]) * S0
    for j, p in enumerate(path):
        S1 = S1 + np.exp(G[-1] - G[j]) * np.outer(k[p], U[p])
    return S1


def verify_workload_unit(w, b: int, h: int):
    hq = h // (w.Hv // w.Hqk)
    return verify_unit(w.q[b, :, hq], w.k[b, :, hq], w.v[b, :, h],
                       w.log_alpha[b, :, h], w.beta[b, :, h], w.parent[b],
                       w.S0[b, h])
