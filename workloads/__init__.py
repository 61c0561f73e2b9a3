"""Seeded synthetic inputs for rollback-free GDN tree verification.

This module only draws random numbers, builds tree shapes and rounds values to
the storage dtype.  It holds none of the method's arithmetic (no recurrence, no
decay products, no solve), so the fp64 oracle and the CUDA path can both read
the inputs it produces without sharing any computation.

Tensor layouts (all C-contiguous):

    q, k        [B, N, Hqk, dk]   values exactly representable in `dtype`
    v           [B, N, Hv,  dv]   same
    log_alpha   [B, N, Hv]        float32, log of the per-step decay alpha_t
    beta        [B, N, Hv]        float32, per-step write strength beta_t
    parent      [B, N]            int32, parent[i] < i, -1 = child of S0
    S0          [B, Hv, dk, dv]   float32 committed state (dv contiguous)
    path        [B, Lmax]         int32 accepted root-to-node path, -1 padded
    path_len    [B]               int32

The draws follow the workload recipe of the tree-verification setting of
"DFlash-TfM: Trees from Marginals" (gist.science/it/paper/2607.06763, section 3,
"Verifica dell'Albero Senza Rollback per GDN"): q, k ~ N(0, 1) then
L2-normalised per (node, head), v ~ N(0, 1), log alpha ~ -U(0.01, 0.5),
beta = sigmoid(N(0, 1)), S0 ~ N(0, 0.1^2).  Tree shapes stand in for the
drafter's trees of that page's section 2 ("Costruzione dell'Albero").
"""

from __future__ import annotations

import heapq
from dataclasses import dataclass, field

import numpy as np

BF16 = "bf16"
F32 = "f32"

# ---------------------------------------------------------------------------
# dtype rounding
# ---------------------------------------------------------------------------


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bfloat16 (ties to even).

    Returns float32 values that are exactly representable in bfloat16, so a
    later cast to torch.bfloat16 is exact.  NaN/Inf are not expected here.
    """
    f = np.ascontiguousarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> np.uint64(16)) & np.uint64(1)
    bits = (bits + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    out = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return out.reshape(np.shape(x))


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == BF16:
        return bf16_round(x)
    if dtype == F32:
        return np.asarray(x, dtype=np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


# ---------------------------------------------------------------------------
# tree shapes (topologically ordered: parent[i] < i, -1 hangs off S0)
# ---------------------------------------------------------------------------


def tree_uniform_parent(rng: np.random.Generator, n: int) -> np.ndarray:
    """parent[i] uniform in {-1, ..., i-1}; may give a forest."""
    return np.array([rng.integers(-1, i) for i in range(n)], dtype=np.int32)


def tree_chain(n: int) -> np.ndarray:
    return np.arange(-1, n - 1, dtype=np.int32)


def tree_star(n: int, rooted: bool = True) -> np.ndarray:
    """rooted: node 0 hangs off S0 and every other node off node 0.
    not rooted: every node hangs off S0 directly."""
    if not rooted:
        return np.full(n, -1, dtype=np.int32)
    p = np.zeros(n, dtype=np.int32)
    p[0] = -1
    return p


def tree_random_capped(rng: np.random.Generator, n: int, max_depth: int,
                       max_branch: int = 4) -> np.ndarray:
    """Random tree with node 0 as root.  Each node draws a branching cap in
    {1..max_branch}; node i attaches to a uniformly chosen earlier node that
    still has spare capacity and depth < max_depth (root depth = 1)."""
    parent = [-1]
    depth = [1]
    cap = [int(rng.integers(1, max_branch + 1))]
    nchild = [0]
    for i in range(1, n):
        cands = [j for j in range(i) if nchild[j] < cap[j] and depth[j] < max_depth]
        if not cands:
            cands = [j for j in range(i) if depth[j] < max_depth]
        j = cands[int(rng.integers(len(cands)))]
        parent.append(j)
        depth.append(depth[j] + 1)
        cap.append(int(rng.integers(1, max_branch + 1)))
        nchild.append(0)
        nchild[j] += 1
    return np.array(parent, dtype=np.int32)


def tree_top_w(rng: np.random.Generator, n: int, w: int = 4,
               max_depth: int = 16) -> np.ndarray:
    """Best-first tree growth that pops the top-w candidates per round.

    The expansion rule of the DFlash-TfM page, section 2 (top-w pops from the
    candidate heap, w expansions at once): node 0 is the root; every tree node
    offers w candidate children whose score is the parent's score plus
    log U(0, 1); each round pops the w best candidates (ties: lower creation
    index) and appends them in pop order; only then do the new nodes offer
    their own candidates.  Nodes at max_depth offer none.
    """
    parent = [-1]
    depth = [1]
    score = [0.0]
    heap: list[tuple[float, int, int]] = []
    created = 0

    def offer(node: int) -> None:
        nonlocal created
        if depth[node] >= max_depth:
            return
        for _ in range(w):
            s = score[node] + float(np.log(rng.uniform(1e-300, 1.0)))
            heapq.heappush(heap, (-s, created, node))
            created += 1

    offer(0)
    while len(parent) < n and heap:
        take = min(w, len(heap), n - len(parent))
        popped = [heapq.heappop(heap) for _ in range(take)]
        fresh = []
        for negs, _, par in popped:
            parent.append(par)
            depth.append(depth[par] + 1)
            score.append(-negs)
            fresh.append(len(parent) - 1)
        for node in fresh:
            offer(node)
    if len(parent) != n:
        raise RuntimeError("top-w growth ran out of candidates")
    return np.array(parent, dtype=np.int32)


def node_depths(parent: np.ndarray) -> np.ndarray:
    d = np.zeros(len(parent), dtype=np.int64)
    for i, p in enumerate(parent):
        d[i] = 1 if p < 0 else d[p] + 1
    return d


def check_tree(parent: np.ndarray) -> None:
    for i, p in enumerate(parent):
        if not (-1 <= p < i):
            raise ValueError(f"parent[{i}] = {p} is not in [-1, {i - 1}]")


def root_path(parent: np.ndarray, node: int) -> list[int]:
    """Nodes of the root-to-node path, root first."""
    out = []
    while node >= 0:
        out.append(int(node))
        node = int(parent[node])
    return out[::-1]


def leaves(parent: np.ndarray) -> np.ndarray:
    has_child = np.zeros(len(parent), dtype=bool)
    for p in parent:
        if p >= 0:
            has_child[p] = True
    return np.nonzero(~has_child)[0]


def random_leaf_path(rng: np.random.Generator, parent: np.ndarray) -> list[int]:
    lv = leaves(parent)
    return root_path(parent, int(lv[int(rng.integers(len(lv)))]))


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------


@dataclass
class Workload:
    name: str
    B: int
    N: int
    Hqk: int
    Hv: int
    dk: int
    dv: int
    dtype: str
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    log_alpha: np.ndarray
    beta: np.ndarray
    parent: np.ndarray
    S0: np.ndarray | None
    path: np.ndarray
    path_len: np.ndarray
    # raw draws for a state warm-up (k, v, log_alpha, beta over T tokens); the
    # harness turns them into S0 with the oracle's sequential recurrence.
    warmup: dict | None = None
    notes: dict = field(default_factory=dict)

    @property
    def Lmax(self) -> int:
        return int(self.path.shape[1])

    def nbytes_inputs(self) -> int:
        es = 2 if self.dtype == BF16 else 4
        return int((self.q.size + self.k.size + self.v.size) * es
                   + (self.log_alpha.size + self.beta.size) * 4
                   + self.parent.size * 4 + self.S0.size * 4
                   + self.path.size * 4 + self.path_len.size * 4)


def _unit_rows(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    x = rng.standard_normal(shape)
    x = x / np.linalg.norm(x, axis=-1, keepdims=True)
    return round_to(x, dtype)


def draw_qkv(rng, B, N, Hqk, Hv, dk, dv, dtype):
    q = _unit_rows(rng, (B, N, Hqk, dk), dtype)
    k = _unit_rows(rng, (B, N, Hqk, dk), dtype)
    v = round_to(rng.standard_normal((B, N, Hv, dv)), dtype)
    return q, k, v


def draw_gates(rng, B, N, Hv, la_lo=0.01, la_hi=0.5, beta_kind="sigmoid"):
    log_alpha = (-rng.uniform(la_lo, la_hi, size=(B, N, Hv))).astype(np.float32)
    if beta_kind == "sigmoid":
        beta = (1.0 / (1.0 + np.exp(-rng.standard_normal((B, N, Hv))))).astype(np.float32)
    elif beta_kind == "uniform":
        beta = rng.uniform(0.01, 0.99, size=(B, N, Hv)).astype(np.float32)
    else:
        raise ValueError(beta_kind)
    return log_alpha, beta


def draw_state(rng, B, Hv, dk, dv, scale=0.1):
    return (scale * rng.standard_normal((B, Hv, dk, dv))).astype(np.float32)


def pack_paths(paths: list[list[int]], lmax: int):
    B = len(paths)
    path = np.full((B, lmax), -1, dtype=np.int32)
    plen = np.zeros(B, dtype=np.int32)
    for b, p in enumerate(paths):
        if len(p) > lmax:
            raise ValueError("path longer than Lmax")
        path[b, : len(p)] = p
        plen[b] = len(p)
    return path, plen


CONFIG_NAMES = {
    0: "tiny-f32-d32-N8",
    1: "decode-B1-Hv32-N16-warm512",
    2: "batched-B8-Hv32-N64-topw4",
    3: "serving-B32-Hv32-N128",
    4: "stress-B64-Hv32-N256-mixed",
}


def make_config(cfg: int, seed: int | None = None) -> Workload:
    """The five workloads of the tree-verification setting, seeded
    (default seed = 1000 + cfg).  Config 1 carries warm-up draws instead of
    S0; the caller builds S0 from them with the oracle's recurrence."""
    if seed is None:
        seed = 1000 + cfg
    rng = np.random.Generator(np.random.PCG64(seed))
    if cfg == 0:
        B, N, Hqk, Hv, d, dt = 1, 8, 1, 1, 32, F32
        parents = [tree_uniform_parent(rng, N)]
        q, k, v = draw_qkv(rng, B, N, Hqk, Hv, d, d, dt)
        la, be = draw_gates(rng, B, N, Hv)
        S0 = draw_state(rng, B, Hv, d, d)
        paths = [random_leaf_path(rng, p) for p in parents]
        lmax, warm = N, None
    elif cfg == 1:
        B, N, Hqk, Hv, d, dt = 1, 16, 16, 32, 128, BF16
        parents = [tree_random_capped(rng, N, max_depth=8)]
        q, k, v = draw_qkv(rng, B, N, Hqk, Hv, d, d, dt)
        la, be = draw_gates(rng, B, N, Hv)
        T = 512
        wq, wk, wv = draw_qkv(rng, B, T, Hqk, Hv, d, d, dt)
        wla, wbe = draw_gates(rng, B, T, Hv)
        warm = dict(T=T, k=wk, v=wv, log_alpha=wla, beta=wbe)
        S0 = None
        paths = [random_leaf_path(rng, p) for p in parents]
        lmax = 8
    elif cfg == 2:
        B, N, Hqk, Hv, d, dt = 8, 64, 16, 32, 128, BF16
        parents = [tree_top_w(rng, N, w=4, max_depth=16) for _ in range(B)]
        q, k, v = draw_qkv(rng, B, N, Hqk, Hv, d, d, dt)
        la, be = draw_gates(rng, B, N, Hv)
        S0 = draw_state(rng, B, Hv, d, d)
        paths = []
        for p in parents:
            full = random_leaf_path(rng, p)
            L = int(rng.integers(1, 17))
            paths.append(full[: min(L, len(full))])
        lmax, warm = 16, None
    elif cfg == 3:
        B, N, Hqk, Hv, d, dt = 32, 128, 16, 32, 128, BF16
        parents = [tree_random_capped(rng, N, max_depth=24) for _ in range(B)]
        q, k, v = draw_qkv(rng, B, N, Hqk, Hv, d, d, dt)
        la, be = draw_gates(rng, B, N, Hv)
        S0 = draw_state(rng, B, Hv, d, d)
        paths = []
        for p in parents:
            full = random_leaf_path(rng, p)
            L = int(rng.integers(1, min(24, len(full)) + 1))
            paths.append(full[:L])
        lmax, warm = 24, None
    elif cfg == 4:
        B, N, Hqk, Hv, d, dt = 64, 256, 16, 32, 128, BF16
        parents = []
        for b in range(B):
            kind = b % 3
            if kind == 0:
                parents.append(tree_chain(N))
            elif kind == 1:
                parents.append(tree_star(N, rooted=(b % 2 == 1)))
            else:
                parents.append(tree_random_capped(rng, N, max_depth=64))
        q, k, v = draw_qkv(rng, B, N, Hqk, Hv, d, d, dt)
        la, be = draw_gates(rng, B, N, Hv, la_lo=0.01, la_hi=4.0, beta_kind="uniform")
        be[B - 1] = np.float32(0.99)  # one sequence with beta = 0.99 everywhere
        S0 = draw_state(rng, B, Hv, d, d)
        paths = []
        for p in parents:
            full = random_leaf_path(rng, p)
            L = int(rng.integers(1, len(full) + 1))
            paths.append(full[:L])
        lmax, warm = 256, None
    else:
        raise ValueError(f"no config {cfg}")
    parent = np.stack(parents).astype(np.int32)
    path, plen = pack_paths(paths, lmax)
    return Workload(name=CONFIG_NAMES[cfg], B=B, N=N, Hqk=Hqk, Hv=Hv, dk=d, dv=d,
                    dtype=dt, q=q, k=k, v=v, log_alpha=la, beta=be, parent=parent,
                    S0=S0, path=path, path_len=plen, warmup=warm,
                    notes=dict(config=cfg, seed=seed))


def make_custom(seed: int, B: int, N: int, Hqk: int, Hv: int, dk: int, dv: int,
                dtype: str = BF16, tree: str = "random", max_depth: int = 24,
                la_range=(0.01, 0.5), beta_kind="sigmoid", s0_scale=0.1,
                lmax: int | None = None) -> Workload:
    """Free-form workload for tests: any shape, any tree family
    ("random", "uniform", "chain", "star", "flatstar", "topw", "mixed")."""
    rng = np.random.Generator(np.random.PCG64(seed))
    parents = []
    for b in range(B):
        kind = tree
        if tree == "mixed":
            kind = ["chain", "star", "random", "uniform", "flatstar", "topw"][b % 6]
        if kind == "random":
            parents.append(tree_random_capped(rng, N, max_depth=max_depth))
        elif kind == "uniform":
            parents.append(tree_uniform_parent(rng, N))
        elif kind == "chain":
            parents.append(tree_chain(N))
        elif kind == "star":
            parents.append(tree_star(N, rooted=True))
        elif kind == "flatstar":
            parents.append(tree_star(N, rooted=False))
        elif kind == "topw":
            parents.append(tree_top_w(rng, N, w=4, max_depth=max(2, max_depth)))
        else:
            raise ValueError(kind)
    q, k, v = draw_qkv(rng, B, N, Hqk, Hv, dk, dv, dtype)
    la, be = draw_gates(rng, B, N, Hv, la_lo=la_range[0], la_hi=la_range[1],
                        beta_kind=beta_kind)
    S0 = draw_state(rng, B, Hv, dk, dv, scale=s0_scale)
    paths = []
    for p in parents:
        full = random_leaf_path(rng, p)
        L = int(rng.integers(1, len(full) + 1))
        paths.append(full[:L])
    if lmax is None:
        lmax = max(1, max(len(p) for p in paths))
    path, plen = pack_paths(paths, lmax)
    return Workload(name=f"custom-{tree}-B{B}-N{N}-d{dk}x{dv}-{dtype}", B=B, N=N,
                    Hqk=Hqk, Hv=Hv, dk=dk, dv=dv, dtype=dtype, q=q, k=k, v=v,
                    log_alpha=la, beta=be, parent=np.stack(parents).astype(np.int32),
                    S0=S0, path=path, path_len=plen, notes=dict(seed=seed))
