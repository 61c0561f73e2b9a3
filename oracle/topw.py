"""Oracle of the draft-tree construction (test infrastructure only: called by the
tests, __graft_entry__.smoke() and bench.py's baseline legs, never by the library).

Method: "DFlash-TfM: Trees from Marginals", section 2 ("Costruzione dell'Albero"):
the DySpec best-first construction, modified to pop the top-w candidates of the
heap and expand all w at once, so that a tree of N nodes takes ceil(N / w)
sequential rounds.

Reading taken (the page gives no more detail):
  - node 0 is the root, score 0, depth 1;
  - every node of depth < max_depth offers c candidate children; candidate j of
    node p scores score(p) + cand_logp[p, j] (fp32 addition, the precision the
    kernel decides in);
  - a round pops the min(w, N - nodes) best live candidates (higher score first,
    ties to the lower key p * c + j, i.e. creation order), appends them as nodes
    in pop order, and only then do the new nodes offer their candidates;
  - a candidate whose score is -inf is never taken; construction stops early when
    no live candidate is left (n_built < N).

Plain Python with heapq; one sequence at a time.  Parity: pinned by
tests/test_topw_oracle.py (brute-force top-N for w = 1, stars, depth limits,
ties, invariants).
"""

from __future__ import annotations

import heapq

import numpy as np


def build_topw_one(cand_logp, N: int, w: int, max_depth: int, c: int | None = None):
    """One tree.  cand_logp is [N, c] float32, or a callable (node, depth) -> c
    log-probabilities, asked once per offering node in offer order (the form the
    pins use for path-dependent candidates).  Returns parent [N] int32 (-1 root),
    cand_index [N] int32 (j of the parent's candidate, -1 root), score [N] float32,
    depth [N] int32, the number of nodes built (entries past it are -2 / -2 / nan /
    0) and round [N] int32 (the round that took the node; 0 for the root)."""
    if callable(cand_logp):
        row = lambda p: np.asarray(cand_logp(p, int(depth[p])), dtype=np.float32)
    else:
        table = np.asarray(cand_logp, dtype=np.float32)
        c = table.shape[1]
        row = lambda p: table[p]
    parent = np.full(N, -2, np.int32)
    cidx = np.full(N, -2, np.int32)
    score = np.full(N, np.nan, np.float32)
    depth = np.zeros(N, np.int32)
    rnd = np.zeros(N, np.int32)
    parent[0], cidx[0], score[0], depth[0] = -1, -1, np.float32(0.0), 1
    heap: list[tuple[float, int]] = []  # (-score, key), key = p * c + j

    def offer(p: int) -> None:
        if depth[p] >= max_depth:
            return
        lp = row(p)
        for j in range(c):
            s = np.float32(score[p] + lp[j])  # fp32 addition, as the kernel
            if s == -np.inf:
                continue  # a candidate of probability 0 is never taken
            heapq.heappush(heap, (-float(s), p * c + j))

    offer(0)
    n, r = 1, 0
    while n < N and heap:
        r += 1
        take = min(w, N - n, len(heap))
        fresh = []
        for _ in range(take):
            negs, key = heapq.heappop(heap)
            p, j = divmod(key, c)
            parent[n], cidx[n], score[n], depth[n] = p, j, np.float32(-negs), depth[p] + 1
            rnd[n] = r
            fresh.append(n)
            n += 1
        for node in fresh:
            offer(node)
    return parent, cidx, score, depth, n, rnd


def build_topw(cand_logp: np.ndarray, w: int, max_depth: int):
    """A batch: cand_logp [B, N, c].  Returns (parent [B, N], cand_index [B, N],
    score [B, N], depth [B, N], n_built [B], round [B, N])."""
    cand_logp = np.asarray(cand_logp, dtype=np.float32)
    B, N, _ = cand_logp.shape
    outs = [build_topw_one(cand_logp[b], N, w, max_depth) for b in range(B)]
    return (np.stack([o[0] for o in outs]), np.stack([o[1] for o in outs]),
            np.stack([o[2] for o in outs]), np.stack([o[3] for o in outs]),
            np.array([o[4] for o in outs], np.int32), np.stack([o[5] for o in outs]))
