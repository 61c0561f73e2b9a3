/*
 * gdn_tree.h -- C ABI of libgdntree: rollback-free tree verification and
 * delayed state commitment for Gated DeltaNet (GDN) layers, on sm_103a.
 *
 * The method is the one of "DFlash-TfM: Trees from Marginals"
 * (gist.science/it/paper/2607.06763), section 3 "Verifica dell'Albero Senza
 * Rollback per GDN":
 *
 *   - GDN recurrence ("Sfida"):
 *       S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 *     S in R^{dk x dv}; the output of a step is o_t = S_t^T q_t.
 *   - The draft tree is topologically ordered; every node's output is the
 *     recurrence run along its own root-to-node path from the committed state
 *     S0, computed in one chunked pass as a masked triangular solve with
 *     ancestor interaction matrices X and Y ("Soluzione").
 *   - The state is committed only at the next decoding iteration, once the
 *     accepted branch is known, so no state is ever rolled back.
 *
 * Closed form used by the kernels (the page prints the system only as
 * "(I+X)U = beta V", its S0 = 0 case): with g_t the sum of log alpha over the
 * root-to-t path P(t) and gamma_t = exp(g_t),
 *     X[t,s] = beta_t exp(g_t - g_s) (k_t . k_s)   for s a strict ancestor of t,
 *     Y[t,s] =        exp(g_t - g_s) (q_t . k_s)   for s in P(t),
 *     (I + X) U = diag(beta) (V - diag(gamma) K S0),
 *     O = diag(gamma) Q S0 + Y U,
 *     S1 = gamma_{p_L} S0 + sum_j exp(g_{p_L} - g_{p_j}) k_{p_j} u_{p_j}^T.
 * Row t of U is u_t = beta_t (v_t - alpha_t S_parent(t)^T k_t): one row per
 * node, shared by every branch through it.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every tensor pointer is a DEVICE pointer owned by the caller; the library
 *    keeps no pointer after the call returns and allocates no device memory.
 *  - Every tensor is dense, row-major (C-contiguous) and 16-byte aligned.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream).  A return of GDN_TREE_OK means the work was enqueued.
 *  - Shape/pointer problems are reported by the return value BEFORE any
 *    launch.  Problems that depend on device data (an invalid tree or path)
 *    are reported per sequence in `dev_status` (int32[B], device memory,
 *    may be NULL); the outputs of such a sequence are left unwritten.  The
 *    call first sets every dev_status[b] to GDN_TREE_STATUS_OK on `stream`
 *    (a stream-ordered fill, no allocation); each of the sequence's (b, h)
 *    units then raises it to the largest code it reports, so a report is
 *    never lost to another unit's.
 *  - The library is thread-safe and holds no global mutable state.
 *
 * Shapes (B sequences, Hqk query/key heads, Hv value heads, Hv % Hqk == 0,
 * v-head h reads q/k head h / (Hv / Hqk)):
 *    q, k        [B, N, Hqk, dk]   bf16 or fp32 (dims.dtype)
 *    v           [B, N, Hv,  dv]   same dtype as q, k
 *    log_alpha   [B, N, Hv]        fp32, log of the decay alpha (<= 0 typical)
 *    beta        [B, N, Hv]        fp32
 *    parent      [B, N]            int32, -1 <= parent[b][i] < i (-1: child of S0)
 *    S0, S1      [B, Hv, dk, dv]   fp32, dv contiguous
 *    o           [B, N, Hv, dv]    same dtype as q
 *    U           [B, Hv, N, dv]    fp32
 *    path        [B, Lmax]         int32 accepted root-to-node path, -1 padded
 *    path_len    [B]               int32, 0 <= path_len[b] <= min(N, Lmax)
 *
 * Limits: 1 <= N <= 1024 and Lmax <= 1024; dk, dv in {16, 32, 48, ..., 128};
 * B, Hv >= 1.  Trees of up to 256 nodes are verified on chip; longer trees go
 * through a two-level chunk pass (chunks of 128 nodes on chip, earlier chunks'
 * U rows read back from U), which is correct for every shape but slower.  For
 * bf16 with dk = dv = 128 and N > 128, a sequence whose tree is one chain (the
 * parent of node t is t - 1) is verified in the chunkwise form of the same
 * closed form (the state carried between 64-node chunks), on the tensor cores.
 * B == 0 or N == 0 is a valid empty call that enqueues nothing.
 */
#ifndef GDN_TREE_H
#define GDN_TREE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* return codes */
#define GDN_TREE_OK 0
#define GDN_TREE_EINVAL (-1)      /* NULL or misaligned pointer, bad dims       */
#define GDN_TREE_EUNSUPPORTED (-2) /* N > 1024, dk/dv outside the list, dtype  */
#define GDN_TREE_ECUDA (-3)       /* a CUDA call (launch, attribute) failed     */

/* per-sequence device status codes written to dev_status[b] */
#define GDN_TREE_STATUS_OK 0
#define GDN_TREE_STATUS_BAD_TREE 1 /* some parent[b][i] outside [-1, i-1]       */
#define GDN_TREE_STATUS_BAD_PATH 2 /* path_len or a path entry out of range, or
                                      (with parent given) not a root chain     */
#define GDN_TREE_STATUS_TIMEOUT 3  /* a bounded on-device wait (a copy, a tensor-core
                                      completion or a solve barrier; 2 s) ran
                                      out: the sequence's outputs, and those of
                                      the sequences the same CTA had not yet
                                      reached (which report it too), are
                                      incomplete; the context stays usable     */
#define GDN_TREE_STATUS_BAD_LAYOUT 4 /* packed layout: the sequence's row range or
                                        state slot is out of range             */

/* element type of q, k, v and o */
#define GDN_TREE_BF16 0
#define GDN_TREE_F32 1

typedef struct {
  int32_t B, N, Hqk, Hv, dk, dv;
  int32_t dtype; /* GDN_TREE_BF16 or GDN_TREE_F32 */
} gdn_tree_dims;

/*
 * gdn_tree_verify -- outputs of every tree node, without touching S0.
 *
 * Defined by the DFlash-TfM page, section 3 "Soluzione": o[b, t, h, :] is
 * S_t^T q_t where S_t is the GDN recurrence run along t's root-to-node path
 * from S0[b, h]; U[b, h, t, :] is the node's write vector u_t (see above).
 * Reads q, k, v, log_alpha, beta, parent, S0; writes o and U.  S0 is never
 * written (the "rollback-free" property).  dev_status[b] (if non-NULL) is set
 * to GDN_TREE_STATUS_OK or GDN_TREE_STATUS_BAD_TREE for every b (or
 * GDN_TREE_STATUS_BAD_LAYOUT / GDN_TREE_STATUS_TIMEOUT, see above).
 */
int gdn_tree_verify(const void *q, const void *k, const void *v,
                    const float *log_alpha, const float *beta,
                    const int32_t *parent, const float *S0, void *o, float *U,
                    gdn_tree_dims dims, int32_t *dev_status, void *stream);

/*
 * gdn_tree_commit -- delayed state commitment of the accepted branch.
 *
 * Defined by the DFlash-TfM page, section 3 (state commitment deferred to the
 * next decoding iteration): S1[b, h] is the state reached by running the GDN
 * recurrence from S0[b, h] along path[b, 0 .. path_len[b]-1], evaluated as
 * gamma_{p_L} S0 + sum_j exp(g_{p_L} - g_{p_j}) k_{p_j} u_{p_j}^T from the U
 * rows a previous gdn_tree_verify wrote for the same tree.  `k` and
 * `log_alpha` must be the arrays that verify saw.  `parent` may be NULL; when
 * given, the path must start at a node with parent -1 and follow parent
 * links, else the sequence gets GDN_TREE_STATUS_BAD_PATH.  path_len[b] == 0
 * gives S1 = S0.  S1 may alias S0 exactly (in-place commit); any other
 * overlap is undefined.  dev_status[b] (if non-NULL) is set for every b, to
 * GDN_TREE_STATUS_OK, BAD_PATH or BAD_LAYOUT, or TIMEOUT if a bounded on-device
 * wait of the tensor-core commit (taken for bf16, dk = dv = 128 and Lmax > 32:
 * its state copy and MMAs) ran out; S1[b, ...] is then left unwritten.
 */
int gdn_tree_commit(const int32_t *path, const int32_t *path_len,
                    const int32_t *parent, const float *U, const void *k,
                    const float *log_alpha, const float *S0, float *S1,
                    gdn_tree_dims dims, int32_t Lmax, int32_t *dev_status,
                    void *stream);

/*
 * gdn_tree_commit_verify -- one decoding iteration: the delayed commitment of
 * the previous tree's accepted path, fused with the verification of the next
 * tree from the state it produces.
 *
 * The DFlash-TfM page, section 3, commits the state "at the next decoding
 * iteration, once the accepted branch is known"; this call is that iteration.
 * It equals gdn_tree_commit(prev_path, prev_path_len, prev_parent, prev_U,
 * prev_k, prev_log_alpha, S_prev -> S1) followed by gdn_tree_verify(q, k, v,
 * log_alpha, beta, parent, S1 -> o, U), but the state is read once and
 * written once (the tensor-core path commits it on chip).
 *
 *   prev_*          the previous tree (prev_N nodes): its accepted path
 *                   [B, Lmax] / [B], optional parent [B, prev_N], the U rows
 *                   verify wrote [B, Hv, prev_N, dv], its k [B, prev_N, Hqk, dk]
 *                   and log_alpha [B, prev_N, Hv]
 *   S_prev -> S1    [B, Hv, dk, dv] fp32; S1 may alias S_prev exactly
 *   q .. parent     the next tree, shapes as for gdn_tree_verify (dims.N nodes)
 *   o, U            its outputs; U may be prev_U itself when prev_N == dims.N
 *                   (each (b, h) slice is then read before it is written); any
 *                   other overlap of U and prev_U returns GDN_TREE_EINVAL
 *   commit_status   [B] or NULL: as gdn_tree_commit's dev_status
 *   verify_status   [B] or NULL: as gdn_tree_verify's dev_status (the fused
 *                   path also sets GDN_TREE_STATUS_BAD_PATH when the commit of
 *                   that sequence failed).  Whenever commit_status reports an
 *                   error, that sequence's S1, o and U are unspecified.
 * Limits as for the two calls; 1 <= prev_N <= 1024; prev_k has the dtype of q.
 */
int gdn_tree_commit_verify(const int32_t *prev_path, const int32_t *prev_path_len,
                           const int32_t *prev_parent, const float *prev_U,
                           const void *prev_k, const float *prev_log_alpha,
                           int32_t prev_N, int32_t Lmax, const float *S_prev, float *S1,
                           const void *q, const void *k, const void *v,
                           const float *log_alpha, const float *beta,
                           const int32_t *parent, void *o, float *U, gdn_tree_dims dims,
                           int32_t *commit_status, int32_t *verify_status, void *stream);

/*
 * gdn_tree_verify_recurrent -- the same outputs as gdn_tree_verify, computed by
 * single-branch recurrent verification: the baseline the tree verification is
 * measured against.
 *
 * The DFlash-TfM page, results section ("Efficienza di Verifica"), compares its
 * fused tree kernel with verifying every branch by its own recurrent pass.  Here
 * every root-to-leaf branch of the tree runs the GDN recurrence of section 3
 * ("Sfida") from its own copy of S0[b, h], node by node, writing o and U of each
 * node it passes; a node shared by several branches is recomputed by each of
 * them, with identical bits.  All arithmetic is fp32.
 *
 * Arguments, layouts, ownership, limits and dev_status exactly as for
 * gdn_tree_verify, except that N <= 256 (the branch's path is held on chip;
 * GDN_TREE_EUNSUPPORTED beyond).  The state of a branch is held on chip;
 * nothing is allocated.
 */
int gdn_tree_verify_recurrent(const void *q, const void *k, const void *v,
                              const float *log_alpha, const float *beta,
                              const int32_t *parent, const float *S0, void *o, float *U,
                              gdn_tree_dims dims, int32_t *dev_status, void *stream);

/*
 * Packed (ragged) batches with a state pool -- the serving layout of the same
 * calls: every sequence has its own tree size, and its recurrent state lives in
 * a slot of a state pool (the DFlash-TfM page runs the verification inside
 * SGLang, section 3 "Implementazione").  The DFlash-TfM page itself prints no
 * layout; the packed variants are this library's.
 *
 *   cu_nodes      [B + 1] int32, device: sequence b owns node rows
 *                 cu_nodes[b] .. cu_nodes[b+1]-1 of the packed arrays, and its
 *                 tree's node t is row cu_nodes[b] + t; 0 <= cu_nodes[b] <=
 *                 cu_nodes[b+1] <= T and cu_nodes[b+1] - cu_nodes[b] <= dims.N
 *   T             rows of the packed arrays (>= 0)
 *   q, k          [T, Hqk, dk];  v, o [T, Hv, dv];  log_alpha, beta [T, Hv];
 *   parent        [T]: parent[cu_nodes[b] + t] is t's parent within sequence b
 *                 (-1 <= parent < t)
 *   U             [Hv, T, dv] fp32: the rows of sequence b, head h are contiguous
 *   state_slot    [B] int32, device, or NULL (slot b): sequence b's state is
 *                 pool[state_slot[b]] of a pool [n_slots, Hv, dk, dv] fp32;
 *                 0 <= state_slot[b] < n_slots.  Commits need distinct slots.
 *   dims          B sequences, N = the largest tree (the capacity the kernels are
 *                 chosen for), heads and dtype as for the fixed layout.
 * A sequence whose row range or slot is out of range gets
 * GDN_TREE_STATUS_BAD_LAYOUT in its status and its outputs are left unwritten.
 * Everything else -- dtypes, alignment, ownership, asynchrony, tree and path
 * validity -- is as for the fixed-layout calls.
 */
int gdn_tree_verify_packed(const void *q, const void *k, const void *v, const float *log_alpha,
                           const float *beta, const int32_t *parent, const int32_t *cu_nodes,
                           int32_t T, const float *state_pool, const int32_t *state_slot,
                           int32_t n_slots, void *o, float *U, gdn_tree_dims dims,
                           int32_t *dev_status, void *stream);

/* Delayed commitment in the packed layout: path/path_len [B, Lmax] / [B] index
 * each sequence's own nodes; pool_out[state_slot[b]] = the state after the path,
 * from pool_in[state_slot[b]] (pool_out may be pool_in: in-place). */
int gdn_tree_commit_packed(const int32_t *path, const int32_t *path_len, const int32_t *parent,
                           const int32_t *cu_nodes, int32_t T, const float *U, const void *k,
                           const float *log_alpha, const float *pool_in, float *pool_out,
                           const int32_t *state_slot, int32_t n_slots, gdn_tree_dims dims,
                           int32_t Lmax, int32_t *dev_status, void *stream);

/* One decoding iteration in the packed layout: the previous tree (prev_cu_nodes,
 * prev_T, prev_N its largest tree) is committed from pool_in into pool_out and
 * the next tree is verified from pool_out, as gdn_tree_commit_verify. */
int gdn_tree_commit_verify_packed(const int32_t *prev_path, const int32_t *prev_path_len,
                                  const int32_t *prev_parent, const int32_t *prev_cu_nodes,
                                  int32_t prev_T, const float *prev_U, const void *prev_k,
                                  const float *prev_log_alpha, int32_t prev_N, int32_t Lmax,
                                  const float *pool_in, float *pool_out,
                                  const int32_t *state_slot, int32_t n_slots, const void *q,
                                  const void *k, const void *v, const float *log_alpha,
                                  const float *beta, const int32_t *parent,
                                  const int32_t *cu_nodes, int32_t T, void *o, float *U,
                                  gdn_tree_dims dims, int32_t *commit_status,
                                  int32_t *verify_status, void *stream);

/*
 * gdn_tree_build_topw -- the draft tree, by top-w best-first growth.
 *
 * The DFlash-TfM page, section 2 ("Costruzione dell'Albero"), builds the draft
 * tree with DySpec's best-first growth, modified to pop the top-w candidates of
 * the heap and expand all w at once: a tree of N nodes in ceil(N / w) rounds.
 * Reading taken: node 0 is the root (score 0, depth 1); every node of depth <
 * max_depth offers c candidate children, candidate j of node p scoring
 * score(p) + cand_logp[b, p, j] (an fp32 addition); a round takes the
 * min(w, N - built) best live candidates (higher score first, ties to the lower
 * p * c + j, i.e. creation order) as new nodes in that order, after which they
 * offer their own candidates.  A -inf candidate is never taken; if candidates run
 * out first, fewer than N nodes are built.
 *
 *   cand_logp   [B, N, c] fp32, device: the log-probabilities of node p's c
 *               candidates (rows of nodes that are never built are not read);
 *               no NaN
 *   parent      [B, N] int32, device, out: the tree (topologically ordered,
 *               -1 for the root), ready for gdn_tree_verify; -2 past n_built
 *   cand_index  [B, N] int32 or NULL, out: j of the parent's candidate each node
 *               is (-1 root, -2 past n_built)
 *   score       [B, N] fp32 or NULL, out: the node's score (NaN past n_built)
 *   n_built     [B] int32 or NULL, out: nodes built per sequence
 * Limits: 1 <= N <= 256, 1 <= c <= 32, 1 <= w <= N, max_depth >= 1, B >= 0.
 * Asynchronous on `stream`; allocates nothing.
 */
int gdn_tree_build_topw(const float *cand_logp, int32_t B, int32_t N, int32_t c, int32_t w,
                        int32_t max_depth, int32_t *parent, int32_t *cand_index, float *score,
                        int32_t *n_built, void *stream);

/* Human-readable text for a return code or a device status code. */
const char *gdn_tree_strerror(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int gdn_tree_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TREE_H */
