/*
 * gdn_oracle.c -- plain fp64 CPU oracle for rollback-free GDN tree verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (DFlash-TfM: Trees from Marginals,
 * gist.science/it/paper/2607.06763, section 3 "Verifica dell'Albero Senza
 * Rollback per GDN"):
 *
 *   GDN recurrence (section 3, "Sfida"):
 *       S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
 *   with S in R^{dk x dv}.  The draft tree is in topological order (section 3,
 *   "Soluzione": every node comes after its ancestors, i.e. parent[i] < i);
 *   S_{t-1} is the state of t's parent, or the committed state S0 when t hangs
 *   off it (parent = -1).
 *   The verified output of node t is o_t = S_t^T q_t: the result of running
 *   the recurrence along t's own root-to-node path, which is exactly the
 *   "single-branch recurrent" verification the page compares against
 *   (section "Risultati Sperimentali", verification efficiency).
 *
 *   Delayed commitment (section 3, state commitment deferred to the next
 *   iteration): once the accepted branch p_1..p_L is known, S1 is the state
 *   reached by running the same recurrence along p_1..p_L from S0.
 *
 *   The per-node write vector u_t = beta_t (v_t - alpha_t S_par^T k_t), with
 *   S_t = alpha_t S_par + k_t u_t^T, is what the page's linear system solves
 *   for; this oracle reports it read straight off the recurrence.
 *
 * Two verify modes, doing the same floating-point operations in the same
 * order, so their results are bitwise identical:
 *   mode 0  literal path walk: for every node, start from S0 and step along
 *           the whole root-to-node path;
 *   mode 1  memoised: S_t is stepped once from the stored S_parent.
 *
 * All values are fp64; inputs are the exact upcast of the bf16 / fp32 data.
 * Build: plain C99, -O2 -ffp-contract=off (no FMA contraction), -pthread.
 *
 * Layouts (row-major):
 *   q, k [B][N][Hqk][dk]; v [B][N][Hv][dv]; log_alpha, beta [B][N][Hv];
 *   parent [B][N] (int32, -1 = child of S0); S0, S1 [B][Hv][dk][dv];
 *   o [B][N][Hv][dv]; U [B][Hv][N][dv]; path [B][Lmax]; path_len [B].
 *   v-head h reads qk-head h / (Hv / Hqk).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ETREE (-2)
#define ORC_EPATH (-3)
#define ORC_ENOMEM (-4)

typedef struct {
  int32_t B, N, Hqk, Hv, dk, dv;
} orc_dims;

/* ---- the recurrence, literally ------------------------------------------ */

/* S <- a (S - b k (k^T S)) + b k v^T.  w is a dv-long scratch. */
static void gdn_step(double *S, const double *k, const double *v, double a,
                     double b, int dk, int dv, double *w) {
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int i = 0; i < dk; ++i) acc += k[i] * S[(size_t)i * dv + j];
    w[j] = acc;
  }
  for (int i = 0; i < dk; ++i) {
    for (int j = 0; j < dv; ++j) {
      double *s = &S[(size_t)i * dv + j];
#ifdef ORC_MUTANT_SIGN
      *s = a * (*s + b * k[i] * w[j]) + b * k[i] * v[j];
#elif defined(ORC_MUTANT_DECAY_ON_WRITE)
      *s = a * ((*s - b * k[i] * w[j]) + b * k[i] * v[j]);
#elif defined(ORC_MUTANT_DROP_WRITE)
      *s = a * (*s - b * k[i] * w[j]);
#else
      *s = a * (*s - b * k[i] * w[j]) + b * k[i] * v[j];
#endif
    }
  }
}

/* o = S^T q */
static void gdn_readout(const double *S, const double *q, double *o, int dk,
                        int dv) {
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int i = 0; i < dk; ++i) {
#ifdef ORC_MUTANT_TRANSPOSE
      /* S q instead of S^T q; indices clamped so that dk != dv stays in bounds */
      acc += S[(size_t)(j < dk ? j : 0) * dv + (i < dv ? i : 0)] * q[i];
#else
      acc += S[(size_t)i * dv + j] * q[i];
#endif
    }
    o[j] = acc;
  }
}

/* u = b (v - a S^T k), S = state of the parent */
static void gdn_write_vector(const double *S, const double *k, const double *v,
                             double a, double b, double *u, int dk, int dv) {
  for (int j = 0; j < dv; ++j) {
    double acc = 0.0;
    for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * k[i];
    u[j] = b * (v[j] - a * acc);
  }
}

/* ---- indexing helpers ---------------------------------------------------- */

typedef struct {
  const double *q, *k, *v, *la, *beta, *S0;
  const int32_t *parent;
  double *o, *U;
  orc_dims d;
  int mode;
  const int32_t *units;
  int n_units;
  int nthreads;
  int tid;
  int status;
} verify_job;

static const double *row_qk(const double *x, const orc_dims *d, int b, int t,
                            int hq) {
  return x + (((size_t)b * d->N + t) * d->Hqk + hq) * d->dk;
}
static const double *row_v(const double *x, const orc_dims *d, int b, int t,
                           int h) {
  return x + (((size_t)b * d->N + t) * d->Hv + h) * d->dv;
}
static double gate(const double *x, const orc_dims *d, int b, int t, int h) {
  return x[((size_t)b * d->N + t) * d->Hv + h];
}

static int tree_ok(const int32_t *parent, int N) {
  for (int i = 0; i < N; ++i)
    if (parent[i] < -1 || parent[i] >= i) return 0;
  return 1;
}

/* verify one (b, h) unit */
static int verify_unit(verify_job *J, int b, int h, double *states,
                       double *S, double *w, int *path) {
  const orc_dims *d = &J->d;
  const int N = d->N, dk = d->dk, dv = d->dv;
  const int hq = h / (d->Hv / d->Hqk);
  const int32_t *par = J->parent + (size_t)b * N;
  const double *S0 = J->S0 + ((size_t)b * d->Hv + h) * dk * dv;
  const size_t dd = (size_t)dk * dv;
  if (!tree_ok(par, N)) return ORC_ETREE;
  for (int t = 0; t < N; ++t) {
    double *o_t = J->o + (((size_t)b * N + t) * d->Hv + h) * dv;
    double *u_t = J->U + (((size_t)b * d->Hv + h) * N + t) * dv;
    const double *k_t = row_qk(J->k, d, b, t, hq);
    const double *v_t = row_v(J->v, d, b, t, h);
    const double a_t = exp(gate(J->la, d, b, t, h));
    const double b_t = gate(J->beta, d, b, t, h);
    if (J->mode == 1) {
      /* memoised: S_t from the stored parent state */
      double *St = states + (size_t)t * dd;
#ifdef ORC_MUTANT_IGNORE_TREE
      const int pt = t - 1; /* treats every tree as a chain */
#else
      const int pt = par[t];
#endif
      const double *Sp = pt < 0 ? S0 : states + (size_t)pt * dd;
      memcpy(St, Sp, dd * sizeof(double));
#ifdef ORC_MUTANT_U_AFTER_STEP
      gdn_step(St, k_t, v_t, a_t, b_t, dk, dv, w);
      gdn_write_vector(St, k_t, v_t, a_t, b_t, u_t, dk, dv);
#else
      gdn_write_vector(St, k_t, v_t, a_t, b_t, u_t, dk, dv);
      gdn_step(St, k_t, v_t, a_t, b_t, dk, dv, w);
#endif
      gdn_readout(St, row_qk(J->q, d, b, t, hq), o_t, dk, dv);
    } else {
      /* literal: walk the root-to-t path from S0 */
      int len = 0;
      for (int s = t; s >= 0; s = par[s]) path[len++] = s;
      memcpy(S, S0, dd * sizeof(double));
      for (int i = len - 1; i >= 0; --i) {
        const int s = path[i];
        const double *k_s = row_qk(J->k, d, b, s, hq);
        const double *v_s = row_v(J->v, d, b, s, h);
        const double a_s = exp(gate(J->la, d, b, s, h));
        const double b_s = gate(J->beta, d, b, s, h);
        if (s == t) gdn_write_vector(S, k_s, v_s, a_s, b_s, u_t, dk, dv);
        gdn_step(S, k_s, v_s, a_s, b_s, dk, dv, w);
      }
      gdn_readout(S, row_qk(J->q, d, b, t, hq), o_t, dk, dv);
    }
  }
  return ORC_OK;
}

static void *verify_worker(void *arg) {
  verify_job *J = (verify_job *)arg;
  const orc_dims *d = &J->d;
  const size_t dd = (size_t)d->dk * d->dv;
  double *states = NULL;
  if (J->mode == 1) states = (double *)malloc((size_t)d->N * dd * sizeof(double));
  double *S = (double *)malloc(dd * sizeof(double));
  double *w = (double *)malloc((size_t)d->dv * sizeof(double));
  int *path = (int *)malloc((size_t)d->N * sizeof(int));
  if ((J->mode == 1 && !states) || !S || !w || !path) {
    J->status = ORC_ENOMEM;
  } else {
    const int total = J->units ? J->n_units : d->B * d->Hv;
    for (int i = J->tid; i < total; i += J->nthreads) {
      const int unit = J->units ? J->units[i] : i;
      const int rc = verify_unit(J, unit / d->Hv, unit % d->Hv, states, S, w, path);
      if (rc != ORC_OK) J->status = rc;
    }
  }
  free(states);
  free(S);
  free(w);
  free(path);
  return NULL;
}

static int dims_ok(const orc_dims *d) {
  return d->B > 0 && d->N > 0 && d->Hqk > 0 && d->Hv > 0 && d->dk > 0 &&
         d->dv > 0 && d->Hv % d->Hqk == 0;
}

/*
 * Verify every node of every (b, h) unit listed in `units` (flat b*Hv + h; all
 * units when NULL).  Writes o and U for those units only.  Returns 0, or a
 * negative code (bad dims, invalid tree, no memory).
 */
int gdn_oracle_verify(const double *q, const double *k, const double *v,
                      const double *log_alpha, const double *beta,
                      const int32_t *parent, const double *S0, double *o,
                      double *U, orc_dims d, int mode, const int32_t *units,
                      int n_units, int nthreads) {
  if (!dims_ok(&d) || (mode != 0 && mode != 1)) return ORC_EINVAL;
  if (nthreads < 1) nthreads = 1;
  verify_job *jobs = (verify_job *)calloc((size_t)nthreads, sizeof(verify_job));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return ORC_ENOMEM;
  }
  for (int i = 0; i < nthreads; ++i) {
    verify_job J = {q, k, v, log_alpha, beta, S0, parent, o, U, d, mode,
                    units, n_units, nthreads, i, ORC_OK};
    jobs[i] = J;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, verify_worker, &jobs[i]);
  verify_worker(&jobs[0]);
  int rc = ORC_OK;
  for (int i = 0; i < nthreads; ++i) {
    if (i > 0) pthread_join(th[i], NULL);
    if (jobs[i].status != ORC_OK) rc = jobs[i].status;
  }
  free(jobs);
  free(th);
  return rc;
}

/* ---- delayed commitment --------------------------------------------------- */

typedef struct {
  const int32_t *path, *path_len, *parent;
  const double *k, *v, *la, *beta, *S0;
  double *S1;
  orc_dims d;
  int Lmax;
  const int32_t *units;
  int n_units, nthreads, tid, status;
} commit_job;

static int path_ok(const int32_t *p, int L, const int32_t *parent, int N,
                   int Lmax) {
  if (L < 0 || L > Lmax || L > N) return 0;
  for (int j = 0; j < L; ++j) {
    if (p[j] < 0 || p[j] >= N) return 0;
    if (parent) {
      const int want = j == 0 ? -1 : p[j - 1];
      if (parent[p[j]] != want) return 0;
    }
  }
  return 1;
}

static void *commit_worker(void *arg) {
  commit_job *J = (commit_job *)arg;
  const orc_dims *d = &J->d;
  const size_t dd = (size_t)d->dk * d->dv;
  double *w = (double *)malloc((size_t)d->dv * sizeof(double));
  if (!w) {
    J->status = ORC_ENOMEM;
    return NULL;
  }
  const int total = J->units ? J->n_units : d->B * d->Hv;
  for (int i = J->tid; i < total; i += J->nthreads) {
    const int unit = J->units ? J->units[i] : i;
    const int b = unit / d->Hv, h = unit % d->Hv;
    const int hq = h / (d->Hv / d->Hqk);
    const int32_t *p = J->path + (size_t)b * J->Lmax;
    const int L = J->path_len[b];
    const int32_t *par = J->parent ? J->parent + (size_t)b * d->N : NULL;
    if (!path_ok(p, L, par, d->N, J->Lmax)) {
      J->status = ORC_EPATH;
      continue;
    }
    double *S = J->S1 + ((size_t)b * d->Hv + h) * dd;
    memcpy(S, J->S0 + ((size_t)b * d->Hv + h) * dd, dd * sizeof(double));
#ifdef ORC_MUTANT_REVERSED_PATH
    for (int j = L - 1; j >= 0; --j) {
#else
    for (int j = 0; j < L; ++j) {
#endif
      const int s = p[j];
      gdn_step(S, row_qk(J->k, d, b, s, hq), row_v(J->v, d, b, s, h),
               exp(gate(J->la, d, b, s, h)), gate(J->beta, d, b, s, h), d->dk,
               d->dv, w);
    }
  }
  free(w);
  return NULL;
}

/*
 * Commit the accepted path of every listed unit: S1 = state after running the
 * recurrence along path[b][0 .. path_len[b]-1] from S0.  `parent` may be NULL
 * (then only index ranges are checked); when given, the path must be a chain
 * that starts at a node hanging off S0.
 */
int gdn_oracle_commit(const int32_t *path, const int32_t *path_len,
                      const int32_t *parent, const double *k, const double *v,
                      const double *log_alpha, const double *beta,
                      const double *S0, double *S1, orc_dims d, int Lmax,
                      const int32_t *units, int n_units, int nthreads) {
  if (!dims_ok(&d) || Lmax < 0) return ORC_EINVAL;
  if (nthreads < 1) nthreads = 1;
  commit_job *jobs = (commit_job *)calloc((size_t)nthreads, sizeof(commit_job));
  pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!jobs || !th) {
    free(jobs);
    free(th);
    return ORC_ENOMEM;
  }
  for (int i = 0; i < nthreads; ++i) {
    commit_job J = {path, path_len, parent, k, v, log_alpha, beta, S0, S1, d,
                    Lmax, units, n_units, nthreads, i, ORC_OK};
    jobs[i] = J;
  }
  for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, commit_worker, &jobs[i]);
  commit_worker(&jobs[0]);
  int rc = ORC_OK;
  for (int i = 0; i < nthreads; ++i) {
    if (i > 0) pthread_join(th[i], NULL);
    if (jobs[i].status != ORC_OK) rc = jobs[i].status;
  }
  free(jobs);
  free(th);
  return rc;
}
