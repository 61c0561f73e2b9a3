// verify_tc.cu -- tensor-core tree verification for bf16 q/k/v, dk = dv = 128,
// trees of up to 128 nodes (sm_103a: TMA + tcgen05 + TMEM).
//
// Method: "DFlash-TfM: Trees from Marginals", section 3 ("Soluzione"): the
// chunked form of the GDN recurrence over the topologically ordered tree,
//     X[t,s] = beta_t e^{g_t - g_s} (k_t . k_s)   s a strict ancestor of t
//     Y[t,s] =        e^{g_t - g_s} (q_t . k_s)   s on the root-to-t path
//     (I + X) U = diag(beta) (V - diag(gamma) K S0)
//     O = diag(gamma) Q S0 + Y U
// The page's fused kernel computes the Gram matrix, solves by tiled forward
// substitution and applies the output stage in one pass; this kernel does the
// same in one launch, laid out for Blackwell:
//
//   a CTA (512 threads, 512 TMEM columns) per (sequence b, v-head h) unit, one
//   fitting an SM; a running CTA takes over the units of CTAs not launched yet
//   (cluster launch control: it cancels them), one unit ahead, so that the SMs
//   stay busy however uneven the units; the next unit's K, Q and state are
//   already being copied while the current unit finishes.  Per unit:
//   1. TMA brings K and Q of the q/k head (128-byte swizzle) and the fp32 state
//      tile (four 32-column boxes).  Fused with the delayed commitment of the
//      previous tree's accepted path, K_P^T diag(w) U_P is one tcgen05 MMA
//      (both operands MN-major: the path's k rows as they are, exact in bf16,
//      and w U split hi + lo), so that S1 = gamma S0 + that is formed row by
//      row (thread = state row) and leaves by TMA store.  The same thread
//      writes the row as S0 = hi + lo, the bf16 operand of the next MMAs.
//   2. tcgen05.mma, accumulators in TMEM:  G_kk = K K^T, G_qk = Q K^T,
//      KS = K S0_hi + K S0_lo, QS = Q S0_hi.
//   3. TMEM -> registers (thread = tree node): the X and Y entries of the node's
//      ancestors (masked, decay-weighted, fp32), R = beta (V - gamma KS) and
//      the output seed gamma QS go to shared memory.
//   4. forward substitution as a dataflow over the tree, a half-warp per node
//      and 8 value columns a lane: u_t = r_t - sum_a X[t,a] u_a and, in the
//      same walk over t's path, o_t = gamma_t (Q S0)_t + sum_s Y[t,s] u_s, both
//      fp32; u_t and o_t are stored straight from the solve.
//
// Precision: K S0, the commit, the solve and Y U are fp32-accurate (U feeds the
// commit's 1e-4 bound); Q S0 uses S0_hi only, ample for the bf16 output.  Waits
// are bounded; a timeout reports a device status.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace gdn {

namespace {

using namespace sm100;

constexpr int kTile = 128;         // padded node count = MMA M
constexpr int kD = 128;            // dk = dv
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kW = kTile / 32;     // ancestor bitset words per node
constexpr uint32_t kTmemCols = 512;
// TMEM columns: the Gram matrices, then K S0 (its columns first hold the fused
// commit's rank-L update), Q S0
constexpr uint32_t kColGkk = 0, kColGqk = 128, kColKS = 256, kColQS = 384;
constexpr uint32_t kColCommit = 256;
constexpr int kIssuer = 128;  // the one thread that issues every copy and MMA (warp 4, lane 0)
constexpr int kCommitChunk = 32;  // fused commit: path entries staged per MMA round
constexpr int kStagers = kThreads - 160;  // warps 5-15
// while every |g_t| of a unit is at most this, e^{g_t - g_s} is formed as
// e^{g_t} e^{-g_s} (both factors, and their product, stay normal fp32 numbers);
// beyond it, from the double-float difference
constexpr float kProductDecayLimit = 40.f;

#ifdef GDN_TC_PROFILE
// per-unit phase timestamps for a profiling build (never in the product build):
// SM clock counts kept in shared memory during the unit, dumped with the unit's
// global-timer span (slots 24, 25) once it is over
constexpr int kMarks = 26;
__device__ unsigned long long g_tc_phase[4096][kMarks];
#define TC_MARK_BY(thread, i)                      \
  do {                                             \
    if (threadIdx.x == (thread)) S.marks[i] = clock64(); \
  } while (0)
#define TC_DUMP()                                                           \
  do {                                                                      \
    if (threadIdx.x == 0 && unit < 4096) {                                  \
      for (int i_ = 0; i_ < 24; ++i_) g_tc_phase[unit][i_] = S.marks[i_];   \
      g_tc_phase[unit][24] = S.gt0;                                         \
      g_tc_phase[unit][25] = globaltimer_ns();                              \
    }                                                                       \
  } while (0)
#define TC_START()                                  \
  do {                                              \
    if (threadIdx.x == 0) S.gt0 = globaltimer_ns(); \
  } while (0)
#else
#define TC_MARK_BY(thread, i) \
  do {                        \
  } while (0)
#define TC_DUMP() \
  do {            \
  } while (0)
#define TC_START() \
  do {             \
  } while (0)
#endif
#define TC_MARK(i) TC_MARK_BY(0, i)

// shared memory map (byte offsets from a 1024-aligned base); three 64 KB regions
// change roles within a unit
constexpr uint32_t kTileBytes = 128 * 128;            // one 64-wide K block: 128 rows x 128 B
constexpr uint32_t kOpBytes = 2 * kTileBytes;         // a 128 x 128 bf16 operand (2 K blocks)
// region 1: K, Q (TMA) until the MMAs that read them end; then X, Y of each
// node's ancestors (packed strictly-lower triangle, float2)
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = 1 * kOpBytes;
constexpr uint32_t OFF_XY = 0;
// region 2: fused, the commit's operand tiles (k rows; w U hi, lo: MN-major);
// then S0 hi, lo (MN-major) until the K S0 / Q S0 MMAs end; then the output
// rows (fp32, seeded with gamma Q S0, finished by the solve)
constexpr uint32_t OFF_R2 = 2 * kOpBytes;
constexpr uint32_t kCommitTile = kCommitChunk * kD * 2;  // 32 path rows of bf16
constexpr uint32_t OFF_CA = OFF_R2;
constexpr uint32_t OFF_CBH = OFF_R2 + kCommitTile;
constexpr uint32_t OFF_CBL = OFF_R2 + 2 * kCommitTile;
constexpr uint32_t OFF_S0H = OFF_R2;
constexpr uint32_t OFF_S0L = OFF_R2 + kOpBytes;
constexpr uint32_t OFF_P = OFF_R2;
// region 3: the fp32 state (TMA: four boxes of 32 columns x 128 rows), S1 in
// place until its TMA store has read it; then R / U (fp32 rows, same layout)
constexpr uint32_t OFF_R3 = 4 * kOpBytes;
constexpr uint32_t OFF_PATH = OFF_R3 + kTile * kD * 4;  // uint8 [node][depth - 1] -> path node
constexpr uint32_t OFF_SMALL = OFF_PATH + kTile * kTile;
#ifdef GDN_TC_PROFILE
constexpr uint32_t kSmallBytes = 16384 + 512;  // room for the phase stamps
#else
constexpr uint32_t kSmallBytes = 16384;
#endif
constexpr uint32_t kSmemBytes = OFF_SMALL + kSmallBytes + 1024;  // + alignment slack

static_assert(kTile * (kTile - 1) / 2 * 8 <= 2 * kOpBytes, "X, Y must fit in region 1");
static_assert(3 * kCommitTile <= 2 * kOpBytes, "commit tiles must fit in region 2");
static_assert(OFF_R3 % 1024 == 0 && OFF_SMALL % 16 == 0, "alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Small {
  int parent[kTile];
  int jump[kTile];  // tree prep: pointer jumping
  df g[kTile];
  float eg[kTile], emg[kTile];  // e^{g_t}, e^{-g_t}
  float beta[kTile];
  float la[kTile];
  float ydiag[kTile];  // Y[t,t] = q_t . k_t
  uint32_t anc[kTile * kW];
  int order[kTile];
  int depth[kTile];
  int level_start[kTile + 2];
  int level_cursor[kTile + 2];
  int level_task[kTile + 2];  // first solve task of each depth
  uint8_t task_pos[kTile];    // solve task k: nodes order[task_pos[k]] .. (task_n[k] of them,
  uint8_t task_n[kTile];      // one or two, of one depth)
  int n_tasks;
  uint64_t node_bar[kTile];  // solve: completes a phase per unit once the node's u is final
  // the next unit's tree and gates, prefetched (cp.async) while this unit runs
  int pre_parent[kTile];
  float pre_beta[kTile];
  float pre_la[kTile];
  // K, Q landed; Gram done; K S0 / Q S0 done; state landed; commit rows staged;
  // commit MMA done
  uint64_t bar_kq, bar_g, bar_ks, bar_s, bar_stage, bar_c;
  uint32_t tmem_base;
  int err;
  int bad;     // the tree failed validation
  int wide_g;  // some |g_t| > kProductDecayLimit
  // phases issued on bar_kq, bar_g, bar_ks, bar_s, bar_c (for the drain)
  int n_kq, n_g, n_ks, n_s, n_c;
  int s1_pending;  // a TMA store of S1 is in flight
  // work stealing: the unit after the current one (n_units: none) in slot it & 1 of
  // iteration it, the response of the cluster-launch-control request in flight (it
  // names the unit after that), its mbarrier and phase count
  uint4 clc_resp;
  uint64_t bar_clc;
  int n_clc;
  int clc_pending;
  int next_unit[2];
  // fused delayed commitment of the previous tree's accepted path
  int cpath[kMaxN];
  int pre_path[kMaxN];  // the next unit's accepted path and its length, prefetched
  int pre_plen;
  float cla[kMaxN];
  float cw[kMaxN];
  float cgamma;
  int cL;
  int cbad;
#ifdef GDN_TC_PROFILE
  unsigned long long marks[24];
  unsigned long long gt0;
#endif
};
static_assert(sizeof(Small) <= kSmallBytes, "small state too large");
// members read or written as 16-byte vectors
static_assert(offsetof(Small, g) % 16 == 0 && offsetof(Small, emg) % 16 == 0,
              "path log-decays are read as float4");
static_assert(offsetof(Small, anc) % 16 == 0, "ancestor rows are read and written as uint4");

// packed strictly-lower triangle of X and Y
__device__ __forceinline__ int x_index(int t, int s) { return (t * (t - 1) >> 1) + s; }

// The issuer: the unit that the work-stealing request in flight took over (the
// cancelled CTA's blockIdx.x), or n_units when none is in flight, when the grid had no
// CTA left to cancel, or when the response did not land within the limit (S.err is
// then set and the request stays pending)
__device__ __forceinline__ int clc_take(Small& S, int n_units, uint64_t limit_ns) {
  if (!S.clc_pending) return n_units;
  if (!mbar_wait(&S.bar_clc, (uint32_t)S.n_clc & 1u, limit_ns)) {
    S.err = 5;
    return n_units;
  }
  ++S.n_clc;
  S.clc_pending = 0;
  int x = 0;
  return clc_cancelled(&S.clc_resp, &x) && x >= 0 && x < n_units ? x : n_units;
}

__device__ __forceinline__ uint32_t pack2f(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// acc + a x, as two packed fp32x2 FMAs (same rounding as four fmaf)
__device__ __forceinline__ float4 fma4(float a, float4 x, float4 acc) {
  const float2 aa = make_float2(a, a);
  const float2 lo = __ffma2_rn(aa, make_float2(x.x, x.y), make_float2(acc.x, acc.y));
  const float2 hi = __ffma2_rn(aa, make_float2(x.z, x.w), make_float2(acc.z, acc.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

// 4-byte asynchronous copy global -> shared (this thread's cp.async group)
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
// 16-byte asynchronous copy global -> shared (L2 only)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

// Where unit (b, h)'s nodes live: its node count n (0 when the sequence's layout
// is invalid, flagged by bad), its first row, its state index, and the node /
// sequence coordinates of its rows in the q/k/v tensor maps.
struct UnitGeom {
  int n, row0, st, c_node, c_seq;
  bool bad;
};
__device__ __forceinline__ UnitGeom unit_geom(const SeqLayout& lay, int b, int Nmax) {
  UnitGeom g;
  const int n = lay.count(b, Nmax), st = lay.state(b);
  g.bad = n < 0 || st < 0;
  g.n = g.bad ? 0 : n;
  g.st = g.bad ? 0 : st;
  g.row0 = g.bad ? 0 : lay.row0(b, Nmax);
  g.c_node = lay.packed() ? g.row0 : 0;
  g.c_seq = lay.packed() ? 0 : b;
  return g;
}

// Tree group: starts the copies of a unit's parent links and gates (node = tid)
// into the prefetch slots; tree_prep of that unit waits for them.
__device__ __forceinline__ void prefetch_tree(Small& S, const int32_t* parent, const float* beta,
                                              const float* log_alpha, const SeqLayout& lay,
                                              int unit, int Nmax, int Hv, int tid) {
  const int b = unit / Hv, h = unit - b * Hv;
  const UnitGeom g = unit_geom(lay, b, Nmax);
  if (tid < g.n) {
    cp_async4(&S.pre_parent[tid], parent + (size_t)g.row0 + tid);
    cp_async4(&S.pre_beta[tid], beta + ((size_t)g.row0 + tid) * Hv + h);
    cp_async4(&S.pre_la[tid], log_alpha + ((size_t)g.row0 + tid) * Hv + h);
  }
  cp_async_commit();
}

// previous tree's accepted path for the fused delayed commitment
struct FusedCommit {
  const int32_t* path;      // [B, Lmax]
  const int32_t* path_len;  // [B]
  const int32_t* parent;    // node rows (see lay), or NULL
  const float* U;           // [B, Hv, N, dv] or [Hv, T, dv]
  const __nv_bfloat16* k;   // node rows x [Hqk, dk]
  const float* log_alpha;   // node rows x [Hv]
  int32_t N, Lmax;          // N: the previous tree's (largest) node count
  float* S1;                // committed states, indexed like the input states (may alias them)
  int32_t* status;          // [B] or NULL
  SeqLayout lay;            // the previous tree's rows (its state index is unused)
};

// reduction barrier over the first kCount threads (named barrier kId): OR of v
template <int kId, int kCount>
__device__ __forceinline__ int bar_or(int v) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.b32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(v), "n"(kId), "n"(kCount)
      : "memory");
  return r;
}

// K and Q of the unit's q/k head into region 1 (bar_kq); issuing thread only
__device__ __forceinline__ void issue_kq(Small& S, uint8_t* smem, const CUtensorMap* tmK,
                                         const CUtensorMap* tmQ, const SeqLayout& lay, int unit,
                                         int Hv, int Hqk, int Nmax) {
  const int b = unit / Hv, h = unit - b * Hv, hq = h / (Hv / Hqk);
  const UnitGeom g = unit_geom(lay, b, Nmax);
  const int cn = g.c_node, cs = g.c_seq;
  mbar_arrive_expect_tx(&S.bar_kq, 4 * kTileBytes);
  tma_load_4d(smem + OFF_K, tmK, &S.bar_kq, 0, hq, cn, cs);
  tma_load_4d(smem + OFF_K + kTileBytes, tmK, &S.bar_kq, 64, hq, cn, cs);
  tma_load_4d(smem + OFF_Q, tmQ, &S.bar_kq, 0, hq, cn, cs);
  tma_load_4d(smem + OFF_Q + kTileBytes, tmQ, &S.bar_kq, 64, hq, cn, cs);
  ++S.n_kq;
}

// the unit's fp32 state (four boxes of 32 columns) into region 3 (bar_s);
// issuing thread only
__device__ __forceinline__ void issue_state(Small& S, uint8_t* smem, const CUtensorMap* tmS,
                                            const SeqLayout& lay, int unit, int Hv, int Nmax) {
  const int b = unit / Hv, h = unit - b * Hv;
  const UnitGeom g = unit_geom(lay, b, Nmax);
  const int su = g.st * Hv + h;
  mbar_arrive_expect_tx(&S.bar_s, 4 * kBoxBytes);
#pragma unroll
  for (int c = 0; c < 4; ++c) tma_load_3d(smem + OFF_R3 + c * kBoxBytes, tmS, &S.bar_s, 32 * c, 0, su);
  ++S.n_s;
}

// Tree group (threads 0..127): takes the unit's prefetched tree and gates,
// validates the tree, then pointer jumping (ceil(log2 depth) rounds) gives every
// node its strict-ancestor bitset and its path log-decay g_t (double-float); its
// depth and its path (sPath row, root first: the ancestors in index order) follow
// from the bitset; finally the nodes are ordered by depth.  An invalid tree is
// replaced by all-roots (nothing of it is stored).  The copies
// for the CTA's next unit (if `next` < `end`) start as soon as the prefetch
// slots have been read.
__device__ __forceinline__ void tree_prep(Small& S, uint8_t* sPath, const int32_t* parent,
                                          const float* beta, const float* log_alpha,
                                          const SeqLayout& lay, int Nmax, int next, int end,
                                          int N, int Hv, int tid, int lane, int warp, int unit) {
  using TreeSync = NamedSync<1, 128>;
  cp_async_wait_all();
  TC_MARK(12);
  int p_in = -1;
  float be_in = 0.f, la_in = 0.f;
  if (tid < N) {
    p_in = S.pre_parent[tid];
    be_in = S.pre_beta[tid];
    la_in = S.pre_la[tid];
  }
  S.beta[tid] = be_in;
  S.la[tid] = la_in;
  S.level_start[tid] = 0;
  if (tid < 2) S.level_start[kTile + tid] = 0;
  const int bad_any = bar_or<1, 128>(tid < N && (p_in < -1 || p_in >= tid));
  S.parent[tid] = bad_any ? -1 : p_in;
  if (tid == 0) S.bad = bad_any;
  // every read of the prefetch slots has completed (their values are used above)
  if (next < end) prefetch_tree(S, parent, beta, log_alpha, lay, next, Nmax, Hv, tid);
  TreeSync()();
  // pointer jumping: after round r, jump[t] is t's 2^r-th ancestor (or -1) and
  // anc[t], g[t] cover the part of t's path below it
  int jmp = tid < N ? S.parent[tid] : -1;
  df g = {la_in, 0.f};
  uint4 a = make_uint4(0u, 0u, 0u, 0u);
  if (jmp >= 0) {
    const uint32_t bit = 1u << (jmp & 31);
    a.x = (jmp >> 5) == 0 ? bit : 0u;
    a.y = (jmp >> 5) == 1 ? bit : 0u;
    a.z = (jmp >> 5) == 2 ? bit : 0u;
    a.w = (jmp >> 5) == 3 ? bit : 0u;
  }
  S.jump[tid] = jmp;
  S.g[tid] = g;
  *reinterpret_cast<uint4*>(&S.anc[tid * kW]) = a;
  while (bar_or<1, 128>(jmp >= 0)) {  // also the barrier after the last round's writes
    int jj = -1;
    df gj = {0.f, 0.f};
    uint4 aj = make_uint4(0u, 0u, 0u, 0u);
    if (jmp >= 0) {
      jj = S.jump[jmp];
      gj = S.g[jmp];
      aj = *reinterpret_cast<const uint4*>(&S.anc[jmp * kW]);
    }
    TreeSync()();
    if (jmp >= 0) {
      g = df_add(g, gj);
      a.x |= aj.x;
      a.y |= aj.y;
      a.z |= aj.z;
      a.w |= aj.w;
      jmp = jj;
      S.jump[tid] = jmp;
      S.g[tid] = g;
      *reinterpret_cast<uint4*>(&S.anc[tid * kW]) = a;
    }
  }
  int dep = 0;
  if (tid < N) {
    dep = __popc(a.x) + __popc(a.y) + __popc(a.z) + __popc(a.w) + 1;
    S.depth[tid] = dep;
    // path: the strict ancestors in index order (root first), then t itself
    uint8_t* row = sPath + tid * kTile;
    const uint32_t aw[4] = {a.x, a.y, a.z, a.w};
    int k = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      for (uint32_t m = aw[w]; m != 0u; m &= m - 1u) row[k++] = (uint8_t)(w * 32 + __ffs(m) - 1);
    }
    row[k] = (uint8_t)tid;
    atomicAdd(&S.level_start[dep], 1);
  }
  int wide = 0;
  if (tid < N) {
    const float gv = df_value(g);
    S.eg[tid] = expf(gv);
    S.emg[tid] = expf(-gv);
    wide = fabsf(gv) > kProductDecayLimit;
  }
  wide = bar_or<1, 128>(wide);  // (also the barrier before the level scan)
  if (tid == 0) S.wide_g = wide;
  if (warp == 0) {
    // exclusive scans of the level counts 0..kTile+1 and of the solve tasks per
    // level (pairs of nodes, ceil(count / 2)), packed in one int (each <= 128);
    // lane owns 5 entries
    int cnt[5], run = 0;
#pragma unroll
    for (int e = 0; e < 5; ++e) {
      const int l = lane * 5 + e;
      cnt[e] = l < kTile + 2 ? S.level_start[l] : 0;
      run += cnt[e] | (((cnt[e] + 1) >> 1) << 16);
    }
    int incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int up = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += up;
    }
    int excl = incl - run;
#pragma unroll
    for (int e = 0; e < 5; ++e) {
      const int l = lane * 5 + e;
      if (l < kTile + 2) {
        S.level_start[l] = excl & 0xffff;
        S.level_cursor[l] = excl & 0xffff;
        S.level_task[l] = excl >> 16;
      }
      excl += cnt[e] | (((cnt[e] + 1) >> 1) << 16);
    }
    if (lane == 31) S.n_tasks = incl >> 16;
  }
  TreeSync()();
  if (tid < N) {
    // position in the depth order; every even rank within the level opens a task
    // of two nodes (one at an odd-sized level's end)
    const int pos = atomicAdd(&S.level_cursor[dep], 1);
    S.order[pos] = tid;
    const int r = pos - S.level_start[dep];
    if ((r & 1) == 0) {
      const int k = S.level_task[dep] + (r >> 1);
      S.task_pos[k] = (uint8_t)pos;
      S.task_n[k] = (uint8_t)(pos + 1 < S.level_start[dep + 1] ? 2 : 1);
    }
  }
}

// w_j = exp(G_L - G_j) and gamma_L = exp(G_L) along the committed path, with
// G_j the inclusive double-float prefix sums of log alpha; one warp
__device__ __forceinline__ void commit_weights(Small& S, int L, int lane) {
  df loc[8];
  df run = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int j = lane * 8 + e;
    run = df_add(run, df{j < L ? S.cla[j] : 0.f, 0.f});
    loc[e] = run;
  }
  df pre = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    df up;
    up.hi = __shfl_up_sync(0xffffffffu, pre.hi, o);
    up.lo = __shfl_up_sync(0xffffffffu, pre.lo, o);
    if (lane >= o) pre = df_add(pre, up);
  }
  df excl;
  excl.hi = __shfl_up_sync(0xffffffffu, pre.hi, 1);
  excl.lo = __shfl_up_sync(0xffffffffu, pre.lo, 1);
  if (lane == 0) excl = df{0.f, 0.f};
  df G[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) G[e] = df_add(excl, loc[e]);
  const int owner = L > 0 ? (L - 1) >> 3 : 0, slot = L > 0 ? (L - 1) & 7 : 0;
  df mine = G[0];
#pragma unroll
  for (int e = 1; e < 8; ++e)
    if (e == slot) mine = G[e];
  df GL;
  GL.hi = __shfl_sync(0xffffffffu, mine.hi, owner);
  GL.lo = __shfl_sync(0xffffffffu, mine.lo, owner);
  if (L == 0) GL = df{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int j = lane * 8 + e;
    if (j < L) S.cw[j] = expf(df_diff(GL, G[e]));
  }
  if (lane == 0) S.cgamma = expf(df_value(GL));
}

// Warps 5-15 (ot = tid - 160): start the copies of a unit's accepted path and
// its length into the prefetch slots (the unit's prologue waits for them).
__device__ __forceinline__ void prefetch_path(const FusedCommit& fc, Small& S, int b, int ot) {
  if (ot < fc.Lmax) cp_async4(&S.pre_path[ot], fc.path + (size_t)b * fc.Lmax + ot);
  if (ot == 0) cp_async4(&S.pre_plen, fc.path_len + b);
  cp_async_commit();
}

// Warps 5-15 (ot = tid - 160), as they finish their part of a unit's solve: the
// next unit's accepted path (landed in the prefetch slots during this unit) sends
// the rows its commit will read (U, k, log alpha, parent link of every entry in
// range) to L2, so that the next unit's prologue finds them there.  The entries
// are only read here; the prologue checks them.
__device__ __forceinline__ void prefetch_path_rows_l2(const FusedCommit& fc, Small& S, int nb,
                                                      int nh, int nhq, int Hqk, int Hv, int ot) {
  cp_async_wait_all();  // this thread's slot entries
  if (ot < fc.Lmax) {
    const int pj = S.pre_path[ot];
    const int pn = fc.lay.count(nb, fc.N);
    if (pj >= 0 && pj < pn) {
      const size_t prow0 = (size_t)fc.lay.row0(nb, fc.N);
      bulk_prefetch_l2(fc.U + (fc.lay.urow0(nb, nh, Hv, fc.N) + pj) * kD, kD * 4);
      bulk_prefetch_l2(fc.k + ((prow0 + pj) * Hqk + nhq) * kD, kD * 2);
      prefetch_l2(fc.log_alpha + (prow0 + pj) * Hv + nh);
      if (fc.parent) prefetch_l2(fc.parent + prow0 + pj);
    }
  }
}

// Fused commit, warps 5-15 (ot = tid - 160): checks the previous tree's
// accepted path of sequence b (range, chain order, parent links), gathers its
// log alpha and forms the path weights.  Sets S.cbad (0 or the sequence's
// commit status) and S.cL; returns whether the commit has rows to stage.
__device__ __forceinline__ bool commit_prologue(const FusedCommit& fc, Small& S, int b, int h,
                                                int Hv, int ot, int warp, int lane, int next_b,
                                                int& L_out) {
  const int pn = fc.lay.count(b, fc.N);  // the previous tree's node count (< 0: bad rows)
  cp_async_wait_all();  // this unit's path, prefetched during the previous unit
  NamedSync<2, kStagers>()();
  const int L = S.pre_plen;
  int pj = -1;
  if (ot < fc.Lmax) pj = S.pre_path[ot];
  int cbad = (pn < 0 || L < 0 || L > pn || L > fc.Lmax);
  if (!cbad && ot < L) {
    cbad |= (pj < 0 || pj >= pn);
    S.cpath[ot] = pj;
  }
  cbad = bar_or<2, kStagers>(cbad);
  if (!cbad && ot < L) {
    const int prev = ot == 0 ? -1 : S.cpath[ot - 1];
    cbad |= (ot > 0 && pj <= prev);
    const size_t prow0 = (size_t)fc.lay.row0(b, fc.N);
    if (fc.parent) cbad |= (fc.parent[prow0 + pj] != prev);
    S.cla[ot] = fc.log_alpha[(prow0 + pj) * Hv + h];
  }
  // every read of the prefetch slots is done: the next unit's path starts coming
  if (next_b >= 0) prefetch_path(fc, S, next_b, ot);
  cbad = bar_or<2, kStagers>(cbad);  // (also: every log alpha is in place)
  if (ot == 0) {
    S.cbad = !cbad ? GDN_TREE_STATUS_OK
                   : (pn < 0 ? GDN_TREE_STATUS_BAD_LAYOUT : GDN_TREE_STATUS_BAD_PATH);
    S.cL = cbad ? 0 : L;
  }
  L_out = cbad ? 0 : L;
  if (cbad || L == 0) return false;
  if (warp == 5) commit_weights(S, L, lane);
  NamedSync<2, kStagers>()();  // the weights are in place
  return true;
}

// Fused commit, warps 5-15: path entries j0 .. j0 + nj - 1 as the rows of the
// commit MMA's MN-major operands: the k rows by cp.async (bf16, as they are,
// exact) and the U rows scaled by w_j, split hi + lo; rows nj .. up to the next
// multiple of 16 are zeroed.  Waits for its own copies and makes its writes
// visible to the tensor cores.
__device__ __forceinline__ void commit_stage(const FusedCommit& fc, const Small& S, uint8_t* smem,
                                             int b, int h, int hq, int Hqk, int Hv, int j0,
                                             int nj, int ot) {
  const size_t prow0 = (size_t)fc.lay.row0(b, fc.N);
  const size_t purow0 = fc.lay.urow0(b, h, Hv, fc.N);
  for (int e = ot; e < nj * 16; e += kStagers) {
    const int jj = e >> 4, c = e & 15;
    cp_async16(smem + OFF_CA + mn_chunk(jj, c),
               fc.k + ((prow0 + S.cpath[j0 + jj]) * Hqk + hq) * kD + 8 * c);
  }
  cp_async_commit();
  const int npad = ((nj + 15) & ~15) - nj;
  for (int e = ot; e < npad * 16; e += kStagers) {
    const int jj = nj + (e >> 4), c = e & 15;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(smem + OFF_CA + mn_chunk(jj, c)) = z;
    *reinterpret_cast<uint4*>(smem + OFF_CBH + mn_chunk(jj, c)) = z;
    *reinterpret_cast<uint4*>(smem + OFF_CBL + mn_chunk(jj, c)) = z;
  }
  for (int e = ot; e < nj * 16; e += kStagers) {
    const int jj = e >> 4, c = e & 15;
    const float w = S.cw[j0 + jj];
    const float4* src =
        reinterpret_cast<const float4*>(fc.U + (purow0 + S.cpath[j0 + jj]) * kD + 8 * c);
    const float4 u0 = src[0], u1 = src[1];
    uint32_t hi[4], lo[4];
    split2(w * u0.x, w * u0.y, hi[0], lo[0]);
    split2(w * u0.z, w * u0.w, hi[1], lo[1]);
    split2(w * u1.x, w * u1.y, hi[2], lo[2]);
    split2(w * u1.z, w * u1.w, hi[3], lo[3]);
    *reinterpret_cast<uint4*>(smem + OFF_CBH + mn_chunk(jj, c)) =
        make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(smem + OFF_CBL + mn_chunk(jj, c)) =
        make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  cp_async_wait_all();
  fence_proxy_async_smem();
}

template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmS,
                 const __grid_constant__ CUtensorMap tmS1, const float* S0,
                 const float* __restrict__ log_alpha, const float* __restrict__ beta,
                 const int32_t* __restrict__ parent, const __nv_bfloat16* __restrict__ v,
                 __nv_bfloat16* __restrict__ o, float* __restrict__ U, gdn_tree_dims d,
                 int32_t* dev_status, SeqLayout lay, FusedCommit fc, WaitHooks hk) {
  const uint64_t kWaitLimitNs = hk.limit_ns;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_addr(smem);
  Small& S = *reinterpret_cast<Small*>(smem + OFF_SMALL);
  float2* sXY = reinterpret_cast<float2*>(smem + OFF_XY);
  uint8_t* sR3 = smem + OFF_R3;
  uint8_t* sP = smem + OFF_P;
  uint8_t* sPath = smem + OFF_PATH;

  const int Nmax = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int n_units = d.B * Hv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // row mapping: thread <-> (tree row / state row t, 32-column quarter cq); warp
  // w may only touch TMEM lanes 32*(w%4) .. 32*(w%4)+31
  const int q4 = warp & 3, cq = warp >> 2;
  const int t = q4 * 32 + lane;
  const int col0 = cq * 32;
  const uint32_t trow_off = (uint32_t)(q4 * 32) << 16;
  int unit = blockIdx.x;

  if (tid == kIssuer) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmS);
    if (kFused) tma_prefetch_desc(&tmS1);
    mbar_init(&S.bar_kq, 1);
    mbar_init(&S.bar_g, 1);
    mbar_init(&S.bar_ks, 1);
    mbar_init(&S.bar_s, 1);
    mbar_init(&S.bar_stage, 1);
    mbar_init(&S.bar_c, 1);
    mbar_init(&S.bar_clc, 1);
    S.err = 0;
    S.n_kq = S.n_g = S.n_ks = S.n_s = S.n_c = 0;
    S.s1_pending = 0;
    S.cbad = 0;
    S.cL = 0;
    S.n_clc = 0;
    S.clc_pending = 0;
    S.next_unit[0] = S.next_unit[1] = n_units;
    mbar_fence_init();
    if (unit < n_units) {
      issue_kq(S, smem, &tmK, &tmQ, lay, unit, Hv, Hqk, Nmax);
      issue_state(S, smem, &tmS, lay, unit, Hv, Nmax);
      // the unit after this one: a CTA of the grid not launched yet, cancelled and
      // taken over (the response lands while the first copies do)
      clc_try_cancel(&S.clc_resp, &S.bar_clc);
      S.clc_pending = 1;
      S.next_unit[0] = clc_take(S, n_units, kWaitLimitNs);
    }
  }
  if constexpr (kFused) {
    if (warp > 4 && unit < n_units) prefetch_path(fc, S, unit / Hv, tid - 160);
  }
  if (warp < 4) {
    if (unit < n_units) prefetch_tree(S, parent, beta, log_alpha, lay, unit, Nmax, Hv, tid);
    mbar_init(&S.node_bar[tid], 1);  // one solve barrier per node (one arrival a phase)
    mbar_fence_init();
  }
  if (warp == 5) tmem_alloc(&S.tmem_base, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = S.tmem_base;
  const uint32_t trow = tmem + trow_off;
  uint32_t stage_ph = 0;  // the issuer's count of bar_stage phases

  uint32_t it = 0;
  for (; unit < n_units; ++it) {
    const uint32_t ph = it & 1u;
    const int b = unit / Hv, h = unit - b * Hv;
    const int hq = h / (Hv / Hqk);
    // the unit after this one, and (requested now, taken at the end of this unit)
    // the one after that
    const int next = S.next_unit[ph];
    if (tid == kIssuer && next < n_units) {
      clc_try_cancel(&S.clc_resp, &S.bar_clc);
      S.clc_pending = 1;
    }
    // this unit's nodes (an invalid sequence layout runs as an empty tree, unwritten)
    const UnitGeom geo = unit_geom(lay, b, Nmax);
    const int N = geo.n;
    const bool live = t < N;
    const int nc0 = S.n_c;  // commit MMA phases before this unit

    // ---- 0. tree group (warps 0-3): the unit's tree.  Operand group (warps 4-15):
    //         the Gram MMAs once K and Q have landed; fused, the previous tree's
    //         accepted path is checked and staged (warps 5-15) and committed on the
    //         tensor cores (warp 4)
    TC_START();
    TC_MARK(0);
    if (warp < 4) {
      tree_prep(S, sPath, parent, beta, log_alpha, lay, Nmax, next, n_units, N, Hv, tid, lane,
                warp, unit);
      TC_MARK(8);
    } else if (warp > 4) {
      if constexpr (kFused) {
        const int ot = tid - 160;
        int L = 0;
        const bool rows = commit_prologue(fc, S, b, h, Hv, ot, warp, lane,
                                          next < n_units ? next / Hv : -1, L);
        TC_MARK_BY(160, 16);
        const int nch = rows ? (L + kCommitChunk - 1) / kCommitChunk : 0;
        for (int c = 0; c < nch; ++c) {
          // the tiles are free once the previous chunk's MMA has read them
          if (c > 0 && !mbar_wait(&S.bar_c, (uint32_t)(nc0 + c - 1) & 1u, kWaitLimitNs)) S.err = 1;
          commit_stage(fc, S, smem, b, h, hq, Hqk, Hv, c * kCommitChunk,
                       min(kCommitChunk, L - c * kCommitChunk), ot);
          NamedSync<2, kStagers>()();
          if (ot == 0) mbar_arrive(&S.bar_stage);
        }
        if (nch == 0 && ot == 0) mbar_arrive(&S.bar_stage);  // nothing to stage: one phase
      }
    } else if (tid == kIssuer) {
      // the next unit's K, Q, v and state head for L2 now, so that their copies
      // (issued when this unit's solve is over) hit L2
      if (next < n_units) {
        const int nb = next / Hv, nh = next - nb * Hv, nhq = nh / (Hv / Hqk);
        const UnitGeom ng = unit_geom(lay, nb, Nmax);
        tma_prefetch_l2_4d(&tmK, 0, nhq, ng.c_node, ng.c_seq);
        tma_prefetch_l2_4d(&tmK, 64, nhq, ng.c_node, ng.c_seq);
        tma_prefetch_l2_4d(&tmQ, 0, nhq, ng.c_node, ng.c_seq);
        tma_prefetch_l2_4d(&tmQ, 64, nhq, ng.c_node, ng.c_seq);
        tma_prefetch_l2_4d(&tmV, 0, nh, ng.c_node, ng.c_seq);
        tma_prefetch_l2_4d(&tmV, 64, nh, ng.c_node, ng.c_seq);
        const float* ns = S0 + ((size_t)ng.st * Hv + nh) * kD * kD;
#pragma unroll
        for (int r = 0; r < 4; ++r) bulk_prefetch_l2(ns + r * (kD * kD / 4), kD * kD);
      }
      if (!mbar_wait(&S.bar_kq, ph, kWaitLimitNs)) {
        S.err = 1;
      } else {
        TC_MARK_BY(kIssuer, 9);
        tc_fence_after_sync();
        umma_128x128x128(tmem + kColGkk, sbase + OFF_K, sbase + OFF_K, false);
        umma_128x128x128(tmem + kColGqk, sbase + OFF_Q, sbase + OFF_K, false);
        umma_commit(&S.bar_g);
        ++S.n_g;
        TC_MARK_BY(kIssuer, 17);
      }
      if constexpr (kFused) {
        // one bar_stage phase per staged chunk (one when there is nothing to stage)
        for (int c = 0;; ++c) {
          if (!mbar_wait(&S.bar_stage, stage_ph & 1u, kWaitLimitNs)) {
            S.err = 1;
            break;
          }
          ++stage_ph;
          const int L = S.cL;
          if (S.cbad || L == 0) break;
          const int nj = min(kCommitChunk, L - c * kCommitChunk);
          tc_fence_after_sync();
          umma_commit_rows(tmem + kColCommit, sbase + OFF_CA, sbase + OFF_CBH, (nj + 15) >> 4,
                           c > 0);
          umma_commit_rows(tmem + kColCommit, sbase + OFF_CA, sbase + OFF_CBL, (nj + 15) >> 4,
                           true);
          umma_commit(&S.bar_c);
          ++S.n_c;
          if ((c + 1) * kCommitChunk >= L) break;
        }
      }
#ifdef GDN_TC_PROFILE
      mbar_wait(&S.bar_g, ph, kWaitLimitNs);
      TC_MARK_BY(kIssuer, 21);
#endif
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (S.err) goto fail;
    TC_MARK(1);

    {
      // ---- 1. the state row t (columns col0 ..) from the TMA tile; fused: S1 =
      //         gamma S0 + K_P^T diag(w) U_P from TMEM, written back for the TMA
      //         store; then S0 = hi + lo (MN-major), eight columns at a time
      const int cstat = kFused ? S.cbad : GDN_TREE_STATUS_OK;
      const bool commit_ok = kFused && cstat == GDN_TREE_STATUS_OK && !geo.bad;
      if (!mbar_wait(&S.bar_s, ph, kWaitLimitNs)) S.err = 2;
      const bool add_commit = kFused && commit_ok && S.cL > 0;  // CTA-uniform
      float gamma = 1.f;
      if (add_commit) {
        if (!mbar_wait(&S.bar_c, (uint32_t)(S.n_c - 1) & 1u, kWaitLimitNs)) S.err = 2;
        tc_fence_after_sync();
        gamma = S.cgamma;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {  // columns col0 + 8 i .. + 7
        uint8_t* p0 = sR3 + u_off(t, cq * 8 + 2 * i);
        uint8_t* p1 = sR3 + u_off(t, cq * 8 + 2 * i + 1);
        float4 a = *reinterpret_cast<const float4*>(p0);
        float4 c = *reinterpret_cast<const float4*>(p1);
        if (add_commit) {
          float dd[8];
          tmem_ld_8cols(trow + kColCommit + col0 + 8 * i, dd);  // warp-collective
          a = make_float4(fmaf(gamma, a.x, dd[0]), fmaf(gamma, a.y, dd[1]),
                          fmaf(gamma, a.z, dd[2]), fmaf(gamma, a.w, dd[3]));
          c = make_float4(fmaf(gamma, c.x, dd[4]), fmaf(gamma, c.y, dd[5]),
                          fmaf(gamma, c.z, dd[6]), fmaf(gamma, c.w, dd[7]));
        }
        if (commit_ok) {  // S1, in place for the TMA store
          *reinterpret_cast<float4*>(p0) = a;
          *reinterpret_cast<float4*>(p1) = c;
        }
        uint32_t hi[4], lo[4];
        split2(a.x, a.y, hi[0], lo[0]);
        split2(a.z, a.w, hi[1], lo[1]);
        split2(c.x, c.y, hi[2], lo[2]);
        split2(c.z, c.w, hi[3], lo[3]);
        *reinterpret_cast<uint4*>(smem + OFF_S0H + mn_chunk(t, cq * 4 + i)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + OFF_S0L + mn_chunk(t, cq * 4 + i)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      TC_MARK(2);
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncthreads();
      if (tid == kIssuer) {
        tc_fence_after_sync();
        if (commit_ok) {
          const int su = geo.st * Hv + h;
#pragma unroll
          for (int c = 0; c < 4; ++c) tma_store_3d(&tmS1, smem + OFF_R3 + c * kBoxBytes, 32 * c, 0, su);
          bulk_commit_group();
          S.s1_pending = 1;
        }
        umma_128x128x128_bmn(tmem + kColQS, sbase + OFF_Q, sbase + OFF_S0H, false);
        umma_128x128x128_bmn(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0H, false);
        umma_128x128x128_bmn(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0L, true);
        umma_commit(&S.bar_ks);
        ++S.n_ks;
        TC_MARK_BY(kIssuer, 22);
      }
      TC_MARK(3);
      if (h == 0 && tid == 0) {
        const int vcode = geo.bad ? GDN_TREE_STATUS_BAD_LAYOUT
                          : cstat ? cstat
                          : S.bad ? GDN_TREE_STATUS_BAD_TREE
                                  : GDN_TREE_STATUS_OK;
        if (dev_status && vcode) atomicMax(dev_status + b, vcode);
        const int ccode = geo.bad ? GDN_TREE_STATUS_BAD_LAYOUT : cstat;
        if (kFused && fc.status && ccode) atomicMax(fc.status + b, ccode);
      }
    }
    // an invalid layout, tree (verified as all-roots) or path leaves the unit's
    // outputs unwritten
    const bool write_out =
        !geo.bad && !S.bad && (!kFused || S.cbad == GDN_TREE_STATUS_OK);

    {
      const float bt = live ? S.beta[t] : 0.f;
      const df gt = live ? S.g[t] : df{0.f, 0.f};
      const float gam = __expf(df_value(gt));
      const uint32_t abits = live ? S.anc[t * kW + cq] : 0u;  // ancestors among my 32 columns
      const bool wide = S.wide_g;  // CTA-uniform

      // ---- 3. X and Y entries of t's ancestors in registers while K S0 / Q S0 run
      //         (X[t,s] = beta_t e^{g_t - g_s} G_kk[t,s], Y[t,s] = e^{g_t - g_s} G_qk[t,s])
      TC_MARK(13);
      if (!mbar_wait(&S.bar_g, ph, kWaitLimitNs)) S.err = 2;
      TC_MARK(14);
      tc_fence_after_sync();
      TC_MARK(10);
      // X while K S0 / Q S0 run, written back over G_kk in TMEM (nothing is held in
      // registers across the wait); Y is formed once they are done
      const float egt = live ? S.eg[t] : 0.f;
      if (!wide) {  // e^{g_t - g_s} = e^{g_t} e^{-g_s}
        float xr[32];
        tmem_ld_32cols(trow + kColGkk + col0, xr);
        TC_MARK(11);
#pragma unroll
        for (int j4 = 0; j4 < 8; ++j4) {
          const float4 m = *reinterpret_cast<const float4*>(&S.emg[col0 + j4 * 4]);
          const float em[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) xr[j4 * 4 + e] *= bt * egt * em[e];
        }
        tmem_st_32cols(trow + kColGkk + col0, xr);
      }
      TC_MARK(4);

      // ---- 4. once K S0 / Q S0 are done (regions 1 and 2 free) and the S1 store
      //         has read region 3: X, Y to region 1, R = beta (V - gamma K S0) to
      //         region 3, output seeds gamma Q S0 to region 2
      uint4 vreg[4];  // this thread's 32 values of v (row t, columns col0 ..)
      if (live) {
        const uint4* vsrc =
            reinterpret_cast<const uint4*>(v + (((size_t)geo.row0 + t) * Hv + h) * kD + col0);
#pragma unroll
        for (int i = 0; i < 4; ++i) vreg[i] = vsrc[i];
      }
      if (!mbar_wait(&S.bar_ks, ph, kWaitLimitNs)) S.err = 2;
      tc_fence_after_sync();
      if (tid == kIssuer && S.s1_pending) {
        bulk_wait_read_all();
        S.s1_pending = 0;
      }
      if (__syncthreads_or(S.err)) goto fail;
      TC_MARK(5);
      {
        float ks[32];
        tmem_ld_32cols(trow + kColKS + col0, ks);  // warp-collective: every lane
        if (live) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t w4[4] = {vreg[q].x, vreg[q].y, vreg[q].z, vreg[q].w};
            float r[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              r[2 * e] = bt * (__uint_as_float(w4[e] << 16) - gam * ks[q * 8 + 2 * e]);
              r[2 * e + 1] =
                  bt * (__uint_as_float(w4[e] & 0xffff0000u) - gam * ks[q * 8 + 2 * e + 1]);
            }
            *reinterpret_cast<float4*>(sR3 + u_off(t, cq * 8 + q * 2)) =
                make_float4(r[0], r[1], r[2], r[3]);
            *reinterpret_cast<float4*>(sR3 + u_off(t, cq * 8 + q * 2 + 1)) =
                make_float4(r[4], r[5], r[6], r[7]);
          }
        }
      }
      if (!wide) {
        float xr[32], yr[32];
        tmem_ld_32cols(trow + kColGkk + col0, xr);  // warp-collective: every lane
        tmem_ld_32cols(trow + kColGqk + col0, yr);
        if (live) {
#pragma unroll
          for (int j4 = 0; j4 < 8; ++j4) {
            const float4 m = *reinterpret_cast<const float4*>(&S.emg[col0 + j4 * 4]);
            const float em[4] = {m.x, m.y, m.z, m.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int j = j4 * 4 + e;
              if ((abits >> j) & 1u)
                sXY[x_index(t, col0 + j)] = make_float2(xr[j], egt * em[e] * yr[j]);
              if (col0 + j == t) S.ydiag[t] = yr[j];
            }
          }
        }
      } else {
        // some |g| of the tree is past the product form's bound: each decay from
        // the double-float difference, eight columns at a time, straight to
        // shared memory (rare trees; kept off the register budget of the
        // common path)
#pragma unroll 1
        for (int j8 = 0; j8 < 4; ++j8) {
          float gk[8], gq[8];
          tmem_ld_8cols(trow + kColGkk + col0 + 8 * j8, gk);  // warp-collective
          tmem_ld_8cols(trow + kColGqk + col0 + 8 * j8, gq);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = 8 * j8 + e;
            const bool need = (abits >> j) & 1u;
            if (live && col0 + j == t) S.ydiag[t] = gq[e];
            float dec = 0.f;
            if (__any_sync(0xffffffffu, need)) dec = need ? __expf(df_diff(gt, S.g[col0 + j])) : 0.f;
            if (need) sXY[x_index(t, col0 + j)] = make_float2(bt * dec * gk[e], dec * gq[e]);
          }
        }
      }
      {
        float qs[32];
        tmem_ld_32cols(trow + kColQS + col0, qs);  // warp-collective: every lane
        if (live) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(sP + u_off(t, cq * 8 + q)) =
                make_float4(gam * qs[4 * q], gam * qs[4 * q + 1], gam * qs[4 * q + 2],
                            gam * qs[4 * q + 3]);
        }
      }
      // nodes past this tree complete their solve phase too, so that every node's
      // barrier stays in step with the unit count
      if (cq == 0 && !live) mbar_arrive(&S.node_bar[t]);
      tc_fence_before_sync();
      __syncthreads();
    }

    // ---- 5. forward substitution as a dataflow over the tree ------------------------
    // u_t = r_t - sum over ancestors a of X[t,a] u_a and o_t = seed_t + sum over
    // t's path of Y[t,s] u_s.  Tasks (two nodes of one depth, one per half-warp)
    // go to the warps in depth order.  For node t a half-warp waits (acquire) on
    // the mbarrier of t's grandparent -- every ancestor but the parent is then
    // final -- sums those terms two at a time, then waits on the parent, adds its
    // term, publishes u_t and arrives on t's mbarrier (release); the parent's and
    // t's own output terms follow.  So a link of the dependency chain costs one
    // term, not the whole ancestor sum.  No cycle of waits can form: the
    // unfinished node of lowest depth order never waits (its ancestors come
    // earlier in that order).
    TC_MARK(6);
    {
      float* Ubh = U + lay.urow0(b, h, Hv, Nmax) * kD;
      __nv_bfloat16* obh = o + ((size_t)geo.row0 * Hv + h) * kD;
      bool timed_out = false;
      // a waiting warp is suspended by the hardware instead of spinning
      auto wait_ready = [&](int node) {
        if (!mbar_wait(&S.node_bar[node], ph, kWaitLimitNs)) timed_out = true;
      };
      // lanes: half-warp hf takes node hf of the task (a single task's second half
      // shadows the first without writing); lane hl of the half owns value columns
      // 4 hl .. 4 hl + 3 and 64 + 4 hl .. 64 + 4 hl + 3 (16-byte chunks hl, hl + 16)
      const int hf = lane >> 4, hl = lane & 15;
      const int n_tasks = S.n_tasks;
      for (int k = warp; k < n_tasks; k += kWarps) {
        const int pos = S.task_pos[k];
        const bool on = hf < S.task_n[k];
        const int tn = S.order[pos + (on ? hf : 0)];
        const int dep = S.depth[tn];  // the task's two nodes share it
        const uint8_t* pth = sPath + tn * kTile;  // pth[dep - 1] = tn, pth[0] = its root
        const float2* xyrow = sXY + x_index(tn, 0);
        float4 acc0 = *reinterpret_cast<const float4*>(sR3 + u_off(tn, hl));
        float4 acc1 = *reinterpret_cast<const float4*>(sR3 + u_off(tn, hl + 16));
        float4 py0 = *reinterpret_cast<const float4*>(sP + u_off(tn, hl));
        float4 py1 = *reinterpret_cast<const float4*>(sP + u_off(tn, hl + 16));
        float yp = 0.f;
        float4 up0 = make_float4(0.f, 0.f, 0.f, 0.f), up1 = up0;
        if (dep > 1) {
          if (dep > 2) wait_ready(pth[dep - 3]);
          int j = 0;
          for (; j + 2 <= dep - 2; j += 2) {
            int aa[2];
            float2 xy[2];
            float4 u0[2], u1[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) aa[e] = pth[j + e];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              xy[e] = xyrow[aa[e]];
              u0[e] = *reinterpret_cast<const float4*>(sR3 + u_off(aa[e], hl));
              u1[e] = *reinterpret_cast<const float4*>(sR3 + u_off(aa[e], hl + 16));
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              acc0 = fma4(-xy[e].x, u0[e], acc0);
              acc1 = fma4(-xy[e].x, u1[e], acc1);
              py0 = fma4(xy[e].y, u0[e], py0);
              py1 = fma4(xy[e].y, u1[e], py1);
            }
          }
          if (j < dep - 2) {
            const int a1 = pth[j];
            const float2 xy1 = xyrow[a1];
            const float4 v0 = *reinterpret_cast<const float4*>(sR3 + u_off(a1, hl));
            const float4 v1 = *reinterpret_cast<const float4*>(sR3 + u_off(a1, hl + 16));
            acc0 = fma4(-xy1.x, v0, acc0);
            acc1 = fma4(-xy1.x, v1, acc1);
            py0 = fma4(xy1.y, v0, py0);
            py1 = fma4(xy1.y, v1, py1);
          }
          const int par = pth[dep - 2];
          const float2 xyp = xyrow[par];
          yp = xyp.y;
          wait_ready(par);
          up0 = *reinterpret_cast<const float4*>(sR3 + u_off(par, hl));
          up1 = *reinterpret_cast<const float4*>(sR3 + u_off(par, hl + 16));
          acc0 = fma4(-xyp.x, up0, acc0);
          acc1 = fma4(-xyp.x, up1, acc1);
          if (on) {
            *reinterpret_cast<float4*>(sR3 + u_off(tn, hl)) = acc0;
            *reinterpret_cast<float4*>(sR3 + u_off(tn, hl + 16)) = acc1;
          }
        }
        __syncwarp();
        if (on && hl == 0 && !(unit == hk.withhold_unit && tn == hk.withhold_node))
          mbar_arrive(&S.node_bar[tn]);
        const float yd = S.ydiag[tn];
        py0 = fma4(yd, acc0, fma4(yp, up0, py0));
        py1 = fma4(yd, acc1, fma4(yp, up1, py1));
        if (write_out && on) {
          float* urow = Ubh + (size_t)tn * kD;
          *reinterpret_cast<float4*>(urow + hl * 4) = acc0;
          *reinterpret_cast<float4*>(urow + 64 + hl * 4) = acc1;
          __nv_bfloat16* orow = obh + (size_t)tn * Hv * kD;
          *reinterpret_cast<uint2*>(orow + hl * 4) =
              make_uint2(pack2f(py0.x, py0.y), pack2f(py0.z, py0.w));
          *reinterpret_cast<uint2*>(orow + 64 + hl * 4) =
              make_uint2(pack2f(py1.x, py1.y), pack2f(py1.z, py1.w));
        }
      }
      TC_MARK_BY(0, 18);
      TC_MARK_BY(480, 19);
      if (timed_out) S.err = 4;
      if constexpr (kFused) {
        if (warp > 4 && next < n_units) {
          const int nb = next / Hv, nh = next - nb * Hv;
          prefetch_path_rows_l2(fc, S, nb, nh, nh / (Hv / Hqk), Hqk, Hv, tid - 160);
        }
      }
    }
    if (tid == kIssuer) S.next_unit[ph ^ 1u] = clc_take(S, n_units, kWaitLimitNs);
    // regions 1 and 3 are free: the next unit's K, Q and state start loading
    tc_fence_before_sync();
    if (__syncthreads_or(S.err)) goto fail;
    tc_fence_after_sync();
    TC_MARK(7);
    TC_DUMP();
    if (tid == kIssuer && next < n_units) {
      issue_kq(S, smem, &tmK, &tmQ, lay, next, Hv, Hqk, Nmax);
      issue_state(S, smem, &tmS, lay, next, Hv, Nmax);
    }
    unit = next;
  }
  goto release;

fail:
  // a bounded wait ran out: report it for this unit's sequence and for the
  // sequences of every unit this CTA has not reached (their outputs stay
  // unwritten), let in-flight copies, stores and MMAs drain (again bounded),
  // then free TMEM
  if (tid == kIssuer) {
    // the units this CTA owns: the current one, the one after it, and the one the
    // request in flight names (a slot not yet rewritten holds the current unit)
    int own[4] = {unit, S.next_unit[it & 1u], S.next_unit[(it & 1u) ^ 1u], n_units};
    if (S.clc_pending) own[3] = clc_take(S, n_units, kWaitLimitNs);
    for (int i = 0; i < 4; ++i) {
      const int u = own[i];
      if (u < 0 || u >= n_units) continue;
      if (dev_status) atomicMax(dev_status + u / Hv, GDN_TREE_STATUS_TIMEOUT);
      if (kFused && fc.status) atomicMax(fc.status + u / Hv, GDN_TREE_STATUS_TIMEOUT);
    }
  }
  cp_async_wait_all();  // this thread's prefetches into shared memory
  if (tid == kIssuer) {
    if (S.n_kq > 0) mbar_wait(&S.bar_kq, (S.n_kq - 1) & 1, kWaitLimitNs);
    if (S.n_g > 0) mbar_wait(&S.bar_g, (S.n_g - 1) & 1, kWaitLimitNs);
    if (S.n_ks > 0) mbar_wait(&S.bar_ks, (S.n_ks - 1) & 1, kWaitLimitNs);
    if (S.n_s > 0) mbar_wait(&S.bar_s, (S.n_s - 1) & 1, kWaitLimitNs);
    if (S.n_c > 0) mbar_wait(&S.bar_c, (S.n_c - 1) & 1, kWaitLimitNs);
  }

release:
  if (tid == kIssuer) bulk_wait_all();  // the last S1 store has landed
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// ---- host side -------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// q, k [B, N, Hqk, 128] or v [B, N, Hv, 128] bf16 (`heads` = Hqk or Hv) -> boxes
// of 64 (columns) x 128 (nodes), 128-byte swizzled; nodes past N read as zeros
// `rows` x `seqs`: N x B for the fixed layout, T x 1 for packed rows
bool encode_rows_map(CUtensorMap* map, const void* base, int rows, int seqs, int heads) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)heads, (cuuint64_t)rows, (cuuint64_t)seqs};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)heads * kD * 2,
                                 (cuuint64_t)rows * heads * kD * 2};
  const cuuint32_t box[4] = {64, 1, kTile, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// fp32 states [n_states, 128, 128] (n_states = (B or n_slots) x Hv) -> boxes of 32
// columns x 128 rows, 128-byte swizzled (four per state)
bool encode_state_map(CUtensorMap* map, const float* base, long long n_states) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kD, (cuuint64_t)n_states};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)kD * kD * 4};
  const cuuint32_t box[3] = {32, kD, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool verify_tc_supported(const gdn_tree_dims& d) {
  return d.dtype == GDN_TREE_BF16 && d.dk == kD && d.dv == kD && d.N >= 1 && d.N <= kTile &&
         (long long)d.B * d.Hv < (1ll << 30) && tensor_map_encoder() != nullptr;
}

namespace {

template <bool kFused>
cudaError_t launch_tc(const VerifyArgs& a, const FusedCommit& fc, cudaStream_t stream) {
  CUtensorMap tmQ, tmK, tmV, tmS, tmS1;
  const int rows = a.lay.packed() ? a.lay.T : a.d.N, seqs = a.lay.packed() ? 1 : a.d.B;
  const long long n_states = (long long)(a.lay.slot ? a.lay.n_slots : a.d.B) * a.d.Hv;
  if (!encode_rows_map(&tmQ, a.q, rows, seqs, a.d.Hqk) ||
      !encode_rows_map(&tmK, a.k, rows, seqs, a.d.Hqk) ||
      !encode_rows_map(&tmV, a.v, rows, seqs, a.d.Hv) ||
      !encode_state_map(&tmS, a.S0, n_states) ||
      !encode_state_map(&tmS1, kFused ? fc.S1 : a.S0, n_states))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(verify_tc_kernel<kFused>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  // a CTA per unit; one fits an SM (the shared memory admits no second), and each
  // running CTA takes over the units of CTAs not launched yet (work stealing), so
  // the SMs stay busy until the units run out, however uneven the units
  const int n_units = a.d.B * a.d.Hv;
  verify_tc_kernel<kFused><<<n_units, kThreads, kSmemBytes, stream>>>(
      tmQ, tmK, tmV, tmS, tmS1, a.S0, a.log_alpha, a.beta, a.parent,
      static_cast<const __nv_bfloat16*>(a.v), static_cast<__nv_bfloat16*>(a.o), a.U, a.d,
      a.dev_status, a.lay, fc, wait_hooks());
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream) {
  return launch_tc<false>(a, FusedCommit{}, stream);
}

bool commit_verify_tc_supported(const gdn_tree_dims& d, int prev_N, int Lmax) {
  // the path prefetch copies min(Lmax, 352) entries into a kMaxN slot
  return verify_tc_supported(d) && prev_N >= 1 && prev_N <= kMaxN && Lmax <= kMaxN;
}

cudaError_t launch_commit_verify_tc(const CommitVerifyArgs& a, cudaStream_t stream) {
  FusedCommit fc{a.prev_path, a.prev_path_len, a.prev_parent, a.prev_U,
                 static_cast<const __nv_bfloat16*>(a.prev_k), a.prev_log_alpha, a.prev_N,
                 a.Lmax, a.S1, a.commit_status, a.prev_lay};
  VerifyArgs v = a.verify;
  v.S0 = a.S_prev;  // the kernel loads the previous state and commits it on chip
  return launch_tc<true>(v, fc, stream);
}

}  // namespace gdn

#ifdef GDN_TC_PROFILE
extern "C" int gdn_tree_debug_tc_phases(unsigned long long* host, int n_units) {
  return (int)cudaMemcpyFromSymbol(
      host, gdn::g_tc_phase,
      sizeof(unsigned long long) * gdn::kMarks * (n_units < 4096 ? n_units : 4096));
}
#endif
