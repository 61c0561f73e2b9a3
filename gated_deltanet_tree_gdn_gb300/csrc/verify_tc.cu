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
//   a persistent grid, one CTA (512 threads, 512 TMEM columns) per SM, walks the
//   (sequence b, v-head h) units; the next unit's operands are already being
//   loaded while the current unit finishes.  Per unit:
//   1. TMA (128-byte swizzle) brings K and Q of the q/k head and v of the unit
//      (issued as soon as the previous unit's solve is over); each thread loads an
//      8 x 4 tile of the fp32 state into registers and writes it as S0 = hi + lo,
//      two bf16 tiles laid out MN-major for the MMA's B operand, so K S0 keeps fp32
//      accuracy (K is exact in bf16).
//      (Fused with the delayed commitment, the tile is first committed in registers
//      and stored as S1.)  No thread waits on its own global loads near shared-memory
//      work: the state tile is its only per-thread load.
//   2. tcgen05.mma, accumulators in TMEM:  G_kk = K K^T, G_qk = Q K^T,
//      KS = K S0_hi + K S0_lo, QS = Q S0_hi.
//   3. TMEM -> registers (thread = tree node): the X and Y entries of the node's
//      ancestors (masked, decay-weighted, fp32), R = beta (V - gamma KS) and the
//      output seed gamma QS go to shared memory.
//   4. forward substitution as a dataflow over the tree, a warp per node and a
//      lane per 4 value columns: u_t = r_t - sum_a X[t,a] u_a, and in the same
//      walk over t's path o_t = gamma_t (Q S0)_t + sum_s Y[t,s] u_s, both fp32;
//      u_t and o_t are stored straight from the solve.
//
// Precision: K S0, the solve and Y U are fp32-accurate (U feeds the commit's
// 1e-4 bound); Q S0 uses S0_hi only, ample for the bf16 output.  Waits are
// bounded; a timeout reports a device status.
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
constexpr uint32_t kColGkk = 0, kColGqk = 128, kColKS = 256, kColQS = 384;
constexpr int kIssuer = 128;  // the one thread that issues every copy and MMA (warp 4, lane 0)
constexpr int kCommitChunk = 32;  // fused commit: path entries staged per round
// while every |g_t| of a unit is at most this, e^{g_t - g_s} is formed as
// e^{g_t} e^{-g_s} (both factors, and their product, stay normal fp32 numbers);
// beyond it, from the double-float difference
constexpr float kProductDecayLimit = 40.f;

#ifdef GDN_TC_PROFILE
// per-unit phase timestamps for a profiling build (never in the product build):
// SM clock counts kept in shared memory during the unit, dumped with the unit's
// global-timer span (slots 16, 17) once it is over
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
// region 1: K, Q (TMA) until the MMAs that read them end; then X, Y
constexpr uint32_t OFF_K = 0;
constexpr uint32_t OFF_Q = 1 * kOpBytes;
constexpr uint32_t OFF_XY = 0;
// region 2: the fused commit's staged path rows; S0^T hi, lo until the K S0 / Q S0
// MMAs end; then the output rows (seeded with gamma Q S0, finished by the solve)
constexpr uint32_t OFF_CK = 2 * kOpBytes;
constexpr uint32_t OFF_CU = 2 * kOpBytes + kCommitChunk * kD * 4;
constexpr uint32_t OFF_CKRAW = 2 * kOpBytes + 2 * kCommitChunk * kD * 4;  // k rows as bf16
constexpr uint32_t OFF_S0H = 2 * kOpBytes;
constexpr uint32_t OFF_S0L = 3 * kOpBytes;
constexpr uint32_t OFF_P = 2 * kOpBytes;
// region 3: v (TMA, 128-byte swizzle, first 32 KB) until it is read; then R / U
constexpr uint32_t OFF_U = 4 * kOpBytes;
constexpr uint32_t OFF_V = OFF_U;
constexpr uint32_t OFF_PATH = OFF_U + kTile * kD * 4;   // uint8 [node][depth - 1] -> path node
constexpr uint32_t OFF_SMALL = OFF_PATH + kTile * kTile;
#ifdef GDN_TC_PROFILE
constexpr uint32_t kSmallBytes = 16384 + 512;  // room for the phase stamps
#else
constexpr uint32_t kSmallBytes = 16384;
#endif
constexpr uint32_t kSmemBytes = OFF_SMALL + kSmallBytes + 1024;  // + alignment slack

static_assert(kTile * (kTile - 1) / 2 * 8 <= 2 * kOpBytes, "X, Y must fit in region 1");
static_assert(2 * kCommitChunk * kD * 4 <= 2 * kOpBytes, "commit staging must fit in region 2");
static_assert(OFF_U % 1024 == 0 && OFF_SMALL % 16 == 0, "alignment");
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
  uint64_t bar_kq, bar_v, bar_g, bar_ks;
  uint32_t tmem_base;
  int err;
  int bad;     // the tree failed validation
  int wide_g;  // some |g_t| > kProductDecayLimit
  int n_kq, n_g, n_ks;  // phases issued on bar_kq (and bar_v), bar_g, bar_ks
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

// byte offset of 16-byte chunk k8 (K elements 8*k8 .. 8*k8+7) of `row` in a
// 128-row, 128-wide K-major bf16 tile stored with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_chunk(int row, int k8) {
  const int kb = k8 >> 3, j = k8 & 7;
  return (uint32_t)(kb * kTileBytes + row * 128 + ((j ^ (row & 7)) << 4));
}

// fp32 128 x 128 row tiles (R / U, output rows): row t, 4-float chunk c4 (0..31),
// chunk index xor-swizzled by the row so that row-per-thread float4 accesses
// are bank-conflict free
__device__ __forceinline__ int u_index(int t, int c4) { return t * kD + ((c4 ^ (t & 7)) << 2); }

// packed strictly-lower triangle of X and Y
__device__ __forceinline__ int x_index(int t, int s) { return (t * (t - 1) >> 1) + s; }

// (a, b) -> bf16x2 hi parts and bf16x2 lo parts (x = hi + lo to ~2^-17)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
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

// issue the 8 K-steps (K = 128) of D (+)= A B^T for two 128x128 K-major tiles
__device__ __forceinline__ void umma_128x128x128(uint32_t d_tmem, uint32_t a_base,
                                                 uint32_t b_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t off = (uint32_t)((s >> 2) * kTileBytes + (s & 3) * 32);
    umma_bf16(d_tmem, desc_sw128_kmajor(a_base + off), desc_sw128_kmajor(b_base + off), idesc,
              (accumulate || s > 0) ? 1u : 0u);
  }
}

// The state operand S0 (K = dk rows x N = dv columns, bf16) is stored MN-major:
// the 16-byte chunk n8 (columns 8 n8 .. 8 n8 + 7) of row k sits in the 1024-byte
// atom of rows 8 (k / 8) .. and columns 64 (n8 / 8) .., atoms of one row group
// 1 KB apart along N and row groups 2 KB apart, chunks swizzled by the row.
constexpr uint32_t kS0Lbo = 1024, kS0Sbo = 2048;
__device__ __forceinline__ uint32_t s0_chunk(int k, int n8) {
  const int r = k & 7;
  return (uint32_t)((k >> 3) * kS0Sbo + (n8 >> 3) * kS0Lbo + r * 128 + (((n8 & 7) ^ r) << 4));
}

// issue the 8 K-steps (K = 128) of D (+)= A S for a 128x128 K-major tile A and
// the MN-major state tile S (a K-step of 16 rows spans two row groups)
__device__ __forceinline__ void umma_128x128x128_s0(uint32_t d_tmem, uint32_t a_base,
                                                    uint32_t s_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32_bmn(128, 128);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t a_off = (uint32_t)((s >> 2) * kTileBytes + (s & 3) * 32);
    umma_bf16(d_tmem, desc_sw128_kmajor(a_base + a_off),
              desc_sw128_mnmajor(s_base + (uint32_t)s * 2 * kS0Sbo, kS0Lbo, kS0Sbo), idesc,
              (accumulate || s > 0) ? 1u : 0u);
  }
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
// waits for all but this thread's most recent cp.async group
__device__ __forceinline__ void cp_async_wait_but_last() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
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

// K and Q of the unit's q/k head into region 1 (bar_kq), its v rows into region 3
// (bar_v); issuing thread only
__device__ __forceinline__ void issue_kqv(Small& S, uint8_t* smem, const CUtensorMap* tmK,
                                          const CUtensorMap* tmQ, const CUtensorMap* tmV,
                                          const SeqLayout& lay, int unit, int Hv, int Hqk,
                                          int Nmax) {
  const int b = unit / Hv, h = unit - b * Hv, hq = h / (Hv / Hqk);
  const UnitGeom g = unit_geom(lay, b, Nmax);
  const int cn = g.c_node, cs = g.c_seq;
  mbar_arrive_expect_tx(&S.bar_kq, 4 * kTileBytes);
  tma_load_4d(smem + OFF_K, tmK, &S.bar_kq, 0, hq, cn, cs);
  tma_load_4d(smem + OFF_K + kTileBytes, tmK, &S.bar_kq, 64, hq, cn, cs);
  tma_load_4d(smem + OFF_Q, tmQ, &S.bar_kq, 0, hq, cn, cs);
  tma_load_4d(smem + OFF_Q + kTileBytes, tmQ, &S.bar_kq, 64, hq, cn, cs);
  mbar_arrive_expect_tx(&S.bar_v, 2 * kTileBytes);
  tma_load_4d(smem + OFF_V, tmV, &S.bar_v, 0, h, cn, cs);
  tma_load_4d(smem + OFF_V + kTileBytes, tmV, &S.bar_v, 64, h, cn, cs);
  ++S.n_kq;
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
  TC_MARK(13);
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
  TC_MARK(14);
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
  TC_MARK(15);
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

// k and U rows of path entries j0 .. j0+nj-1 of the previous tree into the
// staging area as fp32; items i0, i0 + stride, ... of the calling group
__device__ __forceinline__ void commit_stage_rows(const FusedCommit& fc, const Small& S,
                                                  uint8_t* smem, int b, int h, int hq, int Hqk,
                                                  int Hv, int j0, int nj, int i0, int stride) {
  const size_t prow0 = (size_t)fc.lay.row0(b, fc.N);
  const size_t purow0 = fc.lay.urow0(b, h, Hv, fc.N);
  float* sk = reinterpret_cast<float*>(smem + OFF_CK);  // [kCommitChunk][kD]
  float* su = reinterpret_cast<float*>(smem + OFF_CU);  // [kCommitChunk][kD]
  for (int e = i0; e < nj * (kD / 8); e += stride) {
    const int jj = e / (kD / 8), c = (e % (kD / 8)) * 8;
    const uint4 raw = *reinterpret_cast<const uint4*>(
        fc.k + ((prow0 + S.cpath[j0 + jj]) * Hqk + hq) * kD + c);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    float* dst = sk + jj * kD + c;
    const float w = S.cw[j0 + jj];  // weighted as in stage_rows_finish
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dst[2 * q] = w * __uint_as_float(w4[q] << 16);
      dst[2 * q + 1] = w * __uint_as_float(w4[q] & 0xffff0000u);
    }
  }
  for (int e = i0; e < nj * (kD / 4); e += stride) {
    const int jj = e / (kD / 4), c = (e % (kD / 4)) * 4;
    *reinterpret_cast<float4*>(su + jj * kD + c) = *reinterpret_cast<const float4*>(
        fc.U + (purow0 + S.cpath[j0 + jj]) * kD + c);
  }
}

// The first chunk of path rows, asynchronously: the k rows (bf16, as they are) and
// the U rows are copied with cp.async (one group); stage_rows_finish, by the same
// threads, waits for it and widens the k rows to fp32.
__device__ __forceinline__ void stage_rows_issue(const FusedCommit& fc, const Small& S,
                                                 uint8_t* smem, int b, int h, int hq, int Hqk,
                                                 int Hv, int nj, int i0, int stride) {
  const size_t prow0 = (size_t)fc.lay.row0(b, fc.N);
  const size_t purow0 = fc.lay.urow0(b, h, Hv, fc.N);
  uint8_t* kraw = smem + OFF_CKRAW;  // [kCommitChunk][kD] bf16
  float* su = reinterpret_cast<float*>(smem + OFF_CU);
  for (int e = i0; e < nj * (kD / 8); e += stride) {
    const int jj = e / (kD / 8), c = (e % (kD / 8)) * 8;
    cp_async16(kraw + (jj * kD + c) * 2, fc.k + ((prow0 + S.cpath[jj]) * Hqk + hq) * kD + c);
  }
  for (int e = i0; e < nj * (kD / 4); e += stride) {
    const int jj = e / (kD / 4), c = (e % (kD / 4)) * 4;
    cp_async16(su + jj * kD + c, fc.U + (purow0 + S.cpath[jj]) * kD + c);
  }
  cp_async_commit();
}

// widens the staged bf16 k rows to fp32, each scaled by its path weight w_j
// (the products w_j k are the ones the accumulation would form)
__device__ __forceinline__ void stage_rows_finish(const Small& S, uint8_t* smem, int nj, int i0,
                                                  int stride) {
  const uint8_t* kraw = smem + OFF_CKRAW;
  float* sk = reinterpret_cast<float*>(smem + OFF_CK);
  for (int e = i0; e < nj * (kD / 8); e += stride) {
    const int jj = e / (kD / 8), c = (e % (kD / 8)) * 8;
    const float w = S.cw[jj];
    const uint4 raw = *reinterpret_cast<const uint4*>(kraw + (jj * kD + c) * 2);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    float* dst = sk + jj * kD + c;
    *reinterpret_cast<float4*>(dst) =
        make_float4(w * __uint_as_float(w4[0] << 16), w * __uint_as_float(w4[0] & 0xffff0000u),
                    w * __uint_as_float(w4[1] << 16), w * __uint_as_float(w4[1] & 0xffff0000u));
    *reinterpret_cast<float4*>(dst + 4) =
        make_float4(w * __uint_as_float(w4[2] << 16), w * __uint_as_float(w4[2] & 0xffff0000u),
                    w * __uint_as_float(w4[3] << 16), w * __uint_as_float(w4[3] & 0xffff0000u));
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

// Warps 5-15 (ot = tid - 160; warp 4 issues the copies and MMAs meanwhile): checks the previous tree's
// accepted path of sequence b (range, chain order, parent links), gathers its
// log alpha, stages the first chunk of its k / U rows into region 2 and forms
// the path weights.  Sets S.cbad (0 or the sequence's commit status), S.cL.
__device__ __forceinline__ void commit_prologue(const FusedCommit& fc, Small& S, uint8_t* smem,
                                                int b, int h, int hq, int Hqk, int Hv, int ot,
                                                int warp, int lane, int next_b) {
  const int pn = fc.lay.count(b, fc.N);  // the previous tree's node count (< 0: bad rows)
  cp_async_wait_all();  // this unit's path, prefetched during the previous unit
  NamedSync<2, kThreads - 160>()();
  const int L = S.pre_plen;
  int pj = -1;
  if (ot < fc.Lmax) pj = S.pre_path[ot];
  int cbad = (pn < 0 || L < 0 || L > pn || L > fc.Lmax);
  if (!cbad && ot < L) {
    cbad |= (pj < 0 || pj >= pn);
    S.cpath[ot] = pj;
  }
  cbad = bar_or<2, kThreads - 160>(cbad);
  // the entries are in range: the first chunk of k / U rows starts coming while
  // the chain check and log alpha are fetched (rows of a failed check go unused)
  const int nj0 = min(kCommitChunk, L);
  if (!cbad) stage_rows_issue(fc, S, smem, b, h, hq, Hqk, Hv, nj0, ot, kThreads - 160);
  if (!cbad && ot < L) {
    const int prev = ot == 0 ? -1 : S.cpath[ot - 1];
    cbad |= (ot > 0 && pj <= prev);
    const size_t prow0 = (size_t)fc.lay.row0(b, fc.N);
    if (fc.parent) cbad |= (fc.parent[prow0 + pj] != prev);
    S.cla[ot] = fc.log_alpha[(prow0 + pj) * Hv + h];
  }
  // every read of the prefetch slots is done: the next unit's path starts coming
  // (its own cp.async group, left in flight by the wait below)
  if (next_b >= 0) prefetch_path(fc, S, next_b, ot);
  else cp_async_commit();  // an empty group keeps the wait's count right
  cbad = bar_or<2, kThreads - 160>(cbad);  // (also: every log alpha is in place)
  if (ot == 0) {
    S.cbad = !cbad ? GDN_TREE_STATUS_OK
                   : (pn < 0 ? GDN_TREE_STATUS_BAD_LAYOUT : GDN_TREE_STATUS_BAD_PATH);
    S.cL = L;
  }
  if (!cbad) {
    // the weights while the rows land, then the k rows widened and weighted
    if (warp == 5) commit_weights(S, L, lane);
    cp_async_wait_but_last();
    NamedSync<2, kThreads - 160>()();
    stage_rows_finish(S, smem, nj0, ot, kThreads - 160);
  }
}

// K_P^T diag(w) U_P for this thread's 8x4 tile of the state (rows r8*8 .., columns
// c4*4 ..); needs no state, so it runs while the state is still in flight
__device__ __forceinline__ void commit_accumulate(const FusedCommit& fc, const Small& S,
                                                  uint8_t* smem, int b, int h, int hq, int Hqk,
                                                  int Hv, int tid, int r8, int c4,
                                                  float (&acc)[8][4]) {
  const int L = S.cL;
  const float* sk = reinterpret_cast<const float*>(smem + OFF_CK);
  const float* su = reinterpret_cast<const float*>(smem + OFF_CU);
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int j0 = 0; j0 < L; j0 += kCommitChunk) {
    const int nj = min(kCommitChunk, L - j0);
    if (j0 > 0) {  // the first chunk was staged by the operand group
      __syncthreads();
      commit_stage_rows(fc, S, smem, b, h, hq, Hqk, Hv, j0, nj, tid, kThreads);
      __syncthreads();
    }
    for (int jj = 0; jj < nj; ++jj) {
      // the staged k rows already carry their weights w_j
      const float4 k0 = *reinterpret_cast<const float4*>(sk + jj * kD + r8 * 8);
      const float4 k1 = *reinterpret_cast<const float4*>(sk + jj * kD + r8 * 8 + 4);
      const float4 uu = *reinterpret_cast<const float4*>(su + jj * kD + c4 * 4);
      const float kk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
      const float2 u01 = make_float2(uu.x, uu.y), u23 = make_float2(uu.z, uu.w);
#pragma unroll
      for (int i = 0; i < 8; ++i) {  // packed fp32x2 FMAs (same rounding as fmaf)
        const float2 ki = make_float2(kk[i], kk[i]);
        const float2 lo = __ffma2_rn(ki, u01, make_float2(acc[i][0], acc[i][1]));
        const float2 hi = __ffma2_rn(ki, u23, make_float2(acc[i][2], acc[i][3]));
        acc[i][0] = lo.x;
        acc[i][1] = lo.y;
        acc[i][2] = hi.x;
        acc[i][3] = hi.y;
      }
    }
  }
}

// S1 = gamma S0 + acc on this thread's 8x4 tile of the state, in registers (it is
// the state the next tree is verified from), stored to fc.S1
__device__ __forceinline__ void commit_finish(const FusedCommit& fc, const Small& S,
                                              size_t state_unit, int r8, int c4, float4 (&st)[8],
                                              const float (&acc)[8][4]) {
  const float gamma = S.cgamma;
  float* dst = fc.S1 + state_unit * kD * kD + (r8 * 8) * kD + c4 * 4;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    st[i].x = fmaf(gamma, st[i].x, acc[i][0]);
    st[i].y = fmaf(gamma, st[i].y, acc[i][1]);
    st[i].z = fmaf(gamma, st[i].z, acc[i][2]);
    st[i].w = fmaf(gamma, st[i].w, acc[i][3]);
    *reinterpret_cast<float4*>(dst + i * kD) = st[i];
  }
}

// S0 = hi + lo (bf16, MN-major, 128-byte swizzle: s0_chunk) from every thread's 8x4
// tile of the state (rows 8 r8 .., columns 4 c4 ..).  The two lanes of a pair (c4
// even, odd: one 16-byte chunk of columns) swap half their rows, so that each holds
// whole chunks: rows 8 r8 .. + 3 in the even lane, 8 r8 + 4 .. + 7 in the odd one.
// The hi half is written first, so that Q S0_hi and K S0_hi run on the tensor cores
// while the lo half is written; then K S0_lo, and bar_ks tracks all of them.  All
// threads of the CTA.
__device__ __forceinline__ void split_state(uint8_t* smem, uint32_t sbase, Small& S, uint32_t tmem,
                                            int r8, int c4, const float4 (&st)[8], bool issuer,
                                            bool issue) {
  const bool odd = c4 & 1;
  float4 ch[4][2];  // chunk rows: 8 r8 + (odd ? 4 : 0) + i, columns 8 (c4 / 2) .. + 7
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 give = odd ? st[i] : st[4 + i];
    float4 got;
    got.x = __shfl_xor_sync(0xffffffffu, give.x, 1);
    got.y = __shfl_xor_sync(0xffffffffu, give.y, 1);
    got.z = __shfl_xor_sync(0xffffffffu, give.z, 1);
    got.w = __shfl_xor_sync(0xffffffffu, give.w, 1);
    ch[i][0] = odd ? got : st[i];
    ch[i][1] = odd ? st[4 + i] : got;
  }
  const int row0 = 8 * r8 + (odd ? 4 : 0), n8 = c4 >> 1;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t hi[4], lo[4];
      split2(ch[i][0].x, ch[i][0].y, hi[0], lo[0]);
      split2(ch[i][0].z, ch[i][0].w, hi[1], lo[1]);
      split2(ch[i][1].x, ch[i][1].y, hi[2], lo[2]);
      split2(ch[i][1].z, ch[i][1].w, hi[3], lo[3]);
      const uint32_t* part = half == 0 ? hi : lo;
      *reinterpret_cast<uint4*>(smem + (half == 0 ? OFF_S0H : OFF_S0L) + s0_chunk(row0 + i, n8)) =
          make_uint4(part[0], part[1], part[2], part[3]);
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (issuer && issue) {
      tc_fence_after_sync();
      if (half == 0) {
        umma_128x128x128_s0(tmem + kColQS, sbase + OFF_Q, sbase + OFF_S0H, false);
        umma_128x128x128_s0(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0H, false);
      } else {
        umma_128x128x128_s0(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0L, true);
        umma_commit(&S.bar_ks);
        ++S.n_ks;
      }
    }
  }
}

template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const float* S0,
                 const float* __restrict__ log_alpha, const float* __restrict__ beta,
                 const int32_t* __restrict__ parent, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ U, gdn_tree_dims d, int32_t* dev_status, SeqLayout lay,
                 FusedCommit fc, WaitHooks hk) {
  const uint64_t kWaitLimitNs = hk.limit_ns;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_addr(smem);
  Small& S = *reinterpret_cast<Small*>(smem + OFF_SMALL);
  float* sU = reinterpret_cast<float*>(smem + OFF_U);
  float* sP = reinterpret_cast<float*>(smem + OFF_P);
  float2* sXY = reinterpret_cast<float2*>(smem + OFF_XY);
  uint8_t* sPath = smem + OFF_PATH;

  const int Nmax = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int n_units = d.B * Hv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // row mapping: thread <-> (tree row t, 32-column quarter cq); warp w may only
  // touch TMEM lanes 32*(w%4) .. 32*(w%4)+31
  const int q4 = warp & 3, cq = warp >> 2;
  const int t = q4 * 32 + lane;
  const int col0 = cq * 32;
  const uint32_t trow_off = (uint32_t)(q4 * 32) << 16;
  // state mapping: thread <-> 8x4 tile (rows 8 r8 .., columns 4 c4 ..); a warp holds
  // 4 row blocks x 8 column groups, so its loads and stores are 128-byte rows
  const int r8 = (warp >> 2) * 4 + (lane >> 3), c4 = (warp & 3) * 8 + (lane & 7);
  int unit = blockIdx.x;

  if (tid == kIssuer) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmV);
    mbar_init(&S.bar_kq, 1);
    mbar_init(&S.bar_v, 1);
    mbar_init(&S.bar_g, 1);
    mbar_init(&S.bar_ks, 1);
    S.err = 0;
    S.n_kq = 0;
    S.n_g = 0;
    S.n_ks = 0;
    S.cbad = 0;
    mbar_fence_init();
    if (unit < n_units) issue_kqv(S, smem, &tmK, &tmQ, &tmV, lay, unit, Hv, Hqk, Nmax);
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

  for (uint32_t it = 0; unit < n_units; unit += gridDim.x, ++it) {
    const uint32_t ph = it & 1u;
    const int b = unit / Hv, h = unit - b * Hv;
    const int hq = h / (Hv / Hqk);
    const int next = unit + gridDim.x;
    // this unit's nodes (an invalid sequence layout runs as an empty tree, unwritten)
    const UnitGeom geo = unit_geom(lay, b, Nmax);
    const int N = geo.n;
    const bool live = t < N;
    const size_t state_unit = (size_t)geo.st * Hv + h;

    // this thread's 8x4 tile of the state, into registers (L2 hits: prefetched)
    float4 st[8];
    {
      const float4* src =
          reinterpret_cast<const float4*>(S0 + state_unit * kD * kD + (r8 * 8) * kD + c4 * 4);
#pragma unroll
      for (int i = 0; i < 8; ++i) st[i] = __ldg(src + i * (kD / 4));
    }

    // ---- 0. tree group (warps 0-3): the unit's tree.  Operand group (warps 4-15):
    //         the Gram MMAs once K and Q have landed; fused, the previous tree's
    //         accepted path (warps 5-15)
    TC_START();
    TC_MARK(0);
    if (warp < 4) {
      tree_prep(S, sPath, parent, beta, log_alpha, lay, Nmax, next, n_units, N, Hv, tid, lane,
                warp, unit);
      TC_MARK(8);
    } else {
      if constexpr (kFused) {
        if (warp > 4)
          commit_prologue(fc, S, smem, b, h, hq, Hqk, Hv, tid - 160, warp, lane,
                          next < n_units ? next / Hv : -1);
        TC_MARK_BY(160, 16);
      }
      if (tid == kIssuer) {
        // the next unit's K, Q and state head for L2 now, so that their copies (issued
        // when this unit's solve is over) hit L2
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
      }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (S.err) goto fail;
    TC_MARK(1);

    // ---- 1. fused: S1 = gamma S0 + K_P^T diag(w) U_P on the tile in registers, stored
    //         to S1; then (both) S0^T from the tile
    if constexpr (kFused) {
      if (!S.cbad && !geo.bad) {  // (an invalid layout has no state of its own to commit)
        float cacc[8][4];
        commit_accumulate(fc, S, smem, b, h, hq, Hqk, Hv, tid, r8, c4, cacc);
        commit_finish(fc, S, state_unit, r8, c4, st, cacc);
      }
      __syncthreads();  // the staged path rows are read before S0^T goes over them
      TC_MARK(2);
    }
    split_state(smem, sbase, S, tmem, r8, c4, st, tid == kIssuer, true);
    TC_MARK(3);
    const int cstat = kFused ? S.cbad : GDN_TREE_STATUS_OK;
    const bool cbad = cstat != GDN_TREE_STATUS_OK;
    if (h == 0 && tid == 0) {
      const int vcode = geo.bad ? GDN_TREE_STATUS_BAD_LAYOUT
                        : cbad  ? cstat
                        : S.bad ? GDN_TREE_STATUS_BAD_TREE
                                : GDN_TREE_STATUS_OK;
      if (dev_status && vcode) atomicMax(dev_status + b, vcode);
      const int ccode = geo.bad ? GDN_TREE_STATUS_BAD_LAYOUT : cstat;
      if (kFused && fc.status && ccode) atomicMax(fc.status + b, ccode);
    }
    // an invalid layout, tree (verified as all-roots) or path leaves the unit's
    // outputs unwritten
    const bool write_out = !geo.bad && !S.bad && !cbad;

    {
      const uint32_t trow = tmem + trow_off;
      const float bt = live ? S.beta[t] : 0.f;
      const df gt = live ? S.g[t] : df{0.f, 0.f};
      const float gam = __expf(df_value(gt));
      const uint32_t abits = live ? S.anc[t * kW + cq] : 0u;  // ancestors among my 32 columns

      // ---- 3. X and Y entries of t's ancestors in registers while K S0 / Q S0 run
      if (!mbar_wait(&S.bar_g, ph, kWaitLimitNs)) S.err = 2;
      tc_fence_after_sync();
      TC_MARK(10);
      float xr[32], yr[32];
      tmem_ld_32cols(trow + kColGkk + col0, xr);
      tmem_ld_32cols(trow + kColGqk + col0, yr);
      TC_MARK(11);
      float ydiag = 0.f;
      if (!S.wide_g) {  // CTA-uniform: e^{g_t - g_s} = e^{g_t} e^{-g_s}
        const float egt = live ? S.eg[t] : 0.f;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          const float4 m0 = *reinterpret_cast<const float4*>(&S.emg[col0 + j8 * 8]);
          const float4 m1 = *reinterpret_cast<const float4*>(&S.emg[col0 + j8 * 8 + 4]);
          const float em[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int j = j8 * 8 + e;
            if (col0 + j == t) ydiag = yr[j];
            const float dec = ((abits >> j) & 1u) ? egt * em[e] : 0.f;
            xr[j] = bt * dec * xr[j];
            yr[j] = dec * yr[j];
          }
        }
      } else {
#pragma unroll
      for (int j8 = 0; j8 < 4; ++j8) {
        df gs[8];  // path log-decays of columns col0 + 8 j8 .., loaded together
        const float4* g4 = reinterpret_cast<const float4*>(&S.g[col0 + j8 * 8]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 w = g4[e];
          gs[2 * e] = df{w.x, w.y};
          gs[2 * e + 1] = df{w.z, w.w};
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = j8 * 8 + e;
          if (col0 + j == t) ydiag = yr[j];
          const bool need = (abits >> j) & 1u;
          float dec = 0.f;
          if (__any_sync(0xffffffffu, need)) dec = __expf(df_diff(gt, gs[e]));
          xr[j] = bt * dec * xr[j];
          yr[j] = dec * yr[j];
        }
      }
      }
      TC_MARK(4);

      // ---- 4. once K S0 / Q S0 are done (regions 1 and 2 free): X, Y to region 1,
      //         R = beta (V - gamma K S0) to region 3, output seeds gamma Q S0 to region 2
      if (!mbar_wait(&S.bar_ks, ph, kWaitLimitNs)) S.err = 2;
      tc_fence_after_sync();
      uint4 vreg[4];  // this thread's 32 values of v (row t, columns col0 ..), read before
                      // R goes over them
      if (!mbar_wait(&S.bar_v, ph, kWaitLimitNs)) S.err = 2;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        vreg[i] = *reinterpret_cast<const uint4*>(smem + OFF_V + sw128_chunk(t, cq * 4 + i));
      if (__syncthreads_or(S.err)) goto fail;
      TC_MARK(5);
      if (live) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((abits >> j) & 1u) sXY[x_index(t, col0 + j)] = make_float2(xr[j], yr[j]);
        if ((t >> 5) == cq) S.ydiag[t] = ydiag;
      }
      {
        float ks[32];
        tmem_ld_32cols(trow + kColKS + col0, ks);
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
            const int cc = cq * 8 + q * 2;
            *reinterpret_cast<float4*>(sU + u_index(t, cc)) = make_float4(r[0], r[1], r[2], r[3]);
            *reinterpret_cast<float4*>(sU + u_index(t, cc + 1)) =
                make_float4(r[4], r[5], r[6], r[7]);
          }
        }
      }
      {
        float qs[32];
        tmem_ld_32cols(trow + kColQS + col0, qs);
        if (live) {
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(sP + u_index(t, cq * 8 + q)) =
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
    // t's path of Y[t,s] u_s.  Warp w takes the nodes at positions w, w + 16, ... of
    // the depth order.  For node t it waits (acquire) on the mbarrier of t's
    // grandparent -- every ancestor but the parent is then final -- sums those
    // terms four at a time (lane = 4 value columns), then waits on the parent and
    // adds its term, publishes u_t and arrives on t's mbarrier (release); the
    // parent's and t's own output terms follow.  So a link of the dependency chain
    // costs one term, not the whole ancestor sum.  No cycle of waits can form: the
    // unfinished node of lowest depth order never waits (its ancestors come earlier
    // in that order).
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
        float4 acc0 = *reinterpret_cast<const float4*>(sU + u_index(tn, hl));
        float4 acc1 = *reinterpret_cast<const float4*>(sU + u_index(tn, hl + 16));
        float4 py0 = *reinterpret_cast<const float4*>(sP + u_index(tn, hl));
        float4 py1 = *reinterpret_cast<const float4*>(sP + u_index(tn, hl + 16));
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
              u0[e] = *reinterpret_cast<const float4*>(sU + u_index(aa[e], hl));
              u1[e] = *reinterpret_cast<const float4*>(sU + u_index(aa[e], hl + 16));
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
            const float4 v0 = *reinterpret_cast<const float4*>(sU + u_index(a1, hl));
            const float4 v1 = *reinterpret_cast<const float4*>(sU + u_index(a1, hl + 16));
            acc0 = fma4(-xy1.x, v0, acc0);
            acc1 = fma4(-xy1.x, v1, acc1);
            py0 = fma4(xy1.y, v0, py0);
            py1 = fma4(xy1.y, v1, py1);
          }
          const int par = pth[dep - 2];
          const float2 xyp = xyrow[par];
          yp = xyp.y;
          wait_ready(par);
          up0 = *reinterpret_cast<const float4*>(sU + u_index(par, hl));
          up1 = *reinterpret_cast<const float4*>(sU + u_index(par, hl + 16));
          acc0 = fma4(-xyp.x, up0, acc0);
          acc1 = fma4(-xyp.x, up1, acc1);
          if (on) {
            *reinterpret_cast<float4*>(sU + u_index(tn, hl)) = acc0;
            *reinterpret_cast<float4*>(sU + u_index(tn, hl + 16)) = acc1;
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
    // region 1 is free: the next unit's K and Q start loading
    fence_proxy_async_smem();
    tc_fence_before_sync();
    if (__syncthreads_or(S.err)) goto fail;
    tc_fence_after_sync();
    TC_MARK(7);
    TC_DUMP();
    if (tid == kIssuer && next < n_units)
      issue_kqv(S, smem, &tmK, &tmQ, &tmV, lay, next, Hv, Hqk, Nmax);
  }
  goto release;

fail:
  // a bounded wait ran out: report it for this unit's sequence and for the
  // sequences of every unit this CTA has not reached (their outputs stay
  // unwritten), let in-flight copies and MMAs drain (again bounded), then free
  // TMEM
  if (tid == 0) {
    for (int u = unit; u < n_units; u += gridDim.x) {
      if (dev_status) atomicMax(dev_status + u / Hv, GDN_TREE_STATUS_TIMEOUT);
      if (kFused && fc.status) atomicMax(fc.status + u / Hv, GDN_TREE_STATUS_TIMEOUT);
    }
  }
  cp_async_wait_all();  // this thread's prefetches into shared memory
  if (tid == kIssuer) {
    if (S.n_kq > 0) {
      mbar_wait(&S.bar_kq, (S.n_kq - 1) & 1, kWaitLimitNs);
      mbar_wait(&S.bar_v, (S.n_kq - 1) & 1, kWaitLimitNs);
    }
    if (S.n_g > 0) mbar_wait(&S.bar_g, (S.n_g - 1) & 1, kWaitLimitNs);
    if (S.n_ks > 0) mbar_wait(&S.bar_ks, (S.n_ks - 1) & 1, kWaitLimitNs);
  }

release:
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 5) tmem_dealloc(tmem, kTmemCols);
}

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

}  // namespace

bool verify_tc_supported(const gdn_tree_dims& d) {
  return d.dtype == GDN_TREE_BF16 && d.dk == kD && d.dv == kD && d.N >= 1 && d.N <= kTile &&
         (long long)d.B * d.Hv < (1ll << 30) && tensor_map_encoder() != nullptr;
}

namespace {

// streaming multiprocessors of the current device (cached per device)
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int n = (dev >= 0 && dev < 64) ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

template <bool kFused>
cudaError_t launch_tc(const VerifyArgs& a, const FusedCommit& fc, cudaStream_t stream) {
  CUtensorMap tmQ, tmK, tmV;
  const int rows = a.lay.packed() ? a.lay.T : a.d.N, seqs = a.lay.packed() ? 1 : a.d.B;
  if (!encode_rows_map(&tmQ, a.q, rows, seqs, a.d.Hqk) ||
      !encode_rows_map(&tmK, a.k, rows, seqs, a.d.Hqk) ||
      !encode_rows_map(&tmV, a.v, rows, seqs, a.d.Hv))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(verify_tc_kernel<kFused>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  // persistent: one CTA per SM (the shared memory admits no second), each walking
  // units blockIdx.x, blockIdx.x + gridDim.x, ...
  const int n_units = a.d.B * a.d.Hv;
  const int n_sm = sm_count();
  if (n_sm <= 0) return cudaErrorInvalidDevice;
  const int grid = n_units < n_sm ? n_units : n_sm;
  verify_tc_kernel<kFused><<<grid, kThreads, kSmemBytes, stream>>>(
      tmQ, tmK, tmV, a.S0, a.log_alpha, a.beta, a.parent,
      static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status, a.lay, fc, wait_hooks());
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
