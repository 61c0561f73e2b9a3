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
//   1. TMA (128-byte swizzle) brings K and Q of the q/k head and the fp32 state;
//      threads turn S0 into S0^T = hi + lo, two bf16 K-major tiles, so K S0
//      keeps fp32 accuracy (K is exact in bf16).
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
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kIssuer = 128;  // the one thread that issues every copy and MMA (warp 4, lane 0)
constexpr int kS0BoxRows = 32;  // the state arrives as four 32-row boxes
constexpr int kCommitChunk = 32;  // fused commit: path entries staged per round
constexpr uint32_t kSpinLimit = 1u << 24;  // bounded wait on a solve ready flag

#ifdef GDN_TC_PROFILE
// per-unit phase timestamps for a profiling build (never in the product build)
__device__ unsigned long long g_tc_phase[4096][16];
#define TC_MARK_BY(thread, i)                                                           \
  do {                                                                                  \
    if (threadIdx.x == (thread) && unit < 4096) g_tc_phase[unit][i] = globaltimer_ns(); \
  } while (0)
#else
#define TC_MARK_BY(thread, i) \
  do {                        \
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
constexpr uint32_t OFF_S0H = 2 * kOpBytes;
constexpr uint32_t OFF_S0L = 3 * kOpBytes;
constexpr uint32_t OFF_P = 2 * kOpBytes;
// region 3: the raw fp32 state (TMA) until S0^T is formed; then R / U
constexpr uint32_t OFF_U = 4 * kOpBytes;
constexpr uint32_t OFF_PATH = OFF_U + kTile * kD * 4;   // uint8 [node][depth - 1] -> path node
constexpr uint32_t OFF_SMALL = OFF_PATH + kTile * kTile;
constexpr uint32_t kSmallBytes = 12800;
constexpr uint32_t kSmemBytes = OFF_SMALL + kSmallBytes + 1024;  // + alignment slack

static_assert(kTile * (kTile - 1) / 2 * 8 <= 2 * kOpBytes, "X, Y must fit in region 1");
static_assert(2 * kCommitChunk * kD * 4 <= 2 * kOpBytes, "commit staging must fit in region 2");
static_assert(OFF_U % 1024 == 0 && OFF_SMALL % 16 == 0, "alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Small {
  int parent[kTile];
  df g[kTile];
  float beta[kTile];
  float la[kTile];
  float ydiag[kTile];  // Y[t,t] = q_t . k_t
  uint32_t anc[kTile * kW];
  int order[kTile];
  int depth[kTile];
  int level_start[kTile + 2];
  int level_cursor[kTile + 2];
  int ready[kTile];  // solve: node's u is final
  // the next unit's tree and gates, prefetched (cp.async) while this unit runs
  int pre_parent[kTile];
  float pre_beta[kTile];
  float pre_la[kTile];
  uint64_t bar_kq, bar_s0, bar_g, bar_ks;
  uint32_t tmem_base;
  int err;
  int bad;  // the tree failed validation
  int n_loads, n_g, n_ks;  // phases issued on bar_kq / bar_s0, bar_g, bar_ks
  // fused delayed commitment of the previous tree's accepted path
  int cpath[kMaxN];
  float cla[kMaxN];
  float cw[kMaxN];
  float cgamma;
  int cL;
  int cbad;
};
static_assert(sizeof(Small) <= kSmallBytes, "small state too large");
static_assert(offsetof(Small, g) % 16 == 0, "path log-decays are read as float4");

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

__device__ __forceinline__ float4 fma4(float a, float4 x, float4 acc) {
  acc.x = fmaf(a, x.x, acc.x);
  acc.y = fmaf(a, x.y, acc.y);
  acc.z = fmaf(a, x.z, acc.z);
  acc.w = fmaf(a, x.w, acc.w);
  return acc;
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

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
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

// Tree group: starts the copies of a unit's parent links and gates (node = tid)
// into the prefetch slots; tree_prep of that unit waits for them.
__device__ __forceinline__ void prefetch_tree(Small& S, const int32_t* parent, const float* beta,
                                              const float* log_alpha, int unit, int N, int Hv,
                                              int tid) {
  if (tid < N) {
    const int b = unit / Hv, h = unit - b * Hv;
    cp_async4(&S.pre_parent[tid], parent + (size_t)b * N + tid);
    cp_async4(&S.pre_beta[tid], beta + ((size_t)b * N + tid) * Hv + h);
    cp_async4(&S.pre_la[tid], log_alpha + ((size_t)b * N + tid) * Hv + h);
  }
  cp_async_commit();
}

// previous tree's accepted path for the fused delayed commitment
struct FusedCommit {
  const int32_t* path;      // [B, Lmax]
  const int32_t* path_len;  // [B]
  const int32_t* parent;    // [B, N] or NULL
  const float* U;           // [B, Hv, N, dv]
  const __nv_bfloat16* k;   // [B, N, Hqk, dk]
  const float* log_alpha;   // [B, N, Hv]
  int32_t N, Lmax;
  float* S1;                // [B, Hv, dk, dv] committed state (may alias the input state)
  int32_t* status;          // [B] or NULL
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

// K and Q of the unit's q/k head into region 1 (bar_kq), its fp32 state into
// region 3 (bar_s0); issuing thread only
__device__ __forceinline__ void issue_loads(Small& S, uint8_t* smem, const CUtensorMap* tmK,
                                            const CUtensorMap* tmQ, const CUtensorMap* tmS,
                                            int unit, int Hv, int Hqk) {
  const int b = unit / Hv, h = unit - b * Hv, hq = h / (Hv / Hqk);
  mbar_arrive_expect_tx(&S.bar_kq, 4 * kTileBytes);
  tma_load_4d(smem + OFF_K, tmK, &S.bar_kq, 0, hq, 0, b);
  tma_load_4d(smem + OFF_K + kTileBytes, tmK, &S.bar_kq, 64, hq, 0, b);
  tma_load_4d(smem + OFF_Q, tmQ, &S.bar_kq, 0, hq, 0, b);
  tma_load_4d(smem + OFF_Q + kTileBytes, tmQ, &S.bar_kq, 64, hq, 0, b);
  mbar_arrive_expect_tx(&S.bar_s0, kTile * kD * 4);
#pragma unroll
  for (int r = 0; r < kD; r += kS0BoxRows)  // four boxes land in parallel
    tma_load_3d(smem + OFF_U + r * kD * 4, tmS, &S.bar_s0, 0, r, unit);
  ++S.n_loads;
}

// Tree group (threads 0..127): takes the unit's prefetched tree and gates,
// validates the tree, then one upward walk per node gives its depth, its path
// log-decay g_t (double-float) and its strict-ancestor bitset, and a second its
// path (sPath row, root first); finally the nodes are ordered by depth.  An invalid tree is replaced by all-roots (nothing of it is stored).
// Then the copies for the CTA's next unit (`next`, if < n_units) are started.
__device__ __forceinline__ void tree_prep(Small& S, uint8_t* sPath, const int32_t* parent,
                                          const float* beta,
                                          const float* log_alpha, int next, int n_units, int N,
                                          int Hv, int tid, int lane, int warp) {
  using TreeSync = NamedSync<1, 128>;
  cp_async_wait_all();
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
  if (next < n_units) prefetch_tree(S, parent, beta, log_alpha, next, N, Hv, tid);
  TreeSync()();
  int dep = 0;
  if (tid < N) {
    df g = {0.f, 0.f};
    uint32_t a0 = 0u, a1 = 0u, a2 = 0u, a3 = 0u;
    for (int s = tid; s >= 0; s = S.parent[s]) {
      g = df_add(g, df{S.la[s], 0.f});
      const uint32_t bit = (s != tid) ? 1u << (s & 31) : 0u;
      const int w = s >> 5;
      a0 |= w == 0 ? bit : 0u;
      a1 |= w == 1 ? bit : 0u;
      a2 |= w == 2 ? bit : 0u;
      a3 |= w == 3 ? bit : 0u;
      ++dep;
    }
    S.g[tid] = g;
    S.anc[tid * kW + 0] = a0;
    S.anc[tid * kW + 1] = a1;
    S.anc[tid * kW + 2] = a2;
    S.anc[tid * kW + 3] = a3;
    S.depth[tid] = dep;
    // path: sPath[t * 128 + depth(s) - 1] = s for every s on t's path
    int ds = dep - 1;
    for (int s = tid; s >= 0; s = S.parent[s]) sPath[tid * kTile + ds--] = (uint8_t)s;
    atomicAdd(&S.level_start[dep], 1);
  }
  TreeSync()();
  if (warp == 0) {
    // exclusive scan of the level counts 0..kTile+1 (lane owns 5 entries)
    int cnt[5], run = 0;
#pragma unroll
    for (int e = 0; e < 5; ++e) {
      const int l = lane * 5 + e;
      cnt[e] = l < kTile + 2 ? S.level_start[l] : 0;
      run += cnt[e];
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
        S.level_start[l] = excl;
        S.level_cursor[l] = excl;
      }
      excl += cnt[e];
    }
  }
  TreeSync()();
  if (tid < N) S.order[atomicAdd(&S.level_cursor[dep], 1)] = tid;
}

// k and U rows of path entries j0 .. j0+nj-1 of the previous tree into the
// staging area as fp32; items i0, i0 + stride, ... of the calling group
__device__ __forceinline__ void commit_stage_rows(const FusedCommit& fc, const Small& S,
                                                  uint8_t* smem, int b, int h, int hq, int Hqk,
                                                  int Hv, int j0, int nj, int i0, int stride) {
  float* sk = reinterpret_cast<float*>(smem + OFF_CK);  // [kCommitChunk][kD]
  float* su = reinterpret_cast<float*>(smem + OFF_CU);  // [kCommitChunk][kD]
  for (int e = i0; e < nj * (kD / 8); e += stride) {
    const int jj = e / (kD / 8), c = (e % (kD / 8)) * 8;
    const uint4 raw = *reinterpret_cast<const uint4*>(
        fc.k + (((size_t)b * fc.N + S.cpath[j0 + jj]) * Hqk + hq) * kD + c);
    const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
    float* dst = sk + jj * kD + c;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      dst[2 * q] = __uint_as_float(w4[q] << 16);
      dst[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
    }
  }
  for (int e = i0; e < nj * (kD / 4); e += stride) {
    const int jj = e / (kD / 4), c = (e % (kD / 4)) * 4;
    *reinterpret_cast<float4*>(su + jj * kD + c) = *reinterpret_cast<const float4*>(
        fc.U + (((size_t)b * Hv + h) * fc.N + S.cpath[j0 + jj]) * kD + c);
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

// Warps 5-15 (ot = tid - 160; warp 4 issues the copies and MMAs meanwhile): checks the previous tree's
// accepted path of sequence b (range, chain order, parent links), gathers its
// log alpha, stages the first chunk of its k / U rows into region 2 and forms
// the path weights.  Sets S.cbad, S.cL.
__device__ __forceinline__ void commit_prologue(const FusedCommit& fc, Small& S, uint8_t* smem,
                                                int b, int h, int hq, int Hqk, int Hv, int ot,
                                                int warp, int lane) {
  const int L = fc.path_len[b];
  int pj = -1;
  if (ot < fc.Lmax) pj = fc.path[(size_t)b * fc.Lmax + ot];
  int cbad = (L < 0 || L > fc.N || L > fc.Lmax);
  if (!cbad && ot < L) {
    cbad |= (pj < 0 || pj >= fc.N);
    S.cpath[ot] = pj;
  }
  cbad = bar_or<2, kThreads - 160>(cbad);
  if (!cbad && ot < L) {
    const int prev = ot == 0 ? -1 : S.cpath[ot - 1];
    cbad |= (ot > 0 && pj <= prev);
    if (fc.parent) cbad |= (fc.parent[(size_t)b * fc.N + pj] != prev);
    S.cla[ot] = fc.log_alpha[((size_t)b * fc.N + pj) * Hv + h];
  }
  if (!cbad)
    commit_stage_rows(fc, S, smem, b, h, hq, Hqk, Hv, 0, min(kCommitChunk, L), ot, kThreads - 160);
  cbad = bar_or<2, kThreads - 160>(cbad);
  if (ot == 0) {
    S.cbad = cbad;
    S.cL = L;
  }
  if (!cbad && warp == 5) commit_weights(S, L, lane);
}

// K_P^T diag(w) U_P for this thread's 8x4 tile of the state (rows r8*8 .., columns
// c4*4 ..); needs no state, so it runs while the state is still in flight
__device__ __forceinline__ void commit_accumulate(const FusedCommit& fc, const Small& S,
                                                  uint8_t* smem, int b, int h, int hq, int Hqk,
                                                  int Hv, int tid, float (&acc)[8][4]) {
  const int L = S.cL;
  const int r8 = tid / 32, c4 = tid % 32;
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
      const float w = S.cw[j0 + jj];
      const float4 k0 = *reinterpret_cast<const float4*>(sk + jj * kD + r8 * 8);
      const float4 k1 = *reinterpret_cast<const float4*>(sk + jj * kD + r8 * 8 + 4);
      const float4 uu = *reinterpret_cast<const float4*>(su + jj * kD + c4 * 4);
      const float kk[8] = {w * k0.x, w * k0.y, w * k0.z, w * k0.w,
                           w * k1.x, w * k1.y, w * k1.z, w * k1.w};
      const float ul[4] = {uu.x, uu.y, uu.z, uu.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(kk[i], ul[j], acc[i][j]);
    }
  }
}

// S1 = gamma S0 + acc on the raw fp32 state tile in shared memory (updated in
// place: it is the state the next tree is verified from), then stored to fc.S1
// as one bulk copy; all threads of the CTA
__device__ __forceinline__ void commit_finish(const FusedCommit& fc, const Small& S, float* tile,
                                              int unit, int tid, const float (&acc)[8][4]) {
  const int r8 = tid / 32, c4 = tid % 32;
  const float gamma = S.cgamma;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = r8 * 8 + i;
    float4* cell = reinterpret_cast<float4*>(tile + row * kD + c4 * 4);
    const float4 s0 = *cell;
    float4 s1;
    s1.x = fmaf(gamma, s0.x, acc[i][0]);
    s1.y = fmaf(gamma, s0.y, acc[i][1]);
    s1.z = fmaf(gamma, s0.z, acc[i][2]);
    s1.w = fmaf(gamma, s0.w, acc[i][3]);
    *cell = s1;
  }
  fence_proxy_async_smem();
  __syncthreads();  // the committed state is in place before S0^T is formed from it
  // the tile goes back to S1 as one bulk store; thread 0 waits for it to finish
  // reading the tile before that region is reused
  if (tid == 0) {
    bulk_store(fc.S1 + (size_t)unit * kD * kD, tile, kD * kD * 4);
    bulk_commit_group();
  }
}

// S0^T = hi + lo (bf16, K-major, 128-byte swizzle) from the raw fp32 state tile in
// region 3; the hi half is written first, so that Q S0_hi and K S0_hi run on the
// tensor cores while the lo half is written; then K S0_lo, and bar_ks tracks all
// of them.  Called by kCount threads (index gtid, the issuing thread among them)
// that Sync synchronises.
template <int kCount, typename Sync>
__device__ __forceinline__ void split_state(uint8_t* smem, uint32_t sbase, Small& S, uint32_t tmem,
                                            int gtid, bool issuer, bool issue) {
  constexpr int kItems = kD * 16;  // 16-byte output chunks per half
  constexpr int kRounds = (kItems + kCount - 1) / kCount;
  const float* raw = reinterpret_cast<const float*>(smem + OFF_U);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int r = 0; r < kRounds; ++r) {
      const int item = gtid + r * kCount;
      if (kItems % kCount == 0 || item < kItems) {
        const int n = item & (kD - 1), k8 = item >> 7;
        const float* col = raw + (k8 * 8) * kD + n;
        uint32_t part[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint32_t hi, lo;
          split2(col[(2 * i) * kD], col[(2 * i + 1) * kD], hi, lo);
          part[i] = half == 0 ? hi : lo;
        }
        *reinterpret_cast<uint4*>(smem + (half == 0 ? OFF_S0H : OFF_S0L) + sw128_chunk(n, k8)) =
            make_uint4(part[0], part[1], part[2], part[3]);
      }
    }
    fence_proxy_async_smem();
    Sync()();
    if (issuer && issue) {
      tc_fence_after_sync();
      if (half == 0) {
        umma_128x128x128(tmem + kColQS, sbase + OFF_Q, sbase + OFF_S0H, false);
        umma_128x128x128(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0H, false);
      } else {
        umma_128x128x128(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0L, true);
        umma_commit(&S.bar_ks);
        ++S.n_ks;
      }
    }
  }
}

template <bool kFused>
__global__ void __launch_bounds__(kThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmS,
                 const __nv_bfloat16* __restrict__ v, const float* __restrict__ log_alpha,
                 const float* __restrict__ beta, const int32_t* __restrict__ parent,
                 __nv_bfloat16* __restrict__ o, float* __restrict__ U, gdn_tree_dims d,
                 int32_t* dev_status, FusedCommit fc) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_addr(smem);
  Small& S = *reinterpret_cast<Small*>(smem + OFF_SMALL);
  float* sU = reinterpret_cast<float*>(smem + OFF_U);
  float* sP = reinterpret_cast<float*>(smem + OFF_P);
  float2* sXY = reinterpret_cast<float2*>(smem + OFF_XY);
  uint8_t* sPath = smem + OFF_PATH;

  const int N = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int n_units = d.B * Hv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // row mapping: thread <-> (tree row t, 32-column quarter cq); warp w may only
  // touch TMEM lanes 32*(w%4) .. 32*(w%4)+31
  const int q4 = warp & 3, cq = warp >> 2;
  const int t = q4 * 32 + lane;
  const int col0 = cq * 32;
  const bool live = t < N;
  const uint32_t trow_off = (uint32_t)(q4 * 32) << 16;
  int unit = blockIdx.x;

  if (tid == kIssuer) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmS);
    mbar_init(&S.bar_kq, 1);
    mbar_init(&S.bar_s0, 1);
    mbar_init(&S.bar_g, 1);
    mbar_init(&S.bar_ks, 1);
    S.err = 0;
    S.n_loads = 0;
    S.n_g = 0;
    S.n_ks = 0;
    S.cbad = 0;
    mbar_fence_init();
    if (unit < n_units) issue_loads(S, smem, &tmK, &tmQ, &tmS, unit, Hv, Hqk);
  }
  if (warp < 4 && unit < n_units) prefetch_tree(S, parent, beta, log_alpha, unit, N, Hv, tid);
  if (warp == 5) tmem_alloc(&S.tmem_base, kTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = S.tmem_base;

  for (uint32_t it = 0; unit < n_units; unit += gridDim.x, ++it) {
    const uint32_t ph = it & 1u;
    const int b = unit / Hv, h = unit - b * Hv;
    const int hq = h / (Hv / Hqk);

    // ---- 0. tree group (warps 0-3): the unit's tree.  Operand group (warps 4-15):
    //         the Gram MMAs once K and Q have landed; then, plain, S0^T and the
    //         K S0 / Q S0 MMAs (1. below) while the tree group still works; fused,
    //         the previous tree's accepted path (warps 5-15)
    TC_MARK(0);
    if (warp < 4) {
      tree_prep(S, sPath, parent, beta, log_alpha, unit + gridDim.x, n_units, N, Hv, tid, lane, warp);
      TC_MARK(8);
    } else {
      if constexpr (kFused) {
        if (warp > 4) commit_prologue(fc, S, smem, b, h, hq, Hqk, Hv, tid - 160, warp, lane);
      }
      if (tid == kIssuer) {
        if (!mbar_wait(&S.bar_kq, ph, kWaitLimitNs)) {
          S.err = 1;
        } else {
          TC_MARK_BY(kIssuer, 9);
          tc_fence_after_sync();
          umma_128x128x128(tmem + kColGkk, sbase + OFF_K, sbase + OFF_K, false);
          umma_128x128x128(tmem + kColGqk, sbase + OFF_Q, sbase + OFF_K, false);
          umma_commit(&S.bar_g);
          ++S.n_g;
        }
      }
      if constexpr (!kFused) {
        // ---- 1. (plain) S0^T from the landed state, by the operand group
        const bool s0_ok = mbar_wait(&S.bar_s0, ph, kWaitLimitNs);
        if (!s0_ok) S.err = 1;
        split_state<kThreads - 128, NamedSync<2, kThreads - 128>>(
            smem, sbase, S, tmem, tid - 128, tid == kIssuer, s0_ok && S.err == 0);
      }
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (S.err) goto fail;
    TC_MARK(1);

    if constexpr (kFused) {
      // ---- 1. (fused) S1 = gamma S0 + K_P^T diag(w) U_P on the landed state tile (the
      //         product is formed while the state is still in flight), then S0^T from S1
      float cacc[8][4];
      if (!S.cbad) commit_accumulate(fc, S, smem, b, h, hq, Hqk, Hv, tid, cacc);
      if (__syncthreads_or(!mbar_wait(&S.bar_s0, ph, kWaitLimitNs))) goto fail;
      if (!S.cbad) commit_finish(fc, S, sU, unit, tid, cacc);
      TC_MARK(2);
      split_state<kThreads, BlockSync>(smem, sbase, S, tmem, tid, tid == kIssuer, true);
    }
    uint4 vreg[4];  // this thread's 32 values of v (row t, columns col0 ..)
#pragma unroll
    for (int i = 0; i < 4; ++i) vreg[i] = make_uint4(0, 0, 0, 0);
    if (live) {
      const uint4* vrow =
          reinterpret_cast<const uint4*>(v + (((size_t)b * N + t) * Hv + h) * kD + col0);
#pragma unroll
      for (int i = 0; i < 4; ++i) vreg[i] = __ldg(vrow + i);
    }
    TC_MARK(3);
    const bool cbad = kFused && S.cbad;
    if (h == 0 && tid == 0) {
      if (dev_status)
        dev_status[b] = cbad ? GDN_TREE_STATUS_BAD_PATH
                             : (S.bad ? GDN_TREE_STATUS_BAD_TREE : GDN_TREE_STATUS_OK);
      if (kFused && fc.status) fc.status[b] = cbad ? GDN_TREE_STATUS_BAD_PATH : GDN_TREE_STATUS_OK;
    }
    // an invalid tree (verified as all-roots) or path leaves the unit's outputs unwritten
    const bool write_out = !S.bad && !cbad;

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
      TC_MARK(4);

      // ---- 4. once K S0 / Q S0 are done (regions 1 and 2 free): X, Y to region 1,
      //         R = beta (V - gamma K S0) to region 3, output seeds gamma Q S0 to region 2
      if (!mbar_wait(&S.bar_ks, ph, kWaitLimitNs)) S.err = 2;
      tc_fence_after_sync();
      if constexpr (kFused) {
        if (tid == 0) bulk_wait_read_all();  // the S1 store has read the tile R goes into
      }
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
            const int c4 = cq * 8 + q * 2;
            *reinterpret_cast<float4*>(sU + u_index(t, c4)) = make_float4(r[0], r[1], r[2], r[3]);
            *reinterpret_cast<float4*>(sU + u_index(t, c4 + 1)) =
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
      if (cq == 0) S.ready[t] = 0;
      tc_fence_before_sync();
      __syncthreads();
    }

    // ---- 5. forward substitution as a dataflow over the tree ------------------------
    // u_t = r_t - sum over ancestors a of X[t,a] u_a and o_t = seed_t + sum over
    // t's path of Y[t,s] u_s.  Warp w takes the nodes at positions w, w + 16, ... of
    // the depth order.  For node t it waits (acquire) on the ready flag of t's
    // grandparent -- every ancestor but the parent is then final -- sums those
    // terms four at a time (lane = 4 value columns), then waits on the parent and
    // adds its term, publishes u_t and raises t's flag (release); the parent's and
    // t's own output terms follow.  So a link of the dependency chain costs one
    // term, not the whole ancestor sum.  No cycle of waits can form: the
    // unfinished node of lowest depth order never waits (its ancestors come
    // earlier in that order).
    TC_MARK(6);
    {
      int* ready = S.ready;
      float* Ubh = U + (size_t)unit * N * kD;
      __nv_bfloat16* obh = o + ((size_t)b * N * Hv + h) * kD;
      bool timed_out = false;
      auto wait_ready = [&](int node) {
        uint32_t spins = 0;
        while (ld_acquire_shared(ready + node) == 0) {
          if (++spins > kSpinLimit) {
            timed_out = true;
            break;
          }
        }
      };
      for (int i = warp; i < N; i += kWarps) {
        const int tn = S.order[i];
        const int dep = S.depth[tn];
        const uint8_t* pth = sPath + tn * kTile;  // pth[dep - 1] = tn, pth[0] = its root
        const float2* xyrow = sXY + x_index(tn, 0);
        float4 acc = *reinterpret_cast<const float4*>(sU + u_index(tn, lane));
        float4 py = *reinterpret_cast<const float4*>(sP + u_index(tn, lane));
        float yp = 0.f;
        float4 up = make_float4(0.f, 0.f, 0.f, 0.f);
        if (dep > 1) {
          if (dep > 2) wait_ready(pth[dep - 3]);
          int j = 0;
          for (; j + 4 <= dep - 2; j += 4) {
            int aa[4];
            float2 xy[4];
            float4 uu[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) aa[e] = pth[j + e];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              xy[e] = xyrow[aa[e]];
              uu[e] = *reinterpret_cast<const float4*>(sU + u_index(aa[e], lane));
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc = fma4(-xy[e].x, uu[e], acc);
              py = fma4(xy[e].y, uu[e], py);
            }
          }
          for (; j < dep - 2; ++j) {
            const int a1 = pth[j];
            const float2 xy1 = xyrow[a1];
            const float4 u1 = *reinterpret_cast<const float4*>(sU + u_index(a1, lane));
            acc = fma4(-xy1.x, u1, acc);
            py = fma4(xy1.y, u1, py);
          }
          const int par = pth[dep - 2];
          const float2 xyp = xyrow[par];
          yp = xyp.y;
          wait_ready(par);
          up = *reinterpret_cast<const float4*>(sU + u_index(par, lane));
          acc = fma4(-xyp.x, up, acc);
          *reinterpret_cast<float4*>(sU + u_index(tn, lane)) = acc;
        }
        __syncwarp();
        if (lane == 0) st_release_shared(ready + tn, 1);
        py = fma4(yp, up, py);
        py = fma4(S.ydiag[tn], acc, py);
        if (write_out) {
          *reinterpret_cast<float4*>(Ubh + (size_t)tn * kD + lane * 4) = acc;
          *reinterpret_cast<uint2*>(obh + (size_t)tn * Hv * kD + lane * 4) =
              make_uint2(pack2f(py.x, py.y), pack2f(py.z, py.w));
        }
      }
      if (timed_out) S.err = 4;
    }
    // regions 1 and 3 are free: the next unit's operands start loading
    fence_proxy_async_smem();
    tc_fence_before_sync();
    if (__syncthreads_or(S.err)) goto fail;
    tc_fence_after_sync();
    TC_MARK(7);
    if (tid == kIssuer && unit + (int)gridDim.x < n_units)
      issue_loads(S, smem, &tmK, &tmQ, &tmS, unit + gridDim.x, Hv, Hqk);
  }
  goto release;

fail:
  // a bounded wait ran out: report it, let in-flight copies and MMAs drain
  // (again bounded), then free TMEM
  if (tid == 0 && dev_status && unit < n_units)
    atomicMax(dev_status + unit / Hv, GDN_TREE_STATUS_TIMEOUT);
  if (tid == kIssuer) {
    if (S.n_loads > 0) {
      mbar_wait(&S.bar_kq, (S.n_loads - 1) & 1, kWaitLimitNs);
      mbar_wait(&S.bar_s0, (S.n_loads - 1) & 1, kWaitLimitNs);
    }
    if (S.n_g > 0) mbar_wait(&S.bar_g, (S.n_g - 1) & 1, kWaitLimitNs);
    if (S.n_ks > 0) mbar_wait(&S.bar_ks, (S.n_ks - 1) & 1, kWaitLimitNs);
  }

release:
  if constexpr (kFused) {
    if (tid == 0) bulk_wait_all();  // every S1 store is complete before the CTA leaves
  }
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

// q or k [B, N, Hqk, 128] bf16 -> boxes of 64 (K) x 128 (nodes); nodes past N
// read as zeros
bool encode_qk_map(CUtensorMap* map, const void* base, const gdn_tree_dims& d) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)d.Hqk, (cuuint64_t)d.N, (cuuint64_t)d.B};
  const cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)d.Hqk * kD * 2,
                                 (cuuint64_t)d.N * d.Hqk * kD * 2};
  const cuuint32_t box[4] = {64, 1, kTile, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// S0 [B*Hv, dk, dv] fp32 -> 32-row boxes of one (b, h) state, unswizzled
bool encode_state_map(CUtensorMap* map, const float* base, const gdn_tree_dims& d) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)kD, (cuuint64_t)d.B * d.Hv};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * 4, (cuuint64_t)kD * kD * 4};
  const cuuint32_t box[3] = {kD, kS0BoxRows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides,
             box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
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
  CUtensorMap tmQ, tmK, tmS;
  if (!encode_qk_map(&tmQ, a.q, a.d) || !encode_qk_map(&tmK, a.k, a.d) ||
      !encode_state_map(&tmS, a.S0, a.d))
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
      tmQ, tmK, tmS, static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent,
      static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status, fc);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream) {
  return launch_tc<false>(a, FusedCommit{}, stream);
}

bool commit_verify_tc_supported(const gdn_tree_dims& d, int prev_N) {
  return verify_tc_supported(d) && prev_N >= 1 && prev_N <= kMaxN;
}

cudaError_t launch_commit_verify_tc(const CommitVerifyArgs& a, cudaStream_t stream) {
  FusedCommit fc{a.prev_path, a.prev_path_len, a.prev_parent, a.prev_U,
                 static_cast<const __nv_bfloat16*>(a.prev_k), a.prev_log_alpha, a.prev_N,
                 a.Lmax, a.S1, a.commit_status};
  VerifyArgs v = a.verify;
  v.S0 = a.S_prev;  // the kernel loads the previous state and commits it on chip
  return launch_tc<true>(v, fc, stream);
}

}  // namespace gdn

#ifdef GDN_TC_PROFILE
extern "C" int gdn_tree_debug_tc_phases(unsigned long long* host, int n_units) {
  return (int)cudaMemcpyFromSymbol(
      host, gdn::g_tc_phase, sizeof(unsigned long long) * 16 * (n_units < 4096 ? n_units : 4096));
}
#endif
