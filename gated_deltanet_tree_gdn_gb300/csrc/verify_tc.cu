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
//   one CTA (256 threads) per (sequence b, v-head h); 512 TMEM columns.
//   1. TMA (128-byte swizzle) brings K and Q of the q/k head into shared
//      memory; threads turn S0 (fp32) into S0^T = hi + lo, two bf16 K-major
//      tiles, so K S0 keeps fp32 accuracy (K is exact in bf16).
//   2. tcgen05.mma, accumulators in TMEM:  G_kk = K K^T, G_qk = Q K^T,
//      KS = K S0_hi + K S0_lo, QS = Q S0_hi.
//   3. TMEM -> registers (thread = tree node): X (masked, decay-weighted,
//      fp32) and R = beta (V - gamma KS) to shared memory.
//   4. forward substitution over tree depth levels (nodes of one depth are
//      independent): fp32 FMA, warp per node, lane per 4 value columns.
//   5. Y (from G_qk) and U^T go to shared memory as bf16 hi + lo pairs;
//      tcgen05.mma computes Y U in three passes (hi*hi + hi*lo + lo*hi).
//   6. O = gamma QS + Y U from TMEM, stored as bf16; U stored as fp32.
//
// Precision: K S0 and the solve are fp32-accurate (U feeds the commit's 1e-4
// bound); Q S0 uses S0_hi only and Y U the three-pass split, both ample for
// the bf16 output.  Waits are bounded; a timeout reports a device status.
#include <cuda.h>
#include <cudaTypedefs.h>

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
constexpr uint32_t kColGkk = 0, kColGqk = 128, kColKS = 256, kColQS = 384, kColYU = 0;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kIssuer = 128;  // the one thread that issues every MMA (warp 4, lane 0)
constexpr int kS0BoxRows = 32;  // S0 arrives as four 32-row boxes
constexpr int kCommitChunk = 32;  // fused commit: path entries staged per round
constexpr uint32_t kSpinLimit = 1u << 24;  // bounded wait on a solve ready flag

#ifdef GDN_TC_PROFILE
// per-CTA phase timestamps for a profiling build (never in the product build)
__device__ unsigned long long g_tc_phase[4096][16];
#define TC_MARK(i)                                                                   \
  do {                                                                               \
    if (threadIdx.x == 0 && blockIdx.y * gridDim.x + blockIdx.x < 4096)              \
      g_tc_phase[blockIdx.y * gridDim.x + blockIdx.x][i] = globaltimer_ns();         \
  } while (0)
#else
#define TC_MARK(i) \
  do {             \
  } while (0)
#endif

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t kTileBytes = 128 * 128;            // one 64-wide K block: 128 rows x 128 B
constexpr uint32_t kOpBytes = 2 * kTileBytes;         // a 128 x 128 bf16 operand (2 K blocks)
constexpr uint32_t OFF_K = 0;                 // K, Q, S0^T: live until the K S0 / Q S0 MMAs end
constexpr uint32_t OFF_Q = 1 * kOpBytes;
constexpr uint32_t OFF_S0H = 2 * kOpBytes;
constexpr uint32_t OFF_S0L = 3 * kOpBytes;
constexpr uint32_t OFF_YH = 0;                // then Y (hi, lo) over K, Q ...
constexpr uint32_t OFF_YL = 1 * kOpBytes;
constexpr uint32_t OFF_X = 2 * kOpBytes;      // ... X (packed lower triangle, fp32) over S0^T
constexpr uint32_t OFF_UTH = 2 * kOpBytes;    // ... and, after the solve, U^T (hi, lo) over X
constexpr uint32_t OFF_UTL = 3 * kOpBytes;
constexpr uint32_t OFF_U = 4 * kOpBytes;      // raw S0 (TMA), then R / U, fp32, 64 KB
constexpr uint32_t OFF_CK = 2 * kOpBytes;     // fused commit: k rows of the path, before S0^T
constexpr uint32_t OFF_CU = 2 * kOpBytes + kCommitChunk * kD * 4;  // ... and their U rows
constexpr uint32_t OFF_PATH = OFF_U + kTile * kD * 4;   // uint8 [node][depth] -> ancestor
constexpr uint32_t OFF_SMALL = OFF_PATH + kTile * kTile;
constexpr uint32_t kSmallBytes = 11264;
constexpr uint32_t kSmemBytes = OFF_SMALL + kSmallBytes + 1024;  // + alignment slack

static_assert(kTile * (kTile - 1) / 2 * 4 <= 2 * kOpBytes, "X must fit in the S0^T region");
static_assert(OFF_U % 1024 == 0 && OFF_SMALL % 16 == 0, "alignment");
static_assert(kSmemBytes <= 232448, "shared memory budget");

struct Small {
  int parent[kTile];
  int jump[kTile];
  df g[kTile];
  float beta[kTile];
  float la[kTile];
  uint32_t anc[kTile * kW];
  int order[kTile];
  int depth[kTile];
  int level_start[kTile + 2];
  int level_cursor[kTile + 2];
  int ready[kTile];  // solve: node's u is final
  uint64_t bar_kq, bar_s0, bar_g, bar_ks, bar_yu;
  uint32_t tmem_base;
  int max_depth;
  int err;
  int bad;  // the tree failed validation
  int issued;
  // fused delayed commitment of the previous tree's accepted path
  int cpath[kMaxN];
  float cla[kMaxN];
  float cw[kMaxN];
  float cgamma;
  int cL;
  int cbad;  // bit 0: Gram MMAs, bit 1: K S0 / Q S0 MMAs, bit 2: Y U MMAs
};
static_assert(sizeof(Small) <= kSmallBytes, "small state too large");

// byte offset of 16-byte chunk k8 (K elements 8*k8 .. 8*k8+7) of `row` in a
// 128-row, 128-wide K-major bf16 tile stored with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_chunk(int row, int k8) {
  const int kb = k8 >> 3, j = k8 & 7;
  return (uint32_t)(kb * kTileBytes + row * 128 + ((j ^ (row & 7)) << 4));
}

// fp32 R/U tile: row t, 4-float chunk c4 (0..31), chunk index xor-swizzled by
// the row so that row-per-thread float4 accesses are bank-conflict free
__device__ __forceinline__ int u_index(int t, int c4) { return t * kD + ((c4 ^ (t & 7)) << 2); }

// packed strictly-lower triangle of X
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
    if (j0 > 0) {  // the first chunk was staged while the state was in flight
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
                                              int b, int h, int Hv, int tid,
                                              const float (&acc)[8][4]) {
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
    bulk_store(fc.S1 + ((size_t)b * Hv + h) * kD * kD, tile, kD * kD * 4);
    bulk_commit_group();
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
  float* sX = reinterpret_cast<float*>(smem + OFF_X);
  uint8_t* sPath = smem + OFF_PATH;

  const int N = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y;
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // epilogue mapping: thread <-> (tree row t, 32-column quarter cq); warp w
  // may only touch TMEM lanes 32*(w%4) .. 32*(w%4)+31
  const int q4 = warp & 3, cq = warp >> 2;
  const int t = q4 * 32 + lane;
  const bool live = t < N;

  // ---- 0. two groups run side by side until the tensor cores need both:
  //   tree group (warps 0-3): tree loads, validation, one upward walk per node
  //     (depth, path log-decay, ancestor bitset, path table), depth order;
  //   operand group (warps 4-15): bulk loads, TMEM, Gram MMAs, S0^T split, and
  //     the K S0 / Q S0 MMAs as soon as S0^T is in place.
  TC_MARK(0);
  if (tid == kIssuer) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmS);
  }
  if (warp < 4) {
    using TreeSync = NamedSync<1, 128>;
    int p_in = -1;
    float be_in = 0.f, la_in = 0.f;
    if (tid < N) {
      p_in = parent[(size_t)b * N + tid];
      be_in = beta[((size_t)b * N + tid) * Hv + h];
      la_in = log_alpha[((size_t)b * N + tid) * Hv + h];
    }
    S.parent[tid] = p_in;
    S.beta[tid] = be_in;
    S.la[tid] = la_in;
    S.level_start[tid] = 0;
    if (tid < 2) S.level_start[kTile + tid] = 0;
    if (tid == 0) S.max_depth = 0;
    const int bad_me = tid < N && (p_in < -1 || p_in >= tid);
    int bad_any;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 128, p;\n\t"
        "selp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(bad_any)
        : "r"(bad_me)
        : "memory");
    if (tid == 0) S.bad = bad_any;
    if (!bad_any) {
      // walk t -> root once: depth, g_t (double-float), ancestor bits
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
        // path table: sPath[t * 128 + depth(s)] = s for every s on t's path
        int ds = dep;
        for (int s = tid; s >= 0; s = S.parent[s]) sPath[tid * kTile + ds--] = (uint8_t)s;
        atomicAdd(&S.level_start[dep], 1);
        atomicMax(&S.max_depth, dep);
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
  } else {
    using OperandSync = NamedSync<2, kThreads - 128>;
    if (tid == kIssuer) {
      mbar_init(&S.bar_kq, 1);
      mbar_init(&S.bar_s0, 1);
      mbar_init(&S.bar_g, 1);
      mbar_init(&S.bar_ks, 1);
      mbar_init(&S.bar_yu, 1);
      S.err = 0;
      S.issued = 0;
      mbar_fence_init();
      mbar_arrive_expect_tx(&S.bar_kq, 4 * kTileBytes);
      tma_load_4d(smem + OFF_K, &tmK, &S.bar_kq, 0, hq, 0, b);
      tma_load_4d(smem + OFF_K + kTileBytes, &tmK, &S.bar_kq, 64, hq, 0, b);
      tma_load_4d(smem + OFF_Q, &tmQ, &S.bar_kq, 0, hq, 0, b);
      tma_load_4d(smem + OFF_Q + kTileBytes, &tmQ, &S.bar_kq, 64, hq, 0, b);
      mbar_arrive_expect_tx(&S.bar_s0, kTile * kD * 4);
#pragma unroll
      for (int r = 0; r < kD; r += kS0BoxRows)  // four boxes land in parallel
        tma_load_3d(smem + OFF_U + r * kD * 4, &tmS, &S.bar_s0, 0, r, b * Hv + h);
    }
    if (warp == 5) tmem_alloc(&S.tmem_base, kTmemCols);
    tc_fence_before_sync();
    OperandSync()();
    tc_fence_after_sync();
    const uint32_t tm = S.tmem_base;
    if (tid == kIssuer) {
      if (!mbar_wait(&S.bar_kq, 0, kWaitLimitNs)) {
        S.err = 1;
      } else {
        tc_fence_after_sync();
        umma_128x128x128(tm + kColGkk, sbase + OFF_K, sbase + OFF_K, false);
        umma_128x128x128(tm + kColGqk, sbase + OFF_Q, sbase + OFF_K, false);
        umma_commit(&S.bar_g);
        S.issued |= 1;
      }
    }
    if constexpr (kFused) {
      // previous tree's accepted path: range check, chain check, log alpha, and the
      // first chunk of its k / U rows, staged where S0^T will go (still free)
      const int ot = tid - 128;
      const int L = fc.path_len[b];
      int pj = -1;
      if (ot < fc.Lmax) pj = fc.path[(size_t)b * fc.Lmax + ot];
      int cbad = (L < 0 || L > fc.N || L > fc.Lmax);
      if (!cbad && ot < L) {
        cbad |= (pj < 0 || pj >= fc.N);
        S.cpath[ot] = pj;
      }
      cbad = bar_or<2, kThreads - 128>(cbad);
      if (!cbad && ot < L) {
        const int prev = ot == 0 ? -1 : S.cpath[ot - 1];
        cbad |= (ot > 0 && pj <= prev);
        if (fc.parent) cbad |= (fc.parent[(size_t)b * fc.N + pj] != prev);
        S.cla[ot] = fc.log_alpha[((size_t)b * fc.N + pj) * Hv + h];
      }
      if (!cbad)
        commit_stage_rows(fc, S, smem, b, h, hq, Hqk, Hv, 0, min(kCommitChunk, L), ot, kThreads - 128);
      cbad = bar_or<2, kThreads - 128>(cbad);
      if (ot == 0) {
        S.cbad = cbad;
        S.cL = L;
      }
      if (!cbad && warp == 4) commit_weights(S, L, lane);
    }
  }
  // ---- 1. both groups: S0^T = hi + lo (bf16, K-major, 128-byte swizzle) from the
  //         raw S0 tile; the hi half first, so that K S0_hi and Q S0_hi can run on
  //         the tensor cores while the lo half is written --------------------------
  TC_MARK(1);
  tc_fence_before_sync();
  __syncthreads();  // barriers initialised, TMEM allocated, tree group done
  tc_fence_after_sync();
  const uint32_t tmem = S.tmem_base;
  uint4 vreg[4];  // this thread's 32 values of v (row t, columns 32 cq ..), loaded below
  float cacc[8][4];  // fused commit: this thread's part of K_P^T diag(w) U_P
  if constexpr (kFused) {
    if (!S.cbad) commit_accumulate(fc, S, smem, b, h, hq, Hqk, Hv, tid, cacc);
  }
  if (!mbar_wait(&S.bar_s0, 0, kWaitLimitNs)) S.err = 1;
  if constexpr (kFused) {
    // delayed commitment: S1 = gamma S0 + K_P^T diag(w) U_P over the raw state tile,
    // written back in place (it is the state this tree is verified from) and to S1
    if (h == 0 && tid == 0 && fc.status)
      fc.status[b] = S.cbad ? GDN_TREE_STATUS_BAD_PATH : GDN_TREE_STATUS_OK;
    if (S.cbad) {
      if (h == 0 && tid == 0 && dev_status) dev_status[b] = GDN_TREE_STATUS_BAD_PATH;
      goto drain;
    }
    if (!S.err) commit_finish(fc, S, sU, b, h, Hv, tid, cacc);
  }
  TC_MARK(2);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float* raw = sU;  // S0 [dk][dv], row-major, landed by TMA
#pragma unroll
    for (int r = 0; r < (kD * 16) / kThreads; ++r) {
      const int item = tid + r * kThreads;
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
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == kIssuer && S.err == 0) {
      tc_fence_after_sync();
      if (half == 0) {
        umma_128x128x128(tmem + kColQS, sbase + OFF_Q, sbase + OFF_S0H, false);
        umma_128x128x128(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0H, false);
      } else {
        umma_128x128x128(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0L, true);
        umma_commit(&S.bar_ks);
        S.issued |= 2;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) vreg[i] = make_uint4(0, 0, 0, 0);
  if (live) {
    const uint4* vrow =
        reinterpret_cast<const uint4*>(v + (((size_t)b * N + t) * Hv + h) * kD + cq * 32);
#pragma unroll
    for (int i = 0; i < 4; ++i) vreg[i] = __ldg(vrow + i);
  }
  TC_MARK(3);
  if (h == 0 && tid == 0 && dev_status)
    dev_status[b] = S.bad ? GDN_TREE_STATUS_BAD_TREE : GDN_TREE_STATUS_OK;
  if (S.bad) goto drain;
  if (__syncthreads_or(S.err)) goto fail;

  {
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const int col0 = cq * 32;
    const float bt = live ? S.beta[t] : 0.f;
    const df gt = live ? S.g[t] : df{0.f, 0.f};
    const float gam = __expf(df_value(gt));
    const uint32_t abits = live ? S.anc[t * kW + cq] : 0u;  // ancestors among my 32 columns

    // ---- 4. X row segment (registers) while K S0 / Q S0 run ------------------------
    TC_MARK(4);
    if (!mbar_wait(&S.bar_g, 0, kWaitLimitNs)) S.err = 2;
    tc_fence_after_sync();
    float xr[32];
    tmem_ld_32cols(trow + kColGkk + col0, xr);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const bool need = (abits >> j) & 1u;
      float xv = 0.f;
      if (__any_sync(0xffffffffu, need)) {  // skip columns no lane of the warp needs
        const float e = __expf(df_diff(gt, S.g[col0 + j]));
        xv = need ? bt * e * xr[j] : 0.f;
      }
      xr[j] = xv;
    }

    // ---- 5. once K S0 / Q S0 are done (K, Q, S0^T dead): X, R = beta (V - gamma K S0)
    //         and Y (hi, lo) to shared memory -------------------------------------------
    if (!mbar_wait(&S.bar_ks, 0, kWaitLimitNs)) S.err = 2;
    tc_fence_after_sync();
    if constexpr (kFused) {
      if (tid == 0) bulk_wait_read_all();  // the S1 store has read the tile R goes into
    }
    if (__syncthreads_or(S.err)) goto fail;
    TC_MARK(5);
    {
      float ks[32];
      tmem_ld_32cols(trow + kColKS + col0, ks);
      if (cq == 0) S.ready[t] = 0;
      if (live) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if ((abits >> j) & 1u) sX[x_index(t, col0 + j)] = xr[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t w4[4] = {vreg[q].x, vreg[q].y, vreg[q].z, vreg[q].w};
          float r[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            r[2 * e] = bt * (__uint_as_float(w4[e] << 16) - gam * ks[q * 8 + 2 * e]);
            r[2 * e + 1] = bt * (__uint_as_float(w4[e] & 0xffff0000u) - gam * ks[q * 8 + 2 * e + 1]);
          }
          const int c4 = cq * 8 + q * 2;
          *reinterpret_cast<float4*>(sU + u_index(t, c4)) = make_float4(r[0], r[1], r[2], r[3]);
          *reinterpret_cast<float4*>(sU + u_index(t, c4 + 1)) =
              make_float4(r[4], r[5], r[6], r[7]);
        }
      }
    }
    {
      float gq[32];
      tmem_ld_32cols(trow + kColGqk + col0, gq);
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) {
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float y[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = g8 * 8 + 2 * i + e;
            const int s = col0 + j;
            const bool anc_s = live && ((abits >> j) & 1u);
            float yv = (live && s == t) ? gq[j] : 0.f;
            if (__any_sync(0xffffffffu, anc_s)) {
              const float dec = __expf(df_diff(gt, S.g[s]));
              if (anc_s) yv = dec * gq[j];
            }
            y[e] = yv;
          }
          split2(y[0], y[1], hi[i], lo[i]);
        }
        const uint32_t off = sw128_chunk(t, cq * 4 + g8);
        *reinterpret_cast<uint4*>(smem + OFF_YH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + OFF_YL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    tc_fence_before_sync();
    __syncthreads();

    // ---- 6. forward substitution as a dataflow over the tree ------------------------
    // u_t = r_t - sum over ancestors a of X[t,a] u_a.  Warp w takes the nodes at
    // positions w, w + 16, ... of the depth order.  For node t it waits (acquire)
    // on the ready flag of t's grandparent -- every ancestor but the parent is
    // then final -- sums those terms four at a time (lane = 4 value columns),
    // then waits on the parent and adds its term, publishes u_t and raises t's
    // flag (release).  So a link of the dependency chain costs one term, not the
    // whole ancestor sum.  No cycle of waits can form: the unfinished node of
    // lowest depth order never waits (its ancestors come earlier in that order).
    TC_MARK(6);
    {
      int* ready = S.ready;
      float* Ubh = U + ((size_t)b * Hv + h) * N * kD;
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
        const uint8_t* pth = sPath + tn * kTile;
        const float* xrow = sX + x_index(tn, 0);
        float4 acc = *reinterpret_cast<const float4*>(sU + u_index(tn, lane));
        if (dep > 1) {
          if (dep > 2) wait_ready(pth[dep - 2]);
          int j = 1;
          for (; j + 4 <= dep - 1; j += 4) {
            int aa[4];
            float xx[4];
            float4 uu[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) aa[e] = pth[j + e];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              xx[e] = xrow[aa[e]];
              uu[e] = *reinterpret_cast<const float4*>(sU + u_index(aa[e], lane));
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc.x = fmaf(-xx[e], uu[e].x, acc.x);
              acc.y = fmaf(-xx[e], uu[e].y, acc.y);
              acc.z = fmaf(-xx[e], uu[e].z, acc.z);
              acc.w = fmaf(-xx[e], uu[e].w, acc.w);
            }
          }
          for (; j < dep - 1; ++j) {
            const int a1 = pth[j];
            const float x1 = xrow[a1];
            const float4 u1 = *reinterpret_cast<const float4*>(sU + u_index(a1, lane));
            acc.x = fmaf(-x1, u1.x, acc.x);
            acc.y = fmaf(-x1, u1.y, acc.y);
            acc.z = fmaf(-x1, u1.z, acc.z);
            acc.w = fmaf(-x1, u1.w, acc.w);
          }
          const int par = pth[dep - 1];
          const float xp = xrow[par];
          wait_ready(par);
          const float4 up = *reinterpret_cast<const float4*>(sU + u_index(par, lane));
          acc.x = fmaf(-xp, up.x, acc.x);
          acc.y = fmaf(-xp, up.y, acc.y);
          acc.z = fmaf(-xp, up.z, acc.z);
          acc.w = fmaf(-xp, up.w, acc.w);
          *reinterpret_cast<float4*>(sU + u_index(tn, lane)) = acc;
        }
        __syncwarp();
        if (lane == 0) st_release_shared(ready + tn, 1);
        *reinterpret_cast<float4*>(Ubh + (size_t)tn * kD + lane * 4) = acc;
      }
      if (timed_out) S.err = 4;
    }
    if (__syncthreads_or(S.err)) goto fail;

    // ---- 7. U^T (hi, lo) over X ----------------------------------------------------------
    TC_MARK(7);
#pragma unroll
    for (int r = 0; r < (kD * 16) / kThreads; ++r) {
      const int item = tid + r * kThreads;
      const int n = item & (kD - 1), t8 = item >> 7;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int ta = t8 * 8 + 2 * i, tb = ta + 1;
        const float x0 = ta < N ? sU[u_index(ta, n >> 2) + (n & 3)] : 0.f;
        const float x1 = tb < N ? sU[u_index(tb, n >> 2) + (n & 3)] : 0.f;
        split2(x0, x1, hi[i], lo[i]);
      }
      const uint32_t off = sw128_chunk(n, t8);
      *reinterpret_cast<uint4*>(smem + OFF_UTH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + OFF_UTL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();

    // ---- 8. Y U on the tensor cores (three bf16 passes) -------------------------------
    TC_MARK(8);
    if (tid == kIssuer) {
      tc_fence_after_sync();
      umma_128x128x128(tmem + kColYU, sbase + OFF_YH, sbase + OFF_UTH, false);
      umma_128x128x128(tmem + kColYU, sbase + OFF_YH, sbase + OFF_UTL, true);
      umma_128x128x128(tmem + kColYU, sbase + OFF_YL, sbase + OFF_UTH, true);
      umma_commit(&S.bar_yu);
      S.issued |= 4;
    }
    if (!mbar_wait(&S.bar_yu, 0, kWaitLimitNs)) S.err = 3;
    tc_fence_after_sync();
    if (__syncthreads_or(S.err)) goto fail;

    // ---- 9. O = gamma QS + Y U ----------------------------------------------------------
    TC_MARK(9);
    {
      float yu[32], qs[32];
      tmem_ld_32cols(trow + kColYU + col0, yu);
      tmem_ld_32cols(trow + kColQS + col0, qs);
      if (live) {
        uint4* orow = reinterpret_cast<uint4*>(o + (((size_t)b * N + t) * Hv + h) * kD + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = q * 8 + 2 * e;
            w4[e] = pack2f(fmaf(gam, qs[j], yu[j]), fmaf(gam, qs[j + 1], yu[j + 1]));
          }
          orow[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    }
  }
  TC_MARK(10);
  goto release;

fail:
  // a bounded wait ran out: report it, let in-flight copies and MMAs drain
  // (again bounded), then free TMEM
  if (tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_TIMEOUT);
drain:
  if (tid == 0) {
    mbar_wait(&S.bar_kq, 0, kWaitLimitNs);
    mbar_wait(&S.bar_s0, 0, kWaitLimitNs);
    if (S.issued & 1) mbar_wait(&S.bar_g, 0, kWaitLimitNs);
    if (S.issued & 2) mbar_wait(&S.bar_ks, 0, kWaitLimitNs);
    if (S.issued & 4) mbar_wait(&S.bar_yu, 0, kWaitLimitNs);
  }

release:
  if constexpr (kFused) {
    if (tid == 0) bulk_wait_all();  // the S1 store is complete before the CTA leaves
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
         tensor_map_encoder() != nullptr;
}

namespace {

template <bool kFused>
cudaError_t launch_tc(const VerifyArgs& a, const FusedCommit& fc, cudaStream_t stream) {
  CUtensorMap tmQ, tmK, tmS;
  if (!encode_qk_map(&tmQ, a.q, a.d) || !encode_qk_map(&tmK, a.k, a.d) ||
      !encode_state_map(&tmS, a.S0, a.d))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(verify_tc_kernel<kFused>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  verify_tc_kernel<kFused><<<dim3(a.d.Hv, a.d.B), kThreads, kSmemBytes, stream>>>(
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
extern "C" int gdn_tree_debug_tc_phases(unsigned long long* host, int n_ctas) {
  return (int)cudaMemcpyFromSymbol(host, gdn::g_tc_phase,
                                   sizeof(unsigned long long) * 16 * (n_ctas < 4096 ? n_ctas : 4096));
}
#endif
