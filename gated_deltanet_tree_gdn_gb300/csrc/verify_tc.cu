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
constexpr int kThreads = 256;
constexpr int kW = kTile / 32;     // ancestor bitset words per node
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColGkk = 0, kColGqk = 128, kColKS = 256, kColQS = 384, kColYU = 0;
constexpr int kXStride = kTile + 1;  // padded fp32 row of X
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// shared memory map (byte offsets from a 1024-aligned base)
constexpr uint32_t kTileBytes = kTile * 128 * 2 / 2;  // one 64-wide K block: 128 rows x 128 B
constexpr uint32_t kOpBytes = 2 * kTileBytes;         // a 128 x 128 bf16 operand (2 K blocks)
constexpr uint32_t OFF_K = 0;                 // phase A
constexpr uint32_t OFF_Q = 1 * kOpBytes;
constexpr uint32_t OFF_S0H = 2 * kOpBytes;
constexpr uint32_t OFF_S0L = 3 * kOpBytes;
constexpr uint32_t OFF_X = 0;                 // phase B (solve), aliases phase A
constexpr uint32_t OFF_YH = 0;                // phase C (output), aliases A and B
constexpr uint32_t OFF_YL = 1 * kOpBytes;
constexpr uint32_t OFF_UTH = 2 * kOpBytes;
constexpr uint32_t OFF_UTL = 3 * kOpBytes;
constexpr uint32_t OFF_U = 4 * kOpBytes;      // R / U, fp32, 64 KB
constexpr uint32_t OFF_SMALL = OFF_U + kTile * kD * 4;
constexpr uint32_t kSmallBytes = 8192;
constexpr uint32_t kSmemBytes = OFF_SMALL + kSmallBytes + 1024;  // + alignment slack

static_assert(kTile * kXStride * 4 <= 4 * kOpBytes, "X must fit in the operand region");
static_assert(OFF_U % 1024 == 0, "alignment");

struct Small {
  int parent[kTile];
  int jump[kTile];
  df g[kTile];
  float beta[kTile];
  float la[kTile];
  uint32_t anc[kTile * kW];
  int depth[kTile];
  int order[kTile];
  int level_start[kTile + 2];
  int level_cursor[kTile + 2];
  uint64_t bar_tma;
  uint64_t bar_mma;
  uint32_t tmem_base;
  int max_depth;
  int err;
};
static_assert(sizeof(Small) <= kSmallBytes, "small state too large");

// byte offset of element (row, k) inside a 128-row, 128-wide K-major
// bf16 tile with the 128-byte swizzle (two 64-wide K blocks)
__device__ __forceinline__ uint32_t sw128_chunk(int row, int k8) {
  // k8 = index of the 8-element (16-byte) chunk along K, 0..15
  const int kb = k8 >> 3, j = k8 & 7;
  return (uint32_t)(kb * kTileBytes + row * 128 + ((j ^ (row & 7)) << 4));
}

// fp32 R/U tile: row t, 4-float chunk c4 (0..31), chunk index xor-swizzled by
// the row so that row-per-thread float4 accesses are bank-conflict free
__device__ __forceinline__ int u_index(int t, int c4) { return t * kD + ((c4 ^ (t & 7)) << 2); }

__device__ __forceinline__ void split_bf16(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

__device__ __forceinline__ uint32_t pack2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
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

__global__ void __launch_bounds__(kThreads, 1)
verify_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __nv_bfloat16* __restrict__ v, const float* __restrict__ log_alpha,
                 const float* __restrict__ beta, const int32_t* __restrict__ parent,
                 const float* __restrict__ S0, __nv_bfloat16* __restrict__ o,
                 float* __restrict__ U, gdn_tree_dims d, int32_t* dev_status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_addr(smem_raw);
  uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  const uint32_t sbase = smem_addr(smem);
  Small& S = *reinterpret_cast<Small*>(smem + OFF_SMALL);
  float* sU = reinterpret_cast<float*>(smem + OFF_U);
  float* sX = reinterpret_cast<float*>(smem + OFF_X);

  const int N = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y;
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // ---- 1. tree: load + validate (nothing issued yet) ----------------------
  int bad = 0;
  for (int t = tid; t < kTile; t += kThreads) {
    int p = -1;
    float be = 0.f, la = 0.f;
    if (t < N) {
      p = parent[(size_t)b * N + t];
      bad |= (p < -1 || p >= t);
      be = beta[((size_t)b * N + t) * Hv + h];
      la = log_alpha[((size_t)b * N + t) * Hv + h];
    }
    S.parent[t] = p;
    S.beta[t] = be;
    S.la[t] = la;
  }
  if (tid == 0) {
    S.err = 0;
    S.max_depth = 0;
  }
  bad = __syncthreads_or(bad);
  if (h == 0 && tid == 0 && dev_status)
    dev_status[b] = bad ? GDN_TREE_STATUS_BAD_TREE : GDN_TREE_STATUS_OK;
  if (bad) return;

  // ---- 2. TMEM, barriers, TMA of K and Q --------------------------------------
  if (warp == 0) tmem_alloc(&S.tmem_base, kTmemCols);
  if (tid == 32) {
    mbar_init(&S.bar_tma, 1);
    mbar_init(&S.bar_mma, 1);
    mbar_fence_init();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = S.tmem_base;
  if (tid == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmQ);
    mbar_arrive_expect_tx(&S.bar_tma, 4 * kTileBytes);
    tma_load_4d(smem + OFF_K, &tmK, &S.bar_tma, 0, hq, 0, b);
    tma_load_4d(smem + OFF_K + kTileBytes, &tmK, &S.bar_tma, 64, hq, 0, b);
    tma_load_4d(smem + OFF_Q, &tmQ, &S.bar_tma, 0, hq, 0, b);
    tma_load_4d(smem + OFF_Q + kTileBytes, &tmQ, &S.bar_tma, 64, hq, 0, b);
  }

  // ---- 3. ancestor bitsets, path log-decays, depth levels -----------------------
  tree_prepare(S.parent, kTile, kW, S.la, S.jump, S.anc, S.g);
  int my_depth = 0;
  if (tid < kTile + 2) S.level_start[tid] = 0;
  if (tid < N) {
#pragma unroll
    for (int w = 0; w < kW; ++w) my_depth += __popc(S.anc[tid * kW + w]);
    my_depth += 1;
    S.depth[tid] = my_depth;
  }
  __syncthreads();
  if (tid < N) {
    atomicAdd(&S.level_start[my_depth], 1);
    atomicMax(&S.max_depth, my_depth);
  }
  __syncthreads();
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
  __syncthreads();
  if (tid < N) S.order[atomicAdd(&S.level_cursor[my_depth], 1)] = tid;

  // ---- S0^T = hi + lo (bf16, K-major, 128-byte swizzle) --------------------------
  {
    const float* S0bh = S0 + ((size_t)b * Hv + h) * kD * kD;
    for (int item = tid; item < kD * 16; item += kThreads) {
      const int n = item & (kD - 1), k8 = item >> 7;
      float x[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __ldg(S0bh + (size_t)(k8 * 8 + i) * kD + n);
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        __nv_bfloat16 h0, l0, h1, l1;
        split_bf16(x[2 * i], h0, l0);
        split_bf16(x[2 * i + 1], h1, l1);
        hi[i] = pack2(h0, h1);
        lo[i] = pack2(l0, l1);
      }
      const uint32_t off = sw128_chunk(n, k8);
      *reinterpret_cast<uint4*>(smem + OFF_S0H + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + OFF_S0L + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  // ---- 4. Gram, K S0, Q S0 on the tensor cores --------------------------------
  if (tid == 0) {
    if (!mbar_wait(&S.bar_tma, 0, kWaitLimitNs)) {
      S.err = 1;
    } else {
      tc_fence_after_sync();
      umma_128x128x128(tmem + kColGkk, sbase + OFF_K, sbase + OFF_K, false);
      umma_128x128x128(tmem + kColGqk, sbase + OFF_Q, sbase + OFF_K, false);
      umma_128x128x128(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0H, false);
      umma_128x128x128(tmem + kColKS, sbase + OFF_K, sbase + OFF_S0L, true);
      umma_128x128x128(tmem + kColQS, sbase + OFF_Q, sbase + OFF_S0H, false);
      umma_commit(&S.bar_mma);
    }
  }
  __syncthreads();
  if (S.err) goto fail;
  if (!mbar_wait(&S.bar_mma, 0, kWaitLimitNs)) S.err = 2;
  tc_fence_after_sync();
  if (__syncthreads_or(S.err)) goto fail;

  {
    // thread <-> (tree row t, column half): warp w reads TMEM lanes 32*(w%4)..
    const int q4 = warp & 3, half = warp >> 2;
    const int t = q4 * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(q4 * 32) << 16);
    const bool live = t < N;
    const float bt = live ? S.beta[t] : 0.f;
    const df gt = live ? S.g[t] : df{0.f, 0.f};
    const float gam = expf(df_value(gt));
    uint32_t anc[kW];
#pragma unroll
    for (int w = 0; w < kW; ++w) anc[w] = live ? S.anc[t * kW + w] : 0u;

    // ---- 5. X (masked, decay-weighted K K^T) and R ----------------------------
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col0 = half * 64 + c * 32;
      float gk[32];
      tmem_ld_32cols(trow + kColGkk + col0, gk);
      const uint32_t bits = anc[col0 >> 5];
      if (live) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if ((bits >> j) & 1u) {
            const int s = col0 + j;
            sX[t * kXStride + s] = bt * expf(df_diff(gt, S.g[s])) * gk[j];
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col0 = half * 64 + c * 32;
      float ks[32];
      tmem_ld_32cols(trow + kColKS + col0, ks);
      if (live) {
        const uint4* vrow = reinterpret_cast<const uint4*>(
            v + (((size_t)b * N + t) * Hv + h) * kD + col0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 raw = __ldg(vrow + q);
          const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
          float r[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float v0 = __uint_as_float(w4[e] << 16);
            const float v1 = __uint_as_float(w4[e] & 0xffff0000u);
            r[2 * e] = bt * (v0 - gam * ks[q * 8 + 2 * e]);
            r[2 * e + 1] = bt * (v1 - gam * ks[q * 8 + 2 * e + 1]);
          }
          const int c4 = (col0 >> 2) + q * 2;
          *reinterpret_cast<float4*>(sU + u_index(t, c4)) = make_float4(r[0], r[1], r[2], r[3]);
          *reinterpret_cast<float4*>(sU + u_index(t, c4 + 1)) =
              make_float4(r[4], r[5], r[6], r[7]);
        }
      }
    }
    tc_fence_before_sync();
    __syncthreads();

    // ---- 6. forward substitution, level by level -------------------------------
    const int max_depth = S.max_depth;
    for (int lvl = 2; lvl <= max_depth; ++lvl) {
      const int beg = S.level_start[lvl], end = S.level_start[lvl + 1];
      for (int i = beg + warp; i < end; i += kThreads / 32) {
        const int tn = S.order[i];
        float4 acc = *reinterpret_cast<const float4*>(sU + u_index(tn, lane));
#pragma unroll
        for (int w = 0; w < kW; ++w) {
          uint32_t bits = S.anc[tn * kW + w];
          while (bits) {
            const int s = w * 32 + __ffs(bits) - 1;
            bits &= bits - 1;
            const float x = sX[tn * kXStride + s];
            const float4 us = *reinterpret_cast<const float4*>(sU + u_index(s, lane));
            acc.x = fmaf(-x, us.x, acc.x);
            acc.y = fmaf(-x, us.y, acc.y);
            acc.z = fmaf(-x, us.z, acc.z);
            acc.w = fmaf(-x, us.w, acc.w);
          }
        }
        *reinterpret_cast<float4*>(sU + u_index(tn, lane)) = acc;
      }
      __syncthreads();
    }

    // ---- 7. U out; U^T and Y to shared memory as bf16 hi + lo -------------------
    for (int tn = warp; tn < N; tn += kThreads / 32) {
      const float4 u = *reinterpret_cast<const float4*>(sU + u_index(tn, lane));
      *reinterpret_cast<float4*>(U + (((size_t)b * Hv + h) * N + tn) * kD + lane * 4) = u;
    }
    for (int item = tid; item < kD * 16; item += kThreads) {
      const int n = item & (kD - 1), t8 = item >> 7;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float x0 = 0.f, x1 = 0.f;
        const int ta = t8 * 8 + 2 * i, tb = ta + 1;
        if (ta < N) x0 = sU[u_index(ta, n >> 2) + (n & 3)];
        if (tb < N) x1 = sU[u_index(tb, n >> 2) + (n & 3)];
        __nv_bfloat16 h0, l0, h1, l1;
        split_bf16(x0, h0, l0);
        split_bf16(x1, h1, l1);
        hi[i] = pack2(h0, h1);
        lo[i] = pack2(l0, l1);
      }
      const uint32_t off = sw128_chunk(n, t8);
      *reinterpret_cast<uint4*>(smem + OFF_UTH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + OFF_UTL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col0 = half * 64 + c * 32;
      float gq[32];
      tmem_ld_32cols(trow + kColGqk + col0, gq);
      const uint32_t bits = anc[col0 >> 5];
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
            y[e] = 0.f;
            if (live && (((bits >> j) & 1u) || s == t))
              y[e] = (s == t ? 1.f : expf(df_diff(gt, S.g[s]))) * gq[j];
          }
          __nv_bfloat16 h0, l0, h1, l1;
          split_bf16(y[0], h0, l0);
          split_bf16(y[1], h1, l1);
          hi[i] = pack2(h0, h1);
          lo[i] = pack2(l0, l1);
        }
        const uint32_t off = sw128_chunk(t, (col0 >> 3) + g8);
        *reinterpret_cast<uint4*>(smem + OFF_YH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + OFF_YL + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();

    // ---- 8. Y U on the tensor cores (three bf16 passes) ---------------------------
    if (tid == 0) {
      tc_fence_after_sync();
      umma_128x128x128(tmem + kColYU, sbase + OFF_YH, sbase + OFF_UTH, false);
      umma_128x128x128(tmem + kColYU, sbase + OFF_YH, sbase + OFF_UTL, true);
      umma_128x128x128(tmem + kColYU, sbase + OFF_YL, sbase + OFF_UTH, true);
      umma_commit(&S.bar_mma);
    }
    if (!mbar_wait(&S.bar_mma, 1, kWaitLimitNs)) S.err = 3;
    tc_fence_after_sync();
    if (__syncthreads_or(S.err)) goto fail;

    // ---- 9. O = gamma QS + Y U -------------------------------------------------------
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col0 = half * 64 + c * 32;
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
            w4[e] = pack2(__float2bfloat16_rn(fmaf(gam, qs[j], yu[j])),
                          __float2bfloat16_rn(fmaf(gam, qs[j + 1], yu[j + 1])));
          }
          orow[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  return;

fail:
  // a wait ran out: report, let in-flight copies / MMAs drain (bounded), free TMEM
  if (tid == 0) {
    if (dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_TIMEOUT);
    if (S.err == 1) mbar_wait(&S.bar_tma, 0, kWaitLimitNs);          // TMA still in flight
    if (S.err >= 2) mbar_wait(&S.bar_mma, S.err == 3 ? 1 : 0, kWaitLimitNs);  // MMAs
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
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

}  // namespace

bool verify_tc_supported(const gdn_tree_dims& d) {
  return d.dtype == GDN_TREE_BF16 && d.dk == kD && d.dv == kD && d.N >= 1 && d.N <= kTile &&
         tensor_map_encoder() != nullptr;
}

cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream) {
  CUtensorMap tmQ, tmK;
  if (!encode_qk_map(&tmQ, a.q, a.d) || !encode_qk_map(&tmK, a.k, a.d))
    return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(verify_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (err != cudaSuccess) return err;
  verify_tc_kernel<<<dim3(a.d.Hv, a.d.B), kThreads, kSmemBytes, stream>>>(
      tmQ, tmK, static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
      static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status);
  return cudaGetLastError();
}

}  // namespace gdn
