// chain_unit.cuh -- the verification of one (sequence, v-head) unit whose tree is
// one chain (parent of node t is t - 1: the draft is a single branch), bf16 with
// dk = dv = 128, up to kMaxNLong nodes: the chunkwise form of the closed form,
// every product on the tensor cores.  The 256-node kernel and the chunk pass run
// it for their chain units (a CTA of 512 threads each).
//
// Method: "DFlash-TfM: Trees from Marginals", section 3 ("Soluzione"): with
// g_t the log-decay summed along the root-to-t path,
//   R = diag(beta)(V - diag(gamma) K S0),   (I + X) U = R,   O = diag(gamma) Q S0 + Y U,
//   X[t,s] = beta_t e^{g_t - g_s} k_t.k_s (s a strict ancestor of t),
//   Y[t,s] = e^{g_t - g_s} q_t.k_s (s on the root-to-t path).
// On a chain the ancestors of t are 0 .. t-1.  Cut into chunks of C = 64 nodes,
// with the state after the first c0 nodes
//   S_c = e^{g_{c0-1}} S0 + sum_{s < c0} e^{g_{c0-1} - g_s} k_s u_s^T     (g_{-1} = 0),
// the terms of earlier chunks fold into S_c (substitute S_c and the sums agree
// term by term):
//   u_t = beta_t (v_t - e^{g_t - g_{c0-1}} S_c^T k_t) - sum_{c0 <= s < t} X[t,s] u_s,
//   o_t = e^{g_t - g_{c0-1}} S_c^T q_t + sum_{c0 <= s <= t} Y[t,s] u_s,
//   S_{c+1} = e^{g_{c1-1} - g_{c0-1}} S_c + sum_{c0 <= s < c1} e^{g_{c1-1} - g_s} k_s u_s^T.
//
// Every product is transposed so that M = dv = 128 and TMEM lane j is v-column j:
//   P1 = S_c^T K_c^T and P2 = S_c^T Q_c^T   (S_c^T as bf16 hi + lo, two MMAs each),
//   GK = K_c K_c^T and GQ = Q_c K_c^T        (one MMA each; the A rows are K_c / Q_c
//                                             twice, so a row sits in both lane halves),
//   O_c^T    = e P2 + U_c^T Y_c^T              (U and Y as bf16 hi + lo, three MMAs),
//   S_{c+1}^T = decay S_c^T + (U_c^T diag(w)) K_c  (accumulated in TMEM in fp32; the
//                                               U operand as bf16 hi + lo).
// The substitution for u is blocked by 16 rows: a sub-block takes the earlier
// sub-blocks' terms as one product on CUDA cores (a thread per column and four
// rows), then solves among its rows in registers (a thread per column), X
// broadcast from shared memory.  S_{c+1}^T is read back, split into hi + lo and
// becomes the next chunk's operand.
#pragma once

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace gdn {
namespace chain {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kPerThread = kMaxNLong / kThreads;  // nodes a thread in the g scan
constexpr int kD = 128;
constexpr int kC = 64;          // chunk
constexpr int kXStride = 68;    // floats a row of X / Y (16-byte rows, float4 stores conflict free)
static_assert(kMaxNLong % kThreads == 0, "the g scan takes whole nodes a thread");

// shared memory, bytes from a 1024-byte aligned base
constexpr uint32_t OFF_ST = 0;                          // S_c^T hi, lo: K-major, 128 rows (dv) x 128 (dk)
constexpr uint32_t OFF_KT = OFF_ST + 2 * 128 * kD * 2;  // K_c, K-major, 128 rows (64 used)
constexpr uint32_t OFF_QT = OFF_KT + 128 * kD * 2;      // Q_c, the same
constexpr uint32_t OFF_KM = OFF_QT + 128 * kD * 2;      // K_c, MN-major (K = 64 nodes, N = dk)
constexpr uint32_t OFF_XY = OFF_KM + kC * kD * 2;       // X fp32 [64][68], Y hi, lo (K-major 64 x 64);
                                                        // later U^T diag(w) hi, lo
constexpr uint32_t OFF_YH = OFF_XY + kC * kXStride * 4; // Y hi (8 KB), then Y lo
constexpr uint32_t kXYBytes = kC * kXStride * 4 + 2 * kC * kC * 2;
constexpr uint32_t OFF_UC = OFF_XY + kXYBytes;          // the chunk's R, then U: fp32 [64][128]
constexpr uint32_t OFF_AUX = OFF_UC + kC * kD * 4;      // e_t, w_t [64] each; warp totals; flags
constexpr uint32_t OFF_TREE = OFF_AUX + 2048;           // g (df) [N], beta [N]
static_assert(2 * 128 * kC * 2 <= kXYBytes, "U^T diag(w) hi / lo fit where X and Y were");
static_assert(OFF_YH % 1024 == 0, "the Y operand tiles start on a 1024-byte boundary");

__host__ __device__ inline size_t smem_bytes(int N) {
  return OFF_TREE + (size_t)N * (sizeof(df) + sizeof(float)) + 1024;  // + alignment slack
}

// TMEM columns
constexpr uint32_t TM_P1 = 0, TM_P2 = 64, TM_GK = 128, TM_GQ = 192, TM_S = 256;
constexpr uint32_t kTmemCols = 512;

__device__ __forceinline__ void cp_async16c(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_addr(dst)),
               "l"(src)
               : "memory");
}

// D (+)= A B^T, M = 128, N = n, K = 16 ksteps, A and B K-major 128-byte-swizzled
// tiles of 128 rows (B's first n rows used)
__device__ __forceinline__ void umma_kmajor(uint32_t d_tmem, uint32_t a_base, uint32_t b_base,
                                            int n, int ksteps, bool accumulate) {
  const uint32_t idesc = sm100::idesc_bf16_f32(128, n);
  for (int s = 0; s < ksteps; ++s) {
    const uint32_t off = (uint32_t)((s >> 2) * sm100::kSw128TileBytes + (s & 3) * 32);
    sm100::umma_bf16(d_tmem, sm100::desc_sw128_kmajor(a_base + off),
                     sm100::desc_sw128_kmajor(b_base + off), idesc,
                     (accumulate || s > 0) ? 1u : 0u);
  }
}

// D += A B, M = N = 128, K = 64: A K-major (128 rows x 64), B MN-major (64 rows x 128)
__device__ __forceinline__ void umma_update(uint32_t d_tmem, uint32_t a_base, uint32_t b_base) {
  constexpr uint32_t idesc = sm100::idesc_bf16_f32_bmn(128, 128);
#pragma unroll
  for (int s = 0; s < kC / 16; ++s)
    sm100::umma_bf16(d_tmem, sm100::desc_sw128_kmajor(a_base + (uint32_t)s * 32),
                     sm100::desc_sw128_mnmajor(b_base + (uint32_t)s * 2 * sm100::kMnSbo,
                                               sm100::kMnLbo, sm100::kMnSbo),
                     idesc, 1u);
}

__device__ __forceinline__ float bf16_bits_to_f32(unsigned short x) {
  return __uint_as_float((uint32_t)x << 16);
}

// Whole CTA (kThreads threads): verifies unit (b, h) whose N-node tree is one chain.
// smem: the CTA's dynamic shared memory from a 1024-byte aligned base, at least
// smem_bytes(Nmax) long; Ubh: the unit's U rows.  Reports a timeout to dev_status.
__device__ __forceinline__ void run(unsigned char* smem, const __nv_bfloat16* __restrict__ q,
                                    const __nv_bfloat16* __restrict__ k,
                                    const __nv_bfloat16* __restrict__ v,
                                    const float* __restrict__ log_alpha,
                                    const float* __restrict__ beta, const float* __restrict__ S0,
                                    __nv_bfloat16* __restrict__ o, float* __restrict__ Ubh,
                                    int N, int Nmax, size_t row, int st, int b, int h, int Hv,
                                    int Hqk, int32_t* dev_status, const WaitHooks& hk) {
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // TMEM lane group (warp % 4: lanes / v-columns 32 g ..) and quarter (warp / 4)
  const int lg = warp & 3, qd = warp >> 2;
  const int j = 32 * lg + lane;  // this thread's v-column in the column-parallel phases
  float* sX = reinterpret_cast<float*>(smem + OFF_XY);
  float* sUc = reinterpret_cast<float*>(smem + OFF_UC);  // the chunk's rows [t][128]
  float* sE = reinterpret_cast<float*>(smem + OFF_AUX);  // e^{g_t - g_{c0-1}}
  float* sW = sE + kC;                                    // e^{g_{c1-1} - g_t}
  df* sWarpTot = reinterpret_cast<df*>(sW + kC);          // [kWarps]
  int* sFlag = reinterpret_cast<int*>(sWarpTot + kWarps); // [0] status flag, [1] TMEM base
  uint64_t* sBar = reinterpret_cast<uint64_t*>(sFlag + 2);
  df* sG = reinterpret_cast<df*>(smem + OFF_TREE);
  float* sBeta = reinterpret_cast<float*>(sG + Nmax);

  // ---- g by a blocked scan (kPerThread nodes a thread, df sums), beta ---------------
  {
    df loc[kPerThread];
    df run = {0.f, 0.f};
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const int t = kPerThread * tid + i;
      const df x = {t < N ? log_alpha[(row + t) * Hv + h] : 0.f, 0.f};
      run = df_add(run, x);
      loc[i] = run;
      if (t < N) sBeta[t] = beta[(row + t) * Hv + h];
    }
    df inc = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const df y = {__shfl_up_sync(0xffffffffu, inc.hi, off), __shfl_up_sync(0xffffffffu, inc.lo, off)};
      if (lane >= off) inc = df_add(y, inc);
    }
    if (lane == 31) sWarpTot[warp] = inc;
    if (tid == 0) sFlag[0] = 0;
    if (tid == 0) sm100::mbar_init(sBar, 1);
    sm100::mbar_fence_init();
    __syncthreads();
    df base = {0.f, 0.f};
    for (int w = 0; w < warp; ++w) base = df_add(base, sWarpTot[w]);
    const df ex = {__shfl_up_sync(0xffffffffu, inc.hi, 1), __shfl_up_sync(0xffffffffu, inc.lo, 1)};
    if (lane > 0) base = df_add(base, ex);
#pragma unroll
    for (int i = 0; i < kPerThread; ++i) {
      const int t = kPerThread * tid + i;
      if (t < N) sG[t] = df_add(base, loc[i]);
    }
  }
  if (warp == 0) sm100::tmem_alloc(reinterpret_cast<uint32_t*>(sFlag + 1), kTmemCols);

  // the chunk's K and Q tiles (K-major) and its K tile (MN-major)
  auto load_tiles = [&](int c0, bool kq, bool km) {
    const int nc = min(kC, N - c0);
    for (int e = tid; e < kC * 16; e += kThreads) {
      const int r = e >> 4, ch = e & 15;
      if (r < nc) {
        const size_t src = ((row + c0 + r) * Hqk + hq) * kD + 8 * ch;
        if (kq) {  // rows r and r + 64: the Grams' rows land in both TMEM lane halves
          cp_async16c(smem + OFF_KT + sm100::sw128_chunk(r, ch), k + src);
          cp_async16c(smem + OFF_QT + sm100::sw128_chunk(r, ch), q + src);
          cp_async16c(smem + OFF_KT + sm100::sw128_chunk(r + kC, ch), k + src);
          cp_async16c(smem + OFF_QT + sm100::sw128_chunk(r + kC, ch), q + src);
        }
        if (km) cp_async16c(smem + OFF_KM + sm100::mn_chunk(r, ch), k + src);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  load_tiles(0, true, true);

  sm100::tc_fence_before_sync();
  __syncthreads();
  sm100::tc_fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(sFlag[1]);
  const uint32_t tl = tmem + ((uint32_t)(lg * 32) << 16);  // this warp's TMEM lanes

  // ---- S0^T into TMEM (fp32) and into the operand tile (bf16 hi + lo) ---------------
  // thread: row j of S^T, columns 32 qd .. 32 qd + 31
  auto st_to_operand = [&](const float (&col)[32]) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sm100::split2(col[8 * c8 + 2 * e], col[8 * c8 + 2 * e + 1], hi[e], lo[e]);
      const uint32_t off = sm100::sw128_chunk(j, 4 * qd + c8);
      *reinterpret_cast<uint4*>(smem + OFF_ST + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + OFF_ST + 32768 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  };
  {
    const float* s0 = S0 + ((size_t)st * Hv + h) * kD * kD + j;  // column j of S0
    float col[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) col[i] = s0[(size_t)(32 * qd + i) * kD];
    sm100::tmem_st_32cols(tl + TM_S + 32 * qd, col);
    st_to_operand(col);
  }

  bool timed_out = false;
  uint32_t phase = 0;
  auto wait_mma = [&]() {
    if (!sm100::mbar_wait(sBar, phase, hk.limit_ns)) {
      // (bounded again: the MMAs must be done before TMEM or their operands are reused)
      sm100::mbar_wait(sBar, phase, hk.limit_ns);
      timed_out = true;
    }
    phase ^= 1u;
    sm100::tc_fence_after_sync();
  };
  const uint32_t aST = sm100::smem_addr(smem + OFF_ST), aKT = sm100::smem_addr(smem + OFF_KT),
                 aQT = sm100::smem_addr(smem + OFF_QT), aKM = sm100::smem_addr(smem + OFF_KM),
                 aXY = sm100::smem_addr(smem + OFF_XY);
  const int nchunks = (N + kC - 1) / kC;
  const unsigned short* vb = reinterpret_cast<const unsigned short*>(v);
  unsigned short* ob = reinterpret_cast<unsigned short*>(o);
  // v[t][j] for this thread's 16 rows t = 16 qd + i of the chunk (the next chunk's
  // come during the output product)
  float vv[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int t = 16 * qd + i;
    vv[i] = t < min(kC, N) ? bf16_bits_to_f32(vb[((row + t) * Hv + h) * kD + j]) : 0.f;
  }

#pragma unroll 1
  for (int ci = 0; ci < nchunks; ++ci) {
    const int c0 = ci * kC, nc = min(kC, N - c0);
    const bool last = ci + 1 == nchunks;
    const df gref = c0 > 0 ? sG[c0 - 1] : df{0.f, 0.f};
    // ---- the products: P1, P2 (with S_c^T), GK, GQ ----------------------------------
    asm volatile("cp.async.wait_all;" ::: "memory");
    sm100::fence_proxy_async_smem();
    sm100::tc_fence_before_sync();
    __syncthreads();
    sm100::tc_fence_after_sync();
    if (tid == 0) {
      umma_kmajor(tmem + TM_P1, aST, aKT, kC, 8, false);
      umma_kmajor(tmem + TM_P1, aST + 32768, aKT, kC, 8, true);
      umma_kmajor(tmem + TM_P2, aST, aQT, kC, 8, false);
      umma_kmajor(tmem + TM_P2, aST + 32768, aQT, kC, 8, true);
      umma_kmajor(tmem + TM_GK, aKT, aKT, kC, 8, false);
      umma_kmajor(tmem + TM_GQ, aQT, aKT, kC, 8, false);
      sm100::umma_commit(sBar);
    }
    wait_mma();
    // the next chunk's K and Q tiles (these products have read the current ones)
    if (!last) load_tiles(c0 + kC, true, false);

    // ---- e and w; X and Y: row t in TMEM lanes t and 64 + t, so that every warp
    // takes 8 of a row's 64 columns (part qd + 4 (lg / 2)) --------------------------
    if (tid < kC) {
      const int t = tid;
      const bool live = t < nc;
      sE[t] = live ? expf(df_diff(sG[c0 + t], gref)) : 0.f;
      sW[t] = live ? expf(df_diff(sG[c0 + nc - 1], sG[c0 + t])) : 0.f;
    }
    {
      const int t = 32 * (lg & 1) + lane, part = qd + 4 * (lg >> 1);
      const bool live = t < nc;
      const df gt = live ? sG[c0 + t] : df{0.f, 0.f};
      const float bt = live ? sBeta[c0 + t] : 0.f;
      float gk[8], gq[8];
      sm100::tmem_ld_8cols(tl + TM_GK + 8 * part, gk);
      sm100::tmem_ld_8cols(tl + TM_GQ + 8 * part, gq);
      float x[8], y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int s = 8 * part + e;
        x[e] = 0.f;
        y[e] = 0.f;
        if (live && s <= t) {
          const float dec = s == t ? 1.f : expf(df_diff(gt, sG[c0 + s]));
          y[e] = dec * gq[e];
          if (s < t) x[e] = bt * dec * gk[e];
        }
      }
      float* xr = sX + t * kXStride + 8 * part;
      *reinterpret_cast<float4*>(xr) = make_float4(x[0], x[1], x[2], x[3]);
      *reinterpret_cast<float4*>(xr + 4) = make_float4(x[4], x[5], x[6], x[7]);
      // Y as the output product's B operand: row t, chunk part, bf16 hi + lo
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sm100::split2(y[2 * e], y[2 * e + 1], hi[e], lo[e]);
      const uint32_t off = sm100::sw128_chunk(t, part);
      *reinterpret_cast<uint4*>(smem + OFF_YH + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + OFF_YH + kC * 128 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    __syncthreads();  // X, Y, e, w in shared memory
    // ---- r_t = beta_t (v_t - e_t P1[j][t]) for rows t = 16 qd + i ------------------
    {
      float p1[16];
      sm100::tmem_ld_16cols(tl + TM_P1 + 16 * qd, p1);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = 16 * qd + i;
        sUc[t * kD + j] = t < nc ? sBeta[c0 + t] * (vv[i] - sE[t] * p1[i]) : 0.f;
      }
    }
    // S_c^T *= e^{g_{c1-1} - g_{c0-1}} in TMEM, ahead of the update's accumulation (the
    // chunk's products read the operand copy, not TMEM)
    if (!last) {
      const float decay = expf(df_diff(sG[c0 + nc - 1], gref));
      float sv[32];
      sm100::tmem_ld_32cols(tl + TM_S + 32 * qd, sv);
#pragma unroll
      for (int i = 0; i < 32; ++i) sv[i] *= decay;
      sm100::tmem_st_32cols(tl + TM_S + 32 * qd, sv);
    }
    __syncthreads();

    // ---- the substitution (I + X) U = R, blocked by 16 rows ------------------------
    // rows of sub-block sb take the earlier sub-blocks' terms as one product (thread:
    // column jc, rows 16 sb + 4 rq + i), then solve among themselves (threads 0..127,
    // a column each, the 16 rows in registers)
    const int jc = tid & (kD - 1), rq = tid >> 7;
#pragma unroll 1
    for (int sb = 0; sb < 4; ++sb) {
      const int r0 = 16 * sb;
      if (r0 >= nc) break;  // (uniform) rows past the tree stay zero
      if (sb > 0) {
        const int t0 = r0 + 4 * rq;
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
        for (int s4 = 0; s4 < r0 / 4; ++s4) {
          float us[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) us[e] = sUc[(4 * s4 + e) * kD + jc];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float4 x = *reinterpret_cast<const float4*>(sX + (t0 + i) * kXStride + 4 * s4);
            a[i] = fmaf(x.x, us[0], fmaf(x.y, us[1], fmaf(x.z, us[2], fmaf(x.w, us[3], a[i]))));
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) sUc[(t0 + i) * kD + jc] -= a[i];
        __syncthreads();
      }
      if (tid < kD) {
        float u[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = sUc[(r0 + i) * kD + jc];
#pragma unroll
        for (int i = 1; i < 16; ++i) {
          const float* xr = sX + (r0 + i) * kXStride + r0;
          float a0 = 0.f, a1 = 0.f;
#pragma unroll
          for (int s = 0; s < i; ++s) {
            if (s & 1) a1 = fmaf(xr[s], u[s], a1);
            else a0 = fmaf(xr[s], u[s], a0);
          }
          u[i] -= a0 + a1;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) sUc[(r0 + i) * kD + jc] = u[i];
      }
      __syncthreads();
    }

    // ---- O_c^T = e P2 + U_c^T Y_c^T and S_{c+1}^T = decay S_c^T + (U_c^T diag(w)) K_c
    // on the tensor cores, one round trip; the outputs -----------------------------
    // U_c^T and U_c^T diag(w) (bf16 hi + lo, K-major: row jc, entries 16 rq ..) go
    // where S_c^T's operand was (its products are done; it is rewritten below)
#pragma unroll
    for (int k8 = 2 * rq; k8 < 2 * rq + 2; ++k8) {
      float uu[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) uu[e] = sUc[(8 * k8 + e) * kD + jc];
      const uint32_t off = sm100::sw128_chunk(jc, k8);
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sm100::split2(uu[2 * e], uu[2 * e + 1], hi[e], lo[e]);
      *reinterpret_cast<uint4*>(smem + OFF_ST + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(smem + OFF_ST + 16384 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      if (!last) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          sm100::split2(uu[2 * e] * sW[8 * k8 + 2 * e], uu[2 * e + 1] * sW[8 * k8 + 2 * e + 1],
                        hi[e], lo[e]);
        *reinterpret_cast<uint4*>(smem + OFF_ST + 32768 + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + OFF_ST + 49152 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
    }
    sm100::fence_proxy_async_smem();
    sm100::tc_fence_before_sync();
    __syncthreads();
    sm100::tc_fence_after_sync();
    if (tid == 0) {
      const uint32_t aYH = sm100::smem_addr(smem + OFF_YH), aYL = aYH + kC * 128;
      umma_kmajor(tmem + TM_GK, aST, aYH, kC, kC / 16, false);
      umma_kmajor(tmem + TM_GK, aST, aYL, kC, kC / 16, true);
      umma_kmajor(tmem + TM_GK, aST + 16384, aYH, kC, kC / 16, true);
      if (!last) {
        umma_update(tmem + TM_S, aST + 32768, aKM);
        umma_update(tmem + TM_S, aST + 49152, aKM);
      }
      sm100::umma_commit(sBar);
    }
    // the next chunk's v values start coming meanwhile
    float vn[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int t = 16 * qd + i;
      vn[i] = (!last && t < min(kC, N - c0 - kC))
                  ? bf16_bits_to_f32(vb[((row + c0 + kC + t) * Hv + h) * kD + j])
                  : 0.f;
    }
    wait_mma();
    if (!last) load_tiles(c0 + kC, false, true);  // the next MN-major K tile (this one is read)
    {
      // thread: column j, rows 16 qd .. 16 qd + 15
      float pc[16], dc[16];
      sm100::tmem_ld_16cols(tl + TM_P2 + 16 * qd, pc);
      sm100::tmem_ld_16cols(tl + TM_GK + 16 * qd, dc);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int t = 16 * qd + i;
        if (t < nc) {
          const __nv_bfloat16 ov = __float2bfloat16_rn(fmaf(sE[t], pc[i], dc[i]));
          ob[((row + c0 + t) * Hv + h) * kD + j] = *reinterpret_cast<const unsigned short*>(&ov);
          Ubh[(size_t)(c0 + t) * kD + j] = sUc[t * kD + j];
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) vv[i] = vn[i];
    if (last) break;
    // S_{c+1}^T -> the operand tile
    {
      float sv[32];
      sm100::tmem_ld_32cols(tl + TM_S + 32 * qd, sv);
      st_to_operand(sv);
    }
  }
  if (timed_out) atomicOr(sFlag, 1);
  sm100::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && sFlag[0] && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_TIMEOUT);
}

}  // namespace chain
}  // namespace gdn
