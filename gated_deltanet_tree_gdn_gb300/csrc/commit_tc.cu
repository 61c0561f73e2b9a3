// commit_tc.cu -- the delayed state commitment on the tensor cores (bf16 k,
// dk = dv = 128).
//
// "DFlash-TfM: Trees from Marginals", section 3: once the accepted branch
// p_1 .. p_L is known, the state it reaches is
//     S1 = gamma_L S0 + K_P^T diag(w) U_P,
//     w_j = exp(G_L - G_j),  gamma_L = exp(G_L),  G_j = sum_{i<=j} log alpha_{p_i},
// a rank-L update of S0.  Here K_P^T diag(w) U_P is a tcgen05 MMA (M = dk rows of
// the state, N = dv columns, K = path entries, 32 a chunk): the path's k rows as
// they lie in memory are the A operand read MN-major (exact in bf16), and w U,
// split hi + lo in bf16, the B operand, MN-major (two MMAs; the split carries w U
// to ~2^-17).
//
// One CTA (four warps) per (b, h) state, two CTAs an SM (128 TMEM columns
// each):
//  - the state tile streams in by TMA (four 32-column boxes, 128-byte swizzle)
//    the moment the CTA starts;
//  - warp 0 takes the path meanwhile: its entries and length; with the entries
//    in range, their log alpha and parent links (the first 256 entries in one
//    round trip); the chain check; the double-float prefix sums G_j and the
//    weights;
//  - per chunk of 32 entries, every thread stages k rows (cp.async) and U rows,
//    then w U as hi + lo; one thread issues the MMAs into TMEM;
//  - thread = state row: S1 = gamma S0 + D, read from TMEM, in place in the
//    tile, which leaves by TMA store.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace gdn {

namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kThreads = 128;
constexpr int kChunk = 32;  // path entries per MMA chunk
constexpr int kPre = 8;     // 32-entry groups of a path whose entries come together
constexpr uint32_t kTmemCols = 128;

// dynamic shared memory, from a 1024-byte aligned base
constexpr uint32_t OFF_ST = 0;                      // the state tile (4 boxes, 64 KB)
constexpr uint32_t OFF_A = 4 * kBoxBytes;           // k rows, MN-major bf16 (8 KB)
constexpr uint32_t OFF_BH = OFF_A + kChunk * kD * 2;   // w U hi
constexpr uint32_t OFF_BL = OFF_BH + kChunk * kD * 2;  // w U lo
constexpr uint32_t OFF_UR = OFF_BL + kChunk * kD * 2;  // U rows as they are (fp32)
constexpr uint32_t OFF_PATH = OFF_UR + kChunk * kD * 4;  // entries, G hi / w, G lo [cap]

__host__ __device__ inline int path_cap(int Lmax) { return Lmax <= 256 ? 256 : (Lmax + 31) / 32 * 32; }
__host__ __device__ inline size_t commit_tc_smem(int Lmax) {
  return OFF_PATH + 12u * (size_t)path_cap(Lmax) + 1024;  // + alignment slack
}

__device__ __forceinline__ void cp_async16c(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}

// inclusive double-float prefix sum of v across the warp's lanes
__device__ __forceinline__ df warp_scan_df(df v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    df up;
    up.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
    up.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
    if (lane >= o) v = df_add(v, up);
  }
  return v;
}

__global__ void __launch_bounds__(kThreads, 2)
commit_tc_kernel(const __grid_constant__ CUtensorMap tmS, const __grid_constant__ CUtensorMap tmS1,
                 const int32_t* __restrict__ path, const int32_t* __restrict__ path_len,
                 const int32_t* __restrict__ parent, const float* __restrict__ U,
                 const __nv_bfloat16* __restrict__ k, const float* __restrict__ log_alpha,
                 gdn_tree_dims d, int32_t Lmax, int32_t* dev_status, SeqLayout lay,
                 WaitHooks hk) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  __shared__ uint64_t bar_s, bar_m;
  __shared__ uint32_t s_tmem;
  __shared__ float s_gamma;
  __shared__ int s_bad, s_len;

  const int Nmax = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int unit = blockIdx.x, b = unit / Hv, h = unit - b * Hv, hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint64_t limit = hk.limit_ns;
  const int cap = path_cap(Lmax);
  int* s_pj = reinterpret_cast<int*>(smem + OFF_PATH);
  float* s_w = reinterpret_cast<float*>(s_pj + cap);  // G_j.hi, then w_j
  float* s_lo = s_w + cap;                             // G_j.lo

  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N < 0 || st < 0) {
    if (tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_LAYOUT);
    return;
  }
  const size_t row = (size_t)lay.row0(b, Nmax), urow = lay.urow0(b, h, Hv, Nmax);
  const int su = st * Hv + h;

  // ---- the state tile starts coming; TMEM for the update --------------------------
  if (tid == 0) {
    mbar_init(&bar_s, 1);
    mbar_init(&bar_m, 1);
    mbar_fence_init();
    mbar_arrive_expect_tx(&bar_s, 4 * kBoxBytes);
    if (b != hk.withhold_copy_seq) {
#pragma unroll
      for (int c = 0; c < 4; ++c) tma_load_3d(smem + OFF_ST + c * kBoxBytes, &tmS, &bar_s, 32 * c, 0, su);
    }
  }
  if (warp == 0) tmem_alloc(&s_tmem, kTmemCols);

  // ---- warp 0: the path, its checks and weights -------------------------------
  if (warp == 0) {
    const int L = path_len[b];
    int bad = (L < 0 || L > N || L > Lmax);
    const int nL = bad ? 0 : L;
    int pjr[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const int e = 32 * i + lane;
      pjr[i] = e < nL ? path[(size_t)b * Lmax + e] : 0;
    }
    {
      int oor = 0;
#pragma unroll
      for (int i = 0; i < kPre; ++i) oor |= (32 * i + lane < nL) && (pjr[i] < 0 || pjr[i] >= N);
      if (__any_sync(0xffffffffu, oor)) bad = 1;
    }
    const int nLc = bad ? 0 : nL;
    float lar[kPre];
    int parr[kPre];
#pragma unroll
    for (int i = 0; i < kPre; ++i) {
      const int e = 32 * i + lane;
      lar[i] = 0.f;
      parr[i] = -1;
      if (e < nLc) {
        s_pj[e] = pjr[i];
        lar[i] = log_alpha[(row + pjr[i]) * Hv + h];
        if (parent) parr[i] = parent[row + pjr[i]];
      }
    }
    // a root-to-node path is strictly increasing in a topological order and, with
    // the tree given, follows the parent links; G_j by a double-float scan
    df carry = {0.f, 0.f};
    int last = -1;
    for (int c0 = 0; c0 < nLc; c0 += 32) {
      const int e = c0 + lane, ci = c0 >> 5;
      const bool live = e < nLc;
      int pj = 0, par = -1;
      float la = 0.f;
#pragma unroll
      for (int i = 0; i < kPre; ++i)
        if (i == ci) {
          pj = pjr[i];
          la = lar[i];
          par = parr[i];
        }
      if (ci >= kPre) {  // past the first 256 entries: fetched as reached
        pj = live ? path[(size_t)b * Lmax + e] : 0;
        if (__any_sync(0xffffffffu, live && (pj < 0 || pj >= N))) {
          bad = 1;
          break;
        }
        if (live) {
          s_pj[e] = pj;
          la = log_alpha[(row + pj) * Hv + h];
          if (parent) par = parent[row + pj];
        }
      }
      int prev = __shfl_up_sync(0xffffffffu, pj, 1);
      if (lane == 0) prev = last;
      if (__any_sync(0xffffffffu,
                     live && ((e > 0 && pj <= prev) || (parent != nullptr && par != prev)))) {
        bad = 1;
        break;
      }
      const df G = df_add(carry, warp_scan_df(df{live ? la : 0.f, 0.f}, lane));
      if (live) {
        s_w[e] = G.hi;
        s_lo[e] = G.lo;
      }
      carry.hi = __shfl_sync(0xffffffffu, G.hi, 31);
      carry.lo = __shfl_sync(0xffffffffu, G.lo, 31);
      last = __shfl_sync(0xffffffffu, pj, 31);
    }
    if (!bad)
      for (int e = lane; e < nLc; e += 32) s_w[e] = expf(df_diff(carry, df{s_w[e], s_lo[e]}));
    if (lane == 0) {
      s_bad = bad;
      s_len = bad ? 0 : nLc;
      s_gamma = expf(df_value(carry));
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = s_tmem;
  const int L = s_len;
  bool ok = true;

  if (s_bad) {
    if (tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_PATH);
  } else {
    // ---- D = K_P^T diag(w) U_P, 32 path entries a chunk ---------------------------
    const int nch = (L + kChunk - 1) / kChunk;
    for (int ch = 0; ch < nch; ++ch) {
      const int c0 = ch * kChunk, nj = min(kChunk, L - c0), nk = (nj + 15) & ~15;
      // the previous chunk's MMAs have read the tiles
      if (ch > 0 && !mbar_wait(&bar_m, (uint32_t)(ch - 1) & 1u, limit)) ok = false;
      for (int e = tid; e < nj * 16; e += kThreads) {
        const int jj = e >> 4, c = e & 15;
        cp_async16c(smem + OFF_A + mn_chunk(jj, c),
                    k + ((row + s_pj[c0 + jj]) * Hqk + hq) * kD + 8 * c);
      }
      for (int e = tid; e < nj * 32; e += kThreads) {
        const int jj = e >> 5, c = e & 31;
        cp_async16c(smem + OFF_UR + (jj * kD + 4 * c) * 4, U + (urow + s_pj[c0 + jj]) * kD + 4 * c);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      for (int e = tid; e < (nk - nj) * 16; e += kThreads) {  // padding rows
        const int jj = nj + (e >> 4), c = e & 15;
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(smem + OFF_A + mn_chunk(jj, c)) = z;
        *reinterpret_cast<uint4*>(smem + OFF_BH + mn_chunk(jj, c)) = z;
        *reinterpret_cast<uint4*>(smem + OFF_BL + mn_chunk(jj, c)) = z;
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      __syncthreads();
      for (int e = tid; e < nj * 16; e += kThreads) {  // w U as hi + lo
        const int jj = e >> 4, c = e & 15;
        const float w = s_w[c0 + jj];
        const float4* src = reinterpret_cast<const float4*>(smem + OFF_UR + (jj * kD + 8 * c) * 4);
        const float4 u0 = src[0], u1 = src[1];
        uint32_t hi[4], lo[4];
        split2(w * u0.x, w * u0.y, hi[0], lo[0]);
        split2(w * u0.z, w * u0.w, hi[1], lo[1]);
        split2(w * u1.x, w * u1.y, hi[2], lo[2]);
        split2(w * u1.z, w * u1.w, hi[3], lo[3]);
        *reinterpret_cast<uint4*>(smem + OFF_BH + mn_chunk(jj, c)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(smem + OFF_BL + mn_chunk(jj, c)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after_sync();
        const uint32_t a = smem_addr(smem + OFF_A);
        umma_commit_rows(tmem, a, smem_addr(smem + OFF_BH), nk / 16, ch > 0);
        umma_commit_rows(tmem, a, smem_addr(smem + OFF_BL), nk / 16, true);
        umma_commit(&bar_m);
      }
    }
    if (nch > 0 && !mbar_wait(&bar_m, (uint32_t)(nch - 1) & 1u, limit)) ok = false;
    tc_fence_after_sync();

    // ---- S1 = gamma S0 + D, thread = state row, in place in the tile --------------
    if (!mbar_wait(&bar_s, 0, limit)) ok = false;
    if (__syncthreads_and(ok)) {
      const float gamma = s_gamma;
      const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
      for (int cc = 0; cc < 16; ++cc) {  // columns 8 cc .. 8 cc + 7
        float dd[8];
        if (L > 0) {
          tmem_ld_8cols(trow + 8 * cc, dd);  // warp-collective (L is CTA-uniform)
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) dd[e] = 0.f;
        }
        float4* p0 = reinterpret_cast<float4*>(smem + OFF_ST + u_off(tid, 2 * cc));
        float4* p1 = reinterpret_cast<float4*>(smem + OFF_ST + u_off(tid, 2 * cc + 1));
        const float4 a = *p0, c = *p1;
        *p0 = make_float4(fmaf(gamma, a.x, dd[0]), fmaf(gamma, a.y, dd[1]), fmaf(gamma, a.z, dd[2]),
                          fmaf(gamma, a.w, dd[3]));
        *p1 = make_float4(fmaf(gamma, c.x, dd[4]), fmaf(gamma, c.y, dd[5]), fmaf(gamma, c.z, dd[6]),
                          fmaf(gamma, c.w, dd[7]));
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tma_store_3d(&tmS1, smem + OFF_ST + c * kBoxBytes, 32 * c, 0, su);
        bulk_commit_group();
        bulk_wait_all();
      }
    } else if (tid == 0 && dev_status) {
      atomicMax(dev_status + b, GDN_TREE_STATUS_TIMEOUT);  // S1 left unwritten
    }
  }
  // the state copy and the last MMAs are drained (bounded) before the CTA leaves,
  // TMEM freed once every access to it is done
  if (tid == 0) {
    mbar_wait(&bar_s, 0, limit);
    const int nch = s_bad ? 0 : (L + kChunk - 1) / kChunk;
    if (nch > 0) mbar_wait(&bar_m, (uint32_t)(nch - 1) & 1u, limit);
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

bool commit_tc_supported(const gdn_tree_dims& d, int32_t Lmax) {
  return d.dtype == GDN_TREE_BF16 && d.dk == kD && d.dv == kD && Lmax <= 1024 &&
         (long long)d.B * d.Hv < (1ll << 30);
}

cudaError_t launch_commit_tc(const CommitArgs& a, cudaStream_t stream) {
  const long long units = (long long)a.d.B * a.d.Hv;
  if (units == 0) return cudaSuccess;
  const long long n_states = (long long)(a.lay.slot ? a.lay.n_slots : a.d.B) * a.d.Hv;
  CUtensorMap tmS, tmS1;
  if (!encode_state_map(&tmS, a.S0, n_states) || !encode_state_map(&tmS1, a.S1, n_states))
    return cudaErrorNotSupported;
  const size_t smem = commit_tc_smem(a.Lmax);
  cudaError_t err =
      cudaFuncSetAttribute(commit_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  commit_tc_kernel<<<(unsigned)units, kThreads, smem, stream>>>(
      tmS, tmS1, a.path, a.path_len, a.parent, a.U, static_cast<const __nv_bfloat16*>(a.k),
      a.log_alpha, a.d, a.Lmax, a.dev_status, a.lay, wait_hooks());
  return cudaGetLastError();
}

}  // namespace gdn
