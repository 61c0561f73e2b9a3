// verify_generic.cu -- tree verification for any supported shape and dtype
// (fp32 CUDA-core arithmetic).  Used for fp32 inputs and for shapes the
// tensor-core kernel does not take.
//
// Follows the chunked form of "DFlash-TfM: Trees from Marginals", section 3
// ("Soluzione"): ancestor bitsets and path log-decays from the topologically
// ordered tree, R = diag(beta)(V - diag(gamma) K S0), the masked unit-lower
// triangular solve (I + X) U = R by forward substitution over the nodes, and
// the output stage O = diag(gamma) Q S0 + Y U, with the masked, decay-weighted
// Gram entries X[t,s] and Y[t,s] formed on the fly from k_t . k_s and q_t . k_s.
//
// One CTA (256 threads) per (sequence b, v-head h).  S0 (dk x dv) and R/U
// (N x dv) live in shared memory; q/k/v rows are read from global (L2).
#include "common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

struct GenericSmem {
  // byte offsets into dynamic shared memory
  size_t S0, U, parent, jump, g, beta, la, anc, coef, list, part, rows, total;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline GenericSmem generic_smem_layout(int N, int dk, int dv) {
  GenericSmem L;
  const int W = (N + 31) / 32;
  size_t o = 0;
  L.S0 = o;     o = align16(o + sizeof(float) * dk * dv);
  L.U = o;      o = align16(o + sizeof(float) * N * dv);
  L.parent = o; o = align16(o + sizeof(int) * N);
  L.jump = o;   o = align16(o + sizeof(int) * N);
  L.g = o;      o = align16(o + sizeof(df) * N);
  L.beta = o;   o = align16(o + sizeof(float) * N);
  L.la = o;     o = align16(o + sizeof(float) * N);
  L.anc = o;    o = align16(o + sizeof(uint32_t) * N * W);
  L.coef = o;   o = align16(o + sizeof(float) * N);
  L.list = o;   o = align16(o + sizeof(int) * N);
  L.part = o;   o = align16(o + sizeof(float) * kThreads);
  L.rows = o;   o = align16(o + sizeof(float) * kWarps * (dk > dv ? dk : dv));
  L.total = o;
  return L;
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
verify_generic_kernel(const T* __restrict__ q, const T* __restrict__ k,
                      const T* __restrict__ v, const float* __restrict__ log_alpha,
                      const float* __restrict__ beta, const int32_t* __restrict__ parent,
                      const float* __restrict__ S0, T* __restrict__ o,
                      float* __restrict__ U, gdn_tree_dims d, int32_t* dev_status,
                      SeqLayout lay) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int Nmax = d.N, dk = d.dk, dv = d.dv, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y;
  const int hq = h / (Hv / Hqk);
  const int W = (Nmax + 31) / 32;
  const GenericSmem L = generic_smem_layout(Nmax, dk, dv);
  float* sS0 = reinterpret_cast<float*>(smem + L.S0);
  float* sU = reinterpret_cast<float*>(smem + L.U);
  int* sPar = reinterpret_cast<int*>(smem + L.parent);
  int* sJump = reinterpret_cast<int*>(smem + L.jump);
  df* sG = reinterpret_cast<df*>(smem + L.g);
  float* sBeta = reinterpret_cast<float*>(smem + L.beta);
  float* sLa = reinterpret_cast<float*>(smem + L.la);
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(smem + L.anc);
  float* sCoef = reinterpret_cast<float*>(smem + L.coef);
  int* sList = reinterpret_cast<int*>(smem + L.list);
  float* sPart = reinterpret_cast<float*>(smem + L.part);
  float* sRows = reinterpret_cast<float*>(smem + L.rows);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // this sequence's rows and state
  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N < 0 || st < 0) {
    if (h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_LAYOUT);
    return;
  }
  const size_t row = (size_t)lay.row0(b, Nmax);

  // ---- tree: load + validate -------------------------------------------
  int bad = 0;
  for (int t = tid; t < N; t += kThreads) {
    const int p = parent[row + t];
    sPar[t] = p;
    bad |= (p < -1 || p >= t);
    sBeta[t] = beta[(row + t) * Hv + h];
    sLa[t] = log_alpha[(row + t) * Hv + h];
  }
  bad = __syncthreads_or(bad);
  if (bad && h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_TREE);
  if (bad) return;

  tree_prepare(sPar, N, W, sLa, sJump, sAnc, sG);

  // ---- S0 tile into shared memory ----------------------------------------
  const float* S0bh = S0 + ((size_t)st * Hv + h) * dk * dv;
  for (int i = tid * 4; i < dk * dv; i += kThreads * 4)
    *reinterpret_cast<float4*>(sS0 + i) = *reinterpret_cast<const float4*>(S0bh + i);
  __syncthreads();

  const int ncol = (dv + 31) / 32;  // columns per lane: c = lane + 32 m
  float* myRow = sRows + warp * (dk > dv ? dk : dv);

  // ---- R = diag(beta) (V - diag(gamma) K S0), one warp per node ----------
  for (int t = warp; t < N; t += kWarps) {
    const T* kt = k + ((row + t) * Hqk + hq) * dk;
    for (int i = lane; i < dk; i += 32) myRow[i] = to_f32(kt[i]);
    __syncwarp();
    const float gam = expf(df_value(sG[t]));
    const float bt = sBeta[t];
    const T* vt = v + ((row + t) * Hv + h) * dv;
    for (int m = 0; m < ncol; ++m) {
      const int c = lane + 32 * m;
      if (c < dv) {
        float acc = 0.f;
        for (int i = 0; i < dk; ++i) acc = fmaf(myRow[i], sS0[i * dv + c], acc);
        sU[t * dv + c] = bt * (to_f32(vt[c]) - gam * acc);
      }
    }
    __syncwarp();
  }
  __syncthreads();

  // ---- forward substitution: u_t = r_t - sum_{s in anc(t)} X[t,s] u_s ----
  const int ngrp = kThreads / dv;  // dv divides 256 for every supported dv
  for (int t = 1; t < N; ++t) {
    // enumerate ancestors (same order in every thread)
    int nA = 0;
    for (int i = 0; i < W; ++i) nA += __popc(sAnc[t * W + i]);
    if (nA == 0) continue;  // uniform across the block
    if (tid < 32) {
      int base = 0;
      for (int i = 0; i < W; ++i) {
        uint32_t bits = sAnc[t * W + i];
        const int cnt = __popc(bits);
        // lane l writes the l-th set bit of this word
        if (lane < cnt) {
          uint32_t bb = bits;
          for (int r = 0; r < lane; ++r) bb &= bb - 1;
          sList[base + lane] = i * 32 + (__ffs(bb) - 1);
        }
        base += cnt;
      }
    }
    __syncthreads();
    {
      const T* kt = k + ((row + t) * Hqk + hq) * dk;
      const float bt = sBeta[t];
      const df gt = sG[t];
      for (int idx = warp; idx < nA; idx += kWarps) {
        const int s = sList[idx];
        const T* ks = k + ((row + s) * Hqk + hq) * dk;
        float part = 0.f;
        for (int i = lane; i < dk; i += 32) part = fmaf(to_f32(kt[i]), to_f32(ks[i]), part);
        part = warp_sum(part);
        if (lane == 0) sCoef[idx] = bt * expf(df_diff(gt, sG[s])) * part;
      }
    }
    __syncthreads();
    {
      const int grp = tid / dv, c = tid % dv;
      if (grp < ngrp) {
        float acc = 0.f;
        for (int idx = grp; idx < nA; idx += ngrp) acc = fmaf(sCoef[idx], sU[sList[idx] * dv + c], acc);
        sPart[grp * dv + c] = acc;
      }
    }
    __syncthreads();
    if (tid < dv) {
      float acc = 0.f;
      for (int g = 0; g < ngrp; ++g) acc += sPart[g * dv + tid];
      sU[t * dv + tid] -= acc;
    }
    __syncthreads();
  }

  // ---- outputs: o_t = gamma_t S0^T q_t + sum_{s in P(t)} Y[t,s] u_s --------
  for (int t = warp; t < N; t += kWarps) {
    const T* qt = q + ((row + t) * Hqk + hq) * dk;
    for (int i = lane; i < dk; i += 32) myRow[i] = to_f32(qt[i]);
    __syncwarp();
    const df gt = sG[t];
    const float gam = expf(df_value(gt));
    float acc[kMaxD / 32];
#pragma unroll
    for (int m = 0; m < kMaxD / 32; ++m) acc[m] = 0.f;
#pragma unroll
    for (int m = 0; m < kMaxD / 32; ++m) {
      const int c = lane + 32 * m;
      if (m < ncol && c < dv) {
        float a = 0.f;
        for (int i = 0; i < dk; ++i) a = fmaf(myRow[i], sS0[i * dv + c], a);
        acc[m] = gam * a;
      }
    }
    // ancestors in bitset order, then t itself
    for (int i = 0; i <= W; ++i) {
      uint32_t bits = i < W ? sAnc[t * W + i] : 0u;
      const bool self = (i == W);
      while (bits || self) {
        int s;
        if (self) {
          s = t;
        } else {
          s = i * 32 + __ffs(bits) - 1;
          bits &= bits - 1;
        }
        const T* ks = k + ((row + s) * Hqk + hq) * dk;
        float part = 0.f;
        for (int e = lane; e < dk; e += 32) part = fmaf(myRow[e], to_f32(ks[e]), part);
        part = warp_sum(part);
        const float y = (s == t ? 1.f : expf(df_diff(gt, sG[s]))) * part;
#pragma unroll
        for (int m = 0; m < kMaxD / 32; ++m) {
          const int c = lane + 32 * m;
          if (m < ncol && c < dv) acc[m] = fmaf(y, sU[s * dv + c], acc[m]);
        }
        if (self) break;
      }
    }
    T* ot = o + ((row + t) * Hv + h) * dv;
    float* Ut = U + (lay.urow0(b, h, Hv, Nmax) + t) * dv;
#pragma unroll
    for (int m = 0; m < kMaxD / 32; ++m) {
      const int c = lane + 32 * m;
      if (m < ncol && c < dv) {
        ot[c] = from_f32<T>(acc[m]);
        Ut[c] = sU[t * dv + c];
      }
    }
    __syncwarp();
  }
}

}  // namespace

size_t verify_generic_smem_bytes(int N, int dk, int dv) {
  return generic_smem_layout(N, dk, dv).total;
}

cudaError_t launch_verify_generic(const VerifyArgs& a, cudaStream_t stream) {
  const size_t smem = verify_generic_smem_bytes(a.d.N, a.d.dk, a.d.dv);
  const dim3 grid(a.d.Hv, a.d.B);
  cudaError_t err;
  if (a.d.dtype == GDN_TREE_BF16) {
    auto kern = verify_generic_kernel<__nv_bfloat16>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
        static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
        static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status, a.lay);
  } else {
    auto kern = verify_generic_kernel<float>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, smem, stream>>>(
        static_cast<const float*>(a.q), static_cast<const float*>(a.k),
        static_cast<const float*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
        static_cast<float*>(a.o), a.U, a.d, a.dev_status, a.lay);
  }
  return cudaGetLastError();
}

}  // namespace gdn
