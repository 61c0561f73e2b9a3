// verify_long.cu -- tree verification for trees too long for the on-chip
// kernels (up to kMaxNLong nodes): a two-level chunk pass.
//
// Method: "DFlash-TfM: Trees from Marginals", section 3 ("Soluzione"): the
// masked unit-lower-triangular solve (I + X) U = R with
// R = diag(beta)(V - diag(gamma) K S0), and the output O = diag(gamma) Q S0 + Y U,
// where X[t,s] = beta_t e^{g_t - g_s} k_t.k_s for s a strict ancestor of t and
// Y[t,s] = e^{g_t - g_s} q_t.k_s for s on the root-to-t path (t included).
//
// The two levels.  The nodes are cut, in index (topological) order, into chunks
// of kChunk.  The U rows of the chunk in work stay in shared memory; the rows of
// earlier chunks are read back from the U output, which this CTA wrote before
// (a node's ancestors all have smaller indices, so they lie in its own chunk or
// an earlier one).  Within a chunk the nodes go level by level: every strict
// ancestor of a node is shallower, so the nodes of one level are independent and
// take one warp each.  A node's warp forms r_t and the output seed
// gamma_t (S0^T q_t) from the state in shared memory, then walks the root path
// once: for each ancestor s it forms X[t,s] and Y[t,s] from the k, q rows and
// applies u_t -= X[t,s] u_s, o_t += Y[t,s] u_s; the node's own term
// Y[t,t] u_t closes o_t.
//
// One CTA (512 threads) per (sequence b, v-head h); fp32 CUDA-core arithmetic
// for both dtypes.  The work is proportional to the sum of the node depths
// times d: a latency-bound kernel for the shapes the faster kernels leave.
#include <limits.h>

#include "common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 128;  // U rows kept in shared memory
constexpr int kNodesPerThread = kMaxNLong / kThreads;
static_assert(kMaxNLong % kThreads == 0, "pointer jumping assigns whole nodes per thread");
constexpr int kBatch = 4;  // ancestors whose rows are loaded together

struct LongSmem {
  // byte offsets into dynamic shared memory
  size_t S0, U, parent, jump, depth, g, rows, total;
};

__host__ __device__ inline size_t align16l(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline LongSmem long_smem_layout(int N, int dk, int dv) {
  LongSmem L;
  size_t o = 0;
  L.S0 = o;     o = align16l(o + sizeof(float) * dk * dv);
  L.U = o;      o = align16l(o + sizeof(float) * kChunk * dv);
  L.parent = o; o = align16l(o + sizeof(int) * N);
  L.jump = o;   o = align16l(o + sizeof(int) * N);
  L.depth = o;  o = align16l(o + sizeof(int) * N);
  L.g = o;      o = align16l(o + sizeof(df) * N);
  L.rows = o;   o = align16l(o + sizeof(float) * kWarps * 2 * kMaxD);
  L.total = o;
  return L;
}

// four consecutive elements as fp32 (16-byte fp32 or 8-byte bf16 loads)
__device__ __forceinline__ float4 load4(const float* p) {
  return *reinterpret_cast<const float4*>(p);
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float* p, float4 x) {
  *reinterpret_cast<float4*>(p) = x;
}
__device__ __forceinline__ void store4(__nv_bfloat16* p, float4 x) {
  __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
  uint2 raw;
  raw.x = *reinterpret_cast<uint32_t*>(&a);
  raw.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = raw;
}

__device__ __forceinline__ float dot4(float4 a, float4 b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

__device__ __forceinline__ void axpy4(float4& y, float a, float4 x) {
  y.x = fmaf(a, x.x, y.x);
  y.y = fmaf(a, x.y, y.y);
  y.z = fmaf(a, x.z, y.z);
  y.w = fmaf(a, x.w, y.w);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
verify_long_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                   const float* __restrict__ log_alpha, const float* __restrict__ beta,
                   const int32_t* __restrict__ parent, const float* __restrict__ S0,
                   T* __restrict__ o, float* U, gdn_tree_dims d, int32_t* dev_status,
                   SeqLayout lay) {
  // U is read back (earlier chunks' rows) after this CTA wrote it, so it is
  // neither const nor restrict: its loads must not take the read-only path.
  extern __shared__ __align__(16) unsigned char smem[];
  __shared__ int sLevelLo, sLevelHi;
  const int Nmax = d.N, dk = d.dk, dv = d.dv, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y;
  const int hq = h / (Hv / Hqk);
  const LongSmem L = long_smem_layout(Nmax, dk, dv);
  float* sS0 = reinterpret_cast<float*>(smem + L.S0);
  float* sU = reinterpret_cast<float*>(smem + L.U);
  int* sPar = reinterpret_cast<int*>(smem + L.parent);
  int* sJump = reinterpret_cast<int*>(smem + L.jump);
  int* sDepth = reinterpret_cast<int*>(smem + L.depth);
  df* sG = reinterpret_cast<df*>(smem + L.g);
  float* sRows = reinterpret_cast<float*>(smem + L.rows);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N < 0 || st < 0) {
    if (h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_LAYOUT);
    return;
  }
  const size_t row = (size_t)lay.row0(b, Nmax);
  const size_t urow = lay.urow0(b, h, Hv, Nmax);

  // ---- the tree: load, validate, seed the pointer jumping -----------------------
  int bad = 0;
  for (int t = tid; t < N; t += kThreads) {
    const int p = parent[row + t];
    sPar[t] = p;
    sJump[t] = p;
    sDepth[t] = 1;
    sG[t] = df{log_alpha[(row + t) * Hv + h], 0.f};
    bad |= (p < -1 || p >= t);
  }
  bad = __syncthreads_or(bad);
  if (bad && h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_TREE);
  if (bad) return;

  // ---- pointer jumping: g_t = sum of log alpha over P(t), depth_t = |P(t)| --------
  for (int span = 1; span < N; span <<= 1) {
    int j[kNodesPerThread], jj[kNodesPerThread], dj[kNodesPerThread];
    df gj[kNodesPerThread];
    int live = 0;
#pragma unroll
    for (int m = 0; m < kNodesPerThread; ++m) {
      const int t = tid + m * kThreads;
      j[m] = t < N ? sJump[t] : -1;
      if (j[m] >= 0) {
        jj[m] = sJump[j[m]];
        dj[m] = sDepth[j[m]];
        gj[m] = sG[j[m]];
        live = 1;
      }
    }
    if (!__syncthreads_or(live)) break;  // every node reached its root
#pragma unroll
    for (int m = 0; m < kNodesPerThread; ++m) {
      const int t = tid + m * kThreads;
      if (j[m] >= 0) {
        sG[t] = df_add(sG[t], gj[m]);
        sDepth[t] += dj[m];
        sJump[t] = jj[m];
      }
    }
    __syncthreads();
  }

  // ---- the state, fp32, into shared memory ----------------------------------------
  const float* S0bh = S0 + ((size_t)st * Hv + h) * dk * dv;
  for (int i = tid * 4; i < dk * dv; i += kThreads * 4)
    *reinterpret_cast<float4*>(sS0 + i) = *reinterpret_cast<const float4*>(S0bh + i);
  __syncthreads();

  const int c4 = lane * 4;  // this lane's elements of a k/q row and columns of a v/u row
  const bool kin = c4 < dk, vin = c4 < dv;
  float* myK = sRows + warp * 2 * kMaxD;
  float* myQ = myK + kMaxD;

  for (int c0 = 0; c0 < N; c0 += kChunk) {
    const int c1 = min(N, c0 + kChunk);
    // the chunk's depth range
    if (tid == 0) {
      sLevelLo = INT_MAX;
      sLevelHi = 0;
    }
    __syncthreads();
    if (tid < c1 - c0) {
      atomicMin(&sLevelLo, sDepth[c0 + tid]);
      atomicMax(&sLevelHi, sDepth[c0 + tid]);
    }
    __syncthreads();
    const int lvl_lo = sLevelLo, lvl_hi = sLevelHi;

    for (int lvl = lvl_lo; lvl <= lvl_hi; ++lvl) {
      for (int t = c0 + warp; t < c1; t += kWarps) {
        if (sDepth[t] != lvl) continue;  // uniform across the warp
        const size_t tk = ((row + t) * Hqk + hq) * dk;
        const float4 kt = kin ? load4(k + tk + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 qt = kin ? load4(q + tk + c4) : make_float4(0.f, 0.f, 0.f, 0.f);
        if (kin) {
          store4(myK + c4, kt);
          store4(myQ + c4, qt);
        }
        __syncwarp();
        const df gt = sG[t];
        const float gam = expf(df_value(gt));
        const float bt = beta[(row + t) * Hv + h];
        // S0^T k_t and S0^T q_t at this lane's columns
        float4 sk = make_float4(0.f, 0.f, 0.f, 0.f), sq = sk;
        if (vin) {
          for (int i = 0; i < dk; ++i) {
            const float4 s = *reinterpret_cast<const float4*>(sS0 + i * dv + c4);
            axpy4(sk, myK[i], s);
            axpy4(sq, myQ[i], s);
          }
        }
        const float4 vt = vin ? load4(v + ((row + t) * Hv + h) * dv + c4)
                              : make_float4(0.f, 0.f, 0.f, 0.f);
        // r_t = beta_t (v_t - gamma_t S0^T k_t); the output seed gamma_t S0^T q_t
        float4 u = make_float4(bt * (vt.x - gam * sk.x), bt * (vt.y - gam * sk.y),
                               bt * (vt.z - gam * sk.z), bt * (vt.w - gam * sk.w));
        float4 oc = make_float4(gam * sq.x, gam * sq.y, gam * sq.z, gam * sq.w);

        // the strict ancestors, parent first, kBatch at a time
        int s = sPar[t];
        while (s >= 0) {
          int a[kBatch];
#pragma unroll
          for (int e = 0; e < kBatch; ++e) {
            a[e] = s;
            if (s >= 0) s = sPar[s];
          }
          float4 ka[kBatch], ua[kBatch];
          float xk[kBatch], yq[kBatch];
#pragma unroll
          for (int e = 0; e < kBatch; ++e) {
            ka[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            ua[e] = ka[e];
            if (a[e] >= 0) {
              if (kin) ka[e] = load4(k + ((row + a[e]) * Hqk + hq) * dk + c4);
              if (vin)
                ua[e] = a[e] >= c0 ? *reinterpret_cast<const float4*>(sU + (a[e] - c0) * dv + c4)
                                   : *reinterpret_cast<const float4*>(U + (urow + a[e]) * dv + c4);
            }
          }
#pragma unroll
          for (int e = 0; e < kBatch; ++e) {
            xk[e] = dot4(kt, ka[e]);
            yq[e] = dot4(qt, ka[e]);
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1)
#pragma unroll
            for (int e = 0; e < kBatch; ++e) {
              xk[e] += __shfl_xor_sync(0xffffffffu, xk[e], off);
              yq[e] += __shfl_xor_sync(0xffffffffu, yq[e], off);
            }
#pragma unroll
          for (int e = 0; e < kBatch; ++e) {
            if (a[e] >= 0) {
              const float dec = expf(df_diff(gt, sG[a[e]]));
              axpy4(u, -(bt * dec * xk[e]), ua[e]);
              axpy4(oc, dec * yq[e], ua[e]);
            }
          }
        }
        // the node's own term Y[t,t] u_t = (q_t . k_t) u_t
        const float self = warp_sum(dot4(qt, kt));
        axpy4(oc, self, u);
        if (vin) {
          store4(sU + (t - c0) * dv + c4, u);
          store4(U + (urow + t) * dv + c4, u);
          store4(o + ((row + t) * Hv + h) * dv + c4, oc);
        }
        __syncwarp();  // myK / myQ are rewritten by the warp's next node
      }
      __syncthreads();  // this level's U rows are final for the next level
    }
  }
}

}  // namespace

size_t verify_long_smem_bytes(int N, int dk, int dv) {
  return long_smem_layout(N, dk, dv).total;
}

cudaError_t launch_verify_long(const VerifyArgs& a, cudaStream_t stream) {
  const size_t smem = verify_long_smem_bytes(a.d.N, a.d.dk, a.d.dv);
  const dim3 grid(a.d.Hv, a.d.B);
  cudaError_t err;
  if (a.d.dtype == GDN_TREE_BF16) {
    auto kern = verify_long_kernel<__nv_bfloat16>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    kern<<<grid, kThreads, smem, stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
        static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
        static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status, a.lay);
  } else {
    auto kern = verify_long_kernel<float>;
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
