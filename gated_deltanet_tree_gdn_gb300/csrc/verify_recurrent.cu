// verify_recurrent.cu -- the single-branch recurrent verification of a draft
// tree: the baseline the tree verification is measured against.
//
// Method: "DFlash-TfM: Trees from Marginals", results section ("Efficienza di
// Verifica"): the fused tree kernel is compared with verifying every branch by
// its own recurrent pass.  Reading taken here: one pass per root-to-leaf branch,
// each from its own copy of S0, stepping the GDN recurrence of section 3
// ("Sfida"),
//     u_t = beta_t (v_t - alpha_t S^T k_t),   S <- alpha_t S + k_t u_t^T,
//     o_t = S^T q_t,
// node by node; a node shared by several branches is recomputed by each of
// them (with identical operations, so with identical bits).
//
// Layout: one CTA (256 threads) per (node t, v-head h, sequence b); the CTA of a
// node that has a child returns at once, so one CTA per leaf does the work.  The
// branch state lives in registers: thread (r, c) = (tid & 7, tid >> 3) holds rows
// r, r + 8, ... (up to 16) and columns 4c .. 4c + 3, so the k^T S and S^T q
// reductions over rows stay within 8 lanes of a warp (three shuffles).  Every
// step is fp32; the node's k, q, v rows and gates are staged in shared memory,
// and the next node's are loaded while the current step computes.
#include <cuda_bf16.h>

#include "common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerThread = kMaxD / 8;  // 16

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
verify_recurrent_kernel(const T* __restrict__ q, const T* __restrict__ k,
                        const T* __restrict__ v, const float* __restrict__ log_alpha,
                        const float* __restrict__ beta, const int32_t* __restrict__ parent,
                        const float* __restrict__ S0, T* __restrict__ o, float* __restrict__ U,
                        gdn_tree_dims d, int32_t* dev_status) {
  __shared__ int s_path[kMaxN];
  __shared__ float s_k[kMaxD], s_q[kMaxD], s_v[kMaxD];
  __shared__ float s_gate[2];  // alpha, beta of the current node
  __shared__ int s_len;

  const int leaf = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int N = d.N, Hv = d.Hv, Hqk = d.Hqk, dk = d.dk, dv = d.dv;
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, r = tid & 7, c = tid >> 3;
  const int32_t* par = parent + (size_t)b * N;

  // the tree must be topologically ordered; the node must have no child
  int bad = 0, has_child = 0;
  for (int i = tid; i < N; i += kThreads) {
    const int p = par[i];
    bad |= (p < -1 || p >= i);
    has_child |= (p == leaf);
  }
  bad = __syncthreads_or(bad);
  if (bad && leaf == 0 && h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_TREE);
  if (bad || __syncthreads_or(has_child)) return;

  // the branch root -> leaf
  if (tid == 0) {
    int len = 0;
    for (int s = leaf; s >= 0; s = par[s]) ++len;
    int i = len;
    for (int s = leaf; s >= 0; s = par[s]) s_path[--i] = s;
    s_len = len;
  }

  // a fresh copy of S0 for this branch
  const bool col_ok = 4 * c < dv;
  float4 S[kRowsPerThread];
  const float* s0 = S0 + ((size_t)b * Hv + h) * dk * dv;
#pragma unroll
  for (int m = 0; m < kRowsPerThread; ++m) {
    const int row = r + 8 * m;
    S[m] = (col_ok && row < dk) ? *reinterpret_cast<const float4*>(s0 + (size_t)row * dv + 4 * c)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  __syncthreads();
  const int len = s_len;

  // this thread's share of a node's inputs: k[tid] and q[tid] (tid < dk), v[tid - 128]
  // (128 <= tid < 128 + dv); thread 0 also takes the gates alpha, beta
  auto load_node = [&](int t, float& x0, float& x1, float& ga, float& gb) {
    x0 = 0.f;
    x1 = 0.f;
    if (tid < dk) {
      x0 = to_f32(k[(((size_t)b * N + t) * Hqk + hq) * dk + tid]);
      x1 = to_f32(q[(((size_t)b * N + t) * Hqk + hq) * dk + tid]);
    } else if (tid >= 128 && tid - 128 < dv) {
      x0 = to_f32(v[(((size_t)b * N + t) * Hv + h) * dv + (tid - 128)]);
    }
    if (tid == 0) {
      ga = __expf(log_alpha[((size_t)b * N + t) * Hv + h]);
      gb = beta[((size_t)b * N + t) * Hv + h];
    }
  };
  float n0, n1, na = 0.f, nb = 0.f;
  load_node(s_path[0], n0, n1, na, nb);

  for (int i = 0; i < len; ++i) {
    const int t = s_path[i];
    if (tid < dk) {
      s_k[tid] = n0;
      s_q[tid] = n1;
    } else if (tid >= 128 && tid - 128 < dv) {
      s_v[tid - 128] = n0;
    }
    if (tid == 0) {
      s_gate[0] = na;
      s_gate[1] = nb;
    }
    __syncthreads();
    if (i + 1 < len) load_node(s_path[i + 1], n0, n1, na, nb);  // lands during this step
    const float al = s_gate[0], bt = s_gate[1];

    // k^T S over this thread's rows, then over the 8 lanes sharing its columns
    float4 ks = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) {
      const int row = r + 8 * m;
      const float kr = row < dk ? s_k[row] : 0.f;
      ks.x = fmaf(kr, S[m].x, ks.x);
      ks.y = fmaf(kr, S[m].y, ks.y);
      ks.z = fmaf(kr, S[m].z, ks.z);
      ks.w = fmaf(kr, S[m].w, ks.w);
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      ks.x += __shfl_xor_sync(0xffffffffu, ks.x, off);
      ks.y += __shfl_xor_sync(0xffffffffu, ks.y, off);
      ks.z += __shfl_xor_sync(0xffffffffu, ks.z, off);
      ks.w += __shfl_xor_sync(0xffffffffu, ks.w, off);
    }
    // u = beta (v - alpha S^T k);  S <- alpha S + k u^T;  o = S^T q
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col_ok) {
      u.x = bt * (s_v[4 * c] - al * ks.x);
      u.y = bt * (s_v[4 * c + 1] - al * ks.y);
      u.z = bt * (s_v[4 * c + 2] - al * ks.z);
      u.w = bt * (s_v[4 * c + 3] - al * ks.w);
    }
    const float2 aa = make_float2(al, al);
    const float2 u01 = make_float2(u.x, u.y), u23 = make_float2(u.z, u.w);
    float4 os = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int m = 0; m < kRowsPerThread; ++m) {
      const int row = r + 8 * m;
      const float kr = row < dk ? s_k[row] : 0.f;
      const float qr = row < dk ? s_q[row] : 0.f;
      const float2 kk = make_float2(kr, kr);
      const float2 lo = __ffma2_rn(kk, u01, __fmul2_rn(aa, make_float2(S[m].x, S[m].y)));
      const float2 hi = __ffma2_rn(kk, u23, __fmul2_rn(aa, make_float2(S[m].z, S[m].w)));
      S[m] = make_float4(lo.x, lo.y, hi.x, hi.y);
      os.x = fmaf(qr, S[m].x, os.x);
      os.y = fmaf(qr, S[m].y, os.y);
      os.z = fmaf(qr, S[m].z, os.z);
      os.w = fmaf(qr, S[m].w, os.w);
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      os.x += __shfl_xor_sync(0xffffffffu, os.x, off);
      os.y += __shfl_xor_sync(0xffffffffu, os.y, off);
      os.z += __shfl_xor_sync(0xffffffffu, os.z, off);
      os.w += __shfl_xor_sync(0xffffffffu, os.w, off);
    }
    if (r == 0 && col_ok) {
      *reinterpret_cast<float4*>(U + (((size_t)b * Hv + h) * N + t) * dv + 4 * c) = u;
      T* orow = o + (((size_t)b * N + t) * Hv + h) * dv + 4 * c;
      orow[0] = from_f32<T>(os.x);
      orow[1] = from_f32<T>(os.y);
      orow[2] = from_f32<T>(os.z);
      orow[3] = from_f32<T>(os.w);
    }
    __syncthreads();  // the staged rows are read before the next node's go in
  }
}

}  // namespace

cudaError_t launch_verify_recurrent(const VerifyArgs& a, cudaStream_t stream) {
  const dim3 grid(a.d.N, a.d.Hv, a.d.B);
  if (a.d.dtype == GDN_TREE_BF16) {
    verify_recurrent_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
        static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
        static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status);
  } else {
    verify_recurrent_kernel<float><<<grid, kThreads, 0, stream>>>(
        static_cast<const float*>(a.q), static_cast<const float*>(a.k),
        static_cast<const float*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
        static_cast<float*>(a.o), a.U, a.d, a.dev_status);
  }
  return cudaGetLastError();
}

}  // namespace gdn
