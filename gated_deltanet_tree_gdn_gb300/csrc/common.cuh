// common.cuh -- device helpers shared by the libgdntree kernels.
//
// Precision notes that hold for every kernel:
//  * Path log-decays g_t (sums of log alpha along the root-to-t path) are
//    carried as double-float pairs (hi + lo, two fp32 words), so that the
//    differences g_t - g_s that set every decay weight exp(g_t - g_s) keep
//    full fp32 relative accuracy even when |g| grows to hundreds (strong
//    decay over deep chains).  A plain fp32 prefix sum would lose ~1e-4 of
//    relative accuracy there.
//  * A decay weight exp(g_t - g_s), s on t's path, has an argument <= 0 for
//    log alpha <= 0.  It is taken from the double-float difference, except in
//    the tensor-core kernel while every |g_t| of the tree is at most 40: there
//    it is the product exp(g_t) * exp(-g_s) of two per-node factors, both (and
//    the product) normal fp32 numbers within that bound.  Past the bound the
//    product could overflow, so the difference form is used.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gdn_tree.h"

namespace gdn {

constexpr int kMaxN = 256;       // largest tree of the kernels that keep it all on chip
constexpr int kMaxNLong = 1024;  // largest tree of the chunked kernel and of a commit path
constexpr int kMaxD = 128;

// ---- double-float arithmetic (Knuth TwoSum / Dekker FastTwoSum) -----------

struct df {
  float hi, lo;
};

__device__ __forceinline__ df df_add(df a, df b) {
  // TwoSum of the high parts, then fold in the low parts and renormalise.
  float s = __fadd_rn(a.hi, b.hi);
  float bb = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  float hi = __fadd_rn(s, e);
  float lo = __fsub_rn(e, __fsub_rn(hi, s));
  return {hi, lo};
}

// (a - b) rounded to fp32; exact-ish for nearby a, b
__device__ __forceinline__ float df_diff(df a, df b) {
  return __fadd_rn(__fsub_rn(a.hi, b.hi), __fsub_rn(a.lo, b.lo));
}

__device__ __forceinline__ float df_value(df a) { return __fadd_rn(a.hi, a.lo); }

// ---- element loads -----------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---- tree preparation --------------------------------------------------------

// block-wide barrier (the default for tree_prepare)
struct BlockSync {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
  // the barrier, returning whether any thread's x is true
  __device__ __forceinline__ bool any(bool x) const { return __syncthreads_or(x) != 0; }
};

// barrier over the first `count` threads of the block (named barrier `id`)
template <int kId, int kCount>
struct NamedSync {
  __device__ __forceinline__ void operator()() const {
    asm volatile("bar.sync %0, %1;" ::"n"(kId), "n"(kCount) : "memory");
  }
  __device__ __forceinline__ bool any(bool x) const {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)x), "n"(kId), "n"(kCount)
        : "memory");
    return r != 0;
  }
};

//
// For the tree of one sequence (parent[] already in shared memory and
// validated), computes with pointer jumping (ceil(log2 depth) rounds: it stops
// once every node has reached its root):
//   anc[t*W .. t*W+W-1] : bitset of the strict ancestors of t (W = ceil(N/32))
//   g[t]                : double-float sum of log_alpha over the path P(t)
// `jump` is an int scratch of N entries.  Must be called by every thread that
// `sync` synchronises; node t is handled by thread t (needs N such threads).
template <typename Sync = BlockSync>
__device__ __forceinline__ void tree_prepare(const int* s_parent, int N, int W,
                                             const float* s_log_alpha,
                                             int* s_jump, uint32_t* s_anc,
                                             df* s_g, Sync sync = Sync()) {
  const int t = threadIdx.x;
  if (t < N) {
    const int p = s_parent[t];
    s_jump[t] = p;
    s_g[t] = df{s_log_alpha[t], 0.f};
    for (int i = 0; i < W; ++i) s_anc[t * W + i] = 0u;
    if (p >= 0) s_anc[t * W + (p >> 5)] = 1u << (p & 31);
  }
  sync();
  for (int span = 1; span < N; span <<= 1) {
    int j = -1, jj = -1;
    df gj = {0.f, 0.f};
    uint32_t w[kMaxN / 32];
    if (t < N) {
      j = s_jump[t];
      if (j >= 0) {
        jj = s_jump[j];
        gj = s_g[j];
#pragma unroll
        for (int i = 0; i < kMaxN / 32; ++i) w[i] = i < W ? s_anc[j * W + i] : 0u;
      }
    }
    if (!sync.any(j >= 0)) break;  // every node reached its root
    if (t < N && j >= 0) {
      s_g[t] = df_add(s_g[t], gj);
#pragma unroll
      for (int i = 0; i < kMaxN / 32; ++i)
        if (i < W) s_anc[t * W + i] |= w[i];
      s_jump[t] = jj;
    }
    sync();
  }
}

}  // namespace gdn
