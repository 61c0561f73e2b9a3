// tree_topw.cu -- top-w best-first construction of the draft tree.
//
// Method: "DFlash-TfM: Trees from Marginals", section 2 ("Costruzione
// dell'Albero"): the DySpec best-first construction, modified to pop the top-w
// candidates of the heap and expand all w at once, so that a tree of N nodes
// takes ceil(N / w) sequential rounds.
//
//   node 0 is the root (score 0, depth 1); every node of depth < max_depth
//   offers c candidates, candidate j of node p scoring score(p) + logp[p, j]
//   (fp32 addition); a round takes the min(w, N - nodes) best live candidates
//   (higher score first, ties to the lower key p * c + j, i.e. creation order)
//   as new nodes in that order, and only then do they offer their candidates.
//   A -inf candidate is never taken; construction stops when none is left.
//
// One warp per sequence.  Trees of up to 512 candidate slots with w <= 4 keep
// them sorted in registers (tree_topw_warp_kernel); other shapes in shared
// memory indexed by their key (slots of nodes not yet built, and taken
// candidates, hold -inf), a pop being one strided scan per lane and a warp
// argmax over (score, key).
#include <math_constants.h>

#include "common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int kWarpsPerCta = 4;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
tree_topw_kernel(const float* __restrict__ cand_logp, int B, int N, int c, int w, int max_depth,
                 int32_t* __restrict__ parent, int32_t* __restrict__ cand_index,
                 float* __restrict__ score, int32_t* __restrict__ n_built) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarpsPerCta + warp;
  if (b >= B) return;  // whole warps only: nothing below synchronises across warps
  const size_t per_warp = (size_t)N * c * sizeof(float) + (size_t)N * 2 * sizeof(float);
  float* cand = reinterpret_cast<float*>(smem + warp * per_warp);  // [N * c]
  float* nscore = cand + N * c;                                     // [N]
  int* ndepth = reinterpret_cast<int*>(nscore + N);                 // [N]
  const float* lp = cand_logp + (size_t)b * N * c;
  int32_t* par = parent + (size_t)b * N;
  int32_t* cix = cand_index ? cand_index + (size_t)b * N : nullptr;
  float* sco = score ? score + (size_t)b * N : nullptr;
  const float kNegInf = -CUDART_INF_F;

  for (int k = lane; k < N * c; k += 32) cand[k] = kNegInf;
  if (lane == 0) {
    nscore[0] = 0.f;
    ndepth[0] = 1;
    par[0] = -1;
    if (cix) cix[0] = -1;
    if (sco) sco[0] = 0.f;
  }
  __syncwarp();
  if (max_depth > 1)
    for (int j = lane; j < c; j += 32) cand[j] = 0.f + lp[j];
  __syncwarp();

  int n = 1;
  while (n < N) {
    const int take = min(w, N - n);
    int popped = 0;
    for (int r = 0; r < take; ++r) {
      // this lane's best live candidate among keys lane, lane + 32, ...
      float bs = kNegInf;
      int bk = 0x7fffffff;
      for (int k = lane; k < n * c; k += 32) {
        const float s = cand[k];
        if (s > bs || (s == bs && k < bk)) {
          bs = s;
          bk = k;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float os = __shfl_xor_sync(0xffffffffu, bs, off);
        const int ok = __shfl_xor_sync(0xffffffffu, bk, off);
        if (os > bs || (os == bs && ok < bk)) {
          bs = os;
          bk = ok;
        }
      }
      if (bs == kNegInf) break;  // no live candidate (uniform across the warp)
      const int node = n + popped, p = bk / c, j = bk - p * c;
      if (lane == 0) {
        cand[bk] = kNegInf;
        nscore[node] = bs;
        ndepth[node] = ndepth[p] + 1;
        par[node] = p;
        if (cix) cix[node] = j;
        if (sco) sco[node] = bs;
      }
      ++popped;
      __syncwarp();
    }
    if (popped == 0) break;
    // the round's new nodes offer their candidates
    for (int i = lane; i < popped * c; i += 32) {
      const int node = n + i / c, j = i % c;
      if (ndepth[node] < max_depth) cand[node * c + j] = nscore[node] + lp[node * c + j];
    }
    n += popped;
    __syncwarp();
  }
  // nodes that could not be built
  for (int i = n + lane; i < N; i += 32) {
    par[i] = -2;
    if (cix) cix[i] = -2;
    if (sco) sco[i] = CUDART_NAN_F;
  }
  if (lane == 0 && n_built) n_built[b] = n;
}

// Trees of up to 512 candidate slots, w <= 4: one warp per tree.  Lane l owns
// the slots l, l + 32, ..., l + 480 (key = p * c + j): their log-probabilities,
// and its live slots as 64-bit words (the score's order-preserving bits, then
// 511 - key, then the depth the node would have, so that one unsigned comparison
// orders by score and then by lower key; 0 = empty): its best four sorted in
// registers, the rest unsorted in shared memory.  A round takes the warp's four
// best words at once -- a butterfly over the lanes merges their sorted top four --
// the owners drop what was taken and refill from their rest, and the new nodes'
// candidates are inserted by the lanes that own their slots.  Same fp32 sums and
// tie rule as the general kernel, so the same tree.
constexpr int kSlots = 16;
constexpr int kTop = 4;

// fp32 -> uint32 with the same order (no NaN)
__device__ __forceinline__ uint32_t order_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  return u ^ ((u >> 31) ? 0xffffffffu : 0x80000000u);
}
__device__ __forceinline__ float from_order_bits(uint32_t o) {
  return __uint_as_float(o ^ ((o >> 31) ? 0x80000000u : 0xffffffffu));
}
// key < 512, depth < 1024
__device__ __forceinline__ uint64_t cand_word(float s, uint32_t key, uint32_t depth) {
  return ((uint64_t)order_bits(s) << 32) | (uint64_t)(((511u - key) << 10) | depth);
}
__device__ __forceinline__ uint32_t word_key(uint64_t x) { return 511u - ((uint32_t)x >> 10); }
__device__ __forceinline__ int word_depth(uint64_t x) { return (int)((uint32_t)x & 1023u); }
__device__ __forceinline__ float word_score(uint64_t x) {
  return from_order_bits((uint32_t)(x >> 32));
}
__device__ __forceinline__ uint64_t shfl_xor64(uint64_t x, int off) {
  const uint32_t lo = __shfl_xor_sync(0xffffffffu, (uint32_t)x, off);
  const uint32_t hi = __shfl_xor_sync(0xffffffffu, (uint32_t)(x >> 32), off);
  return ((uint64_t)hi << 32) | lo;
}
__device__ __forceinline__ void cswap_desc(uint64_t& a, uint64_t& b) {
  const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
  a = hi;
  b = lo;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32, 1)
tree_topw_warp_kernel(const float* __restrict__ cand_logp, int B, int N, int c, int w,
                      int max_depth, int32_t* __restrict__ parent,
                      int32_t* __restrict__ cand_index, float* __restrict__ score,
                      int32_t* __restrict__ n_built) {
  __shared__ float s_lp[kWarpsPerCta][kSlots * 32];
  // each lane's live words past its best four, unsorted: slot i of lane l at [i][l]
  __shared__ uint64_t s_bag[kWarpsPerCta][kSlots][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarpsPerCta + warp;
  if (b >= B) return;  // whole warps only: nothing below synchronises across warps
  float* lp = s_lp[warp];  // the tree's candidate log-probabilities, by key
  uint64_t (*bag)[32] = s_bag[warp];
  const float* lpb = cand_logp + (size_t)b * N * c;
  int32_t* par = parent + (size_t)b * N;
  int32_t* cix = cand_index ? cand_index + (size_t)b * N : nullptr;
  float* sco = score ? score + (size_t)b * N : nullptr;
  const float kNegInf = -CUDART_INF_F;
  const int nslots = N * c;
  // key / c as a multiply and shift (exact for key * c < 2^16: key < 512, c <= 32)
  const uint32_t cinv = 65536u / (uint32_t)c + 1u;
  auto node_of = [&](uint32_t key) { return (int)((key * cinv) >> 16); };

#pragma unroll
  for (int m = 0; m < kSlots; ++m) {
    const int k = lane + 32 * m;
    lp[k] = k < nslots ? lpb[k] : kNegInf;
  }
  // this lane's live words: its best four sorted in registers (0 = empty), the rest
  // in the bag, all below top[3] (so the bag is empty while top has room)
  uint64_t top[kTop] = {0, 0, 0, 0};
  int nb = 0;
  auto insert = [&](uint64_t x) {
    if (x > top[kTop - 1]) {
      const uint64_t out = top[kTop - 1];
      const int at = (top[0] > x) + (top[1] > x) + (top[2] > x);
      top[3] = at == 3 ? x : top[2];
      top[2] = at == 2 ? x : (at < 2 ? top[1] : top[2]);
      top[1] = at == 1 ? x : (at < 1 ? top[0] : top[1]);
      if (at == 0) top[0] = x;
      if (out != 0) bag[nb++][lane] = out;
    } else {
      bag[nb++][lane] = x;
    }
  };
  // the root (node 0, score 0, depth 1) offers its candidates (keys 0 .. c-1)
  if (max_depth > 1) {
    for (int k = lane; k < c; k += 32) {
      const float s = 0.f + lp[k];
      if (s != kNegInf) insert(cand_word(s, (uint32_t)k, 2u));
    }
  }
  if (lane == 0) {
    par[0] = -1;
    if (cix) cix[0] = -1;
    if (sco) sco[0] = 0.f;
  }
  __syncwarp();

  int n = 1;
  while (n < N) {
    const int take = min(w, N - n);
    // the warp's four best words: every lane ends with the same sorted list
    uint64_t t[kTop] = {top[0], top[1], top[2], top[3]};
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint64_t o[kTop];
#pragma unroll
      for (int i = 0; i < kTop; ++i) o[i] = shfl_xor64(t[i], off);
      // top four of two sorted lists: the larger of a[i] and b[3 - i] (a bitonic
      // sequence), then sorted
#pragma unroll
      for (int i = 0; i < kTop; ++i) t[i] = t[i] > o[kTop - 1 - i] ? t[i] : o[kTop - 1 - i];
      cswap_desc(t[0], t[2]);
      cswap_desc(t[1], t[3]);
      cswap_desc(t[0], t[1]);
      cswap_desc(t[2], t[3]);
    }
    int popped = 0, mine = 0;
#pragma unroll
    for (int i = 0; i < kTop; ++i) {
      if (i < take && t[i] != 0) {
        ++popped;
        mine += (int)(word_key(t[i]) & 31u) == lane;
      }
    }
    if (popped == 0) break;  // no live candidate (uniform across the warp)
    // this lane's taken words are the front of top: shift, then refill from the bag
    // with its best words in turn
    if (mine > 0) {
#pragma unroll
      for (int i = 0; i < kTop; ++i) {
        uint64_t x = 0;
#pragma unroll
        for (int q = 1; q <= kTop; ++q)
          if (mine == q && i + q < kTop) x = top[i + q];
        top[i] = x;
      }
      for (int r = kTop - mine; r < kTop && nb > 0; ++r) {
        // the bag's best: every slot loaded at once, then a pairwise maximum with its
        // slot (empty slots count as 0)
        uint64_t y[kSlots];
        int yi[kSlots];
#pragma unroll
        for (int i = 0; i < kSlots; ++i) {
          y[i] = i < nb ? bag[i][lane] : 0;
          yi[i] = i;
        }
#pragma unroll
        for (int span = kSlots / 2; span > 0; span >>= 1) {
#pragma unroll
          for (int i = 0; i < span; ++i) {
            const bool hi = y[i + span] > y[i];
            y[i] = hi ? y[i + span] : y[i];
            yi[i] = hi ? yi[i + span] : yi[i];
          }
        }
        bag[yi[0]][lane] = bag[nb - 1][lane];
        --nb;
#pragma unroll
        for (int i = 0; i < kTop; ++i)
          if (i == r) top[i] = y[0];
      }
    }
    // the new nodes n + i (i < popped): every lane has their words, depths included
    int nd[kTop];
#pragma unroll
    for (int i = 0; i < kTop; ++i) nd[i] = i < popped ? word_depth(t[i]) : 0;
    // lane i < popped records node n + i
    if (lane < popped) {
      const uint64_t x = lane == 0 ? t[0] : lane == 1 ? t[1] : lane == 2 ? t[2] : t[3];
      const uint32_t key = word_key(x);
      const int node = n + lane, p = node_of(key), j = (int)key - p * c;
      par[node] = p;
      if (cix) cix[node] = j;
      if (sco) sco[node] = word_score(x);
    }
    // the new nodes offer their candidates: keys n c .. (n + popped) c - 1, the
    // ones of this lane's slots (one insertion each)
    const int k0 = n * c, k1 = (n + popped) * c;
    for (int k = k0 + ((lane - k0) & 31); k < k1; k += 32) {
      const int i = node_of((uint32_t)k) - n;
      const uint64_t x = i == 0 ? t[0] : i == 1 ? t[1] : i == 2 ? t[2] : t[3];
      const int d = i == 0 ? nd[0] : i == 1 ? nd[1] : i == 2 ? nd[2] : nd[3];
      if (d < max_depth) {
        const float s = word_score(x) + lp[k];
        if (s != kNegInf) insert(cand_word(s, (uint32_t)k, (uint32_t)d + 1u));
      }
    }
    __syncwarp();
    n += popped;
  }
  // nodes that could not be built
  for (int i = n + lane; i < N; i += 32) {
    par[i] = -2;
    if (cix) cix[i] = -2;
    if (sco) sco[i] = CUDART_NAN_F;
  }
  if (lane == 0 && n_built) n_built[b] = n;
}

}  // namespace

size_t tree_topw_smem_bytes(int N, int c) {
  return (size_t)kWarpsPerCta * ((size_t)N * c * sizeof(float) + (size_t)N * 2 * sizeof(float));
}

cudaError_t launch_tree_topw(const float* cand_logp, int B, int N, int c, int w, int max_depth,
                             int32_t* parent, int32_t* cand_index, float* score, int32_t* n_built,
                             cudaStream_t stream) {
  const int grid = (B + kWarpsPerCta - 1) / kWarpsPerCta;
  if (N * c <= kSlots * 32 && w <= kTop) {
    tree_topw_warp_kernel<<<grid, kWarpsPerCta * 32, 0, stream>>>(
        cand_logp, B, N, c, w, max_depth, parent, cand_index, score, n_built);
    return cudaGetLastError();
  }
  const size_t smem = tree_topw_smem_bytes(N, c);
  cudaError_t err = cudaFuncSetAttribute(tree_topw_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  tree_topw_kernel<<<grid, kWarpsPerCta * 32, smem, stream>>>(cand_logp, B, N, c, w, max_depth,
                                                               parent, cand_index, score, n_built);
  return cudaGetLastError();
}

}  // namespace gdn
