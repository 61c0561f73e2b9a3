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
// One warp per sequence.  Rounds of at most 32 offers (w * c <= 32) keep the
// live candidates as one sorted list (tree_topw_list_kernel); other shapes in
// shared memory indexed by their key (slots of nodes not yet built, and taken
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

// Rounds that offer at most 32 candidates (w * c <= 32), trees of up to 256 nodes:
// a CTA of two or four warps per tree keeps its live candidates as one list in shared
// memory, sorted best first, as 64-bit order-preserving words (the fp32 score's bits
// made monotone in the high half; in the low half kKeyTop - key, so that one
// unsigned comparison orders by score and then by lower key, and the depth the node
// would have; 0 = none).  The list is cut to the N - built best: a candidate ranked at
// or below the number of nodes still to build is never taken, since every round
// takes only candidates ranked above it.  A round's takes are then the list's front,
// and its offers (one word per lane, formed by every warp alike) are merged in: each
// offer is broadcast in turn and compared with every listed word (each warp holds its
// share of the list), which gives each listed word the number of offers above it
// (it moves down by that much) and, counted over the warps, each offer the number of
// listed words above it (its place is that plus the offers above it).  The built
// nodes' words are kept and written out once at the end.  Same fp32 sums and tie
// rule as the general kernel, so the same tree.
constexpr uint32_t kKeyTop = (1u << 21) - 1u;  // keys < 2^21, depths < 2^11

// fp32 -> uint32 with the same order (no NaN)
__device__ __forceinline__ uint32_t order_bits(float x) {
  const uint32_t u = __float_as_uint(x);
  return u ^ ((u >> 31) ? 0xffffffffu : 0x80000000u);
}
__device__ __forceinline__ float from_order_bits(uint32_t o) {
  return __uint_as_float(o ^ ((o >> 31) ? 0x80000000u : 0xffffffffu));
}
__device__ __forceinline__ uint64_t cand_word(float s, uint32_t key, uint32_t depth) {
  return ((uint64_t)order_bits(s) << 32) | (uint64_t)(((kKeyTop - key) << 11) | depth);
}
__device__ __forceinline__ uint32_t word_key(uint64_t x) { return kKeyTop - ((uint32_t)x >> 11); }
__device__ __forceinline__ int word_depth(uint64_t x) { return (int)((uint32_t)x & 2047u); }
__device__ __forceinline__ float word_score(uint64_t x) {
  return from_order_bits((uint32_t)(x >> 32));
}

constexpr int kListOffers = 32;  // offers a round can make (w * c)

__device__ __forceinline__ uint64_t shfl64(uint64_t x, int src) {
  const uint32_t lo = __shfl_sync(0xffffffffu, (uint32_t)x, src);
  const uint32_t hi = __shfl_sync(0xffffffffu, (uint32_t)(x >> 32), src);
  return ((uint64_t)hi << 32) | lo;
}

// 4-byte global -> shared copy that the thread does not wait for (cp.async.wait_all)
__device__ __forceinline__ void copy4_async(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   (uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}

inline size_t topw_list_smem_bytes(int N, int c, int slots, int warps) {
  return (size_t)(32 * warps * (slots + 1) + N) * sizeof(uint64_t) +
         (size_t)32 * warps * sizeof(int) + (size_t)N * c * sizeof(float);
}

// kSlots: listed words per thread and kListWarps: warps per tree (the list holds up
// to 32 kListWarps kSlots >= N words; warp v's slots are (s kListWarps + v) 32 + lane);
// kOffers: offers scanned per round (>= w * c).
template <int kSlots, int kOffers, int kListWarps>
__global__ void __launch_bounds__(32 * kListWarps)
tree_topw_list_kernel(const float* __restrict__ cand_logp, int N, int c, int w, int max_depth,
                      int32_t* __restrict__ parent, int32_t* __restrict__ cand_index,
                      float* __restrict__ score, int32_t* __restrict__ n_built) {
  constexpr int kThreads = 32 * kListWarps, kCap = kThreads * kSlots;
  extern __shared__ __align__(16) unsigned char smem[];
  uint64_t* list = reinterpret_cast<uint64_t*>(smem);  // [kCap] live words, best first
  uint64_t* sink = list + kCap;                         // [kThreads] stores of dropped words
  uint64_t* node = sink + kThreads;                     // [N] the built nodes' words
  int* part = reinterpret_cast<int*>(node + N);         // [warps][32] per warp: listed
                                                        //   words below offer lane
  float* lp = reinterpret_cast<float*>(part + kThreads);  // [N * c], by key
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, b = blockIdx.x;
  const float* lpb = cand_logp + (size_t)b * N * c;
  const float kNegInf = -CUDART_INF_F;

  // every copy in flight at once, then one wait
  for (int k = tid; k < N * c; k += kThreads) copy4_async(lp + k, lpb + k);
  asm volatile("cp.async.wait_all;" ::: "memory");
  if (tid == 0) node[0] = cand_word(0.f, 0u, 1u);  // the root: score 0, depth 1
  const int from = lane / c;  // the taken node whose candidate lane - from * c this lane offers
  __syncthreads();

  int n0 = 0, nt = 1, len = 0;  // the round's first node, its takes, the list's length
  int built;
  for (;;) {
    const int n = n0 + nt;  // nodes built with the round's takes
    if (n >= N) {
      built = n;
      break;
    }
    // the takes (nodes n0 .. n - 1) offer their candidates: keys n0 c .. n c - 1, one
    // per lane (every warp forms the same words)
    uint64_t my = 0;
    if (lane < nt * c) {
      const int key = n0 * c + lane;
      const float l = lp[key];
      const uint64_t x = node[n0 + from];
      const int d = word_depth(x);
      const float s = word_score(x) + l;
      if (d < max_depth && s != kNegInf) my = cand_word(s, (uint32_t)key, (uint32_t)d + 1u);
    }
    // this warp's listed words (an empty slot holds the largest word, so that no offer
    // counts as above it)
    uint64_t m[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
      const int k = (s * kListWarps + warp) * 32 + lane;
      m[s] = k < len ? list[k] : ~0ull;
    }
    // each offer y in turn, broadcast from its lane: the offers above this lane's
    // offer, the offers above each of this thread's listed words, and this warp's
    // listed words below y (words are distinct: the listed words above y are the rest)
    int rank = 0, below_mine = 0, cnt[kSlots];
#pragma unroll
    for (int s = 0; s < kSlots; ++s) cnt[s] = 0;
    // every offer's broadcast first, so that the shuffles' latency is paid once
    uint64_t ys[kOffers];
#pragma unroll
    for (int j = 0; j < kOffers; ++j) ys[j] = shfl64(my, j);
#pragma unroll
    for (int j = 0; j < kOffers; ++j) {
      const uint64_t y = ys[j];
      rank += (int)(y > my);
      int below = 0;
#pragma unroll
      for (int s = 0; s < kSlots; ++s) {
        const bool g = y > m[s];
        cnt[s] += (int)g;
        below += __popc(__ballot_sync(0xffffffffu, g));
      }
      if (lane == j) below_mine = below;
    }
    part[tid] = below_mine;
    const int total = len + __popc(__ballot_sync(0xffffffffu, my != 0));
    const int left = N - n;  // nodes still to build
    const int take = min(w, left), keep = min(total, left);
    __syncthreads();  // every read of the list is done, every warp's count is in
    // merged place pos: the next round's takes are nodes n .. n + take - 1, the list
    // keeps places take .. keep - 1, the rest is dropped (into this thread's sink slot)
    auto dest = [&](int pos, bool live) {
      return !live ? sink + tid
                   : pos < take ? node + n + pos : pos < keep ? list + (pos - take) : sink + tid;
    };
#pragma unroll
    for (int s = 0; s < kSlots; ++s) {
      const int k = (s * kListWarps + warp) * 32 + lane;
      *dest(k + cnt[s], k < len) = m[s];
    }
    if (warp == 0) {
      int below = 0;
#pragma unroll
      for (int v = 0; v < kListWarps; ++v) below += part[v * 32 + lane];
      *dest(rank + len - below, my != 0) = my;
    }
    __syncthreads();
    n0 = n;
    nt = min(take, total);
    len = keep > take ? keep - take : 0;
    if (nt == 0) {  // no live candidate (uniform across the CTA)
      built = n;
      break;
    }
  }
  // every node's record, from its word
  int32_t* par = parent + (size_t)b * N;
  int32_t* cix = cand_index ? cand_index + (size_t)b * N : nullptr;
  float* sco = score ? score + (size_t)b * N : nullptr;
  for (int i = tid; i < N; i += kThreads) {
    int p = -2, j = -2;
    float v = CUDART_NAN_F;
    if (i == 0) {
      p = -1, j = -1, v = 0.f;
    } else if (i < built) {
      const uint64_t x = node[i];
      const int key = (int)word_key(x);
      p = key / c, j = key - p * c, v = word_score(x);
    }
    par[i] = p;
    if (cix) cix[i] = j;
    if (sco) sco[i] = v;
  }
  if (tid == 0 && n_built) n_built[b] = built;
}

template <int kSlots, int kListWarps>
cudaError_t launch_topw_list(const float* cand_logp, int B, int N, int c, int w, int max_depth,
                             int32_t* parent, int32_t* cand_index, float* score, int32_t* n_built,
                             cudaStream_t stream) {
  const size_t smem = topw_list_smem_bytes(N, c, kSlots, kListWarps);
  if (w * c <= 16)
    tree_topw_list_kernel<kSlots, 16, kListWarps><<<B, 32 * kListWarps, smem, stream>>>(
        cand_logp, N, c, w, max_depth, parent, cand_index, score, n_built);
  else
    tree_topw_list_kernel<kSlots, 32, kListWarps><<<B, 32 * kListWarps, smem, stream>>>(
        cand_logp, N, c, w, max_depth, parent, cand_index, score, n_built);
  return cudaGetLastError();
}

}  // namespace

size_t tree_topw_smem_bytes(int N, int c) {
  return (size_t)kWarpsPerCta * ((size_t)N * c * sizeof(float) + (size_t)N * 2 * sizeof(float));
}

cudaError_t launch_tree_topw(const float* cand_logp, int B, int N, int c, int w, int max_depth,
                             int32_t* parent, int32_t* cand_index, float* score, int32_t* n_built,
                             cudaStream_t stream) {
  if (w * c <= kListOffers && N <= 256) {
    // two warps up to 64 nodes (fewer threads at each barrier), four with one listed
    // word a thread up to 128, four with two up to 256 (measured faster than eight
    // with one)
    if (N <= 64)
      return launch_topw_list<1, 2>(cand_logp, B, N, c, w, max_depth, parent, cand_index,
                                    score, n_built, stream);
    if (N <= 128)
      return launch_topw_list<1, 4>(cand_logp, B, N, c, w, max_depth, parent, cand_index,
                                    score, n_built, stream);
    return launch_topw_list<2, 4>(cand_logp, B, N, c, w, max_depth, parent, cand_index, score,
                                  n_built, stream);
  }
  const int grid = (B + kWarpsPerCta - 1) / kWarpsPerCta;
  const size_t smem = tree_topw_smem_bytes(N, c);
  cudaError_t err = cudaFuncSetAttribute(tree_topw_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  tree_topw_kernel<<<grid, kWarpsPerCta * 32, smem, stream>>>(cand_logp, B, N, c, w, max_depth,
                                                               parent, cand_index, score, n_built);
  return cudaGetLastError();
}

}  // namespace gdn
