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
// One warp per sequence.  The candidates live in shared memory indexed by their
// key (slots of nodes not yet built, and taken candidates, hold -inf); a pop is
// one strided scan per lane and a warp argmax over (score, key).
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

}  // namespace

size_t tree_topw_smem_bytes(int N, int c) {
  return (size_t)kWarpsPerCta * ((size_t)N * c * sizeof(float) + (size_t)N * 2 * sizeof(float));
}

cudaError_t launch_tree_topw(const float* cand_logp, int B, int N, int c, int w, int max_depth,
                             int32_t* parent, int32_t* cand_index, float* score, int32_t* n_built,
                             cudaStream_t stream) {
  const size_t smem = tree_topw_smem_bytes(N, c);
  cudaError_t err = cudaFuncSetAttribute(tree_topw_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  const int grid = (B + kWarpsPerCta - 1) / kWarpsPerCta;
  tree_topw_kernel<<<grid, kWarpsPerCta * 32, smem, stream>>>(cand_logp, B, N, c, w, max_depth,
                                                               parent, cand_index, score, n_built);
  return cudaGetLastError();
}

}  // namespace gdn
