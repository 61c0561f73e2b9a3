// commit.cu -- delayed state commitment of the accepted branch.
//
// "DFlash-TfM: Trees from Marginals", section 3: the recurrent state is
// committed at the next decoding iteration, once the accepted branch is known,
// so the verification never had to touch (or roll back) S0.  Unrolling the GDN
// recurrence along the accepted root-to-node path p_1..p_L with the verify's
// write vectors u gives
//     S1 = gamma_L S0 + sum_j w_j k_{p_j} u_{p_j}^T,
//     w_j = exp(G_L - G_j),  gamma_L = exp(G_L),  G_j = sum_{i<=j} log alpha_{p_i},
// a rank-L update of S0 that streams S0 in and S1 out once (HBM-bound).
//
// Grid: (Hv, B, dk / kRows).  Each CTA owns kRows rows of one (b, h) state and
// all dv columns; thread (r, c4) keeps a 4x4 register tile: rows r*4..r*4+3,
// columns c4*4..c4*4+3.  Its S0 tile is loaded first, so that the state stream
// overlaps the path-dependent loads; those come in one round (path and its
// length together, then parent links, log alpha, k rows and U rows), and the
// path's k rows (restricted to the CTA's rows) and U rows are staged through
// shared memory in chunks of kChunk path entries.
#include "common.cuh"
#include "kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kRows = 32;    // state rows per CTA
constexpr int kChunk = 32;   // path entries staged per round

template <typename T>
__global__ void __launch_bounds__(kThreads)
commit_kernel(const int32_t* __restrict__ path, const int32_t* __restrict__ path_len,
              const int32_t* __restrict__ parent, const float* __restrict__ U,
              const T* __restrict__ k, const float* __restrict__ log_alpha,
              const float* S0, float* S1, gdn_tree_dims d, int32_t Lmax,
              int32_t* dev_status) {
  // S0 and S1 may alias (in-place commit): every element is read and then
  // written by the same thread, so they are not __restrict__.
  __shared__ int sPath[kMaxN];
  __shared__ float sLa[kMaxN];         // log alpha along the path
  __shared__ float sW[kMaxN];          // w_j
  __shared__ __align__(16) float sK[kChunk][kRows];     // k_{p_j}[row0 + r]
  __shared__ __align__(16) float sU[kChunk][kMaxD];     // u_{p_j}
  __shared__ float sGamma;

  const int N = d.N, dk = d.dk, dv = d.dv, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y, row0 = blockIdx.z * kRows;
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = min(kRows, dk - row0);

  // ---- S0 tile prefetch: thread (r4, c4) owns rows r4*4.., columns c4*4.. ----
  const int r4 = tid / 32, c4 = tid % 32;
  const bool active = (r4 * 4 < rows) && (c4 < dv / 4);
  const size_t sbase = ((size_t)b * Hv + h) * dk * dv;
  float4 s0v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    s0v[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (active)
      s0v[i] = *reinterpret_cast<const float4*>(S0 + sbase + (size_t)(row0 + r4 * 4 + i) * dv + c4 * 4);
  }

  // ---- path length and entries, loaded together ------------------------------
  const int L = path_len[b];
  int pj = -1;
  if (tid < Lmax) pj = path[(size_t)b * Lmax + tid];
  int bad = (L < 0 || L > N || L > Lmax);
  if (!bad && tid < L) {
    bad |= (pj < 0 || pj >= N);
    sPath[tid] = pj;
  }
  bad = __syncthreads_or(bad);
  if (!bad && tid < L) {
    // a root-to-node path is strictly increasing in a topological order; with
    // the tree given it must also follow the parent links
    const int prev = tid == 0 ? -1 : sPath[tid - 1];
    bad |= (tid > 0 && pj <= prev);
    if (parent) bad |= (parent[(size_t)b * N + pj] != prev);
    sLa[tid] = log_alpha[((size_t)b * N + pj) * Hv + h];
  }
  bad = __syncthreads_or(bad);
  if (h == 0 && blockIdx.z == 0 && tid == 0 && dev_status)
    dev_status[b] = bad ? GDN_TREE_STATUS_BAD_PATH : GDN_TREE_STATUS_OK;
  if (bad) return;

  // ---- G_j: inclusive double-float prefix sums of log alpha along the path ------
  if (warp == 0) {
    // lane l owns entries l*8 .. l*8+7 (L <= 256)
    df loc[8];
    df run = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = lane * 8 + e;
      run = df_add(run, df{j < L ? sLa[j] : 0.f, 0.f});
      loc[e] = run;
    }
    df pre = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      df up;
      up.hi = __shfl_up_sync(0xffffffffu, pre.hi, o);
      up.lo = __shfl_up_sync(0xffffffffu, pre.lo, o);
      if (lane >= o) pre = df_add(pre, up);
    }
    df excl;
    excl.hi = __shfl_up_sync(0xffffffffu, pre.hi, 1);
    excl.lo = __shfl_up_sync(0xffffffffu, pre.lo, 1);
    if (lane == 0) excl = df{0.f, 0.f};
    df G[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) G[e] = df_add(excl, loc[e]);
    // G_L lives in the lane that owns entry L-1
    const int owner = L > 0 ? (L - 1) >> 3 : 0, slot = L > 0 ? (L - 1) & 7 : 0;
    df mine = G[0];
#pragma unroll
    for (int e = 1; e < 8; ++e)
      if (e == slot) mine = G[e];
    df GL;
    GL.hi = __shfl_sync(0xffffffffu, mine.hi, owner);
    GL.lo = __shfl_sync(0xffffffffu, mine.lo, owner);
    if (L == 0) GL = df{0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int j = lane * 8 + e;
      if (j < L) sW[j] = expf(df_diff(GL, G[e]));
    }
    if (lane == 0) sGamma = expf(df_value(GL));
  }

  // ---- S1 = gamma S0 + K_P^T diag(w) U_P over this CTA's rows ---------------------
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int j0 = 0; j0 < L; j0 += kChunk) {
    const int nj = min(kChunk, L - j0);
    if (j0 > 0) __syncthreads();
    for (int e = tid; e < nj * rows; e += kThreads) {
      const int jj = e / rows, r = e % rows;
      sK[jj][r] = to_f32(k[(((size_t)b * N + sPath[j0 + jj]) * Hqk + hq) * dk + row0 + r]);
    }
    for (int e = tid; e < nj * (dv / 4); e += kThreads) {
      const int jj = e / (dv / 4), c = (e % (dv / 4)) * 4;
      *reinterpret_cast<float4*>(&sU[jj][c]) = *reinterpret_cast<const float4*>(
          U + (((size_t)b * Hv + h) * N + sPath[j0 + jj]) * dv + c);
    }
    __syncthreads();
    if (active) {
      for (int jj = 0; jj < nj; ++jj) {
        const float w = sW[j0 + jj];
        const float4 kr = *reinterpret_cast<const float4*>(&sK[jj][r4 * 4]);
        const float4 uu = *reinterpret_cast<const float4*>(&sU[jj][c4 * 4]);
        const float kk[4] = {w * kr.x, w * kr.y, w * kr.z, w * kr.w};
        const float ul[4] = {uu.x, uu.y, uu.z, uu.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(kk[i], ul[j], acc[i][j]);
      }
    }
  }
  __syncthreads();  // sGamma (L == 0 skips the chunk loop)
  const float gamma = sGamma;
  if (active) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const size_t off = sbase + (size_t)(row0 + r4 * 4 + i) * dv + c4 * 4;
      float4 s1;
      s1.x = fmaf(gamma, s0v[i].x, acc[i][0]);
      s1.y = fmaf(gamma, s0v[i].y, acc[i][1]);
      s1.z = fmaf(gamma, s0v[i].z, acc[i][2]);
      s1.w = fmaf(gamma, s0v[i].w, acc[i][3]);
      *reinterpret_cast<float4*>(S1 + off) = s1;
    }
  }
}

}  // namespace

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream) {
  const dim3 grid(a.d.Hv, a.d.B, (a.d.dk + kRows - 1) / kRows);
  if (a.d.dtype == GDN_TREE_BF16) {
    commit_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
        a.path, a.path_len, a.parent, a.U, static_cast<const __nv_bfloat16*>(a.k),
        a.log_alpha, a.S0, a.S1, a.d, a.Lmax, a.dev_status);
  } else {
    commit_kernel<float><<<grid, kThreads, 0, stream>>>(
        a.path, a.path_len, a.parent, a.U, static_cast<const float*>(a.k),
        a.log_alpha, a.S0, a.S1, a.d, a.Lmax, a.dev_status);
  }
  return cudaGetLastError();
}

}  // namespace gdn
