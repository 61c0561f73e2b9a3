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
// Grid: (Hv, B, dk / 64), 256 threads, four CTAs per SM.  Each CTA owns 64 rows
// of one (b, h) state, bulk-copied into shared memory the moment the CTA
// starts, so that the state
// stream overlaps the path-dependent gathers, which take two steps: the path
// and its length together, then (with indices range-checked) the parent-link
// check, log alpha and the k and U rows of the path all at once.  Thread
// (r8, c4) keeps an 8x4 register tile (rows r8*8.., columns c4*4..); k and U
// rows are staged through shared memory in chunks of kChunk path entries.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerCta = 64;  // each CTA owns half of a (b, h) state's rows
constexpr int kChunk = 32;   // path entries staged per pass

// dynamic shared memory: S0 rows (kRowsPerCta x dv fp32) | k rows [kChunk][kRowsPerCta] |
// u rows [kChunk][dv] | path, log alpha, w_j [path capacity] each
constexpr size_t kSmemBytes =
    (size_t)(kRowsPerCta * kMaxD + kChunk * kRowsPerCta + kChunk * kMaxD) * sizeof(float);

// path capacity: Lmax rounded up to a whole scan block (at least kMaxN)
__host__ __device__ inline int path_capacity(int Lmax) { return Lmax <= kMaxN ? kMaxN : (Lmax + 255) / 256 * 256; }

// One warp: G[e] = base + (inclusive prefix sum of la[j0 ..] up to entry
// j0 + lane*8 + e), double-float, entries at or past L counting as 0.  Each lane
// reads only its own eight entries.
__device__ __forceinline__ void warp_scan_256(const float* la, int j0, int L, df base, int lane,
                                              df (&G)[8]) {
  df loc[8];
  df run = {0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int j = j0 + lane * 8 + e;
    run = df_add(run, df{j < L ? la[j] : 0.f, 0.f});
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
  excl = df_add(base, excl);
#pragma unroll
  for (int e = 0; e < 8; ++e) G[e] = df_add(excl, loc[e]);
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 4)
commit_kernel(const int32_t* __restrict__ path, const int32_t* __restrict__ path_len,
              const int32_t* __restrict__ parent, const float* __restrict__ U,
              const T* __restrict__ k, const float* __restrict__ log_alpha,
              const float* S0, float* S1, gdn_tree_dims d, int32_t Lmax,
              int32_t* dev_status, SeqLayout lay, WaitHooks hk) {
  const uint64_t kWaitLimitNs = hk.limit_ns;  // bound on the S0 copy wait
  // S0 and S1 may alias (in-place commit): the whole state is copied into
  // shared memory before any element of S1 is written.
  extern __shared__ __align__(128) float smem_f[];
  float* sS0 = smem_f;                            // [rows][dv]
  float* sK = sS0 + kRowsPerCta * kMaxD;          // [kChunk][rows]
  float* sU = sK + kChunk * kRowsPerCta;          // [kChunk][dv]
  const int cap = path_capacity(Lmax);
  int* sPath = reinterpret_cast<int*>(sU + kChunk * kMaxD);  // [cap]
  float* sLa = reinterpret_cast<float*>(sPath + cap);         // log alpha (then G_j.lo)
  float* sW = sLa + cap;                                      // w_j (G_j.hi during the scan)
  __shared__ uint64_t sBar;
  __shared__ float sGamma;

  const int Nmax = d.N, dk = d.dk, dv = d.dv, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y, row0 = blockIdx.z * kRowsPerCta;
  const int hq = h / (Hv / Hqk);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = min(kRowsPerCta, dk - row0);
  // this sequence's tree rows and state
  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N < 0 || st < 0) {
    if (h == 0 && blockIdx.z == 0 && tid == 0 && dev_status)
      atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_LAYOUT);
    return;
  }
  const size_t row = (size_t)lay.row0(b, Nmax);
  const size_t urow = lay.urow0(b, h, Hv, Nmax);
  const size_t sbase = ((size_t)st * Hv + h) * dk * dv;

  // ---- this CTA's rows of the (b, h) state start streaming in at once ----------
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)(rows * dv * sizeof(float));
    sm100::mbar_init(&sBar, 1);
    sm100::mbar_fence_init();
    sm100::mbar_arrive_expect_tx(&sBar, bytes);
    if (b != hk.withhold_copy_seq) sm100::bulk_load(sS0, S0 + sbase + (size_t)row0 * dv, bytes, &sBar);
  }

  // ---- gather 1: path length and entries (range-checked); the first kThreads
  //      entries are loaded together with the length ------------------------------
  const int L = path_len[b];
  int pj = -1;
  if (tid < Lmax) pj = path[(size_t)b * Lmax + tid];
  int bad = (L < 0 || L > N || L > Lmax);
  if (!bad && tid < L) {
    bad |= (pj < 0 || pj >= N);
    sPath[tid] = pj;
  }
  if (!bad) {
    for (int j = tid + kThreads; j < L; j += kThreads) {  // paths past kThreads entries
      const int pv = path[(size_t)b * Lmax + j];
      bad |= (pv < 0 || pv >= N);
      sPath[j] = pv;
    }
  }
  bad = __syncthreads_or(bad);

  // ---- gather 2: chain check, log alpha, and the first chunk of k / u rows,
  //      all issued together (indices are in range from here on) ----------------
  // a root-to-node path is strictly increasing in a topological order; with the
  // tree given it must also follow the parent links
  if (!bad && tid < L) {
    const int prev = tid == 0 ? -1 : sPath[tid - 1];
    bad |= (tid > 0 && pj <= prev);
    if (parent) bad |= (parent[row + pj] != prev);
    sLa[tid] = log_alpha[(row + pj) * Hv + h];
  }
  if (!bad) {
    for (int j = tid + kThreads; j < L; j += kThreads) {
      const int pv = sPath[j], prev = sPath[j - 1];
      bad |= (pv <= prev);
      if (parent) bad |= (parent[row + pv] != prev);
      sLa[j] = log_alpha[(row + pv) * Hv + h];
    }
  }
  auto stage = [&](int j0, int nj) {
    for (int e = tid; e < nj * (rows / 4); e += kThreads) {
      const int jj = e / (rows / 4), c = (e % (rows / 4)) * 4;
      const T* kr = k + ((row + sPath[j0 + jj]) * Hqk + hq) * dk + row0 + c;
      *reinterpret_cast<float4*>(sK + jj * kRowsPerCta + c) =
          make_float4(to_f32(kr[0]), to_f32(kr[1]), to_f32(kr[2]), to_f32(kr[3]));
    }
    for (int e = tid; e < nj * (dv / 4); e += kThreads) {
      const int jj = e / (dv / 4), c = (e % (dv / 4)) * 4;
      *reinterpret_cast<float4*>(sU + jj * dv + c) = *reinterpret_cast<const float4*>(
          U + (urow + sPath[j0 + jj]) * dv + c);
    }
  };
  if (!bad) stage(0, min(kChunk, L));
  bad = __syncthreads_or(bad);
  if (bad && h == 0 && blockIdx.z == 0 && tid == 0 && dev_status)
    atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_PATH);
  if (bad) {
    if (tid == 0) sm100::mbar_wait(&sBar, 0, kWaitLimitNs);  // drain the copy
    return;
  }

  // ---- G_j: inclusive double-float prefix sums of log alpha along the path ------
  if (warp == 0) {
    if (L <= 256) {
      // lane l owns entries l*8 .. l*8+7
      df G[8];
      warp_scan_256(sLa, 0, L, df{0.f, 0.f}, lane, G);
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
    } else {
      // blocks of 256 entries with a running carry; G_j parks in (sW, sLa)
      df carry = {0.f, 0.f};
      for (int j0 = 0; j0 < L; j0 += 256) {
        df G[8];
        warp_scan_256(sLa, j0, L, carry, lane, G);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = j0 + lane * 8 + e;
          if (j < L) {
            sW[j] = G[e].hi;
            sLa[j] = G[e].lo;
          }
        }
        __syncwarp();
        const int last = min(L, j0 + 256) - 1;
        carry = df{sW[last], sLa[last]};
      }
      const df GL = carry;
      for (int j = lane; j < L; j += 32) sW[j] = expf(df_diff(GL, df{sW[j], sLa[j]}));
      if (lane == 0) sGamma = expf(df_value(GL));
    }
  }
  __syncthreads();

  // ---- S1 = gamma S0 + K_P^T diag(w) U_P ------------------------------------------
  // thread (r8, c4): rows r8*8 .. r8*8+7, columns c4*4 .. c4*4+3
  const int r8 = tid / 32, c4 = tid % 32;
  const bool active = (r8 * 8 < rows) && (c4 * 4 < dv);
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int j0 = 0; j0 < L; j0 += kChunk) {
    const int nj = min(kChunk, L - j0);
    if (j0 > 0) {
      __syncthreads();
      stage(j0, nj);
      __syncthreads();
    }
    if (active) {
      for (int jj = 0; jj < nj; ++jj) {
        const float w = sW[j0 + jj];
        const float4 k0 = *reinterpret_cast<const float4*>(sK + jj * kRowsPerCta + r8 * 8);
        const float4 k1 = *reinterpret_cast<const float4*>(sK + jj * kRowsPerCta + r8 * 8 + 4);
        const float4 uu = *reinterpret_cast<const float4*>(sU + jj * dv + c4 * 4);
        const float kk[8] = {w * k0.x, w * k0.y, w * k0.z, w * k0.w,
                             w * k1.x, w * k1.y, w * k1.z, w * k1.w};
        const float ul[4] = {uu.x, uu.y, uu.z, uu.w};
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(kk[i], ul[j], acc[i][j]);
      }
    }
  }
  const float gamma = sGamma;
  const bool landed = sm100::mbar_wait(&sBar, 0, kWaitLimitNs);
  if (!landed) {
    if (tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_TIMEOUT);
    return;  // S1 left unwritten
  }
  if (active) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = r8 * 8 + i;
      const float4 s0 = *reinterpret_cast<const float4*>(sS0 + row * dv + c4 * 4);
      float4 s1;
      s1.x = fmaf(gamma, s0.x, acc[i][0]);
      s1.y = fmaf(gamma, s0.y, acc[i][1]);
      s1.z = fmaf(gamma, s0.z, acc[i][2]);
      s1.w = fmaf(gamma, s0.w, acc[i][3]);
      *reinterpret_cast<float4*>(S1 + sbase + (size_t)(row0 + row) * dv + c4 * 4) = s1;
    }
  }
}

}  // namespace

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream) {
  const dim3 grid(a.d.Hv, a.d.B, (a.d.dk + kRowsPerCta - 1) / kRowsPerCta);
  const size_t smem = kSmemBytes + (size_t)path_capacity(a.Lmax) * 3 * sizeof(float);
  const WaitHooks hk = wait_hooks();
  cudaError_t err;
  if (a.d.dtype == GDN_TREE_BF16) {
    err = cudaFuncSetAttribute(commit_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    commit_kernel<__nv_bfloat16><<<grid, kThreads, smem, stream>>>(
        a.path, a.path_len, a.parent, a.U, static_cast<const __nv_bfloat16*>(a.k),
        a.log_alpha, a.S0, a.S1, a.d, a.Lmax, a.dev_status, a.lay, hk);
  } else {
    err = cudaFuncSetAttribute(commit_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    commit_kernel<float><<<grid, kThreads, smem, stream>>>(
        a.path, a.path_len, a.parent, a.U, static_cast<const float*>(a.k),
        a.log_alpha, a.S0, a.S1, a.d, a.Lmax, a.dev_status, a.lay, hk);
  }
  return cudaGetLastError();
}

}  // namespace gdn
