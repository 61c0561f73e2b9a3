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
// One warp per block of 32 state rows (16 where dk is not a multiple of 32) of
// one (b, h) state; no block-wide barrier anywhere, so that the latency of one
// warp's two dependent gathers hides behind the other warps of the SM.  A warp
// starts its S0 rows streaming into its shared-memory slot at once (cp.async,
// no registers held), together with the path and its length; then, with the
// entries known to be in range, the log alpha and parent links of the path
// (into registers, one entry per lane) and the path's k and U rows (into the
// warp's slots, eight entries at a time) all come in one round trip.  The
// weights follow from a double-float prefix sum across the lanes; the block is
// formed eight rows at a time and S1 leaves straight from the registers that
// form it.  Only S0 in, S1 out and the path's rows cross HBM, each once.
#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace gdn {

namespace {

constexpr int kWarps = 2;  // warps per CTA
constexpr int kThreads = 32 * kWarps;
constexpr int kRB = 8;     // state rows formed at a time (a pass)
constexpr int kMaxRows = 32;  // state rows of a warp's block
constexpr int kPre = 8;       // 32-entry chunks of a path whose entries are fetched together

// path entries whose k / U rows are on chip at a time (eight), and the slots
// holding them: one for paths of up to 32 entries (the common case: the most warps
// an SM), two (the next batch copied while one is used) for longer ones
__host__ __device__ inline int batch_size(int Lmax) { return 8; }
__host__ __device__ inline int batch_slots(int Lmax) { return Lmax > 32 ? 2 : 1; }

// state rows of a warp's block: 32, or 16 where dk is not a multiple of 32
__host__ __device__ inline int block_rows(int dk) { return dk % kMaxRows == 0 ? kMaxRows : 16; }

// path entries a warp keeps (pj, G_j.hi then w_j, G_j.lo): Lmax rounded up to 32
__host__ __device__ inline int path_capacity(int Lmax) { return Lmax <= 32 ? 32 : (Lmax + 31) / 32 * 32; }

// per warp, in bytes: S0 rows [kMaxRows][dv] fp32 | per slot: U rows [batch][dv]
// fp32, k rows [batch][kMaxRows] (as given) | pj, G.hi / w, G.lo [cap] each
__host__ __device__ inline uint32_t slot_bytes(int dv, int tsize, int Lmax) {
  return (uint32_t)batch_size(Lmax) * (dv * 4 + kMaxRows * tsize);
}
__host__ __device__ inline uint32_t warp_smem_bytes(int dv, int tsize, int Lmax) {
  return (uint32_t)kMaxRows * dv * 4 + batch_slots(Lmax) * slot_bytes(dv, tsize, Lmax) +
         3u * path_capacity(Lmax) * 4;
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_addr(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// every cp.async group of this thread but the most recent has completed
__device__ __forceinline__ void cp_async_wait_but_last() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// inclusive double-float prefix sum of v across the warp's lanes
__device__ __forceinline__ df warp_inclusive_scan(df v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    df up;
    up.hi = __shfl_up_sync(0xffffffffu, v.hi, o);
    up.lo = __shfl_up_sync(0xffffffffu, v.lo, o);
    if (lane >= o) v = df_add(v, up);
  }
  return v;
}

// the kRB entries of a staged k row, as fp32
__device__ __forceinline__ void load_k(const __nv_bfloat16* p, float (&v)[kRB]) {
  const uint4 q = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ void load_k(const float* p, float (&v)[kRB]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 c = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 8)
commit_kernel(const int32_t* __restrict__ path, const int32_t* __restrict__ path_len,
              const int32_t* __restrict__ parent, const float* __restrict__ U,
              const T* __restrict__ k, const float* __restrict__ log_alpha,
              const float* S0, float* S1, gdn_tree_dims d, int32_t Lmax,
              int32_t* dev_status, SeqLayout lay) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int Nmax = d.N, dk = d.dk, dv = d.dv, Hv = d.Hv, Hqk = d.Hqk;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = path_capacity(Lmax);
  const int batch = batch_size(Lmax), nslot = batch_slots(Lmax);
  const uint32_t sb = slot_bytes(dv, (int)sizeof(T), Lmax);
  uint8_t* ws = smem + (size_t)warp * warp_smem_bytes(dv, (int)sizeof(T), Lmax);
  float* s_s = reinterpret_cast<float*>(ws);  // [R][dv]
  uint8_t* s_slots = ws + kMaxRows * dv * 4;
  auto slot_u = [&](int sl) { return reinterpret_cast<float*>(s_slots + sl * sb); };  // [batch][dv]
  auto slot_k = [&](int sl) { return reinterpret_cast<T*>(slot_u(sl) + batch * dv); };  // [batch][R]
  int* s_pj = reinterpret_cast<int*>(s_slots + nslot * sb);  // [cap]
  float* s_hi = reinterpret_cast<float*>(s_pj + cap);      // [cap]: G_j.hi, then w_j
  float* s_lo = s_hi + cap;                                // [cap]: G_j.lo

  // this warp's block: rows R rb .. R rb + R - 1 of state (b, h)
  const int R = block_rows(dk), rbs = dk / R;
  const long long item = (long long)blockIdx.x * kWarps + warp;
  if (item >= (long long)d.B * Hv * rbs) return;
  const int rb = (int)(item % rbs);
  const int unit = (int)(item / rbs), b = unit / Hv, h = unit - b * Hv, hq = h / (Hv / Hqk);
  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N < 0 || st < 0) {
    if (lane == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_LAYOUT);
    return;
  }
  const size_t row = (size_t)lay.row0(b, Nmax), urow = lay.urow0(b, h, Hv, Nmax);
  // lane c < dv/4 owns columns 4c .. 4c+3 of the block's rows
  const bool owner = lane < dv / 4;
  const size_t sbase = ((size_t)st * Hv + h) * dk * dv + (size_t)rb * R * dv;

  // ---- round trip 1: the block's S0 rows (into the slot), the path length and
  // its first 32 entries.  S0 and S1 may alias (in-place commit): the block's
  // rows are all on chip before any of its S1 rows is stored, and no two warps
  // share a row.
  for (int q = lane; q < R * dv / 4; q += 32) cp_async16(s_s + 4 * q, S0 + sbase + 4 * q);
  const int L = path_len[b];
  const int pj0 = lane < Lmax ? path[(size_t)b * Lmax + lane] : 0;

  // k (the block's R entries) and U rows of path entries j0 .. j0 + nj - 1
  // into slot sl, by 16-byte copies (one cp.async group)
  auto stage = [&](int j0, int nj, int sl) {
    const int uq = dv / 4, kq = R * (int)sizeof(T) / 16;
    float* su = slot_u(sl);
    T* sk = slot_k(sl);
    for (int q = lane; q < nj * uq; q += 32) {
      const int jj = q / uq, c = q - jj * uq;
      cp_async16(su + jj * dv + 4 * c, U + (urow + s_pj[j0 + jj]) * dv + 4 * c);
    }
    for (int q = lane; q < nj * kq; q += 32) {
      const int jj = q / kq, c = q - jj * kq;
      const T* src = k + ((row + s_pj[j0 + jj]) * Hqk + hq) * dk + rb * R;
      cp_async16(reinterpret_cast<uint8_t*>(sk + jj * R) + 16 * c,
                 reinterpret_cast<const uint8_t*>(src) + 16 * c);
    }
    cp_async_commit();
  };

  // ---- round trip 2, 32 entries (one a lane) at a time: range check; the
  // first batch of k / U rows; log alpha and parent links; chain check (a
  // root-to-node path is strictly increasing in a topological order and, with
  // the tree given, follows the parent links); G_j, the inclusive double-float
  // prefix sums of log alpha along the path
  int bad = (L < 0 || L > N || L > Lmax);
  const int nL = bad ? 0 : L;
  // the entries of the path's first kPre chunks come together (one a lane a
  // chunk), then their log alpha and parent links together; chunks past those
  // are fetched as they are reached
  int pjr[kPre];
  pjr[0] = pj0;
#pragma unroll
  for (int i = 1; i < kPre; ++i) {
    const int e = 32 * i + lane;
    pjr[i] = e < nL ? path[(size_t)b * Lmax + e] : 0;
  }
  {
    int oor = 0;
#pragma unroll
    for (int i = 0; i < kPre; ++i) oor |= (32 * i + lane < nL) && (pjr[i] < 0 || pjr[i] >= N);
    if (__any_sync(0xffffffffu, oor)) bad = 1;
  }
  const int nLc = bad ? 0 : nL;  // (entries known to be in range from here on)
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
  if (nLc > 0) {  // the first batch's rows start coming
    __syncwarp();
    stage(0, min(batch, nLc), 0);
  }
  df carry = {0.f, 0.f};
  int last = -1;  // the previous chunk's last entry
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
    if (ci >= kPre) {
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
    const df G = df_add(carry, warp_inclusive_scan(df{la, 0.f}, lane));
    if (live) {
      s_hi[e] = G.hi;
      s_lo[e] = G.lo;
    }
    // (lanes past the path add zeros: lane 31 holds G of the chunk's last entry)
    carry.hi = __shfl_sync(0xffffffffu, G.hi, 31);
    carry.lo = __shfl_sync(0xffffffffu, G.lo, 31);
    last = __shfl_sync(0xffffffffu, pj, 31);
  }
  if (bad) {
    cp_async_wait_all();  // the S0 rows and the copies of a batch already staged
    if (lane == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_PATH);
    return;  // S1 left unwritten
  }

  // ---- w_j = exp(G_L - G_j), gamma_L = exp(G_L) (G_L = carry; each lane
  // rewrites the entries it wrote)
  for (int e = lane; e < nL; e += 32) s_hi[e] = expf(df_diff(carry, df{s_hi[e], s_lo[e]}));
  const float gamma = expf(df_value(carry));

  // ---- S1 = gamma S0 + K_P^T diag(w) U_P on the block's rows, kRB rows (a
  // pass) at a time; paths past one batch of entries keep the partial sums of
  // the earlier batches in the S0 slot
  const int nb = nL == 0 ? 1 : (nL + batch - 1) / batch;
  for (int bi = 0; bi < nb; ++bi) {
    const int j0 = bi * batch, nj = min(batch, nL - j0);
    const int sl = nslot == 2 ? (bi & 1) : 0;
    if (nslot == 2) {
      // two slots: batch bi + 1 is copied into the other slot (free: batch bi - 1
      // was formed from it) while batch bi is formed
      if (bi + 1 < nb) {
        __syncwarp();
        stage(j0 + batch, min(batch, nL - j0 - batch), sl ^ 1);
        cp_async_wait_but_last();
      } else {
        cp_async_wait_all();
      }
    } else {
      if (bi > 0) {  // one slot: the next batch's rows, here and now
        __syncwarp();
        stage(j0, nj, 0);
      }
      cp_async_wait_all();
    }
    __syncwarp();  // every lane's copies (and weights) in place
    const float* s_u = slot_u(sl);
    const T* s_k = slot_k(sl);
    if (owner) {
      const bool first = bi == 0, final_ = bi == nb - 1;
      for (int r0 = 0; r0 < R; r0 += kRB) {
        float acc[kRB][4];
#pragma unroll
        for (int i = 0; i < kRB; ++i)
#pragma unroll
          for (int c = 0; c < 4; ++c) acc[i][c] = 0.f;
        for (int jj = 0; jj < nj; ++jj) {
          const float w = s_hi[j0 + jj];
          const float4 uv = *reinterpret_cast<const float4*>(s_u + jj * dv + 4 * lane);
          float kv[kRB];
          load_k(s_k + jj * R + r0, kv);
#pragma unroll
          for (int i = 0; i < kRB; ++i) {
            const float kk = w * kv[i];
            acc[i][0] = fmaf(kk, uv.x, acc[i][0]);
            acc[i][1] = fmaf(kk, uv.y, acc[i][1]);
            acc[i][2] = fmaf(kk, uv.z, acc[i][2]);
            acc[i][3] = fmaf(kk, uv.w, acc[i][3]);
          }
        }
#pragma unroll
        for (int i = 0; i < kRB; ++i) {
          float4* sp = reinterpret_cast<float4*>(s_s + (r0 + i) * dv + 4 * lane);
          const float4 s = *sp;
          const float4 v =
              first ? make_float4(fmaf(gamma, s.x, acc[i][0]), fmaf(gamma, s.y, acc[i][1]),
                                  fmaf(gamma, s.z, acc[i][2]), fmaf(gamma, s.w, acc[i][3]))
                    : make_float4(s.x + acc[i][0], s.y + acc[i][1], s.z + acc[i][2],
                                  s.w + acc[i][3]);
          if (final_)
            __stcs(reinterpret_cast<float4*>(S1 + sbase + (size_t)(r0 + i) * dv + 4 * lane), v);
          else
            *sp = v;
        }
      }
    }
  }
}

}  // namespace

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  int n = (dev >= 0 && dev < 64) ? cached[dev].load(std::memory_order_relaxed) : 0;
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

cudaError_t launch_commit_warp(const CommitArgs& a, cudaStream_t stream) {
  const long long n_blocks = (long long)a.d.B * a.d.Hv * (a.d.dk / block_rows(a.d.dk));
  if (n_blocks == 0) return cudaSuccess;
  const long long grid = (n_blocks + kWarps - 1) / kWarps;
  if (grid > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  const int tsize = a.d.dtype == GDN_TREE_BF16 ? 2 : 4;
  const size_t smem = (size_t)kWarps * warp_smem_bytes(a.d.dv, tsize, a.Lmax);
  cudaError_t err;
  if (a.d.dtype == GDN_TREE_BF16) {
    err = cudaFuncSetAttribute(commit_kernel<__nv_bfloat16>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    commit_kernel<__nv_bfloat16><<<(unsigned)grid, kThreads, smem, stream>>>(
        a.path, a.path_len, a.parent, a.U, static_cast<const __nv_bfloat16*>(a.k),
        a.log_alpha, a.S0, a.S1, a.d, a.Lmax, a.dev_status, a.lay);
  } else {
    err = cudaFuncSetAttribute(commit_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem);
    if (err != cudaSuccess) return err;
    commit_kernel<float><<<(unsigned)grid, kThreads, smem, stream>>>(
        a.path, a.path_len, a.parent, a.U, static_cast<const float*>(a.k),
        a.log_alpha, a.S0, a.S1, a.d, a.Lmax, a.dev_status, a.lay);
  }
  return cudaGetLastError();
}

}  // namespace gdn
