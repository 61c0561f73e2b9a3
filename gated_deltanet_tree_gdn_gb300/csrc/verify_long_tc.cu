// verify_long_tc.cu -- tree verification of bf16 trees longer than the on-chip
// kernels take (up to kMaxNLong nodes) with dk = dv = 128: the two-level chunk
// pass with R and the output seeds on the tensor cores.
//
// Method: "DFlash-TfM: Trees from Marginals", section 3 ("Soluzione"): with
// g_t the log-decay summed along the root-to-t path and gamma_t = e^{g_t},
//   R = diag(beta)(V - diag(gamma) K S0),   (I + X) U = R,
//   O = diag(gamma) Q S0 + Y U,
//   X[t,s] = beta_t e^{g_t - g_s} k_t.k_s   (s a strict ancestor of t),
//   Y[t,s] = e^{g_t - g_s} q_t.k_s         (s on the root-to-t path, t included).
//
// One CTA (512 threads) per (sequence b, v-head h).  The tree's parent links are
// checked; pointer jumping gives g, the depths and, kept level by level, the
// ancestor at every power-of-two distance (so a node's ancestor at any depth is a
// few lookups away; 38 bytes of shared memory a node, no bitsets).  S0 is split
// once into bf16 hi + lo (MN-major, 128-byte swizzle) and stays in shared memory.
// The nodes are cut in index (a topological) order into chunks of 128; for each
// chunk
//  1. its K and Q rows land as 128-row K-major tiles (cp.async; rows past the
//     tree zero); one thread issues K S0_hi + K S0_lo and Q S0_hi + Q S0_lo
//     (tcgen05.mma) into 256 TMEM columns; the warps read them back by TMEM lane
//     group, a thread per node: r_t = beta_t (v_t - gamma_t (K S0)_t) goes to the
//     chunk's U rows in shared memory (where the tiles were), the seed
//     gamma_t (Q S0)_t to t's row of U in global memory;
//  2. the chunk's nodes, in depth order, take a warp each as a streaming
//     dataflow.  The node's path goes root first, 32 entries at a time, an entry
//     a lane.  X[t,s] and Y[t,s] come from warp dots of k_s with k_t and q_t (the k
//     rows load whole, eight entries' sixteen sums reduced across the lanes
//     together).  The terms u_t -= X[t,s] u_s and o_t += Y[t,s] u_s follow: rows
//     of earlier chunks from U in global memory, eight at a time (final since the
//     chunk boundary's block barrier), then rows of this chunk from shared memory,
//     four at a time after a bounded wait on the mbarrier of the last of the four
//     (a path's nodes complete in path order).  The node's own term closes o_t;
//     u_t replaces the seed in U and joins the chunk's rows, and the node's
//     barrier is arrived on.
// The unfinished node of lowest depth order in a chunk never waits on an
// unfinished node, so the waits cannot cycle.
//
// Units whose tree is one chain are verified by verify_chain_kernel (this file,
// launched first; the chunkwise form of chain_unit.cuh) and left by the chunk pass.
#include <algorithm>

#include "chain_unit.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kD = 128;      // dk = dv
constexpr int kChunk = 128;  // nodes a chunk: one M = 128 tile
constexpr int kNodesPerThread = kMaxNLong / kThreads;
static_assert(kMaxNLong % kThreads == 0, "pointer jumping assigns whole nodes per thread");
constexpr int kTmemCols = 256;
// ancestor tables for the distances 2^0 .. 2^10 (every distance below kMaxNLong)
constexpr int kLiftLevels = 11;
static_assert((1 << (kLiftLevels - 1)) >= kMaxNLong, "a distance needs at most kLiftLevels - 1 bits");

struct LongTcSmem {
  // byte offsets into dynamic shared memory, from a 1024-byte aligned base
  size_t SK, T, V, lift, depth, g, beta, order, bar, flag, total;
};

__host__ __device__ inline size_t align16t(size_t x) { return (x + 15) & ~size_t(15); }

__host__ __device__ inline LongTcSmem long_tc_smem_layout(int N) {
  LongTcSmem L;
  size_t o = 0;
  L.SK = o;     o += sizeof(float) * kD * kD;       // S0 (fp32), then its hi / lo operands
  L.T = o;      o += sizeof(float) * kChunk * kD;   // K, Q tiles; then the chunk's R / U rows
  L.V = o;      o += sizeof(uint16_t) * kChunk * kD;  // the chunk's v rows (bf16, swizzled)
  L.lift = o;   o = align16t(o + sizeof(int16_t) * kLiftLevels * N);  // [level][node]
  L.depth = o;  o = align16t(o + sizeof(int) * N);
  L.g = o;      o = align16t(o + sizeof(df) * N);
  L.beta = o;   o = align16t(o + sizeof(float) * N);
  L.order = o;  o = align16t(o + sizeof(int) * kChunk);
  L.bar = o;    o = align16t(o + sizeof(uint64_t) * kChunk);
  L.flag = o;   o = align16t(o + sizeof(uint64_t) * 2);  // status flag, TMEM base; MMA barrier
  L.total = o + 1024;  // + alignment slack
  return L;
}

// byte offset of 16-byte chunk c (of 16) of row r in the staged v rows (chunks
// XOR-swizzled by the row, so that 32 threads reading one chunk of 32 rows meet
// two at a bank group at most)
__device__ __forceinline__ uint32_t v_chunk(int r, int c) {
  return (uint32_t)r * (kD * 2) + (uint32_t)((c ^ (r & 15)) << 4);
}

__device__ __forceinline__ void cp_async16t(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_addr(dst)),
               "l"(src)
               : "memory");
}

__device__ __forceinline__ void bf16x8_to_f32t(const uint4 q, float (&v)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// four bf16 elements (as loaded) as fp32
__device__ __forceinline__ float4 bf16x4_to_f32t(uint2 raw) {
  return make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                     __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u));
}

__device__ __forceinline__ float dot4t(float4 a, float4 b) {
  return fmaf(a.w, b.w, fmaf(a.z, b.z, fmaf(a.y, b.y, a.x * b.x)));
}

// acc + a x, as two packed fp32x2 FMAs (same rounding as four fmaf)
__device__ __forceinline__ float4 fma4t(float a, float4 x, float4 acc) {
  const float2 aa = make_float2(a, a);
  const float2 lo = __ffma2_rn(aa, make_float2(x.x, x.y), make_float2(acc.x, acc.y));
  const float2 hi = __ffma2_rn(aa, make_float2(x.z, x.w), make_float2(acc.z, acc.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__global__ void __launch_bounds__(kThreads, 1)
verify_long_tc_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                      const __nv_bfloat16* __restrict__ v, const float* __restrict__ log_alpha,
                      const float* __restrict__ beta, const int32_t* __restrict__ parent,
                      const float* __restrict__ S0, __nv_bfloat16* __restrict__ o, float* U,
                      gdn_tree_dims d, int32_t* dev_status, SeqLayout lay, WaitHooks hk,
                      int skip_chains) {
  // U is read back (seeds, earlier chunks' rows) after this CTA wrote it, so it is
  // neither const nor restrict: its loads must not take the read-only path.
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  const int Nmax = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y;
  const int hq = h / (Hv / Hqk);
  const int unit = b * Hv + h;
  const LongTcSmem L = long_tc_smem_layout(Nmax);
  unsigned char* sSK = smem + L.SK;
  unsigned char* sT = smem + L.T;
  unsigned char* sV = smem + L.V;
  int16_t* sLift = reinterpret_cast<int16_t*>(smem + L.lift);  // [0]: the parent links
  int* sDepth = reinterpret_cast<int*>(smem + L.depth);
  df* sG = reinterpret_cast<df*>(smem + L.g);
  float* sBeta = reinterpret_cast<float*>(smem + L.beta);
  int* sOrder = reinterpret_cast<int*>(smem + L.order);
  uint64_t* sBar = reinterpret_cast<uint64_t*>(smem + L.bar);
  int* sFlag = reinterpret_cast<int*>(smem + L.flag);  // [0] status flag, [1] TMEM base
  uint64_t* sBarMma = reinterpret_cast<uint64_t*>(smem + L.flag) + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N < 0 || st < 0) {
    if (h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_LAYOUT);
    return;
  }
  const size_t row = (size_t)lay.row0(b, Nmax);
  float* Ubh = U + lay.urow0(b, h, Hv, Nmax) * kD;
  if (skip_chains && N > 0) {  // one chain: verify_chain_kernel's (before any copy starts)
    int notchain = 0;
    for (int t = tid; t < N; t += kThreads) notchain |= parent[row + t] != t - 1;
    if (!__syncthreads_or(notchain)) return;
  }

  // S0 starts streaming into shared memory (fp32) at once
  const float* S0bh = S0 + ((size_t)st * Hv + h) * kD * kD;
  for (int i = tid; i < kD * kD / 4; i += kThreads) cp_async16t(sSK + 16 * i, S0bh + 4 * i);
  asm volatile("cp.async.commit_group;" ::: "memory");

  // ---- the tree: load, validate, seed the pointer jumping -------------------------
  int bad = 0;
  for (int t = tid; t < N; t += kThreads) {
    const int p = parent[row + t];
    sLift[t] = (int16_t)p;
    sDepth[t] = 1;
    sG[t] = df{log_alpha[(row + t) * Hv + h], 0.f};
    sBeta[t] = beta[(row + t) * Hv + h];
    bad |= (p < -1 || p >= t);
  }
  if (tid == 0) sFlag[0] = 0;
  if (tid < kChunk) sm100::mbar_init(&sBar[tid], 1);
  if (tid == 0) sm100::mbar_init(sBarMma, 1);
  sm100::mbar_fence_init();
  bad = __syncthreads_or(bad);
  if (bad) {
    if (h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_TREE);
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }
  // the tree is valid: TMEM for the chunk's two accumulators
  if (warp == 0) sm100::tmem_alloc(reinterpret_cast<uint32_t*>(sFlag + 1), kTmemCols);

  // ---- pointer jumping: g_t = sum of log alpha over P(t), depth_t = |P(t)|; level
  // i + 1 of the ancestor table (distance 2^(i+1)) from level i.  A level past the
  // last one built is never read: every distance asked for is below the depth.
  for (int i = 0; i + 1 < kLiftLevels; ++i) {
    const int16_t* lv = sLift + (size_t)i * Nmax;
    int j[kNodesPerThread], jj[kNodesPerThread], dj[kNodesPerThread];
    df gj[kNodesPerThread];
    int live = 0;
#pragma unroll
    for (int m = 0; m < kNodesPerThread; ++m) {
      const int t = tid + m * kThreads;
      j[m] = t < N ? lv[t] : -1;
      jj[m] = -1;
      if (j[m] >= 0) {
        jj[m] = lv[j[m]];
        dj[m] = sDepth[j[m]];
        gj[m] = sG[j[m]];
        live = 1;
      }
    }
    if (!__syncthreads_or(live)) break;  // every node reached its root
#pragma unroll
    for (int m = 0; m < kNodesPerThread; ++m) {
      const int t = tid + m * kThreads;
      if (t < N) sLift[(size_t)(i + 1) * Nmax + t] = (int16_t)jj[m];
      if (j[m] >= 0) {
        sG[t] = df_add(sG[t], gj[m]);
        sDepth[t] += dj[m];
      }
    }
    __syncthreads();
  }

  // ---- S0 = hi + lo (bf16), MN-major (K = dk rows, N = dv columns), in place ---------
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  {
    float sv[4][8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int qd = j * kThreads + tid, i = qd >> 4, n8 = qd & 15;  // a warp: two whole rows
      const float4 a = *reinterpret_cast<const float4*>(sSK + (i * kD + 8 * n8) * 4);
      const float4 c = *reinterpret_cast<const float4*>(sSK + (i * kD + 8 * n8 + 4) * 4);
      sv[j][0] = a.x; sv[j][1] = a.y; sv[j][2] = a.z; sv[j][3] = a.w;
      sv[j][4] = c.x; sv[j][5] = c.y; sv[j][6] = c.z; sv[j][7] = c.w;
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int qd = j * kThreads + tid, i = qd >> 4, n8 = qd & 15;  // a warp: two whole rows
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) sm100::split2(sv[j][2 * e], sv[j][2 * e + 1], hi[e], lo[e]);
      *reinterpret_cast<uint4*>(sSK + sm100::mn_chunk(i, n8)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(sSK + 32768 + sm100::mn_chunk(i, n8)) =
          make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
  }
  sm100::tc_fence_before_sync();
  __syncthreads();
  sm100::tc_fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(sFlag[1]);

  bool timed_out = false;
  const int c4 = lane * 4;  // this lane's elements of a k / q row and columns of a u row
  // the chunk's row tl of R / U (fp32, 128-byte swizzled boxes of 32 columns)
  auto urow_s = [&](int tl) { return reinterpret_cast<float4*>(sT + sm100::u_off(tl, lane)); };

  for (int c0 = 0, ci = 0; c0 < N; c0 += kChunk, ++ci) {
    const int nc = min(kChunk, N - c0);
    const uint32_t parity = (uint32_t)(ci & 1);
    // ---- 1. the chunk's K and Q tiles and v rows; R and the seeds on the tensor cores
    for (int e = tid; e < 2 * kChunk * 16; e += kThreads) {
      const int ch = e & 15, rq = e >> 4, isq = rq >> 7, r = rq & (kChunk - 1);
      unsigned char* dst = sT + isq * 32768 + sm100::sw128_chunk(r, ch);
      if (r < nc)
        cp_async16t(dst, (isq ? q : k) + ((row + c0 + r) * Hqk + hq) * kD + 8 * ch);
      else
        *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int e = tid; e < nc * 16; e += kThreads) {
      const int ch = e & 15, r = e >> 4;
      cp_async16t(sV + v_chunk(r, ch), v + ((row + c0 + r) * Hv + h) * kD + 8 * ch);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    // the chunk's depth order (index order within a depth)
    if (tid < nc) {
      const int dep = sDepth[c0 + tid];
      int rank = 0;
      for (int j = 0; j < nc; ++j) {
        const int dj = sDepth[c0 + j];
        rank += (dj < dep) || (dj == dep && j < tid);
      }
      sOrder[rank] = tid;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    sm100::fence_proxy_async_smem();
    sm100::tc_fence_before_sync();
    __syncthreads();
    sm100::tc_fence_after_sync();
    // TMEM columns: K S0 0..127, Q S0 128..255 (node r of the chunk in lane r)
    if (tid == 0) {
      const uint32_t kt = sm100::smem_addr(sT), qt = kt + 32768, sb = sm100::smem_addr(sSK);
      sm100::umma_128x128x128_bmn(tmem, kt, sb, false);
      sm100::umma_128x128x128_bmn(tmem, kt, sb + 32768, true);
      sm100::umma_128x128x128_bmn(tmem + 128, qt, sb, false);
      sm100::umma_128x128x128_bmn(tmem + 128, qt, sb + 32768, true);
      sm100::umma_commit(sBarMma);
    }
    if (!sm100::mbar_wait(sBarMma, parity, hk.limit_ns)) {
      // (bounded again: the MMAs must be done before TMEM is read or freed)
      sm100::mbar_wait(sBarMma, parity, hk.limit_ns);
      timed_out = true;
    }
    sm100::tc_fence_after_sync();
    {
      // warp w reads accumulator (w / 4) % 2 (K S0, Q S0), columns 64 (w / 8) ..
      // +63, for its TMEM lane group w % 4: thread = node
      const int acc = (warp >> 2) & 1, lg = warp & 3, half = warp >> 3;
      const int tl = lg * 32 + lane, t = c0 + tl;
      const bool live = tl < nc;
      const float gam = live ? expf(df_value(sG[t])) : 0.f;
      const float bt = live ? sBeta[t] : 0.f;
      const uint32_t taddr = tmem + ((uint32_t)(lg * 32) << 16) + 128 * acc + 64 * half;
#pragma unroll 1
      for (int c32 = 0; c32 < 2; ++c32) {
        float r[32];
        sm100::tmem_ld_32cols(taddr + 32 * c32, r);  // warp-collective: every lane
        if (!live) continue;
        const int col0 = 64 * half + 32 * c32;
        if (acc == 0) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            float vv[8];
            bf16x8_to_f32t(*reinterpret_cast<const uint4*>(sV + v_chunk(tl, col0 / 8 + m)), vv);
            const int cc = col0 / 4 + 2 * m;
            *reinterpret_cast<float4*>(sT + sm100::u_off(tl, cc)) =
                make_float4(bt * (vv[0] - gam * r[8 * m]), bt * (vv[1] - gam * r[8 * m + 1]),
                            bt * (vv[2] - gam * r[8 * m + 2]), bt * (vv[3] - gam * r[8 * m + 3]));
            *reinterpret_cast<float4*>(sT + sm100::u_off(tl, cc + 1)) =
                make_float4(bt * (vv[4] - gam * r[8 * m + 4]), bt * (vv[5] - gam * r[8 * m + 5]),
                            bt * (vv[6] - gam * r[8 * m + 6]), bt * (vv[7] - gam * r[8 * m + 7]));
          }
        } else {
          float4* sr = reinterpret_cast<float4*>(Ubh + (size_t)t * kD + col0);
#pragma unroll
          for (int m = 0; m < 8; ++m)
            sr[m] = make_float4(gam * r[4 * m], gam * r[4 * m + 1], gam * r[4 * m + 2],
                                gam * r[4 * m + 3]);
        }
      }
    }
    sm100::tc_fence_before_sync();
    __syncthreads();  // R rows and seeds in place; TMEM free for the next chunk

    // the next chunk's k, q and v rows start coming into L2 during this solve
    if (c0 + kChunk < N) {
      const int n1 = min(kChunk, N - c0 - kChunk);
      for (int e = tid; e < 3 * n1; e += kThreads) {
        const int which = e / n1, r = c0 + kChunk + e - which * n1;
        const __nv_bfloat16* src = which == 2 ? v + ((row + r) * Hv + h) * kD
                                              : (which ? q : k) + ((row + r) * Hqk + hq) * kD;
        sm100::bulk_prefetch_l2(src, kD * 2);
      }
    }
    // ---- 2. the chunk's solve: a warp per node, depth order, streaming waits ------
    // k_t and q_t of the warp's next node, loaded one node ahead
    auto kq_of = [&](int task, uint2& kr, uint2& qr) {
      kr = qr = make_uint2(0u, 0u);
      if (task < nc) {
        const size_t tk = ((row + c0 + sOrder[task]) * Hqk + hq) * kD + c4;
        kr = *reinterpret_cast<const uint2*>(k + tk);
        qr = *reinterpret_cast<const uint2*>(q + tk);
      }
    };
    uint2 knext, qnext;
    kq_of(warp, knext, qnext);
    for (int task = warp; task < nc; task += kWarps) {
      const int tl = sOrder[task], t = c0 + tl;
      const int nA = sDepth[t] - 1;  // strict ancestors
      const df gt = sG[t];
      const float bt = sBeta[t];
      const float4 kt = bf16x4_to_f32t(knext), qt = bf16x4_to_f32t(qnext);
      kq_of(task + kWarps, knext, qnext);
      float* urow = Ubh + (size_t)t * kD + c4;
      const float4 seed = *reinterpret_cast<const float4*>(urow);
      float4 u = *urow_s(tl);  // r_t
      float4 au = make_float4(0.f, 0.f, 0.f, 0.f), ao = au;
      // the path root first, 32 entries at a time: entry n is the ancestor at depth
      // n + 1, in lane n % 32
      for (int n0 = 0; n0 < nA; n0 += 32) {
        const int cnt = min(32, nA - n0);
        int a = t;
        if (lane < cnt) {
          for (int m = nA - n0 - lane, bit = 0; m; m >>= 1, ++bit)
            if (m & 1) a = sLift[(size_t)bit * Nmax + a];
        }
        // entries of earlier chunks: a prefix (indices fall along a path)
        const int nE = __popc(__ballot_sync(0xffffffffu, lane < cnt && a < c0));
        // the first eight earlier-chunk u rows start coming
        float4 ue[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int ss = __shfl_sync(0xffffffffu, a, jj);
          ue[jj] = jj < nE ? *reinterpret_cast<const float4*>(Ubh + (size_t)ss * kD + c4)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // X[t,a] and Y[t,a] before their factors: the dots of k_a with k_t and q_t,
        // eight entries at a time as warp dots (a lane holds 4 of the 128 elements,
        // the k rows load whole), the sixteen sums reduced across the lanes at once:
        // each exchange step halves the values a lane carries, so that lane L ends
        // with value L / 2 (entry L / 4; its k dot for L / 2 even, its q dot for odd)
        float dkk = 0.f, dqk = 0.f;
        for (int j0 = 0; j0 < cnt; j0 += 16) {
          // sixteen k rows in flight at once (one round trip for paths of up to 16
          // entries), then two groups of eight dots
          uint2 kr[16];
#pragma unroll
          for (int jj = 0; jj < 16; ++jj) {
            const int ss = __shfl_sync(0xffffffffu, a, (j0 + jj) & 31);
            kr[jj] = j0 + jj < cnt
                         ? *reinterpret_cast<const uint2*>(k + ((row + ss) * Hqk + hq) * kD + c4)
                         : make_uint2(0u, 0u);
          }
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int j1 = j0 + 8 * half;
            if (j1 >= cnt) break;  // (uniform)
            float vs[16];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const float4 ks = bf16x4_to_f32t(kr[8 * half + jj]);
              vs[2 * jj] = dot4t(kt, ks);
              vs[2 * jj + 1] = dot4t(qt, ks);
            }
#pragma unroll
            for (int w = 8; w >= 1; w >>= 1) {  // 16 -> 8 -> 4 -> 2 -> 1 values a lane
              const bool up = (lane >> 1) & w;  // this lane keeps the upper half
#pragma unroll
              for (int i = 0; i < w; ++i) {
                const float keep = up ? vs[w + i] : vs[i];
                const float send = up ? vs[i] : vs[w + i];
                vs[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2 * w);
              }
            }
            vs[0] += __shfl_xor_sync(0xffffffffu, vs[0], 1);
            // entry j1 + i: its k dot in lane 4 i, its q dot in lane 4 i + 2
            const int i = lane - j1;
            const float xk = __shfl_sync(0xffffffffu, vs[0], (4 * i) & 31);
            const float yq = __shfl_sync(0xffffffffu, vs[0], (4 * i + 2) & 31);
            if (i >= 0 && i < 8) {
              dkk = xk;
              dqk = yq;
            }
          }
        }
        float xe = 0.f, ye = 0.f;
        if (lane < cnt) {
          const float dec = expf(df_diff(gt, sG[a]));
          xe = bt * dec * dkk;
          ye = dec * dqk;
        }
        // the earlier chunks' terms (final rows, no wait), eight at a time
        for (int j0 = 0; j0 < nE; j0 += 8) {
          if (j0 > 0) {
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const int ss = __shfl_sync(0xffffffffu, a, (j0 + jj) & 31);
              ue[jj] = j0 + jj < nE ? *reinterpret_cast<const float4*>(Ubh + (size_t)ss * kD + c4)
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
#pragma unroll
          for (int jj = 0; jj < 8; ++jj) {
            const float xx = __shfl_sync(0xffffffffu, xe, (j0 + jj) & 31);
            const float yy = __shfl_sync(0xffffffffu, ye, (j0 + jj) & 31);
            const bool use = j0 + jj < nE;
            au = fma4t(use ? -xx : 0.f, ue[jj], au);
            ao = fma4t(use ? yy : 0.f, ue[jj], ao);
          }
        }
        // this chunk's terms, four entries at a time: the rows must be final first;
        // the last of the four is the deepest, and a path's nodes complete in path
        // order, so its being final makes all four final
        for (int j0 = nE; j0 < cnt; j0 += 4) {
          const int m = min(4, cnt - j0);
          const int alast = __shfl_sync(0xffffffffu, a, j0 + m - 1);
          if (!sm100::mbar_wait(&sBar[alast - c0], parity, hk.limit_ns)) timed_out = true;
          float4 us[4];
          float xj[4], yj[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int ss = __shfl_sync(0xffffffffu, a, (j0 + jj) & 31);
            const float xx = __shfl_sync(0xffffffffu, xe, (j0 + jj) & 31);
            const float yy = __shfl_sync(0xffffffffu, ye, (j0 + jj) & 31);
            const bool use = jj < m;
            xj[jj] = use ? xx : 0.f;
            yj[jj] = use ? yy : 0.f;
            us[jj] = *urow_s(use ? ss - c0 : tl);
          }
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            au = fma4t(-xj[jj], us[jj], au);
            ao = fma4t(yj[jj], us[jj], ao);
          }
        }
      }
      u.x += au.x;
      u.y += au.y;
      u.z += au.z;
      u.w += au.w;
      // the node's own term Y[t,t] u_t = (q_t . k_t) u_t
      const float self = warp_sum(dot4t(qt, kt));
      ao = fma4t(self, u, ao);
      *urow_s(tl) = u;
      *reinterpret_cast<float4*>(urow) = u;
      __nv_bfloat16* orow = o + ((row + t) * Hv + h) * kD + c4;
      const __nv_bfloat162 p01 = __floats2bfloat162_rn(seed.x + ao.x, seed.y + ao.y);
      const __nv_bfloat162 p23 = __floats2bfloat162_rn(seed.z + ao.z, seed.w + ao.w);
      *reinterpret_cast<uint2*>(orow) = make_uint2(*reinterpret_cast<const uint32_t*>(&p01),
                                                   *reinterpret_cast<const uint32_t*>(&p23));
      __syncwarp();  // every lane's part of u_t is in place before the arrival
      if (lane == 0 && !(unit == hk.withhold_unit && t == hk.withhold_node))
        sm100::mbar_arrive(&sBar[tl]);
    }
    __syncthreads();  // the chunk's U rows are final in global memory; its region is reused
  }
  if (timed_out) atomicOr(sFlag, 1);
  sm100::tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) sm100::tmem_dealloc(tmem, kTmemCols);
  if (tid == 0 && sFlag[0] && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_TIMEOUT);
}

// The units of trees past 256 nodes whose tree is one chain, in the chunkwise form
// (launched ahead of the chunk pass, which then leaves them; a separate kernel, so
// that the chunk pass keeps its own register allocation).  Other units leave at once.
__global__ void __launch_bounds__(kThreads, 1)
verify_chain_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, const float* __restrict__ log_alpha,
                    const float* __restrict__ beta, const int32_t* __restrict__ parent,
                    const float* __restrict__ S0, __nv_bfloat16* __restrict__ o, float* U,
                    gdn_tree_dims d, int32_t* dev_status, SeqLayout lay, WaitHooks hk) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  const int Nmax = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N <= 0 || st < 0) return;  // (a bad layout is the chunk pass's to report)
  const size_t row = (size_t)lay.row0(b, Nmax);
  int notchain = 0;
  for (int t = tid; t < N; t += kThreads) notchain |= parent[row + t] != t - 1;
  if (__syncthreads_or(notchain)) return;
  chain::run(smem, q, k, v, log_alpha, beta, S0, o, U + lay.urow0(b, h, Hv, Nmax) * kD, N, Nmax,
             row, st, b, h, Hv, Hqk, dev_status, hk);
}

}  // namespace

bool verify_long_tc_supported(const gdn_tree_dims& d) {
  return d.dtype == GDN_TREE_BF16 && d.dk == kD && d.dv == kD && d.N >= 1 && d.N <= kMaxNLong &&
         long_tc_smem_layout(d.N).total <= 227 * 1024;
}

cudaError_t launch_verify_long_tc(const VerifyArgs& a, cudaStream_t stream) {
  const size_t smem = long_tc_smem_layout(a.d.N).total;
  if (a.chains) {
    const size_t csmem = chain::smem_bytes(a.d.N);
    cudaError_t err = cudaFuncSetAttribute(verify_chain_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)csmem);
    if (err != cudaSuccess) return err;
    verify_chain_kernel<<<dim3(a.d.Hv, a.d.B), kThreads, csmem, stream>>>(
        static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
        static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
        static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status, a.lay, wait_hooks());
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  const dim3 grid(a.d.Hv, a.d.B);
  cudaError_t err = cudaFuncSetAttribute(verify_long_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  verify_long_tc_kernel<<<grid, kThreads, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
      static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status, a.lay, wait_hooks(),
      a.chains ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace gdn
