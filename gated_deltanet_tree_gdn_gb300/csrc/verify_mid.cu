// verify_mid.cu -- tree verification for bf16 trees of up to 256 nodes with
// dk = dv = 128: the trees the tensor-core kernel (up to 128 nodes) does not take.
//
// Method: "DFlash-TfM: Trees from Marginals", section 3 ("Soluzione"): with
// g_t the log-decay summed along the root-to-t path and gamma_t = e^{g_t},
//   R = diag(beta)(V - diag(gamma) K S0),   (I + X) U = R,
//   O = diag(gamma) Q S0 + Y U,
//   X[t,s] = beta_t e^{g_t - g_s} k_t.k_s   (s a strict ancestor of t),
//   Y[t,s] = e^{g_t - g_s} q_t.k_s         (s on the root-to-t path, t included).
//
// One CTA (512 threads) per (sequence b, v-head h), in four stages:
//  1. the tree: parent links checked; strict-ancestor bitsets and g by pointer
//     jumping; depths, and the nodes grouped by depth (the solve's task order);
//  2. R and the output seeds gamma_t q_t^T S0 for every node at once, on the
//     tensor cores: K and Q (two 128-row tiles each, 128-byte swizzled K-major)
//     and S0 = hi + lo (bf16, MN-major) in shared memory, K S0_hi + K S0_lo and
//     Q S0_hi into the 512 TMEM columns by tcgen05.mma, read back by row (a
//     thread per node, warps by TMEM lane group); R stays in shared memory, the
//     seeds park in the node's U row in global memory (overwritten by u_t at
//     the end);
//  3. K into shared memory (bf16, 16-byte chunks XOR-swizzled by row, so that
//     32 lanes reading 32 rows at once hit distinct banks);
//  4. the solve as a streaming dataflow over the tree, one warp per node in
//     depth order: lane j forms X[t,s] and Y[t,s] for the path entries
//     s = j, j+32, ... from the k rows on chip (no wait: K is static); then the
//     warp walks t's path from the root, four ancestors at a time, waiting
//     (bounded, on an mbarrier) only for the last of the four -- a path's nodes
//     complete in path order -- and sums their terms into u_t and o_t (lane owns
//     4 of the 128 columns); u_t is published and t's mbarrier arrived on, and
//     o_t = seed + sum Y u closes the node.  A node keeps pace with its
//     ancestors as they complete, so a link of a deep chain costs one group of
//     terms, not the whole ancestor sum.
// The unfinished node of lowest depth order never waits on an unfinished node,
// so the waits cannot cycle.
#include <algorithm>

#include "chain_unit.cuh"
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace gdn {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kD = 128;          // dk = dv
constexpr int kMidN = 256;       // largest tree
constexpr int kGroups = kMidN / 32;  // ancestor groups of 32 (one ancestor a lane)
static_assert(kMidN <= kMaxN, "tree_prepare's bitsets hold kMaxN nodes");

struct MidSmem {
  // byte offsets into dynamic shared memory
  size_t U, SK, stage, parent, jump, g, beta, la, anc, depth, order, bar, flag, total;
};

__host__ __device__ inline size_t align16m(size_t x) { return (x + 15) & ~size_t(15); }

// from a 1024-byte aligned base: the U region (the K, Q operand tiles of stage 2,
// then R / U) holds kMidN rows whatever the tree's size, since the four tiles
// fill it
__host__ __device__ inline MidSmem mid_smem_layout(int N) {
  MidSmem L;
  const int W = (N + 31) / 32;
  size_t o = 0;
  L.U = o;      o = align16m(o + sizeof(float) * kMidN * kD);       // K, Q tiles; R, then U
  L.SK = o;     o = align16m(o + sizeof(float) * kD * kD);          // S0, hi / lo; then K
  L.stage = o;  o = align16m(o + sizeof(float) * kWarps * kD);      // q_t of each warp
  L.parent = o; o = align16m(o + sizeof(int) * N);
  L.jump = o;   o = align16m(o + sizeof(int) * N);
  L.g = o;      o = align16m(o + sizeof(df) * N);
  L.beta = o;   o = align16m(o + sizeof(float) * N);
  L.la = o;     o = align16m(o + sizeof(float) * N);
  L.anc = o;    o = align16m(o + sizeof(uint32_t) * N * W);
  L.depth = o;  o = align16m(o + sizeof(int) * N);
  L.order = o;  o = align16m(o + sizeof(int) * (N + kMidN + 1));   // order, then level starts
  L.bar = o;    o = align16m(o + sizeof(uint64_t) * N);
  L.flag = o;   o = align16m(o + sizeof(uint64_t) * 2);  // status flag, TMEM base; MMA barrier
  L.total = o + 1024;  // + alignment slack
  return L;
}

// float offset of 4-float chunk c4 (of 32) of row t in the R / U rows: the chunk
// sits at slot c4 ^ (t % 32) of its row, so that 32 threads storing one chunk of 32
// consecutive rows (stage 2) and 32 lanes reading one row (the solve) both meet
// no bank conflict
__device__ __forceinline__ int u_at(int t, int c4) { return t * kD + 4 * (c4 ^ (t & 31)); }

// byte offset of 16-byte chunk c (of 16) of k row r in the swizzled K tile
__device__ __forceinline__ uint32_t k_chunk(int r, int c) {
  return (uint32_t)r * (kD * 2) + (uint32_t)((c ^ (r & 15)) << 4);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4 q, float (&v)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// acc + a x, as two packed fp32x2 FMAs (same rounding as four fmaf)
__device__ __forceinline__ float4 fma4m(float a, float4 x, float4 acc) {
  const float2 aa = make_float2(a, a);
  const float2 lo = __ffma2_rn(aa, make_float2(x.x, x.y), make_float2(acc.x, acc.y));
  const float2 hi = __ffma2_rn(aa, make_float2(x.z, x.w), make_float2(acc.z, acc.w));
  return make_float4(lo.x, lo.y, hi.x, hi.y);
}

__device__ __forceinline__ void cp_async16m(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sm100::smem_addr(dst)),
               "l"(src)
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
verify_mid_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                  const __nv_bfloat16* __restrict__ v, const float* __restrict__ log_alpha,
                  const float* __restrict__ beta, const int32_t* __restrict__ parent,
                  const float* __restrict__ S0, __nv_bfloat16* __restrict__ o,
                  float* __restrict__ U, gdn_tree_dims d, int32_t* dev_status, SeqLayout lay,
                  WaitHooks hk, int chains) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (sm100::smem_addr(smem_raw) & 1023u)) & 1023u);
  const int Nmax = d.N, Hv = d.Hv, Hqk = d.Hqk;
  const int h = blockIdx.x, b = blockIdx.y;
  const int hq = h / (Hv / Hqk);
  const int unit = b * Hv + h;
  const MidSmem L = mid_smem_layout(Nmax);
  float* sU = reinterpret_cast<float*>(smem + L.U);
  unsigned char* sSK = smem + L.SK;
  float* sStage = reinterpret_cast<float*>(smem + L.stage);
  int* sPar = reinterpret_cast<int*>(smem + L.parent);
  int* sJump = reinterpret_cast<int*>(smem + L.jump);
  df* sG = reinterpret_cast<df*>(smem + L.g);
  float* sBeta = reinterpret_cast<float*>(smem + L.beta);
  float* sLa = reinterpret_cast<float*>(smem + L.la);
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(smem + L.anc);
  int* sDepth = reinterpret_cast<int*>(smem + L.depth);
  int* sOrder = reinterpret_cast<int*>(smem + L.order);
  int* sLevel = sOrder + Nmax;  // [kMidN + 1]
  uint64_t* sBar = reinterpret_cast<uint64_t*>(smem + L.bar);
  int* sFlag = reinterpret_cast<int*>(smem + L.flag);  // [0] status flag, [1] TMEM base
  uint64_t* sBarMma = reinterpret_cast<uint64_t*>(smem + L.flag) + 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // this sequence's rows and state
  const int N = lay.count(b, Nmax), st = lay.state(b);
  if (N < 0 || st < 0) {
    if (h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_LAYOUT);
    return;
  }
  const int W = (N + 31) / 32;
  const size_t row = (size_t)lay.row0(b, Nmax);
  float* Ubh = U + lay.urow0(b, h, Hv, Nmax) * kD;
  // this thread's node: parent link and gates, loaded once
  int pt = -1;
  float bet = 0.f, lat = 0.f;
  if (tid < N) {
    pt = parent[row + tid];
    bet = beta[(row + tid) * Hv + h];
    lat = log_alpha[(row + tid) * Hv + h];
  }
  // one chain: the chunkwise path (no copy of this path has started)
  if (chains && N > 0 && !__syncthreads_or(tid < N && pt != tid - 1)) {
    chain::run(smem, q, k, v, log_alpha, beta, S0, o, Ubh, N, Nmax, row, st, b, h, Hv, Hqk,
               dev_status, hk);
    return;
  }

  // S0, K and Q start streaming into shared memory at once: S0 as it is (fp32),
  // K and Q as 128-row tiles in the tensor cores' K-major 128-byte-swizzled
  // layout (K_A, Q_A, K_B, Q_B; rows past the tree zero)
  const int ntiles = N > 128 ? 2 : 1;
  // the v rows (read at the readout of R) start coming into L2
  for (int r = tid; r < N; r += kThreads)
    sm100::bulk_prefetch_l2(v + ((row + r) * Hv + h) * kD, kD * 2);
  const float* S0bh = S0 + ((size_t)st * Hv + h) * kD * kD;
  for (int i = tid; i < kD * kD / 4; i += kThreads)
    cp_async16m(sSK + 16 * i, S0bh + 4 * i);
  const int nrows = 128 * ntiles;
  for (int e = tid; e < 2 * nrows * 16; e += kThreads) {
    const int c = e & 15, rq = e >> 4, isq = rq / nrows, r = rq - isq * nrows;  // r: node
    unsigned char* dst =
        smem + L.U + (size_t)(r >> 7) * 65536 + isq * 32768 + sm100::sw128_chunk(r & 127, c);
    if (r < N)
      cp_async16m(dst, (isq ? q : k) + ((row + r) * Hqk + hq) * kD + 8 * c);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");

  // ---- 1. the tree ------------------------------------------------------------
  int bad = 0;
  if (tid < N) {
    sPar[tid] = pt;
    bad = (pt < -1 || pt >= tid);
    sBeta[tid] = bet;
    sLa[tid] = lat;
  }
  if (tid <= kMidN) sLevel[tid] = 0;
  if (tid == 0) sFlag[0] = 0;
  bad = __syncthreads_or(bad);
  if (bad) {
    if (h == 0 && tid == 0 && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_BAD_TREE);
    asm volatile("cp.async.wait_all;" ::: "memory");
    return;
  }
  // the tree is valid: the CTA takes the SM's 512 TMEM columns (one CTA an SM)
  if (warp == 0) sm100::tmem_alloc(reinterpret_cast<uint32_t*>(sFlag + 1), 512);
  tree_prepare(sPar, N, W, sLa, sJump, sAnc, sG);
  // depth, level sizes, then the nodes grouped by depth
  if (tid < N) {
    int dep = 1;
    for (int i = 0; i < W; ++i) dep += __popc(sAnc[tid * W + i]);
    sDepth[tid] = dep;
    atomicAdd(&sLevel[dep], 1);
    sm100::mbar_init(&sBar[tid], 1);
  }
  if (tid == 0) sm100::mbar_init(sBarMma, 1);
  sm100::mbar_fence_init();
  __syncthreads();
  if (warp == 0) {  // exclusive scan of the level sizes, in place (depths 1 .. N)
    int carry = 0;
    for (int base = 0; base <= kMidN; base += 32) {
      const int i = base + lane;
      const int c = i <= kMidN ? sLevel[i] : 0;
      int x = c;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (i <= kMidN) sLevel[i] = carry + x - c;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
  }
  __syncthreads();
  {
    // each level's nodes claim consecutive slots from its start: one atomic per group
    // of a warp's lanes of equal depth (any order within a level serves the solve, and
    // no node's result depends on it)
    const int dep = tid < N ? sDepth[tid] : -1;
    const unsigned peers = __match_any_sync(0xffffffffu, dep);
    const int leader = __ffs(peers) - 1;
    int base = 0;
    if (lane == leader && dep >= 0) base = atomicAdd(&sLevel[dep], __popc(peers));
    base = __shfl_sync(0xffffffffu, base, leader);
    if (dep >= 0) sOrder[base + __popc(peers & ((1u << lane) - 1u))] = tid;
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- 2. R = diag(beta)(V - diag(gamma) K S0) and seeds gamma Q S0 -----------
  // S0 = hi + lo (bf16), MN-major (K = dk rows, N = dv columns), in place of the
  // fp32 tile: every thread takes its 32 values into registers first
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
  sm100::fence_proxy_async_smem();
  sm100::tc_fence_before_sync();
  __syncthreads();
  sm100::tc_fence_after_sync();
  const uint32_t tmem = static_cast<uint32_t>(sFlag[1]);
  // TMEM columns: K S0 of tile A 0..127 and of tile B 128..255, Q S0 256..383 and
  // 384..511 (node r of a tile in lane r)
  if (tid == 0) {
    const uint32_t ub = sm100::smem_addr(smem + L.U), sb = sm100::smem_addr(sSK);
    for (int tl = 0; tl < ntiles; ++tl) {
      const uint32_t kt = ub + tl * 65536, qt = kt + 32768;
      sm100::umma_128x128x128_bmn(tmem + 128 * tl, kt, sb, false);
      sm100::umma_128x128x128_bmn(tmem + 128 * tl, kt, sb + 32768, true);
      sm100::umma_128x128x128_bmn(tmem + 256 + 128 * tl, qt, sb, false);
    }
    sm100::umma_commit(sBarMma);
  }
  if (!sm100::mbar_wait(sBarMma, 0, hk.limit_ns)) {
    // (bounded again: the MMAs must be done before TMEM is read or freed)
    sm100::mbar_wait(sBarMma, 0, hk.limit_ns);
    if (tid == 0) sFlag[0] = 1;
  }
  sm100::tc_fence_after_sync();
  {
    // warp w reads accumulator w / 4 (K S0 tile A, B; Q S0 tile A, B) for its
    // TMEM lane group w % 4: lane = node.  The v rows come in and the seeds go out
    // through a 4 KB staging block of the warp in the (now free) state region, so
    // that their global accesses are whole 64 / 128-byte row segments.
    const int acc = warp >> 2, lg = warp & 3;
    if ((acc & 1) < ntiles) {  // (warp-uniform)
      const int t0 = (acc & 1) * 128 + lg * 32, t = t0 + lane;
      const bool live = t < N;
      const float gam = live ? expf(df_value(sG[t])) : 0.f;
      const float bt = live ? sBeta[t] : 0.f;
      const uint32_t taddr = tmem + ((uint32_t)(lg * 32) << 16) + 128 * acc;
      unsigned char* stg = sSK + warp * 4096;
#pragma unroll 1
      for (int c32 = 0; c32 < 4; ++c32) {
        if (acc < 2) {
          // v[t0 + r][32 c32 ..]: lane -> row 8 i + lane / 4, 16-byte chunk lane % 4
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int r = 8 * i + (lane >> 2), c = lane & 3;
            if (t0 + r < N)
              *reinterpret_cast<uint4*>(stg + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) =
                  *reinterpret_cast<const uint4*>(v + ((row + t0 + r) * Hv + h) * kD + 32 * c32 + 8 * c);
          }
        }
        float r[32];
        sm100::tmem_ld_32cols(taddr + 32 * c32, r);  // warp-collective: every lane
        __syncwarp();
        if (acc < 2) {
          if (live) {
#pragma unroll
            for (int m = 0; m < 4; ++m) {
              float vv[8];
              bf16x8_to_f32(*reinterpret_cast<const uint4*>(
                                stg + lane * 64 + ((m ^ ((lane >> 1) & 3)) << 4)), vv);
              *reinterpret_cast<float4*>(sU + u_at(t, 8 * c32 + 2 * m)) =
                  make_float4(bt * (vv[0] - gam * r[8 * m]), bt * (vv[1] - gam * r[8 * m + 1]),
                              bt * (vv[2] - gam * r[8 * m + 2]), bt * (vv[3] - gam * r[8 * m + 3]));
              *reinterpret_cast<float4*>(sU + u_at(t, 8 * c32 + 2 * m + 1)) =
                  make_float4(bt * (vv[4] - gam * r[8 * m + 4]), bt * (vv[5] - gam * r[8 * m + 5]),
                              bt * (vv[6] - gam * r[8 * m + 6]), bt * (vv[7] - gam * r[8 * m + 7]));
            }
          }
        } else {
          // the seeds gamma_t (Q S0)_t into the staging (row = lane), then out by rows
#pragma unroll
          for (int m = 0; m < 8; ++m)
            *reinterpret_cast<float4*>(stg + lane * 128 + ((m ^ (lane & 7)) << 4)) =
                make_float4(gam * r[4 * m], gam * r[4 * m + 1], gam * r[4 * m + 2],
                            gam * r[4 * m + 3]);
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int rr = 4 * i + (lane >> 3), c = lane & 7;
            if (t0 + rr < N)
              *reinterpret_cast<float4*>(Ubh + (size_t)(t0 + rr) * kD + 32 * c32 + 4 * c) =
                  *reinterpret_cast<const float4*>(stg + rr * 128 + ((c ^ (rr & 7)) << 4));
          }
        }
        __syncwarp();  // the staging is read before the next 32 columns use it
      }
    }
  }
  sm100::tc_fence_before_sync();
  __syncthreads();  // TMEM read, S0 no longer needed
  if (warp == 0) sm100::tmem_dealloc(tmem, 512);

  // ---- 3. K into shared memory (bf16, swizzled) ---------------------------------
  for (int e = tid; e < N * 16; e += kThreads) {
    const int r = e >> 4, c = e & 15;
    cp_async16m(sSK + k_chunk(r, c), k + ((row + r) * Hqk + hq) * kD + 8 * c);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // ---- 4. the solve -----------------------------------------------------------
  bool timed_out = false;
  auto wait_final = [&](int node) {
    if (!sm100::mbar_wait(&sBar[node], 0, hk.limit_ns)) timed_out = true;
  };
  float* qs = sStage + warp * kD;
  // q of the warp's next node, loaded one node ahead
  auto q_of = [&](int task) {
    return task < N ? *reinterpret_cast<const uint2*>(q + ((row + sOrder[task]) * Hqk + hq) * kD +
                                                      4 * lane)
                    : make_uint2(0u, 0u);
  };
  // the seed of the warp's next node (parked in its U row), also one node ahead
  auto seed_of = [&](int task) {
    return task < N ? *reinterpret_cast<const float4*>(Ubh + (size_t)sOrder[task] * kD + 4 * lane)
                    : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  uint2 qnext = q_of(warp);
  float4 seednext = seed_of(warp);
  for (int task = warp; task < N; task += kWarps) {
    const int t = sOrder[task];
    const int nA = sDepth[t] - 1;  // strict ancestors
    const df gt = sG[t];
    const float bt = sBeta[t];
    float* urow = Ubh + (size_t)t * kD + 4 * lane;
    const float4 seed = seednext;
    seednext = seed_of(task + kWarps);
    // q_t into the warp's stage (fp32); the next node's q starts coming
    {
      const uint2 qq = qnext;
      *reinterpret_cast<float4*>(qs + 4 * lane) =
          make_float4(__uint_as_float(qq.x << 16), __uint_as_float(qq.x & 0xffff0000u),
                      __uint_as_float(qq.y << 16), __uint_as_float(qq.y & 0xffff0000u));
      qnext = q_of(task + kWarps);
    }
    __syncwarp();
    if (nA <= 1) {
      // a root or a root's child: its dots as warp dots (a lane holds elements
      // 4 lane .. 4 lane + 3), no path table
      auto k4 = [&](int r) {  // row r's four elements of this lane, fp32
        const uint2 w2 = *reinterpret_cast<const uint2*>(sSK + k_chunk(r, lane >> 1) + (lane & 1) * 8);
        return make_float4(__uint_as_float(w2.x << 16), __uint_as_float(w2.x & 0xffff0000u),
                           __uint_as_float(w2.y << 16), __uint_as_float(w2.y & 0xffff0000u));
      };
      const float4 qt4 = *reinterpret_cast<const float4*>(qs + 4 * lane);
      const float4 kt4 = k4(t);
      float qk = qt4.x * kt4.x + qt4.y * kt4.y + qt4.z * kt4.z + qt4.w * kt4.w;
      float xk = 0.f, yq = 0.f;
      const int p = nA == 1 ? sPar[t] : -1;
      if (p >= 0) {
        const float4 kp4 = k4(p);
        xk = kt4.x * kp4.x + kt4.y * kp4.y + kt4.z * kp4.z + kt4.w * kp4.w;
        yq = qt4.x * kp4.x + qt4.y * kp4.y + qt4.z * kp4.z + qt4.w * kp4.w;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        qk += __shfl_xor_sync(0xffffffffu, qk, off);
        xk += __shfl_xor_sync(0xffffffffu, xk, off);
        yq += __shfl_xor_sync(0xffffffffu, yq, off);
      }
      float4 ut = *reinterpret_cast<const float4*>(sU + u_at(t, lane));  // r_t
      float4 ao = make_float4(0.f, 0.f, 0.f, 0.f);
      if (p >= 0) {
        const float dec = expf(df_diff(gt, sG[p]));
        wait_final(p);
        const float4 up = *reinterpret_cast<const float4*>(sU + u_at(p, lane));
        ut = fma4m(-(bt * dec * xk), up, ut);
        ao = fma4m(dec * yq, up, ao);
      }
      *reinterpret_cast<float4*>(sU + u_at(t, lane)) = ut;
      __syncwarp();
      if (lane == 0 && !(unit == hk.withhold_unit && t == hk.withhold_node))
        sm100::mbar_arrive(&sBar[t]);
      ao = fma4m(qk, ut, ao);  // the node's own term (q_t . k_t) u_t
      __nv_bfloat16* orow = o + ((row + t) * Hv + h) * kD + 4 * lane;
      const __nv_bfloat162 p01 = __floats2bfloat162_rn(seed.x + ao.x, seed.y + ao.y);
      const __nv_bfloat162 p23 = __floats2bfloat162_rn(seed.z + ao.z, seed.w + ao.w);
      *reinterpret_cast<uint2*>(orow) = make_uint2(*reinterpret_cast<const uint32_t*>(&p01),
                                                   *reinterpret_cast<const uint32_t*>(&p23));
      *reinterpret_cast<float4*>(urow) = ut;
      __syncwarp();  // the stage is read before the next node's q_t lands in it
      continue;
    }
    // X[t,s] and Y[t,s] for path entry n (strict ancestors in index order, then
    // t itself), left in lane n % 32 as the n / 32-th of sn / xn / yn
    int sn[kGroups];
    float xn[kGroups], yn[kGroups];
    const uint32_t* anc = sAnc + t * W;
    // the n-th strict ancestor of t (n < nA): the n-th set bit of its bitset
    auto nth_ancestor = [&](int n) {
      int left = n;
      for (int wi = 0; wi < W; ++wi) {
        uint32_t bits = anc[wi];
        const int c = __popc(bits);
        if (left < c) {
          // the left-th set bit (from bit 0): halve the window by the count below
          int pos = 0;
#pragma unroll
          for (int half = 16; half > 0; half >>= 1) {
            const int below = __popc(bits & ((1u << half) - 1u));
            if (left >= below) {
              left -= below;
              bits >>= half;
              pos += half;
            }
          }
          return wi * 32 + pos;
        }
        left -= c;
      }
      return t;
    };
    // the two dots of entry s over 16-byte chunks c0 .. c1 - 1
    auto dots = [&](int s, int c0, int c1, float& dkk, float& dqk) {
      for (int c = c0; c < c1; ++c) {
        float ks[8], kt[8];
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sSK + k_chunk(s, c)), ks);
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(sSK + k_chunk(t, c)), kt);
        const float4 q0 = *reinterpret_cast<const float4*>(qs + 8 * c);
        const float4 q1 = *reinterpret_cast<const float4*>(qs + 8 * c + 4);
        const float qv[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dkk = fmaf(kt[e], ks[e], dkk);
          dqk = fmaf(qv[e], ks[e], dqk);
        }
      }
    };
    const int nP = nA + 1;  // path entries
    if (nP <= 16) {
      // a short path: 32 / P lanes share an entry (P >= nP a power of two), each
      // taking 16 / (32 / P) of the 16 chunks, and sum across those lanes
      int P = 2;
      while (P < nP) P <<= 1;
      const int Lp = 32 / P, e = lane / Lp, part = lane % Lp, cpl = 16 / Lp;
      const int s = e < nA ? nth_ancestor(e) : t;
      float dkk = 0.f, dqk = 0.f;
      if (e < nP) dots(s, part * cpl, part * cpl + cpl, dkk, dqk);
      for (int off = 1; off < Lp; off <<= 1) {
        dkk += __shfl_xor_sync(0xffffffffu, dkk, off);
        dqk += __shfl_xor_sync(0xffffffffu, dqk, off);
      }
      const float dec = s == t ? 1.f : expf(df_diff(gt, sG[s]));
      const float x = s == t ? 0.f : bt * dec * dkk, y = dec * dqk;
      const int src = (lane < nP ? lane : 0) * Lp;
      sn[0] = __shfl_sync(0xffffffffu, s, src);
      xn[0] = __shfl_sync(0xffffffffu, x, src);
      yn[0] = __shfl_sync(0xffffffffu, y, src);
#pragma unroll
      for (int gi = 1; gi < kGroups; ++gi) {
        sn[gi] = -1;
        xn[gi] = yn[gi] = 0.f;
      }
    } else {
      // one entry a lane
#pragma unroll
      for (int gi = 0; gi < kGroups; ++gi) {
        const int n = gi * 32 + lane;
        sn[gi] = -1;
        xn[gi] = yn[gi] = 0.f;
        if (gi * 32 > nA) continue;  // (uniform)
        const int s = n < nA ? nth_ancestor(n) : t;
        if (n <= nA) {
          float dkk = 0.f, dqk = 0.f;
          dots(s, 0, 16, dkk, dqk);
          const float dec = s == t ? 1.f : expf(df_diff(gt, sG[s]));
          sn[gi] = s;
          xn[gi] = s == t ? 0.f : bt * dec * dkk;
          yn[gi] = dec * dqk;
        }
      }
    }
    // the terms of the strict ancestors (entries 0 .. nA-1, root first), four at a
    // time as they become final: a path's nodes complete in path order, so the
    // last of the four being final makes all four final
    float4 au = make_float4(0.f, 0.f, 0.f, 0.f), ao = au;
    float ymine = 0.f;  // Y[t,t], in the lane that formed entry nA
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi)
      if (gi * 32 + lane == nA) ymine = yn[gi];
    const float yself = __shfl_sync(0xffffffffu, ymine, nA & 31);
#pragma unroll
    for (int gi = 0; gi < kGroups; ++gi) {
      const int cnt = min(32, nA - gi * 32);  // (<= 0 past the path: no work)
      for (int j0 = 0; j0 < cnt; j0 += 4) {
        const int m = min(4, cnt - j0);
        wait_final(__shfl_sync(0xffffffffu, sn[gi], j0 + m - 1));
        const float* uj[4];
        float xj[4], yj[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int ss = __shfl_sync(0xffffffffu, sn[gi], (j0 + jj) & 31);
          const float xx = __shfl_sync(0xffffffffu, xn[gi], (j0 + jj) & 31);
          const float yy = __shfl_sync(0xffffffffu, yn[gi], (j0 + jj) & 31);
          const bool use = jj < m;
          uj[jj] = sU + u_at(use ? ss : 0, lane);
          xj[jj] = use ? xx : 0.f;
          yj[jj] = use ? yy : 0.f;
        }
        float4 us[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) us[jj] = *reinterpret_cast<const float4*>(uj[jj]);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          au = fma4m(-xj[jj], us[jj], au);
          ao = fma4m(yj[jj], us[jj], ao);
        }
      }
    }
    float4 ut = *reinterpret_cast<const float4*>(sU + u_at(t, lane));  // r_t
    ut.x += au.x;
    ut.y += au.y;
    ut.z += au.z;
    ut.w += au.w;
    *reinterpret_cast<float4*>(sU + u_at(t, lane)) = ut;
    __syncwarp();
    if (lane == 0 && !(unit == hk.withhold_unit && t == hk.withhold_node))
      sm100::mbar_arrive(&sBar[t]);
    // o_t = seed_t + sum over the path of Y[t,s] u_s; u_t replaces the seed in U
    ao = fma4m(yself, ut, ao);
    const float o0 = seed.x + ao.x, o1 = seed.y + ao.y, o2 = seed.z + ao.z, o3 = seed.w + ao.w;
    __nv_bfloat16* orow = o + ((row + t) * Hv + h) * kD + 4 * lane;
    const __nv_bfloat162 p01 = __floats2bfloat162_rn(o0, o1), p23 = __floats2bfloat162_rn(o2, o3);
    *reinterpret_cast<uint2*>(orow) = make_uint2(*reinterpret_cast<const uint32_t*>(&p01),
                                                 *reinterpret_cast<const uint32_t*>(&p23));
    *reinterpret_cast<float4*>(urow) = ut;
    __syncwarp();  // the stage is read before the next node's q_t lands in it
  }
  if (timed_out) atomicOr(sFlag, 1);
  __syncthreads();
  if (tid == 0 && sFlag[0] && dev_status) atomicMax(dev_status + b, GDN_TREE_STATUS_TIMEOUT);
}

}  // namespace

bool verify_mid_supported(const gdn_tree_dims& d) {
  return d.dtype == GDN_TREE_BF16 && d.dk == kD && d.dv == kD && d.N >= 1 && d.N <= kMidN &&
         mid_smem_layout(d.N).total <= 227 * 1024;
}

cudaError_t launch_verify_mid(const VerifyArgs& a, cudaStream_t stream) {
  size_t smem = mid_smem_layout(a.d.N).total;
  if (a.chains) smem = std::max(smem, chain::smem_bytes(a.d.N));
  const dim3 grid(a.d.Hv, a.d.B);
  cudaError_t err = cudaFuncSetAttribute(verify_mid_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  verify_mid_kernel<<<grid, kThreads, smem, stream>>>(
      static_cast<const __nv_bfloat16*>(a.q), static_cast<const __nv_bfloat16*>(a.k),
      static_cast<const __nv_bfloat16*>(a.v), a.log_alpha, a.beta, a.parent, a.S0,
      static_cast<__nv_bfloat16*>(a.o), a.U, a.d, a.dev_status, a.lay, wait_hooks(),
      a.chains ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace gdn
