// sm100.cuh -- thin inline-PTX wrappers for the Blackwell (sm_100 family,
// built here for sm_103a) features the tensor-core kernel uses: mbarriers,
// TMA tiled loads, tcgen05 MMA with TMEM accumulators, TMEM loads, and the
// shared-memory matrix descriptor for 128-byte-swizzled K-major tiles.
//
// Every wait in here is bounded by a wall-clock limit (globaltimer); callers
// turn a timeout into an error status instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace gdn {
namespace sm100 {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarrier ---------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// one arrival (release semantics at CTA scope)
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; gives up after
// limit_ns nanoseconds and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---- CTA-scope flags in shared memory --------------------------------------------

__device__ __forceinline__ int ld_acquire_shared(const int* p) {
  int v;
  asm volatile("ld.acquire.cta.shared::cta.b32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_shared(int* p, int v) {
  asm volatile("st.release.cta.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

// ---- TMA ----------------------------------------------------------------------

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 4-D tiled load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar))
      : "memory");
}

// 3-D tiled store of one box from shared memory, tracked in this thread's bulk
// async-group (bulk_commit_group / bulk_wait_read_all / bulk_wait_all).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0,
                                             int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::
                   "l"(map),
               "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(src))
               : "memory");
}

// L2 prefetch of one 4-D / 3-D tensor-map box (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int c0, int c1, int c2,
                                                   int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(map),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}

// L2 prefetch of the line holding p
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

// L2 prefetch of `bytes` (multiple of 16, 16-byte aligned address)
__device__ __forceinline__ void bulk_prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Plain (untiled) bulk copy global -> shared of `bytes` (multiple of 16, both
// addresses 16-byte aligned), completing on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Plain (untiled) bulk copy shared -> global of `bytes` (multiple of 16, both
// addresses 16-byte aligned), tracked in this thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until every bulk store of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until every bulk store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor cores, TMA).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- cluster launch control (work stealing) -------------------------------------

// One thread: asks the hardware scheduler to cancel a CTA of this grid that has not
// been launched yet.  The 16-byte response lands at `resp` (16-byte aligned shared
// memory) and completes a phase of `bar` by its byte count (this thread arms it).
__device__ __forceinline__ void clc_try_cancel(void* resp, uint64_t* bar) {
  mbar_arrive_expect_tx(bar, 16);
  asm volatile(
      "clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes.b128 "
      "[%0], [%1];" ::"r"(smem_addr(resp)),
      "r"(smem_addr(bar))
      : "memory");
}

// Decodes a landed response: true when a CTA was cancelled, its blockIdx.x in *ctaid_x
// (the cancelled CTA never runs: its work is the caller's).
__device__ __forceinline__ bool clc_cancelled(const void* resp, int* ctaid_x) {
  uint32_t ok = 0, x = 0;
  asm volatile(
      "{\n"
      " .reg .b128 r;\n"
      " .reg .pred p;\n"
      " .reg .b64 lo, hi;\n"
      " ld.shared.v2.b64 {lo, hi}, [%2];\n"
      " mov.b128 r, {lo, hi};\n"
      " clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 p, r;\n"
      " selp.u32 %0, 1, 0, p;\n"
      " @p clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, r;\n"
      "}"
      : "=r"(ok), "=r"(x)
      : "r"(smem_addr(resp))
      : "memory");
  *ctaid_x = (int)x;
  return ok != 0;
}

// ---- TMEM -------------------------------------------------------------------

// Whole warp: allocate ncols TMEM columns, base address written to *dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-collective: 32 consecutive fp32 columns of this warp's 32 TMEM lanes
// (lane i of the warp gets lane (base lane + i)).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-collective: 32 consecutive fp32 columns into this warp's 32 TMEM lanes
// (lane i of the warp writes lane (base lane + i)); waits for the stores.
__device__ __forceinline__ void tmem_st_32cols(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Warp-collective: 16 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Warp-collective: 8 consecutive fp32 columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld_8cols(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// ---- UMMA (tcgen05.mma) ---------------------------------------------------------

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 64 bf16 (128 bytes), 8-row atoms of 1024 bytes
// (stride byte offset 1024), atom base 1024-byte aligned.  Advancing K by 16
// elements inside an atom adds 32 bytes to the start address.
__device__ __forceinline__ uint64_t desc_sw128_kmajor(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address, bits 0-13
  d |= (uint64_t)(16u >> 4) << 16;           // leading byte offset (unused here)
  d |= (uint64_t)(1024u >> 4) << 32;         // stride byte offset, bits 32-45
  d |= (uint64_t)1 << 46;                    // descriptor version for sm_100
  d |= (uint64_t)2 << 61;                    // layout: 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor for an MN-major operand stored with the
// 128-byte swizzle: atoms of 8 K-rows x 64 bf16 (128 bytes, the MN elements
// contiguous) = 1024 bytes, swizzled like the K-major atom; `lbo` = byte offset
// between atoms along MN (64-element blocks), `sbo` = between atoms along K
// (8-row groups).  Atom bases 1024-byte aligned.
__device__ __forceinline__ uint64_t desc_sw128_mnmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);     // start address, bits 0-13
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;  // leading byte offset, bits 16-29
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;  // stride byte offset, bits 32-45
  d |= (uint64_t)1 << 46;                       // descriptor version for sm_100
  d |= (uint64_t)2 << 61;                       // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: A, B bf16 K-major, D fp32, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                        // D format: f32
         | (1u << 7)                      // A format: bf16
         | (1u << 10)                     // B format: bf16
         | ((uint32_t)(N >> 3) << 17)     // N / 8
         | ((uint32_t)(M >> 4) << 24);    // M / 16
}

// The same with B MN-major (B given as K x N, N contiguous).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_bmn(int M, int N) {
  return idesc_bf16_f32(M, N) | (1u << 16);  // transpose B
}

// The same with A and B both MN-major (A given as K x M, B as K x N, the M / N
// elements contiguous).
__host__ __device__ constexpr uint32_t idesc_bf16_f32_amn_bmn(int M, int N) {
  return idesc_bf16_f32(M, N) | (1u << 15) | (1u << 16);  // transpose A and B
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ---- operand layouts and MMA sequences shared by the tensor-core kernels -------

// one 64-wide K block of a 128-row K-major bf16 tile: 128 rows x 128 bytes
constexpr uint32_t kSw128TileBytes = 128 * 128;

// byte offset of 16-byte chunk k8 (K elements 8*k8 .. 8*k8+7) of `row` in a
// 128-row, 128-wide K-major bf16 tile stored with the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128_chunk(int row, int k8) {
  const int kb = k8 >> 3, j = k8 & 7;
  return (uint32_t)(kb * kSw128TileBytes + row * 128 + ((j ^ (row & 7)) << 4));
}

// (a, b) -> bf16x2 hi parts and bf16x2 lo parts (x = hi + lo to ~2^-17)
__device__ __forceinline__ void split2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// issue the 8 K-steps (K = 128) of D (+)= A B^T for two 128x128 K-major tiles
__device__ __forceinline__ void umma_128x128x128(uint32_t d_tmem, uint32_t a_base,
                                                 uint32_t b_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t off = (uint32_t)((s >> 2) * kSw128TileBytes + (s & 3) * 32);
    umma_bf16(d_tmem, desc_sw128_kmajor(a_base + off), desc_sw128_kmajor(b_base + off), idesc,
              (accumulate || s > 0) ? 1u : 0u);
  }
}

// An MN-major bf16 operand (K rows x 128 MN columns): the 16-byte chunk n8
// (columns 8 n8 .. 8 n8 + 7) of row k sits in the 1024-byte atom of rows
// 8 (k / 8) .. and columns 64 (n8 / 8) .., atoms of one row group 1 KB apart
// along MN and row groups 2 KB apart, chunks swizzled by the row.  The state
// operand S0 (K = dk) and the fused commit's k rows and w U rows (K = path
// entries) use it.
constexpr uint32_t kMnLbo = 1024, kMnSbo = 2048;
__device__ __forceinline__ uint32_t mn_chunk(int k, int n8) {
  const int r = k & 7;
  return (uint32_t)((k >> 3) * kMnSbo + (n8 >> 3) * kMnLbo + r * 128 + (((n8 & 7) ^ r) << 4));
}

// issue the 8 K-steps (K = 128) of D (+)= A B for a 128x128 K-major tile A and
// a 128-row MN-major tile B (a K-step of 16 rows spans two row groups)
__device__ __forceinline__ void umma_128x128x128_bmn(uint32_t d_tmem, uint32_t a_base,
                                                     uint32_t b_base, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32_bmn(128, 128);
#pragma unroll
  for (int s = 0; s < 8; ++s) {
    const uint32_t a_off = (uint32_t)((s >> 2) * kSw128TileBytes + (s & 3) * 32);
    umma_bf16(d_tmem, desc_sw128_kmajor(a_base + a_off),
              desc_sw128_mnmajor(b_base + (uint32_t)s * 2 * kMnSbo, kMnLbo, kMnSbo), idesc,
              (accumulate || s > 0) ? 1u : 0u);
  }
}

// issue the K-steps (16 path entries each) of D (+)= A^T B for MN-major tiles of
// `ksteps` * 16 rows: A = the path's k rows, B = its w U rows
__device__ __forceinline__ void umma_commit_rows(uint32_t d_tmem, uint32_t a_base,
                                                 uint32_t b_base, int ksteps, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32_amn_bmn(128, 128);
  for (int s = 0; s < ksteps; ++s) {
    const uint32_t off = (uint32_t)s * 2 * kMnSbo;
    umma_bf16(d_tmem, desc_sw128_mnmajor(a_base + off, kMnLbo, kMnSbo),
              desc_sw128_mnmajor(b_base + off, kMnLbo, kMnSbo), idesc,
              (accumulate || s > 0) ? 1u : 0u);
  }
}

// fp32 128-row tiles of 128 columns (a state, R / U rows) as four TMA boxes of
// 32 columns x 128 rows with the 128-byte swizzle
constexpr uint32_t kBoxBytes = 32 * 4 * 128;  // 16 KB
// fp32 128 x 128 row tiles (the state, R / U) in the layout of four TMA boxes of
// 32 columns x 128 rows with the 128-byte swizzle: row t, 4-float chunk c4
// (0..31) sits in box c4 / 8, its 16-byte slot xor-swizzled by the row, so that
// a row-per-thread float4 access and a half-warp reading one row's 16 chunks are
// both bank-conflict free
__device__ __forceinline__ uint32_t u_off(int t, int c4) {
  return (uint32_t)((c4 >> 3) * kBoxBytes + t * 128 + (((c4 & 7) ^ (t & 7)) << 4));
}

// Arrive once on `bar` when all previously issued MMAs of this thread are done.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

}  // namespace sm100
}  // namespace gdn
