// gdn_tree_api.cu -- the extern "C" entry points of libgdntree.
//
// Every shape, dtype, pointer and alignment check happens here, on the host,
// before anything is enqueued; the kernels only check what depends on device
// data (tree and path validity) and report it through dev_status.
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/gdn_tree.h"
#include "chain_unit.cuh"
#include "kernels.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// [a0, a0 + bytes) and [a1, a1 + bytes) overlap without being the same range
bool partial_overlap(const void* p0, const void* p1, size_t bytes) {
  const char* a0 = reinterpret_cast<const char*>(p0);
  const char* a1 = reinterpret_cast<const char*>(p1);
  return a0 != a1 && a0 < a1 + bytes && a1 < a0 + bytes;
}

// [a0, a0 + b0) and [a1, a1 + b1) overlap at all
bool any_overlap(const void* p0, size_t b0, const void* p1, size_t b1) {
  const char* a0 = reinterpret_cast<const char*>(p0);
  const char* a1 = reinterpret_cast<const char*>(p1);
  return b0 && b1 && a0 < a1 + b1 && a1 < a0 + b0;
}

// packed-layout arguments: offsets and slots (device pointers), row count, slots
int check_packed(const int32_t* cu, int32_t T, const int32_t* slot, int32_t n_slots, int B,
                 gdn::SeqLayout* lay) {
  if (T < 0 || n_slots < 0) return GDN_TREE_EINVAL;
  if (cu == nullptr || !aligned4(cu)) return GDN_TREE_EINVAL;
  if (slot != nullptr && !aligned4(slot)) return GDN_TREE_EINVAL;
  if (slot == nullptr && n_slots < B) return GDN_TREE_EINVAL;
  lay->cu = cu;
  lay->slot = slot;
  lay->T = T;
  lay->n_slots = n_slots;
  return GDN_TREE_OK;
}

bool supported_head_dim(int d) { return d >= 16 && d <= gdn::kMaxDHost && d % 16 == 0; }

int check_dims(const gdn_tree_dims& d) {
  if (d.B < 0 || d.N < 0 || d.Hqk <= 0 || d.Hv <= 0 || d.dk <= 0 || d.dv <= 0)
    return GDN_TREE_EINVAL;
  if (d.Hv % d.Hqk != 0) return GDN_TREE_EINVAL;
  if (d.dtype != GDN_TREE_BF16 && d.dtype != GDN_TREE_F32) return GDN_TREE_EUNSUPPORTED;
  if (d.N > gdn::kMaxNLongHost) return GDN_TREE_EUNSUPPORTED;
  if (!supported_head_dim(d.dk) || !supported_head_dim(d.dv)) return GDN_TREE_EUNSUPPORTED;
  // every flat index must fit comfortably in the kernels' size_t arithmetic and
  // the grid's y dimension
  if (d.B > 65535) return GDN_TREE_EUNSUPPORTED;
  return GDN_TREE_OK;
}

// Per-sequence status words start at GDN_TREE_STATUS_OK; the kernels raise
// them with atomicMax, so that no unit's report can be lost to another's.
cudaError_t clear_status(int32_t* st, int B, cudaStream_t stream) {
  return st ? cudaMemsetAsync(st, 0, (size_t)B * sizeof(int32_t), stream) : cudaSuccess;
}

}  // namespace

namespace gdn {

WaitHooks wait_hooks() {
  WaitHooks h;
  if (const char* e = getenv("GDN_TREE_TEST_WAIT_LIMIT_NS")) {
    const unsigned long long v = strtoull(e, nullptr, 10);
    if (v > 0 && v < h.limit_ns) h.limit_ns = v;
  }
  if (const char* e = getenv("GDN_TREE_TEST_WITHHOLD_COPY")) h.withhold_copy_seq = atoi(e);
  if (const char* e = getenv("GDN_TREE_TEST_WITHHOLD_NODE")) {
    int u = -1, n = -1;
    if (sscanf(e, "%d:%d", &u, &n) == 2) {
      h.withhold_unit = u;
      h.withhold_node = n;
    }
  }
  return h;
}

// GDN_TREE_KERNEL=generic forces the general CUDA-core kernel, =mid the
// 256-node bf16 one, =long the chunked pass (its tensor-core form where it takes
// the shape) and =long_cuda the chunked pass on CUDA cores (used by the tests to
// cover every kernel on the same shapes); the default picks the tensor-core
// kernel whenever it takes the shape, then the 256-node bf16 kernel, the general
// on-chip kernel up to kMaxNHost nodes and the chunked pass beyond.
static bool kernel_forced(const char* name) {
  const char* e = getenv("GDN_TREE_KERNEL");
  return e && strcmp(e, name) == 0;
}
static bool long_forced() { return kernel_forced("long") || kernel_forced("long_cuda"); }
static bool force_generic() {
  return kernel_forced("generic") || long_forced() || kernel_forced("mid");
}

// the tensor-core kernel takes the shape (packed rows: at least one row, for its
// tensor maps)
static bool tc_takes(const VerifyArgs& a) {
  return !force_generic() && verify_tc_supported(a.d) && (!a.lay.packed() || a.lay.T > 0);
}

// past 128 nodes (bf16, d = 128) the units whose tree is one chain take the
// chunkwise path inside the 256-node kernel or the chunk pass
bool verify_chain_path_fits(const gdn_tree_dims& d) {
  return d.dtype == GDN_TREE_BF16 && d.dk == 128 && d.dv == 128 && d.N >= 1 &&
         d.N <= kMaxNLongHost && chain::smem_bytes(d.N) <= 227 * 1024;
}

cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t stream) {
  if (tc_takes(a)) return launch_verify_tc(a, stream);
  VerifyArgs t = a;
  const bool forced = getenv("GDN_TREE_KERNEL") && *getenv("GDN_TREE_KERNEL") &&
                      !kernel_forced("auto");
  const bool mid = !kernel_forced("generic") && !long_forced() && verify_mid_supported(a.d);
  const bool long_tc = (a.d.N > kMaxNHost || long_forced()) && !kernel_forced("long_cuda") &&
                       !kernel_forced("generic") && verify_long_tc_supported(a.d);
  t.chains = !forced && verify_chain_path_fits(a.d);
  if (mid) return launch_verify_mid(t, stream);
  if (long_tc) return launch_verify_long_tc(t, stream);
  if (a.d.N > kMaxNHost || long_forced()) return launch_verify_long(a, stream);
  return launch_verify_generic(a, stream);
}

// paths of more than 32 entries take the tensor-core commit (the rank-L update is
// then real work: a chain's 256-entry path is ~1 M FMAs a 32-row block); shorter
// ones the CUDA-core kernel, whose warps hide the gathers' latency better
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream) {
  if (!kernel_forced("generic") && a.Lmax > 32 && commit_tc_supported(a.d, a.Lmax))
    return launch_commit_tc(a, stream);
  return launch_commit_warp(a, stream);
}

cudaError_t launch_commit_verify(const CommitVerifyArgs& a, cudaStream_t stream) {
  if (tc_takes(a.verify) && commit_verify_tc_supported(a.verify.d, a.prev_N, a.Lmax))
    return launch_commit_verify_tc(a, stream);
  // two launches on the same stream: commit S_prev -> S1, then verify from S1
  gdn_tree_dims dp = a.verify.d;
  dp.N = a.prev_N;
  SeqLayout cl = a.prev_lay;  // the previous tree's rows, the verification's state slots
  cl.slot = a.verify.lay.slot;
  cl.n_slots = a.verify.lay.n_slots;
  const CommitArgs c{a.prev_path, a.prev_path_len, a.prev_parent, a.prev_U, a.prev_k,
                     a.prev_log_alpha, a.S_prev, a.S1, dp, a.Lmax, a.commit_status, cl};
  cudaError_t err = launch_commit(c, stream);
  if (err != cudaSuccess) return err;
  VerifyArgs v = a.verify;
  v.S0 = a.S1;
  return launch_verify(v, stream);
}

}  // namespace gdn

extern "C" {

int gdn_tree_verify(const void* q, const void* k, const void* v, const float* log_alpha,
                    const float* beta, const int32_t* parent, const float* S0, void* o,
                    float* U, gdn_tree_dims dims, int32_t* dev_status, void* stream) {
  const int rc = check_dims(dims);
  if (rc != GDN_TREE_OK) return rc;
  if (dims.B == 0 || dims.N == 0) return GDN_TREE_OK;  // nothing to do
  const void* ptrs[] = {q, k, v, log_alpha, beta, parent, S0, o, U};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return GDN_TREE_EINVAL;
  gdn::VerifyArgs a{q, k, v, log_alpha, beta, parent, S0, o, U, dims, dev_status};
  if (clear_status(dev_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_TREE_ECUDA;
  const cudaError_t err = gdn::launch_verify(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

int gdn_tree_verify_recurrent(const void* q, const void* k, const void* v,
                              const float* log_alpha, const float* beta,
                              const int32_t* parent, const float* S0, void* o, float* U,
                              gdn_tree_dims dims, int32_t* dev_status, void* stream) {
  const int rc = check_dims(dims);
  if (rc != GDN_TREE_OK) return rc;
  if (dims.N > gdn::kMaxNHost) return GDN_TREE_EUNSUPPORTED;  // the path table is on chip
  if (dims.B == 0 || dims.N == 0) return GDN_TREE_OK;  // nothing to do
  const void* ptrs[] = {q, k, v, log_alpha, beta, parent, S0, o, U};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return GDN_TREE_EINVAL;
  if (dims.Hv > 65535) return GDN_TREE_EUNSUPPORTED;  // the grid's y dimension
  gdn::VerifyArgs a{q, k, v, log_alpha, beta, parent, S0, o, U, dims, dev_status};
  if (clear_status(dev_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_TREE_ECUDA;
  const cudaError_t err = gdn::launch_verify_recurrent(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

int gdn_tree_commit(const int32_t* path, const int32_t* path_len, const int32_t* parent,
                    const float* U, const void* k, const float* log_alpha, const float* S0,
                    float* S1, gdn_tree_dims dims, int32_t Lmax, int32_t* dev_status,
                    void* stream) {
  const int rc = check_dims(dims);
  if (rc != GDN_TREE_OK) return rc;
  if (Lmax < 0) return GDN_TREE_EINVAL;
  if (dims.B == 0) return GDN_TREE_OK;
  if (Lmax > gdn::kMaxNLongHost) return GDN_TREE_EUNSUPPORTED;
  const void* ptrs[] = {path_len, U, k, log_alpha, S0, S1};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  if (Lmax > 0 && (path == nullptr || (reinterpret_cast<uintptr_t>(path) & 3u)))
    return GDN_TREE_EINVAL;
  if (parent && (reinterpret_cast<uintptr_t>(parent) & 3u)) return GDN_TREE_EINVAL;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return GDN_TREE_EINVAL;
  // S1 may be S0 exactly; a partial overlap would race between CTAs
  const size_t bytes = (size_t)dims.B * dims.Hv * dims.dk * dims.dv * sizeof(float);
  const char* a0 = reinterpret_cast<const char*>(S0);
  const char* a1 = reinterpret_cast<const char*>(S1);
  if (a0 != a1 && a0 < a1 + bytes && a1 < a0 + bytes) return GDN_TREE_EINVAL;
  gdn::CommitArgs a{path, path_len, parent, U, k, log_alpha, S0, S1, dims, Lmax, dev_status};
  if (clear_status(dev_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_TREE_ECUDA;
  const cudaError_t err = gdn::launch_commit(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

int gdn_tree_commit_verify(const int32_t* prev_path, const int32_t* prev_path_len,
                           const int32_t* prev_parent, const float* prev_U, const void* prev_k,
                           const float* prev_log_alpha, int32_t prev_N, int32_t Lmax,
                           const float* S_prev, float* S1, const void* q, const void* k,
                           const void* v, const float* log_alpha, const float* beta,
                           const int32_t* parent, void* o, float* U, gdn_tree_dims dims,
                           int32_t* commit_status, int32_t* verify_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != GDN_TREE_OK) return rc;
  gdn_tree_dims dp = dims;
  dp.N = prev_N;
  if (prev_N < 0 || Lmax < 0) return GDN_TREE_EINVAL;
  rc = check_dims(dp);
  if (rc != GDN_TREE_OK) return rc;
  if (Lmax > gdn::kMaxNLongHost) return GDN_TREE_EUNSUPPORTED;
  if (dims.B == 0) return GDN_TREE_OK;
  if (prev_N == 0 || dims.N == 0) return GDN_TREE_EUNSUPPORTED;
  const void* ptrs[] = {prev_path_len, prev_U, prev_k, prev_log_alpha, S_prev, S1,
                        q, k, v, log_alpha, beta, parent, o, U};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  if (Lmax > 0 && (prev_path == nullptr || (reinterpret_cast<uintptr_t>(prev_path) & 3u)))
    return GDN_TREE_EINVAL;
  const void* small[] = {prev_parent, commit_status, verify_status};
  for (const void* p : small)
    if (p && (reinterpret_cast<uintptr_t>(p) & 3u)) return GDN_TREE_EINVAL;
  const size_t sbytes = (size_t)dims.B * dims.Hv * dims.dk * dims.dv * sizeof(float);
  const char* a0 = reinterpret_cast<const char*>(S_prev);
  const char* a1 = reinterpret_cast<const char*>(S1);
  if (a0 != a1 && a0 < a1 + sbytes && a1 < a0 + sbytes) return GDN_TREE_EINVAL;
  // U may be prev_U itself only when both trees have the same node count: then
  // each (b, h) slice sits at the same place in both and is read before it is
  // written.  Any other overlap would let one unit's U rows land on another
  // unit's previous rows before those are read.
  const size_t ubytes = (size_t)dims.B * dims.Hv * dims.N * dims.dv * sizeof(float);
  const size_t pubytes = (size_t)dims.B * dims.Hv * prev_N * dims.dv * sizeof(float);
  if (!(U == prev_U && prev_N == dims.N) && any_overlap(U, ubytes, prev_U, pubytes))
    return GDN_TREE_EINVAL;
  gdn::CommitVerifyArgs a{prev_path, prev_path_len, prev_parent, prev_U, prev_k, prev_log_alpha,
                          prev_N, Lmax, S_prev, S1, commit_status,
                          gdn::VerifyArgs{q, k, v, log_alpha, beta, parent, S1, o, U, dims,
                                          verify_status}};
  if (clear_status(commit_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      clear_status(verify_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_TREE_ECUDA;
  const cudaError_t err = gdn::launch_commit_verify(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

int gdn_tree_verify_packed(const void* q, const void* k, const void* v, const float* log_alpha,
                           const float* beta, const int32_t* parent, const int32_t* cu_nodes,
                           int32_t T, const float* state_pool, const int32_t* state_slot,
                           int32_t n_slots, void* o, float* U, gdn_tree_dims dims,
                           int32_t* dev_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != GDN_TREE_OK) return rc;
  gdn::SeqLayout lay;
  rc = check_packed(cu_nodes, T, state_slot, n_slots, dims.B, &lay);
  if (rc != GDN_TREE_OK) return rc;
  if (dims.B == 0 || dims.N == 0) return GDN_TREE_OK;  // nothing to do
  const void* ptrs[] = {q, k, v, log_alpha, beta, parent, state_pool, o, U};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  if (dev_status && !aligned4(dev_status)) return GDN_TREE_EINVAL;
  gdn::VerifyArgs a{q, k, v, log_alpha, beta, parent, state_pool, o, U, dims, dev_status, lay};
  if (clear_status(dev_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_TREE_ECUDA;
  const cudaError_t err = gdn::launch_verify(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

int gdn_tree_commit_packed(const int32_t* path, const int32_t* path_len, const int32_t* parent,
                           const int32_t* cu_nodes, int32_t T, const float* U, const void* k,
                           const float* log_alpha, const float* pool_in, float* pool_out,
                           const int32_t* state_slot, int32_t n_slots, gdn_tree_dims dims,
                           int32_t Lmax, int32_t* dev_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != GDN_TREE_OK) return rc;
  gdn::SeqLayout lay;
  rc = check_packed(cu_nodes, T, state_slot, n_slots, dims.B, &lay);
  if (rc != GDN_TREE_OK) return rc;
  if (Lmax < 0) return GDN_TREE_EINVAL;
  if (dims.B == 0) return GDN_TREE_OK;
  if (Lmax > gdn::kMaxNLongHost) return GDN_TREE_EUNSUPPORTED;
  const void* ptrs[] = {path_len, pool_in, pool_out};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  if (T > 0) {
    const void* rows[] = {U, k, log_alpha};
    for (const void* p : rows)
      if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  }
  if (Lmax > 0 && (path == nullptr || !aligned4(path))) return GDN_TREE_EINVAL;
  if (parent && !aligned4(parent)) return GDN_TREE_EINVAL;
  if (dev_status && !aligned4(dev_status)) return GDN_TREE_EINVAL;
  const int slots = state_slot ? n_slots : dims.B;
  if (partial_overlap(pool_in, pool_out, (size_t)slots * dims.Hv * dims.dk * dims.dv * 4))
    return GDN_TREE_EINVAL;
  gdn::CommitArgs a{path, path_len, parent, U, k, log_alpha, pool_in, pool_out,
                    dims, Lmax, dev_status, lay};
  if (clear_status(dev_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_TREE_ECUDA;
  const cudaError_t err = gdn::launch_commit(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

int gdn_tree_commit_verify_packed(const int32_t* prev_path, const int32_t* prev_path_len,
                                  const int32_t* prev_parent, const int32_t* prev_cu_nodes,
                                  int32_t prev_T, const float* prev_U, const void* prev_k,
                                  const float* prev_log_alpha, int32_t prev_N, int32_t Lmax,
                                  const float* pool_in, float* pool_out,
                                  const int32_t* state_slot, int32_t n_slots, const void* q,
                                  const void* k, const void* v, const float* log_alpha,
                                  const float* beta, const int32_t* parent,
                                  const int32_t* cu_nodes, int32_t T, void* o, float* U,
                                  gdn_tree_dims dims, int32_t* commit_status,
                                  int32_t* verify_status, void* stream) {
  int rc = check_dims(dims);
  if (rc != GDN_TREE_OK) return rc;
  gdn_tree_dims dp = dims;
  dp.N = prev_N;
  if (prev_N < 0 || Lmax < 0) return GDN_TREE_EINVAL;
  rc = check_dims(dp);
  if (rc != GDN_TREE_OK) return rc;
  gdn::SeqLayout lay, prev_lay;
  rc = check_packed(cu_nodes, T, state_slot, n_slots, dims.B, &lay);
  if (rc != GDN_TREE_OK) return rc;
  rc = check_packed(prev_cu_nodes, prev_T, state_slot, n_slots, dims.B, &prev_lay);
  if (rc != GDN_TREE_OK) return rc;
  if (Lmax > gdn::kMaxNLongHost) return GDN_TREE_EUNSUPPORTED;
  if (dims.B == 0) return GDN_TREE_OK;
  if (prev_N == 0 || dims.N == 0) return GDN_TREE_EUNSUPPORTED;
  const void* ptrs[] = {prev_path_len, prev_U, prev_k, prev_log_alpha, pool_in, pool_out,
                        q, k, v, log_alpha, beta, parent, o, U};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return GDN_TREE_EINVAL;
  if (Lmax > 0 && (prev_path == nullptr || !aligned4(prev_path))) return GDN_TREE_EINVAL;
  const void* small[] = {prev_parent, commit_status, verify_status};
  for (const void* p : small)
    if (p && !aligned4(p)) return GDN_TREE_EINVAL;
  const int slots = state_slot ? n_slots : dims.B;
  if (partial_overlap(pool_in, pool_out, (size_t)slots * dims.Hv * dims.dk * dims.dv * 4))
    return GDN_TREE_EINVAL;
  // the next tree's U must not overlap the previous one's (their row ranges differ)
  if (any_overlap(U, (size_t)dims.Hv * T * dims.dv * 4, prev_U,
                  (size_t)dims.Hv * prev_T * dims.dv * 4))
    return GDN_TREE_EINVAL;
  gdn::CommitVerifyArgs a{prev_path, prev_path_len, prev_parent, prev_U, prev_k, prev_log_alpha,
                          prev_N, Lmax, pool_in, pool_out, commit_status,
                          gdn::VerifyArgs{q, k, v, log_alpha, beta, parent, pool_out, o, U, dims,
                                          verify_status, lay},
                          prev_lay};
  if (clear_status(commit_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess ||
      clear_status(verify_status, dims.B, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return GDN_TREE_ECUDA;
  const cudaError_t err = gdn::launch_commit_verify(a, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

int gdn_tree_build_topw(const float* cand_logp, int32_t B, int32_t N, int32_t c, int32_t w,
                        int32_t max_depth, int32_t* parent, int32_t* cand_index, float* score,
                        int32_t* n_built, void* stream) {
  if (B < 0 || N < 1 || c < 1 || w < 1 || max_depth < 1) return GDN_TREE_EINVAL;
  if (N > gdn::kMaxNHost || c > 32 || w > N) return GDN_TREE_EUNSUPPORTED;
  if (B == 0) return GDN_TREE_OK;
  if (cand_logp == nullptr || parent == nullptr || !aligned4(cand_logp) || !aligned4(parent))
    return GDN_TREE_EINVAL;
  const void* opt[] = {cand_index, score, n_built};
  for (const void* p : opt)
    if (p && !aligned4(p)) return GDN_TREE_EINVAL;
  const cudaError_t err = gdn::launch_tree_topw(cand_logp, B, N, c, w, max_depth, parent,
                                                cand_index, score, n_built,
                                                static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? GDN_TREE_OK : GDN_TREE_ECUDA;
}

const char* gdn_tree_strerror(int code) {
  switch (code) {
    case GDN_TREE_OK: return "ok";
    case GDN_TREE_EINVAL: return "invalid argument (NULL or misaligned pointer, bad dims)";
    case GDN_TREE_EUNSUPPORTED: return "unsupported shape or dtype";
    case GDN_TREE_ECUDA: return "CUDA launch failed";
    case GDN_TREE_STATUS_BAD_TREE: return "device status: parent[] is not topologically ordered";
    case GDN_TREE_STATUS_BAD_PATH: return "device status: accepted path is invalid";
    case GDN_TREE_STATUS_TIMEOUT: return "device status: an on-device wait timed out";
    case GDN_TREE_STATUS_BAD_LAYOUT:
      return "device status: the sequence's packed row range or state slot is out of range";
    default: return "unknown code";
  }
}

int gdn_tree_version(void) { return 100; }

}  // extern "C"
