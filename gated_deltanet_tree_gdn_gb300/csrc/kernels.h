// kernels.h -- internal launch interface between the C-ABI layer and the
// kernels of libgdntree (not installed, not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn_tree.h"

namespace gdn {

constexpr int kMaxNHost = 256;       // largest tree of the on-chip kernels
constexpr int kMaxNLongHost = 1024;  // largest tree of the chunked kernel and commit path
constexpr int kMaxDHost = 128;  // largest dk / dv

// Where the rows and the state of sequence b live.
//  - fixed layout (cu == nullptr): every sequence has dims.N nodes; node rows of
//    q, k, v, o, log_alpha, beta, parent are at b * N + t; U is [B, Hv, N, dv].
//  - packed (ragged) layout: sequence b owns rows cu[b] .. cu[b+1] - 1 of the
//    packed arrays ([T, ...]); dims.N is the largest tree; U is [Hv, T, dv].
//  - the state of sequence b is S[slot[b]] of a state pool (slot == nullptr:
//    S[b]); n_slots bounds the slots.
struct SeqLayout {
  const int32_t* cu = nullptr;
  const int32_t* slot = nullptr;
  int32_t T = 0;
  int32_t n_slots = 0;

  __host__ __device__ bool packed() const { return cu != nullptr; }
#ifdef __CUDACC__
  // first row and node count of sequence b (count < 0: invalid offsets)
  __device__ __forceinline__ int row0(int b, int N) const { return cu ? cu[b] : b * N; }
  __device__ __forceinline__ int count(int b, int N) const {
    if (!cu) return N;
    const int a = cu[b], e = cu[b + 1];
    return (a < 0 || e < a || e > T || e - a > N) ? -1 : e - a;
  }
  // state index of sequence b (-1: out of range)
  __device__ __forceinline__ int state(int b) const {
    if (!slot) return b;
    const int s = slot[b];
    return (s < 0 || s >= n_slots) ? -1 : s;
  }
  // row (in units of dv floats) of node 0 of unit (b, h) in U
  __device__ __forceinline__ size_t urow0(int b, int h, int Hv, int N) const {
    return cu ? (size_t)h * T + cu[b] : ((size_t)b * Hv + h) * N;
  }
#endif
};

struct VerifyArgs {
  const void *q, *k, *v;
  const float *log_alpha, *beta;
  const int32_t* parent;
  const float* S0;
  void* o;
  float* U;
  gdn_tree_dims d;
  int32_t* dev_status;
  SeqLayout lay = {};
  // the 256-node kernel and the chunk pass run the units whose tree is one chain in
  // the chunkwise form (bf16, dk = dv = 128)
  bool chains = false;
};

struct CommitArgs {
  const int32_t *path, *path_len, *parent;
  const float* U;
  const void* k;
  const float *log_alpha, *S0;
  float* S1;
  gdn_tree_dims d;
  int32_t Lmax;
  int32_t* dev_status;
  SeqLayout lay = {};
};

// delayed commitment of the previous tree's accepted path fused with the
// verification of the next tree (the next tree is verified from S1)
struct CommitVerifyArgs {
  const int32_t *prev_path, *prev_path_len, *prev_parent;
  const float* prev_U;
  const void* prev_k;
  const float* prev_log_alpha;
  int32_t prev_N, Lmax;
  const float* S_prev;
  float* S1;
  int32_t* commit_status;
  VerifyArgs verify;  // verify.S0 is ignored (the state is S1)
  SeqLayout prev_lay = {};  // the previous tree's rows (state slots: verify.lay's)
};

// Bound of the on-device waits, and test-only controls that make one run out.
// Normal calls use the defaults (2 s, nothing withheld); a test sets them
// through the environment (read at every launch by wait_hooks()):
//   GDN_TREE_TEST_WAIT_LIMIT_NS=<ns>       the bound of every wait
//   GDN_TREE_TEST_WITHHOLD_NODE=<unit>:<node>  the tensor-core, 256-node and
//       tensor-core chunk-pass verifications of unit (b * Hv + h) never arrive on
//       that node's solve barrier, so the waits of its descendants (in its chunk,
//       for the chunk pass) run out (thread arrivals only: no copy or MMA is left
//       in flight)
//   GDN_TREE_TEST_WITHHOLD_COPY=<b>        the tensor-core commit of sequence b
//       expects its state copy but never issues it, so the wait for it runs out
struct WaitHooks {
  uint64_t limit_ns = 2000000000ull;
  int withhold_unit = -1, withhold_node = -1;
  int withhold_copy_seq = -1;
};
WaitHooks wait_hooks();

// picks the kernel for the shape and dtype
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t stream);

size_t verify_generic_smem_bytes(int N, int dk, int dv);
cudaError_t launch_verify_generic(const VerifyArgs& a, cudaStream_t stream);

// trees longer than kMaxNHost: the two-level chunk pass
size_t verify_long_smem_bytes(int N, int dk, int dv);
cudaError_t launch_verify_long(const VerifyArgs& a, cudaStream_t stream);

// the chunkwise path for units whose tree is one chain fits beside the tree kernels
bool verify_chain_path_fits(const gdn_tree_dims& d);

// bf16 trees of up to kMaxNLongHost nodes with dk = dv = 128: the chunk pass with
// R and the output seeds on the tensor cores
bool verify_long_tc_supported(const gdn_tree_dims& d);
cudaError_t launch_verify_long_tc(const VerifyArgs& a, cudaStream_t stream);

// bf16 trees of up to 256 nodes with dk = dv = 128 (R and the seeds on the tensor
// cores, the solve on CUDA cores, on chip)
bool verify_mid_supported(const gdn_tree_dims& d);
cudaError_t launch_verify_mid(const VerifyArgs& a, cudaStream_t stream);

// 128-byte-swizzled TMA maps of fp32 states [n_states, 128, 128] as four boxes of
// 32 columns x 128 rows each (false when the driver's encoder is unavailable)
bool encode_state_map(CUtensorMap* map, const float* base, long long n_states);

bool verify_tc_supported(const gdn_tree_dims& d);
cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream);

// the commit: on the tensor cores (bf16 k, dk = dv = 128) unless the CUDA-core
// kernels are forced, else one warp per 32-row block on CUDA cores
cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream);
cudaError_t launch_commit_warp(const CommitArgs& a, cudaStream_t stream);
bool commit_tc_supported(const gdn_tree_dims& d, int32_t Lmax);
cudaError_t launch_commit_tc(const CommitArgs& a, cudaStream_t stream);

// streaming multiprocessors of the current device (cached per device; 0: no device)
int sm_count();

// top-w best-first draft-tree construction
size_t tree_topw_smem_bytes(int N, int c);
cudaError_t launch_tree_topw(const float* cand_logp, int B, int N, int c, int w, int max_depth,
                             int32_t* parent, int32_t* cand_index, float* score, int32_t* n_built,
                             cudaStream_t stream);

// single-branch recurrent verification (the measurement baseline)
cudaError_t launch_verify_recurrent(const VerifyArgs& a, cudaStream_t stream);

bool commit_verify_tc_supported(const gdn_tree_dims& d, int prev_N, int Lmax);
cudaError_t launch_commit_verify_tc(const CommitVerifyArgs& a, cudaStream_t stream);
cudaError_t launch_commit_verify(const CommitVerifyArgs& a, cudaStream_t stream);

}  // namespace gdn
