// kernels.h -- internal launch interface between the C-ABI layer and the
// kernels of libgdntree (not installed, not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/gdn_tree.h"

namespace gdn {

constexpr int kMaxNHost = 256;  // largest tree the kernels take
constexpr int kMaxDHost = 128;  // largest dk / dv

struct VerifyArgs {
  const void *q, *k, *v;
  const float *log_alpha, *beta;
  const int32_t* parent;
  const float* S0;
  void* o;
  float* U;
  gdn_tree_dims d;
  int32_t* dev_status;
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
};

// picks the kernel for the shape and dtype
cudaError_t launch_verify(const VerifyArgs& a, cudaStream_t stream);

size_t verify_generic_smem_bytes(int N, int dk, int dv);
cudaError_t launch_verify_generic(const VerifyArgs& a, cudaStream_t stream);

bool verify_tc_supported(const gdn_tree_dims& d);
cudaError_t launch_verify_tc(const VerifyArgs& a, cudaStream_t stream);

cudaError_t launch_commit(const CommitArgs& a, cudaStream_t stream);

// single-branch recurrent verification (the measurement baseline)
cudaError_t launch_verify_recurrent(const VerifyArgs& a, cudaStream_t stream);

bool commit_verify_tc_supported(const gdn_tree_dims& d, int prev_N);
cudaError_t launch_commit_verify_tc(const CommitVerifyArgs& a, cudaStream_t stream);
cudaError_t launch_commit_verify(const CommitVerifyArgs& a, cudaStream_t stream);

}  // namespace gdn
