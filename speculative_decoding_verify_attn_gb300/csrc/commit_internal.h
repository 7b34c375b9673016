// Internal interface between the C ABI (api.cpp) and the commit kernel (commit.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

namespace specv {

constexpr int kCommitMaxNodes = 64;

struct CommitParams {
  int mode, B, Hkv, D, nq, Lmax, bf16;
  void* k;
  void* v;
  int64_t kv_sb, kv_sh;  // elements
  int32_t* kv_len;
  const int32_t* num_accepted;
  const int32_t* path_nodes;
  int64_t path_sb;
  int path_cols;
  uint32_t* status;
};

size_t commit_smem_bytes(int nq, int D, int bf16);
cudaError_t launch_commit(const CommitParams& p, cudaStream_t stream);

}  // namespace specv
