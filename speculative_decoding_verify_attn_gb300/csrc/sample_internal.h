// Internal interface between the C ABI (api.cpp) and the sampling kernels (sample.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace specv {

constexpr int kSampleThreads = 256;
constexpr int kSmallVocab = 2048;   // V at or below: one warp per sequence does the whole step
constexpr int kMinChunk = 2048;     // smallest vocabulary chunk per CTA (workspace is sized for it)
constexpr int kMaxGamma = 32;
constexpr int kMaxTreeNodes = 64;

struct SampleParams {
  int mode, B, V;
  int gamma;           // chain: number of drafts; tree: unused
  int rows_t, rows_d;  // target / draft logit rows per sequence
  const float* tl;
  int64_t tl_sb;
  const float* dl;
  int64_t dl_sb;
  const int32_t* tok;
  int64_t tok_sb;
  const float* u;
  int64_t u_sb;
  int out_cols;
  int32_t* out_tok;
  int32_t* out_nacc;
  int32_t* out_nodes;
  int chunk, nchunks;  // vocabulary chunk per CTA (large-V path)
  // workspace
  uint32_t* status;
  float* st_m;      // [B][rows_t + rows_d][nchunks] chunk maxima
  double* st_s;     // [B][rows][nchunks] sum of exp(x - chunk max)
  int32_t* st_arg;  // [B][rows][nchunks] chunk argmax (greedy)
  double* res_sum;  // [B][nchunks] residual mass per chunk
  int32_t* res_last;  // [B][nchunks] last index with positive residual in the chunk, or -1
  int32_t* ticket;  // [B]
  // tree (greedy tree mode)
  int N;
  int8_t parent[kMaxTreeNodes];
  int8_t depth[kMaxTreeNodes];
};

size_t sample_workspace_bytes(int mode, int B, int rows_t, int rows_d, int V);
void sample_workspace_carve(void* ws, SampleParams* p);
cudaError_t launch_sample(SampleParams& p, int num_sms, cudaStream_t stream);

}  // namespace specv
