// Internal interface between the C ABI (api.cpp) and the sampling kernels (sample.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace specv {

constexpr int kSampleThreads = 256;
constexpr int kSmallVocab = 2048;   // V at or below: one warp per sequence does the whole step
constexpr int kStatChunk = 1024;    // statistics item: 1024 logits of one row, one warp
// statistics CTA: warps, each with its own ring of item slots, and the items each keeps in flight
// (4 KB each).  Twenty warps of two slots (a 160 KB ring) measured faster than sixteen of three or
// twenty-four of two (192 KB rings) at every batch tried, and as fast as rings of 8 KB items.
constexpr int kStatWarps = 20;
constexpr int kStatSlots = 2;
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
  int schunks;         // statistics pass: kStatChunk items per row
  int num_sms;
  // workspace
  uint32_t* status;
  int status_zeroed;  // the caller has already cleared *status for this call (no reset here)
  float* st_m;      // [B][rows_t + rows_d][schunks] item maxima
  float2* st_s;     // [B][rows][schunks] sum of exp(x - item max) as a float-float (hi, lo) pair
  int32_t* st_arg;  // [B][rows][schunks] item argmax (greedy)
  float* sel;       // [B][rows] chain: logit of draft token x_i in target row i (at i) and in
                    // draft row i (at rows_t + i), recorded by the statistics pass
  // tree (greedy tree mode)
  int N;
  int8_t parent[kMaxTreeNodes];
  int8_t depth[kMaxTreeNodes];
};

size_t sample_workspace_bytes(int mode, int B, int rows_t, int rows_d, int V);
void sample_workspace_carve(void* ws, SampleParams* p);
cudaError_t launch_sample(SampleParams& p, int num_sms, cudaStream_t stream);
// stochastic tree walk (sample_tree.cu), one CTA per sequence
cudaError_t launch_sample_tree(const SampleParams& p, cudaStream_t stream);

}  // namespace specv
