// Internal interface between the C ABI (api.cpp) and the fused LM-head kernels (lmhead.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace specv {

constexpr int kLmMaxRows = 256;     // B * R hidden rows per call (N of one MMA)
constexpr int kLmMaxNodes = 64;

struct LmheadParams {
  int mode;               // SPEC_SAMPLE_* (greedy: argmax keys; stochastic: logits)
  int B, R, d, V;         // R rows per sequence (gamma + 1 or N)
  int nrows, npad;        // B * R, padded to a multiple of 16
  int n_vtiles;           // ceil(V / 128)
  int tiles_per_pass;     // vocabulary tiles whose accumulators fit in TMEM together
  int w_stages, h_stages; // ring depths in copies (lmhead_layout)
  int kgroup;             // K chunks a tile takes in a row (one accumulator chain of 4 kgroup MMAs)
  int wbox, hbox;         // K chunks per weight / hidden-row copy (one 3-D tensor-map box)
  const int32_t* tok;     // draft tokens [B][gamma] (chain) or node tokens [B][N] (tree)
  int64_t tok_sb;
  int out_cols;
  int32_t* out_tok;
  int32_t* out_nacc;
  int32_t* out_nodes;
  uint32_t* status;
  void* rec;              // [nrows] 64-bit (value, id) keys of the running row maxima
  float* logits;          // stochastic modes: [nrows][V] fp32 target logits written by the GEMM
  int8_t parent[kLmMaxNodes];
  int8_t depth[kLmMaxNodes];
};

struct LmLayout {
  int w_stages, h_stages, kgroup, wbox, hbox;
  size_t smem;            // dynamic shared memory of the GEMM
};
LmLayout lmhead_layout(int npad);
size_t lmhead_workspace_bytes(int nrows);
void lmhead_workspace_carve(void* ws, LmheadParams* p);
cudaError_t launch_lmhead(const LmheadParams& p, const CUtensorMap* tmW, const CUtensorMap* tmH, int num_sms,
                          cudaStream_t stream);
// Stochastic modes: the GEMM alone, writing p.logits (the sampling kernels follow).
cudaError_t launch_lmhead_logits(const LmheadParams& p, const CUtensorMap* tmW, const CUtensorMap* tmH, int num_sms,
                                 cudaStream_t stream);

}  // namespace specv
