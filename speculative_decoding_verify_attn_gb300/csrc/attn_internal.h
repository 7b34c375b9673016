// Internal interface between the C ABI (api.cpp) and the attention kernels (attn.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace specv {

// Keys per TMA stage and pipeline depth of the bf16 split-KV kernel (3 x 64 KB for D = 128).
constexpr int kKeyTile = 128;
constexpr int kStages = 3;
// Consumer warps per CTA (two per SM sub-partition) plus one TMA producer warp.
constexpr int kConsumerWarps = 8;
// Query rows one CTA row-group holds (up to 4 row tiles of 16 for mma.sync).
constexpr int kRowsPerGroup = 64;
// Upper bound on CTAs along the key axis (two per SM on a 160-SM part); the workspace is sized
// for it and launches never exceed it.
constexpr int kMaxGridX = 320;
// Minimum 128-key tiles a CTA takes, so that short total work does not spread over every SM.
constexpr int kMinTilesPerCta = 2;

enum MaskMode : int { kMaskNone = 0, kMaskChain = 1, kMaskTree = 2 };

// Everything a partial/merge kernel needs; passed by value as a __grid_constant__ parameter.
struct AttnParams {
  int B, Hq, Hkv, G, D, nq, rows;  // rows = nq * G query rows per (sequence, kv head)
  int mask;                        // MaskMode
  int Lmax;                        // verify: cache capacity; window: W
  int is_window;                   // lengths come from pos (min(pos, W); pos < 1 invalid)
  const int32_t* lens;             // kv_len or pos, device [B]
  const void* q;
  int64_t q_sb, q_st, q_sh;
  const void* k;
  const void* v;
  int64_t kv_sb, kv_sh;
  float scale_log2;                // scale * log2(e)
  void* o;
  int64_t o_sb, o_st, o_sh;
  int o_bf16;
  int grid_x;                      // CTAs along the key axis (same value in partial and merge)
  int rows_per_group;              // query rows per CTA row group (blockIdx.y), <= kRowsPerGroup
  int nks;                         // key slices per row tile (bf16 path), same for every row group
  int direct;                      // bf16 path: each CTA owns whole segments and writes o itself
  int segs_per_cta;                // direct mode: segments per CTA
  int tc_groups;                   // tensor-core path: row groups per key range (CTA = range x group)
  float* part_o;                   // [slots][nks][rows][D]  (slot = segment + CTA index)
  float2* part_ml;                 // [slots][nks][rows]  (m in log2 units, l)
  uint32_t* status;
  // window with a fused ring append: the partial kernels mask the slot of token pos - 1 (about
  // to be overwritten) and the merge kernel (or, in direct mode, the partial kernel) adds the new
  // key (k_new, v_new) to the softmax and stores it into that slot.  has_new = 0: no append.
  int has_new;
  int n_sinks;                     // window: attention-sink slots at the front of the ring
  int kv_bf16;                     // q, k_new, v_new element type (same as the cache)
  const void* k_new;
  const void* v_new;
  int64_t new_sb, new_sh;
  // verify with a fused append: the nq new tokens' K/V (k_new, v_new as [B, nq, Hkv, D] with
  // strides new_sb, new_st, new_sh) go to positions lens[b] - nq .. lens[b] - 1 first
  int verify_append;
  int64_t new_st;
  int debug_no_loads;              // test hook: the producers issue no K/V copies (waits run out)
  int kv_pair;                     // draft window kernel: tmK maps K and V together (one copy per tile)
  int kv_swap;                     //   ... with V at the lower address, so a tile lands V first
  int q_tma;                       // pair kernel: the first part's Q rows come by TMA (tmQ)
  unsigned long long anc[64];      // tree: bit m of anc[i] set iff node m is on i's root path
};

// Workspace layout for the attention kernels (bytes), for a given number of segments and rows.
size_t attn_workspace_bytes(int segments, int rows, int D);
void attn_workspace_carve(void* ws, int segments, int rows, int D, AttnParams* p);

// Launch helpers; return a cudaError_t.  tmK/tmV are used by the bf16 path only; tmQ (may be
// null) by the pair kernel only, over Q as [B, nq, Hq, D] with boxes of 64 x G heads x 128 / G
// positions (see q_tma_possible).
cudaError_t launch_attention(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV, int kv_bf16,
                             cudaStream_t stream, const CUtensorMap* tmQ = nullptr);
// Whether a Q tensor map for the pair kernel applies: D 128, every row block 128 rows of whole
// GQA groups (G divides 128, nq * G a multiple of 128, more than 128 rows).
bool q_tma_possible(int D, int G, int nq);

// tcgen05 partial kernel (attn_tc.cu): D = 128, bf16, up to 128 query rows per row group; two
// softmax warpgroups on alternate tiles, so each part leaves kTcSlices records.
constexpr int kTcSlices = 2;
cudaError_t launch_partial_tc(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                              cudaStream_t stream);
size_t attn_tc_smem_bytes();

// tcgen05 kernel for more than 128 rows per kv head (attn_tc_pair.cu): a pair of 128-row blocks per
// CTA, Q in shared memory, two S buffers and O per block in TMEM, 64-key tiles (its tensor maps
// use 64-key boxes); one record per row and part, o as column-major [D][128] blocks.
constexpr int kPairTileKeys = 64;
cudaError_t launch_partial_tc_pair(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                   const CUtensorMap* tmQ, cudaStream_t stream);
size_t attn_tc_pair_smem_bytes();
// Keys per TMA box the bf16 tensor maps of a launch need (rows = query rows per kv head).
int attn_tile_keys(int rows, int D);
// merge of the pair kernel's records (column-major o blocks)
cudaError_t launch_merge_pair(const AttnParams& p, cudaStream_t stream);
// The same for the draft window: 64-key boxes where the small per-segment window kernel runs.
int window_tile_keys(int rows, int D, int kv_bf16);
bool window_uses_small_kernel(int rows, int D, int kv_bf16);

}  // namespace specv
