// C ABI of libspecverify: argument validation, workspace sizing, TMA descriptor encoding and
// kernel launches.  Nothing here allocates memory or keeps mutable state between calls (the
// driver entry point for tensor-map encoding is looked up once and never changes).
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "attn_internal.h"
#include "commit_internal.h"
#include "lmhead_internal.h"
#include "sample_internal.h"
#include "spec_verify.h"

namespace {

using specv::AttnParams;
using specv::SampleParams;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Tree: parent[0] == -1, 0 <= parent[i] < i.  Fills ancestor masks and depths; returns max depth
// or -1 if malformed.
int build_tree(const int32_t* parent, int N, unsigned long long* anc, int8_t* par8, int8_t* depth8) {
  if (!parent || N < 1 || N > 64) return -1;
  if (parent[0] != -1) return -1;
  int depth[64];
  depth[0] = 0;
  if (anc) anc[0] = 1ull;
  if (par8) par8[0] = -1;
  int maxd = 0;
  for (int i = 1; i < N; ++i) {
    const int p = parent[i];
    if (p < 0 || p >= i) return -1;
    depth[i] = depth[p] + 1;
    if (anc) anc[i] = anc[p] | (1ull << i);
    if (par8) par8[i] = (int8_t)p;
    if (depth[i] > maxd) maxd = depth[i];
  }
  if (depth8)
    for (int i = 0; i < N; ++i) depth8[i] = (int8_t)depth[i];
  return maxd;
}

bool encode_kv_map(CUtensorMap* m, const void* base, int D, int L, int Hkv, int B, int64_t stride_h,
                   int64_t stride_b, int box_keys = specv::kKeyTile) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  // (column, key, half of D, head, batch): a box is a whole tile, its halves one after the other
  cuuint64_t dims[5] = {64, (cuuint64_t)L, (cuuint64_t)D / 64, (cuuint64_t)Hkv, (cuuint64_t)B};
  cuuint64_t strides[4] = {(cuuint64_t)D * 2, 128, (cuuint64_t)stride_h * 2, (cuuint64_t)stride_b * 2};
  cuuint32_t box[5] = {64, (cuuint32_t)box_keys, (cuuint32_t)D / 64, 1, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// K and V together, for the draft window kernel: (column, key, half of D, tensor, segment) over the
// lower-addressed of the two rings, the fourth dimension stepping to the other ring; segment
// s = b * Hkv + g (rings whose batch stride is Hkv head strides).  A box is one tile of both
// tensors.  Returns false (the caller falls back to one map per tensor) when the rings are 2^40
// bytes or more apart; *swap = 1 when V is the lower-addressed ring (a tile then lands V first).
bool encode_kv_pair_map(CUtensorMap* m, const void* k, const void* v, int D, int L, int segs, int64_t stride_h,
                        int box_keys, int* swap) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || k == v) return false;
  const uintptr_t ka = reinterpret_cast<uintptr_t>(k), va = reinterpret_cast<uintptr_t>(v);
  const uintptr_t lo = ka < va ? ka : va, dist = ka < va ? va - ka : ka - va;
  if (dist >= (uintptr_t(1) << 40) || (dist % 16) != 0) return false;
  cuuint64_t dims[5] = {64, (cuuint64_t)L, (cuuint64_t)D / 64, 2, (cuuint64_t)segs};
  cuuint64_t strides[4] = {(cuuint64_t)D * 2, 128, (cuuint64_t)dist, (cuuint64_t)stride_h * 2};
  cuuint32_t box[5] = {64, (cuuint32_t)box_keys, (cuuint32_t)D / 64, 2, 1};
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, reinterpret_cast<void*>(lo), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  *swap = va < ka ? 1 : 0;
  return true;
}

// Q of the verify call as [B, nq, Hq, D] bf16 for the pair kernel: a box is one half of D (64
// elements, 128-byte swizzle) of the G heads of one kv head over 128 / G consecutive positions,
// i.e. 128 consecutive query rows of a row block in the kernel's row order.
bool encode_q_map(CUtensorMap* m, const spec_attn_args* a) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int G = a->Hq / a->Hkv;
  cuuint64_t dims[4] = {(cuuint64_t)a->D, (cuuint64_t)a->Hq, (cuuint64_t)a->nq, (cuuint64_t)a->B};
  cuuint64_t strides[3] = {(cuuint64_t)a->q_stride_h * 2, (cuuint64_t)a->q_stride_t * 2, (cuuint64_t)a->q_stride_b * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)G, (cuuint32_t)(128 / G), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(a->q), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// bf16 [rows, cols] row-major (cols contiguous, a multiple of 64) viewed as (column in chunk, row,
// chunk of 64 columns): a box is box_rows rows x box_chunks chunks, landing chunk after chunk,
// each chunk's rows 128 bytes apart with the 128-byte swizzle
bool encode_chunk_map(CUtensorMap* m, const void* base, int cols, int rows, int box_rows, int box_chunks) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, (cuuint64_t)rows, (cuuint64_t)cols / 64};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, 128};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, (cuuint32_t)box_chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int num_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  return sms;
}

// ------------------------------------------------------------------ attention validation
struct AttnShape {
  int B, Hq, Hkv, D, nq, Lmax, q_dtype, kv_dtype, o_dtype;
};

int check_attn_shape(const AttnShape& s) {
  if (s.B < 1 || s.B > 4096 || s.Hq < 1 || s.Hkv < 1 || s.nq < 1 || s.Lmax < 1) return SPEC_ERR_INVALID_ARG;
  if (s.Hq % s.Hkv != 0) return SPEC_ERR_INVALID_ARG;
  if (s.D != 64 && s.D != 128) return SPEC_ERR_UNSUPPORTED;
  if ((long long)s.nq * (s.Hq / s.Hkv) > 1024) return SPEC_ERR_UNSUPPORTED;
  if (s.kv_dtype != SPEC_F32 && s.kv_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (s.q_dtype != s.kv_dtype) return SPEC_ERR_UNSUPPORTED;
  if (s.o_dtype != SPEC_F32 && s.o_dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

int check_kv_layout(const void* k, const void* v, int kv_dtype, int64_t sb, int64_t sh) {
  if (!k || !v) return SPEC_ERR_INVALID_ARG;
  if (sb < 0 || sh < 0) return SPEC_ERR_INVALID_ARG;
  if (kv_dtype == SPEC_BF16) {
    if (!aligned(k, 16) || !aligned(v, 16) || (sb % 8) != 0 || (sh % 8) != 0) return SPEC_ERR_INVALID_ARG;
  } else {
    if (!aligned(k, 4) || !aligned(v, 4)) return SPEC_ERR_INVALID_ARG;
  }
  return SPEC_OK;
}

int check_q_layout(const void* q, int dtype, int64_t s0, int64_t s1, int64_t s2) {
  if (!q || s0 < 0 || s1 < 0 || s2 < 0) return SPEC_ERR_INVALID_ARG;
  if (dtype == SPEC_BF16 && (!aligned(q, 16) || (s0 % 8) || (s1 % 8) || (s2 % 8))) return SPEC_ERR_INVALID_ARG;
  if (dtype == SPEC_F32 && !aligned(q, 4)) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

int check_o_layout(const void* o, int dtype, int64_t s0, int64_t s1, int64_t s2) {
  if (!o || s0 < 0 || s1 < 0 || s2 < 0) return SPEC_ERR_INVALID_ARG;
  if (!aligned(o, dtype == SPEC_BF16 ? 2 : 4)) return SPEC_ERR_INVALID_ARG;
  return SPEC_OK;
}

int check_workspace(void* ws, size_t have, size_t need) {
  if (need == 0) return SPEC_ERR_INVALID_ARG;
  if (!ws || have < need || !aligned(ws, 256)) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

float resolve_scale(float scale, int D) { return scale != 0.f ? scale : 1.0f / sqrtf((float)D); }

}  // namespace

extern "C" {

int spec_abi_version(void) { return 6; }

size_t spec_abi_struct_size(int which) {
  switch (which) {
    case 0: return sizeof(spec_attn_args);
    case 1: return sizeof(spec_window_args);
    case 2: return sizeof(spec_sample_args);
    case 3: return sizeof(spec_commit_args);
    case 4: return sizeof(spec_lmhead_args);
    default: return 0;
  }
}

const char* spec_status_string(int s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported configuration";
    case SPEC_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case SPEC_ERR_CUDA: return "CUDA error";
    case SPEC_ERR_SCRATCH_LIMIT: return "problem needs more scratch than the no-allocation entry point holds";
    default: return "unknown status";
  }
}

// ------------------------------------------------------------------ spec_verify_attn
size_t spec_verify_attn_workspace(const spec_attn_args* a) {
  if (!a) return 0;
  AttnShape s{a->B, a->Hq, a->Hkv, a->D, a->nq, a->Lmax, a->q_dtype, a->kv_dtype, a->o_dtype};
  if (check_attn_shape(s) != SPEC_OK) return 0;
  return specv::attn_workspace_bytes(a->B * a->Hkv, a->nq * (a->Hq / a->Hkv), a->D);
}

int spec_verify_attn(const spec_attn_args* a, spec_stream_t stream) {
  if (!a) return SPEC_ERR_INVALID_ARG;
  AttnShape s{a->B, a->Hq, a->Hkv, a->D, a->nq, a->Lmax, a->q_dtype, a->kv_dtype, a->o_dtype};
  int st = check_attn_shape(s);
  if (st != SPEC_OK) return st;
  if (a->Lmax < a->nq) return SPEC_ERR_INVALID_ARG;
  if ((st = check_q_layout(a->q, a->q_dtype, a->q_stride_b, a->q_stride_t, a->q_stride_h)) != SPEC_OK) return st;
  if ((st = check_kv_layout(a->k, a->v, a->kv_dtype, a->kv_stride_b, a->kv_stride_h)) != SPEC_OK) return st;
  if ((st = check_o_layout(a->o, a->o_dtype, a->o_stride_b, a->o_stride_t, a->o_stride_h)) != SPEC_OK) return st;
  if (!a->kv_len) return SPEC_ERR_INVALID_ARG;
  if (!isfinite(a->scale)) return SPEC_ERR_INVALID_ARG;
  if ((a->debug_flags & ~SPEC_DEBUG_NO_LOADS) != 0) return SPEC_ERR_INVALID_ARG;
  if ((a->k_new == nullptr) != (a->v_new == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (a->k_new) {
    // the append moves 16-byte chunks: both row sets 16-byte aligned
    const int64_t el = a->kv_dtype == SPEC_BF16 ? 2 : 4;
    const int64_t st[5] = {a->new_stride_b, a->new_stride_t, a->new_stride_h, a->kv_stride_b, a->kv_stride_h};
    for (int64_t x : st)
      if (x < 0 || (x * el) % 16 != 0) return SPEC_ERR_INVALID_ARG;
    const uintptr_t ptrs[4] = {(uintptr_t)a->k_new, (uintptr_t)a->v_new, (uintptr_t)a->k, (uintptr_t)a->v};
    for (uintptr_t x : ptrs)
      if (x % 16 != 0) return SPEC_ERR_INVALID_ARG;
  }
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.mask = specv::kMaskChain;
  if (a->tree_parent) {
    if (a->nq > 64) return SPEC_ERR_UNSUPPORTED;
    if (build_tree(a->tree_parent, a->nq, p.anc, nullptr, nullptr) < 0) return SPEC_ERR_INVALID_ARG;
    p.mask = specv::kMaskTree;
  }
  const size_t need = spec_verify_attn_workspace(a);
  if ((st = check_workspace(a->workspace, a->workspace_bytes, need)) != SPEC_OK) return st;

  p.B = a->B; p.Hq = a->Hq; p.Hkv = a->Hkv; p.G = a->Hq / a->Hkv; p.D = a->D; p.nq = a->nq;
  p.rows = a->nq * p.G;
  p.Lmax = a->Lmax;
  p.is_window = 0;
  p.lens = a->kv_len;
  p.q = a->q; p.q_sb = a->q_stride_b; p.q_st = a->q_stride_t; p.q_sh = a->q_stride_h;
  p.k = a->k; p.v = a->v; p.kv_sb = a->kv_stride_b; p.kv_sh = a->kv_stride_h;
  p.scale_log2 = resolve_scale(a->scale, a->D) * 1.4426950408889634f;
  p.o = a->o; p.o_sb = a->o_stride_b; p.o_st = a->o_stride_t; p.o_sh = a->o_stride_h;
  p.o_bf16 = a->o_dtype == SPEC_BF16;
  p.kv_bf16 = a->kv_dtype == SPEC_BF16;
  p.verify_append = a->k_new != nullptr;
  p.debug_no_loads = (a->debug_flags & SPEC_DEBUG_NO_LOADS) != 0;
  p.k_new = a->k_new; p.v_new = a->v_new;
  p.new_sb = a->new_stride_b; p.new_st = a->new_stride_t; p.new_sh = a->new_stride_h;
  specv::attn_workspace_carve(a->workspace, p.B * p.Hkv, p.rows, p.D, &p);

  CUtensorMap tmK, tmV;
  const int bf16 = a->kv_dtype == SPEC_BF16;
  if (bf16) {
    const int box = specv::attn_tile_keys(p.rows, a->D);
    if (!encode_kv_map(&tmK, a->k, a->D, a->Lmax, a->Hkv, a->B, a->kv_stride_h, a->kv_stride_b, box) ||
        !encode_kv_map(&tmV, a->v, a->D, a->Lmax, a->Hkv, a->B, a->kv_stride_h, a->kv_stride_b, box))
      return SPEC_ERR_CUDA;
  }
  // the pair kernel (more than 128 query rows per kv head) takes its first Q rows by TMA when the
  // rows of a block are whole GQA groups and the strides suit a tensor map; otherwise its threads
  // load them
  CUtensorMap tmQ;
  bool qmap = false;
  if (bf16 && a->q_dtype == SPEC_BF16 && specv::q_tma_possible(a->D, p.G, a->nq) && aligned(a->q, 16) &&
      (a->q_stride_h * 2) % 16 == 0 && (a->q_stride_t * 2) % 16 == 0 && (a->q_stride_b * 2) % 16 == 0)
    qmap = encode_q_map(&tmQ, a);
  cudaError_t e = specv::launch_attention(p, bf16 ? &tmK : nullptr, bf16 ? &tmV : nullptr, bf16,
                                          reinterpret_cast<cudaStream_t>(stream), qmap ? &tmQ : nullptr);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// ------------------------------------------------------------------ spec_draft_window_attn
size_t spec_draft_window_attn_workspace(const spec_window_args* a) {
  if (!a) return 0;
  AttnShape s{a->B, a->Hq, a->Hkv, a->D, 1, a->W, a->q_dtype, a->kv_dtype, a->o_dtype};
  if (check_attn_shape(s) != SPEC_OK) return 0;
  return specv::attn_workspace_bytes(a->B * a->Hkv, a->Hq / a->Hkv, a->D);
}

int spec_draft_window_attn(const spec_window_args* a, spec_stream_t stream) {
  if (!a) return SPEC_ERR_INVALID_ARG;
  AttnShape s{a->B, a->Hq, a->Hkv, a->D, 1, a->W, a->q_dtype, a->kv_dtype, a->o_dtype};
  int st = check_attn_shape(s);
  if (st != SPEC_OK) return st;
  if ((st = check_q_layout(a->q, a->q_dtype, a->q_stride_b, 0, a->q_stride_h)) != SPEC_OK) return st;
  if ((st = check_kv_layout(a->k_ring, a->v_ring, a->kv_dtype, a->ring_stride_b, a->ring_stride_h)) != SPEC_OK)
    return st;
  if ((st = check_o_layout(a->o, a->o_dtype, a->o_stride_b, 0, a->o_stride_h)) != SPEC_OK) return st;
  if (!a->pos) return SPEC_ERR_INVALID_ARG;
  if ((a->k_new == nullptr) != (a->v_new == nullptr)) return SPEC_ERR_INVALID_ARG;
  if (a->k_new && (a->new_stride_b < 0 || a->new_stride_h < 0)) return SPEC_ERR_INVALID_ARG;
  if (!isfinite(a->scale)) return SPEC_ERR_INVALID_ARG;
  if (a->n_sinks < 0 || a->n_sinks >= a->W) return SPEC_ERR_INVALID_ARG;
  const size_t need = spec_draft_window_attn_workspace(a);
  if ((st = check_workspace(a->workspace, a->workspace_bytes, need)) != SPEC_OK) return st;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const int bf16 = a->kv_dtype == SPEC_BF16;
  AttnParams p;
  memset(&p, 0, sizeof(p));
  p.B = a->B; p.Hq = a->Hq; p.Hkv = a->Hkv; p.G = a->Hq / a->Hkv; p.D = a->D; p.nq = 1;
  p.rows = p.G;
  p.mask = specv::kMaskNone;
  p.Lmax = a->W;
  p.is_window = 1;
  p.lens = a->pos;
  p.q = a->q; p.q_sb = a->q_stride_b; p.q_st = 0; p.q_sh = a->q_stride_h;
  p.k = a->k_ring; p.v = a->v_ring; p.kv_sb = a->ring_stride_b; p.kv_sh = a->ring_stride_h;
  p.scale_log2 = resolve_scale(a->scale, a->D) * 1.4426950408889634f;
  p.o = a->o; p.o_sb = a->o_stride_b; p.o_st = 0; p.o_sh = a->o_stride_h;
  p.o_bf16 = a->o_dtype == SPEC_BF16;
  p.kv_bf16 = bf16;
  p.has_new = a->k_new != nullptr;
  p.n_sinks = a->n_sinks;
  p.k_new = a->k_new; p.v_new = a->v_new;
  p.new_sb = a->new_stride_b; p.new_sh = a->new_stride_h;
  specv::attn_workspace_carve(a->workspace, p.B * p.Hkv, p.rows, p.D, &p);
  CUtensorMap tmK, tmV;
  if (bf16) {
    const int box = specv::window_tile_keys(p.rows, a->D, bf16);
    // the small window kernel takes K and V of a tile in one copy when the rings' heads are
    // contiguous over the batch (one segment index) and the two rings lie under 2^40 bytes apart
    if (specv::window_uses_small_kernel(p.rows, a->D, bf16) && a->ring_stride_b == (int64_t)a->Hkv * a->ring_stride_h &&
        encode_kv_pair_map(&tmK, a->k_ring, a->v_ring, a->D, a->W, a->B * a->Hkv, a->ring_stride_h, box, &p.kv_swap)) {
      p.kv_pair = 1;
      tmV = tmK;
    } else if (!encode_kv_map(&tmK, a->k_ring, a->D, a->W, a->Hkv, a->B, a->ring_stride_h, a->ring_stride_b, box) ||
               !encode_kv_map(&tmV, a->v_ring, a->D, a->W, a->Hkv, a->B, a->ring_stride_h, a->ring_stride_b, box)) {
      return SPEC_ERR_CUDA;
    }
  }
  cudaError_t e = specv::launch_attention(p, bf16 ? &tmK : nullptr, bf16 ? &tmV : nullptr, bf16, cs);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// ------------------------------------------------------------------ spec_sample
static int sample_rows(const spec_sample_args* a, int* rows_t, int* rows_d) {
  switch (a->mode) {
    case SPEC_SAMPLE_CHAIN:
      if (a->n < 1 || a->n > specv::kMaxGamma) return SPEC_ERR_UNSUPPORTED;
      *rows_t = a->n + 1; *rows_d = a->n;
      return SPEC_OK;
    case SPEC_SAMPLE_CHAIN_GREEDY:
      if (a->n < 0 || a->n > specv::kMaxGamma) return SPEC_ERR_UNSUPPORTED;
      *rows_t = a->n + 1; *rows_d = 0;
      return SPEC_OK;
    case SPEC_SAMPLE_TREE_GREEDY:
      if (a->n < 1 || a->n > specv::kMaxTreeNodes) return SPEC_ERR_UNSUPPORTED;
      *rows_t = a->n; *rows_d = 0;
      return SPEC_OK;
    case SPEC_SAMPLE_TREE:
      if (a->n < 1 || a->n > specv::kMaxTreeNodes) return SPEC_ERR_UNSUPPORTED;
      *rows_t = a->n; *rows_d = a->n;
      return SPEC_OK;
    default: return SPEC_ERR_INVALID_ARG;
  }
}

size_t spec_sample_workspace(const spec_sample_args* a) {
  if (!a) return 0;
  int rt, rd;
  if (sample_rows(a, &rt, &rd) != SPEC_OK) return 0;
  if (a->B < 1 || a->V < 1 || a->V > (1 << 20)) return 0;
  return specv::sample_workspace_bytes(a->mode, a->B, rt, rd, a->V);
}

int spec_sample(const spec_sample_args* a, spec_stream_t stream) {
  if (!a) return SPEC_ERR_INVALID_ARG;
  int rt, rd;
  int st = sample_rows(a, &rt, &rd);
  if (st != SPEC_OK) return st;
  if (a->B < 1 || a->V < 1) return SPEC_ERR_INVALID_ARG;
  if (a->V > (1 << 20) || (a->V % 4) != 0) return SPEC_ERR_UNSUPPORTED;
  if (a->V > specv::kSmallVocab && a->B > 65535) return SPEC_ERR_UNSUPPORTED;
  if (!a->target_logits || !aligned(a->target_logits, 16) || a->tl_stride_b < 0 || (a->tl_stride_b % 4))
    return SPEC_ERR_INVALID_ARG;
  if (!a->out_tokens || !a->out_num_accepted) return SPEC_ERR_INVALID_ARG;
  if (a->mode == SPEC_SAMPLE_CHAIN || a->mode == SPEC_SAMPLE_TREE) {
    if (!a->draft_logits || !aligned(a->draft_logits, 16) || a->dl_stride_b < 0 || (a->dl_stride_b % 4))
      return SPEC_ERR_INVALID_ARG;
    if (!a->uniforms || a->u_stride_b < 0) return SPEC_ERR_INVALID_ARG;
  }
  if ((a->mode != SPEC_SAMPLE_CHAIN_GREEDY || a->n > 0) && (!a->draft_tokens || a->tok_stride_b < 0))
    return SPEC_ERR_INVALID_ARG;
  SampleParams p;
  memset(&p, 0, sizeof(p));
  const bool tree = a->mode == SPEC_SAMPLE_TREE_GREEDY || a->mode == SPEC_SAMPLE_TREE;
  if (tree) {
    const int maxd = build_tree(a->tree_parent, a->n, nullptr, p.parent, p.depth);
    if (maxd < 0) return SPEC_ERR_INVALID_ARG;
    if (a->out_cols < maxd + 1) return SPEC_ERR_INVALID_ARG;
    p.N = a->n;
  } else if (a->out_cols < a->n + 1) {
    return SPEC_ERR_INVALID_ARG;
  }
  const size_t need = spec_sample_workspace(a);
  if ((st = check_workspace(a->workspace, a->workspace_bytes, need)) != SPEC_OK) return st;
  const int sms = num_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;

  p.mode = a->mode; p.B = a->B; p.V = a->V;
  p.gamma = tree ? 0 : a->n;
  p.rows_t = rt; p.rows_d = rd;
  p.tl = a->target_logits; p.tl_sb = a->tl_stride_b;
  p.dl = a->draft_logits; p.dl_sb = a->dl_stride_b;
  p.tok = a->draft_tokens; p.tok_sb = a->tok_stride_b;
  p.u = a->uniforms; p.u_sb = a->u_stride_b;
  p.out_cols = a->out_cols; p.out_tok = a->out_tokens; p.out_nacc = a->out_num_accepted;
  p.out_nodes = a->out_path_nodes;
  specv::sample_workspace_carve(a->workspace, &p);
  cudaError_t e = specv::launch_sample(p, sms, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}


// ------------------------------------------------------------------ spec_lmhead_sample
static bool lmhead_stochastic(int mode) { return mode == SPEC_SAMPLE_CHAIN || mode == SPEC_SAMPLE_TREE; }

static int lmhead_rows(const spec_lmhead_args* a, int* R) {
  if (a->mode == SPEC_SAMPLE_CHAIN_GREEDY || a->mode == SPEC_SAMPLE_CHAIN) {
    const int lo = a->mode == SPEC_SAMPLE_CHAIN ? 1 : 0;
    if (a->n < lo || a->n > specv::kMaxGamma) return SPEC_ERR_UNSUPPORTED;
    *R = a->n + 1;
    return SPEC_OK;
  }
  if (a->mode == SPEC_SAMPLE_TREE_GREEDY || a->mode == SPEC_SAMPLE_TREE) {
    if (a->n < 1 || a->n > specv::kLmMaxNodes) return SPEC_ERR_UNSUPPORTED;
    *R = a->n;
    return SPEC_OK;
  }
  return SPEC_ERR_INVALID_ARG;
}

// Workspace of the fused LM-head: the status word and the row keys; in stochastic modes then the
// logits (unless the caller takes them in out_logits) and the sampling kernels' workspace.
struct LmWs {
  size_t keys, logits, sample, total;
};
static bool lmhead_ws(const spec_lmhead_args* a, int R, LmWs* w) {
  const int nrows = a->B * R;
  w->keys = specv::lmhead_workspace_bytes(nrows);
  w->logits = 0;
  w->sample = 0;
  if (lmhead_stochastic(a->mode)) {
    w->keys = (w->keys + 255) / 256 * 256;
    if (a->V > (1 << 20) || (a->V % 4) != 0) return false;
    if (!a->out_logits) w->logits = ((size_t)nrows * a->V * sizeof(float) + 255) / 256 * 256;
    // target rows R, draft rows n (chain: gamma, tree: N)
    w->sample = specv::sample_workspace_bytes(a->mode, a->B, R, a->n, a->V);
  }
  w->total = w->keys + w->logits + w->sample;
  return true;
}

size_t spec_lmhead_sample_workspace(const spec_lmhead_args* a) {
  if (!a) return 0;
  int R;
  if (lmhead_rows(a, &R) != SPEC_OK) return 0;
  if (a->B < 1 || a->V < 1 || a->V > (1 << 24) || (int64_t)a->B * R > specv::kLmMaxRows) return 0;
  LmWs w;
  if (!lmhead_ws(a, R, &w)) return 0;
  return w.total;
}

int spec_lmhead_sample(const spec_lmhead_args* a, spec_stream_t stream) {
  if (!a) return SPEC_ERR_INVALID_ARG;
  int R;
  int st = lmhead_rows(a, &R);
  if (st != SPEC_OK) return st;
  if (a->B < 1 || a->V < 1 || a->d < 64 || (a->d % 64) != 0 || a->d > 65536) return SPEC_ERR_INVALID_ARG;
  if (a->V > (1 << 24) || (int64_t)a->B * R > specv::kLmMaxRows) return SPEC_ERR_UNSUPPORTED;
  if (!a->hidden || !a->weight || !aligned(a->hidden, 16) || !aligned(a->weight, 16)) return SPEC_ERR_INVALID_ARG;
  if (!a->out_tokens || !a->out_num_accepted) return SPEC_ERR_INVALID_ARG;
  const bool stochastic = lmhead_stochastic(a->mode);
  const bool tree = a->mode == SPEC_SAMPLE_TREE_GREEDY || a->mode == SPEC_SAMPLE_TREE;
  if ((tree || a->n > 0) && (!a->draft_tokens || a->tok_stride_b < 0)) return SPEC_ERR_INVALID_ARG;
  if (stochastic) {
    if (a->V > (1 << 20) || (a->V % 4) != 0) return SPEC_ERR_UNSUPPORTED;
    if (!a->draft_logits || !aligned(a->draft_logits, 16) || a->dl_stride_b < 0 || (a->dl_stride_b % 4))
      return SPEC_ERR_INVALID_ARG;
    if (!a->uniforms || a->u_stride_b < 0) return SPEC_ERR_INVALID_ARG;
    if (a->out_logits && !aligned(a->out_logits, 16)) return SPEC_ERR_INVALID_ARG;
  }
  specv::LmheadParams p;
  memset(&p, 0, sizeof(p));
  SampleParams sp;
  memset(&sp, 0, sizeof(sp));
  int maxd = 0;
  if (tree) {
    maxd = build_tree(a->tree_parent, a->n, nullptr, p.parent, p.depth);
    if (maxd < 0) return SPEC_ERR_INVALID_ARG;
    if (a->out_cols < maxd + 1) return SPEC_ERR_INVALID_ARG;
    memcpy(sp.parent, p.parent, sizeof(sp.parent));
    memcpy(sp.depth, p.depth, sizeof(sp.depth));
  } else if (a->out_cols < a->n + 1) {
    return SPEC_ERR_INVALID_ARG;
  }
  LmWs w;
  if (!lmhead_ws(a, R, &w)) return SPEC_ERR_UNSUPPORTED;
  if ((st = check_workspace(a->workspace, a->workspace_bytes, w.total)) != SPEC_OK) return st;
  const int sms = num_sms();
  if (sms <= 0) return SPEC_ERR_CUDA;
  p.mode = a->mode; p.B = a->B; p.R = R; p.d = a->d; p.V = a->V;
  p.nrows = a->B * R;
  p.npad = (p.nrows + 15) / 16 * 16;
  p.n_vtiles = (a->V + 127) / 128;
  p.tiles_per_pass = 512 / p.npad;
  const specv::LmLayout lay = specv::lmhead_layout(p.npad);
  p.w_stages = lay.w_stages; p.h_stages = lay.h_stages; p.kgroup = lay.kgroup;
  p.wbox = lay.wbox; p.hbox = lay.hbox;
  p.tok = a->draft_tokens; p.tok_sb = a->tok_stride_b;
  p.out_cols = a->out_cols; p.out_tok = a->out_tokens; p.out_nacc = a->out_num_accepted; p.out_nodes = a->out_path_nodes;
  specv::lmhead_workspace_carve(a->workspace, &p);
  CUtensorMap tmW, tmH;
  if (!encode_chunk_map(&tmW, a->weight, a->d, a->V, 128, p.wbox) ||
      !encode_chunk_map(&tmH, a->hidden, a->d, p.nrows, p.npad, p.hbox))
    return SPEC_ERR_CUDA;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (!stochastic) {
    cudaError_t e = specv::launch_lmhead(p, &tmW, &tmH, sms, cs);
    return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
  }
  // stochastic: the GEMM writes the target logits, then the kernels of spec_sample in that mode;
  // both flag into the one status word at byte 0, cleared once here
  uint8_t* base = reinterpret_cast<uint8_t*>(a->workspace);
  p.logits = a->out_logits ? a->out_logits : reinterpret_cast<float*>(base + w.keys);
  cudaError_t e = cudaMemsetAsync(p.status, 0, 256, cs);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  e = specv::launch_lmhead_logits(p, &tmW, &tmH, sms, cs);
  if (e != cudaSuccess) return SPEC_ERR_CUDA;
  sp.mode = a->mode; sp.B = a->B; sp.V = a->V;
  sp.gamma = tree ? 0 : a->n;
  sp.rows_t = R;
  sp.rows_d = a->n;
  sp.N = tree ? a->n : 0;
  sp.tl = p.logits; sp.tl_sb = (int64_t)R * a->V;
  sp.dl = a->draft_logits; sp.dl_sb = a->dl_stride_b;
  sp.tok = a->draft_tokens; sp.tok_sb = a->tok_stride_b;
  sp.u = a->uniforms; sp.u_sb = a->u_stride_b;
  sp.out_cols = a->out_cols; sp.out_tok = a->out_tokens; sp.out_nacc = a->out_num_accepted;
  sp.out_nodes = a->out_path_nodes;
  // the sampling workspace follows; its kernels report into the call's status word
  specv::sample_workspace_carve(base + w.keys + w.logits, &sp);
  sp.status = p.status;
  sp.status_zeroed = 1;
  e = specv::launch_sample(sp, sms, cs);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// ------------------------------------------------------------------ spec_commit
size_t spec_commit_workspace(const spec_commit_args* a) {
  if (!a) return 0;
  return 256;
}

int spec_commit(const spec_commit_args* a, spec_stream_t stream) {
  if (!a) return SPEC_ERR_INVALID_ARG;
  if (a->mode != SPEC_COMMIT_CHAIN && a->mode != SPEC_COMMIT_TREE) return SPEC_ERR_INVALID_ARG;
  if (a->B < 1 || a->nq < 1 || a->Lmax < a->nq || !a->kv_len || !a->num_accepted) return SPEC_ERR_INVALID_ARG;
  if (a->B > 65535) return SPEC_ERR_UNSUPPORTED;
  if (a->mode == SPEC_COMMIT_TREE) {
    if (a->nq > specv::kCommitMaxNodes) return SPEC_ERR_UNSUPPORTED;
    if (a->kv_dtype != SPEC_BF16 && a->kv_dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
    const int bf16 = a->kv_dtype == SPEC_BF16;
    if (!a->k || !a->v || !a->path_nodes || a->Hkv < 1 || a->D < 2 || a->D > 256 || (a->D % 2)) return SPEC_ERR_INVALID_ARG;
    if (a->path_cols < 1 || (a->B > 1 && a->path_stride_b < a->path_cols)) return SPEC_ERR_INVALID_ARG;
    if (a->kv_stride_b < 0 || a->kv_stride_h < 0) return SPEC_ERR_INVALID_ARG;
    if (!aligned(a->k, 4) || !aligned(a->v, 4)) return SPEC_ERR_INVALID_ARG;
    if (bf16 && ((a->kv_stride_b % 2) || (a->kv_stride_h % 2))) return SPEC_ERR_INVALID_ARG;
  }
  int st = check_workspace(a->workspace, a->workspace_bytes, spec_commit_workspace(a));
  if (st != SPEC_OK) return st;
  specv::CommitParams p;
  memset(&p, 0, sizeof(p));
  p.mode = a->mode; p.B = a->B; p.Hkv = a->Hkv; p.D = a->D; p.nq = a->nq; p.Lmax = a->Lmax;
  p.bf16 = a->kv_dtype == SPEC_BF16;
  p.k = a->k; p.v = a->v; p.kv_sb = a->kv_stride_b; p.kv_sh = a->kv_stride_h;
  p.kv_len = a->kv_len; p.num_accepted = a->num_accepted;
  p.path_nodes = a->path_nodes; p.path_sb = a->path_stride_b; p.path_cols = a->path_cols;
  p.status = reinterpret_cast<uint32_t*>(a->workspace);
  return specv::launch_commit(p, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"
