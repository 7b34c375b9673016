// Split-KV ("flash-decode") attention for speculative verify and for the draft ring window.
//
// Work decomposition (one launch, balanced over the whole batch): the key ranges of all
// (sequence b, kv head g) segments are laid end to end, total = Hkv * sum_b len_b keys, and CTA c
// takes the global range [c*T, (c+1)*T), T = max(ceil(total / grid_x), kMinKeysPerCta).  A CTA
// walks the segments its range touches; for each piece ("part") it produces the un-normalised
// flash-attention partial (m, l, o) of every query row of that segment, stored at slot s + c
// (s = b*Hkv + g; along the monotone walk s + c is unique, so S + grid_x slots suffice).  The
// merge kernel combines the parts of a segment with a log-sum-exp weighted sum.  The whole GQA
// group of a kv head (nq * G query rows) shares every K/V tile a CTA loads, so each KV byte is
// read from HBM once.
//
// bf16 K/V: TMA (cp.async.bulk.tensor, 128-byte swizzle, no multicast) fills a 3-stage ring of
// 128-key K and V tiles guarded by mbarriers; one producer warp issues the copies, eight consumer
// warps (row tiles x key slices of each tile) run QK^T and PV with mma.sync m16n8k16 (fp32
// accumulate) and an fp32 online softmax in the log2 domain.  fp32 K/V: a plain CUDA-core kernel (one warp per query row).
//
// Masks: chain row j sees keys 0 .. len - nq + j; tree node j sees the context [0, len - nq)
// and the tree keys whose node is on its root path (bitmask); window: every valid ring slot.
// Cache slots at or beyond len are never trusted: their scores are masked by select, and the
// matching V rows are zeroed before P.V, so NaN garbage there cannot leak into the output.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "common.cuh"

namespace specv {

// key slices per row tile for row groups of `rows_per_group` rows: kConsumerWarps / 16-row tiles
static inline int slices_for_rows(int rows_per_group) {
  return rows_per_group <= 16 ? kConsumerWarps : (rows_per_group <= 32 ? kConsumerWarps / 2 : kConsumerWarps / 4);
}

// ------------------------------------------------------------------ bf16 partial kernel

template <int D, int MASK, int NKS>
__device__ void consumer_loop(const AttnParams& p, uint8_t* stages, uint8_t* sQw, uint64_t* full, uint64_t* empty,
                              int warp, int lane, int row0, int rows_here, volatile int* s_abort) {
  constexpr int KT = kKeyTile;
  constexpr int KS = KT / NKS;     // keys of each tile this warp handles
  constexpr int NT = KS / 8;       // score n-tiles
  constexpr int KSTEPS = D / 16;   // k-steps over the head dim
  constexpr int DT = D / 8;        // output n-tiles
  constexpr int TILE = KT * D * 2;
  const int rt = warp / NKS, ks = warp % NKS;
  const int r_lo = rt * 16 + (lane >> 2), r_hi = r_lo + 8;
  const int j_lo = min((row0 + r_lo) / p.G, p.nq - 1), j_hi = min((row0 + r_hi) / p.G, p.nq - 1);
  const unsigned long long anc_lo = (MASK == kMaskTree) ? p.anc[j_lo] : 0ull;
  const unsigned long long anc_hi = (MASK == kMaskTree) ? p.anc[j_hi] : 0ull;
  const __nv_bfloat16* qbase = reinterpret_cast<const __nv_bfloat16*>(p.q);

  Walker w;
  walker_init(p, blockIdx.x, w);
  int stage = 0;
  uint32_t phase = 0;
  int b, g, kb, ke, len;
  while (walker_next(p, w, b, g, kb, ke, len)) {
    // ---- this warp's 16 query rows of (b, g) into its own swizzled shared-memory region
    // (padding rows are zero); A fragments are read back with ldmatrix per k-step pair
    __syncwarp();
    for (int idx = lane; idx < 16 * (D / 8); idx += 32) {
      const int r = idx / (D / 8), c = idx % (D / 8);
      const int rr = rt * 16 + r;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (rr < rows_here) {
        const int ro = row0 + rr;
        val = *reinterpret_cast<const uint4*>(qbase + b * p.q_sb + (ro / p.G) * p.q_st + (g * p.G + ro % p.G) * p.q_sh +
                                              c * 8);
      }
      *reinterpret_cast<uint4*>(sQw + r * (D * 2) + ((c ^ (r & 7)) << 4)) = val;
    }
    __syncwarp();
    float o[DT][4];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m_lo = neg_inf(), m_hi = neg_inf(), l_lo = 0.f, l_hi = 0.f;
    const int tail_start = len - p.nq;

    for (int key0 = kb; key0 < ke; key0 += KT) {
      if (!mbar_wait_bounded(&full[stage], phase, s_abort)) {
        *s_abort = 1;
        atomicOr(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
        return;
      }
      const uint8_t* sK = stages + stage * 2 * TILE;
      const uint8_t* sV = sK + TILE;
      float s[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; kk += 2) {
        uint32_t qa[4], qb[4];
        {
          const int r = ((lane >> 3) & 1) * 8 + (lane & 7);
          const int c0 = kk * 2 + (lane >> 4);
          ldmatrix_x4(smem_u32(sQw + r * (D * 2) + ((c0 ^ (r & 7)) << 4)), qa[0], qa[1], qa[2], qa[3]);
          const int c1 = c0 + 2;
          ldmatrix_x4(smem_u32(sQw + r * (D * 2) + ((c1 ^ (r & 7)) << 4)), qb[0], qb[1], qb[2], qb[3]);
        }
        const int d0 = kk * 16 + (lane >> 3) * 8;
        const int c = (d0 & 63) >> 3;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const int r = ks * KS + nt * 8 + (lane & 7);
          uint32_t b0, b1, b2, b3;
          ldmatrix_x4(smem_u32(sK + (d0 >> 6) * (KT * 128) + r * 128 + ((c ^ (r & 7)) << 4)), b0, b1, b2, b3);
          mma_bf16_16816(s[nt], qa, b0, b1);
          mma_bf16_16816(s[nt], qb, b2, b3);
        }
      }
      const bool tail_tile = key0 + KT > ke;
      const bool needs_mask = tail_tile || (MASK != kMaskNone && key0 + KT > tail_start);
      float mx_lo = neg_inf(), mx_hi = neg_inf();
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x = s[nt][e] * p.scale_log2;
          if (needs_mask) {
            const int kk = key0 + ks * KS + nt * 8 + 2 * (lane & 3) + (e & 1);
            const bool vis = (e < 2) ? key_visible<MASK>(kk, ke, tail_start, j_lo, anc_lo)
                                     : key_visible<MASK>(kk, ke, tail_start, j_hi, anc_hi);
            if (!vis) x = neg_inf();
          }
          s[nt][e] = x;
        }
        mx_lo = fmaxf(mx_lo, fmaxf(s[nt][0], s[nt][1]));
        mx_hi = fmaxf(mx_hi, fmaxf(s[nt][2], s[nt][3]));
      }
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
      mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
      mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
      const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
      const float mu_lo = (mn_lo == neg_inf()) ? 0.f : mn_lo;
      const float mu_hi = (mn_hi == neg_inf()) ? 0.f : mn_hi;
      const float a_lo = exp2f(m_lo - mu_lo), a_hi = exp2f(m_hi - mu_hi);
      m_lo = mn_lo;
      m_hi = mn_hi;
      float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - mu_lo);
        s[nt][1] = exp2f(s[nt][1] - mu_lo);
        s[nt][2] = exp2f(s[nt][2] - mu_hi);
        s[nt][3] = exp2f(s[nt][3] - mu_hi);
        sum_lo += s[nt][0] + s[nt][1];
        sum_hi += s[nt][2] + s[nt][3];
      }
      l_lo = l_lo * a_lo + sum_lo;
      l_hi = l_hi * a_hi + sum_hi;
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        o[dt][0] *= a_lo; o[dt][1] *= a_lo;
        o[dt][2] *= a_hi; o[dt][3] *= a_hi;
      }
#pragma unroll
      for (int s2 = 0; s2 < KS / 16; ++s2) {
        uint32_t a[4];
        a[0] = pack_bf16(s[2 * s2][0], s[2 * s2][1]);
        a[1] = pack_bf16(s[2 * s2][2], s[2 * s2][3]);
        a[2] = pack_bf16(s[2 * s2 + 1][0], s[2 * s2 + 1][1]);
        a[3] = pack_bf16(s[2 * s2 + 1][2], s[2 * s2 + 1][3]);
        const int r = ks * KS + s2 * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        // keys of this thread's B-fragment halves (for zeroing V rows past the part end)
        const int kf = key0 + ks * KS + s2 * 16 + 2 * (lane & 3);
#pragma unroll
        for (int dn = 0; dn < DT; dn += 2) {
          const int d0 = (dn + (lane >> 4)) * 8;
          const int c = (d0 & 63) >> 3;
          uint32_t v0, v1, v2, v3;
          ldmatrix_x4_trans(smem_u32(sV + (d0 >> 6) * (KT * 128) + r * 128 + ((c ^ (r & 7)) << 4)), v0, v1, v2, v3);
          if (tail_tile) {
            const uint32_t m0 = (kf < ke ? 0x0000ffffu : 0u) | (kf + 1 < ke ? 0xffff0000u : 0u);
            const uint32_t m1 = (kf + 8 < ke ? 0x0000ffffu : 0u) | (kf + 9 < ke ? 0xffff0000u : 0u);
            v0 &= m0; v1 &= m1; v2 &= m0; v3 &= m1;
          }
          mma_bf16_16816(o[dn], a, v0, v1);
          mma_bf16_16816(o[dn + 1], a, v2, v3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == kStages) { stage = 0; phase ^= 1u; }
    }
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
    l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    const int64_t slot = (int64_t)(b * p.Hkv + g) + blockIdx.x;
    const int64_t rec_base = (slot * kMaxSlices + ks) * p.rows + row0;
    if (r_lo < rows_here) {
      const int64_t rec = rec_base + r_lo;
      if ((lane & 3) == 0) p.part_ml[rec] = make_float2(m_lo, l_lo);
      float* dst = p.part_o + rec * D + 2 * (lane & 3);
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) *reinterpret_cast<float2*>(dst + dt * 8) = make_float2(o[dt][0], o[dt][1]);
    }
    if (r_hi < rows_here) {
      const int64_t rec = rec_base + r_hi;
      if ((lane & 3) == 0) p.part_ml[rec] = make_float2(m_hi, l_hi);
      float* dst = p.part_o + rec * D + 2 * (lane & 3);
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) *reinterpret_cast<float2*>(dst + dt * 8) = make_float2(o[dt][2], o[dt][3]);
    }
  }
}

template <int D, int MASK, int NKS>
__global__ void __launch_bounds__((kConsumerWarps + 1) * 32, 1)
    attn_partial_bf16(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                      const __grid_constant__ AttnParams p) {
  constexpr int TILE = kKeyTile * D * 2;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[2 * kStages];
  __shared__ int s_abort;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* stages = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sQ = stages + kStages * 2 * TILE;  // kConsumerWarps regions of 16 rows x D bf16
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * p.rows_per_group;
  const int rows_here = min(p.rows_per_group, p.rows - row0);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane issues every TMA copy of this CTA's walk
    Walker w;
    walker_init(p, blockIdx.x, w);
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      int b, g, kb, ke, len;
      bool ok = true;
      while (ok && walker_next(p, w, b, g, kb, ke, len)) {
        for (int key0 = kb; key0 < ke; key0 += kKeyTile) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, &s_abort)) {
            s_abort = 1;
            atomicOr(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* sK = stages + stage * 2 * TILE;
          uint8_t* sV = sK + TILE;
          mbar_arrive_expect_tx(&full[stage], 2u * TILE);
#pragma unroll
          for (int h = 0; h < D / 64; ++h) {
            tma_load_4d(sK + h * (kKeyTile * 128), &tmK, &full[stage], h * 64, key0, g, b);
            tma_load_4d(sV + h * (kKeyTile * 128), &tmV, &full[stage], h * 64, key0, g, b);
          }
          ++issued;
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
      }
      if (!ok || s_abort) {
        // drain: wait (bounded) for the copies still in flight into this CTA's shared memory
        for (int i = 1; i <= min(issued, kStages); ++i) {
          int st = stage - i, ph = (int)phase;
          if (st < 0) { st += kStages; ph ^= 1; }
          mbar_wait_bounded(&full[st], (uint32_t)ph, nullptr);
        }
      }
    }
    return;
  }
  consumer_loop<D, MASK, NKS>(p, stages, sQ + warp * (16 * D * 2), full, empty, warp, lane, row0, rows_here, &s_abort);
}

// ------------------------------------------------------------------ fp32 partial kernel
template <int D, int MASK>
__global__ void __launch_bounds__(128) attn_partial_f32(const __grid_constant__ AttnParams p) {
  constexpr int PER = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * p.rows_per_group;
  const int rows_here = min(p.rows_per_group, p.rows - row0);
  const float* qb = reinterpret_cast<const float*>(p.q);
  const float* kb_ = reinterpret_cast<const float*>(p.k);
  const float* vb_ = reinterpret_cast<const float*>(p.v);
  Walker w;
  walker_init(p, blockIdx.x, w);
  int b, g, kb, ke, len;
  while (walker_next(p, w, b, g, kb, ke, len)) {
    const int tail_start = len - p.nq;
    const float* kseg = kb_ + b * p.kv_sb + g * p.kv_sh;
    const float* vseg = vb_ + b * p.kv_sb + g * p.kv_sh;
    for (int r = warp; r < rows_here; r += 4) {
      const int rr = row0 + r, j = rr / p.G, h = g * p.G + rr % p.G;
      const unsigned long long anc = (MASK == kMaskTree) ? p.anc[j] : 0ull;
      float qv[PER], acc[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        qv[i] = qb[b * p.q_sb + j * p.q_st + h * p.q_sh + lane + 32 * i] * p.scale_log2;
        acc[i] = 0.f;
      }
      float m = neg_inf(), l = 0.f;
      for (int kk = kb; kk < ke; ++kk) {
        if (!key_visible<MASK>(kk, ke, tail_start, j, anc)) continue;
        const float* kp = kseg + (int64_t)kk * D;
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) dot = fmaf(qv[i], kp[lane + 32 * i], dot);
        dot = warp_sum(dot);
        const float mn = fmaxf(m, dot);
        const float a = exp2f(m - mn), pw = exp2f(dot - mn);
        l = l * a + pw;
        const float* vp = vseg + (int64_t)kk * D;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = fmaf(pw, vp[lane + 32 * i], acc[i] * a);
        m = mn;
      }
      const int64_t slot = (int64_t)(b * p.Hkv + g) + blockIdx.x;
      const int64_t rec = (slot * kMaxSlices + 0) * p.rows + rr;
      if (lane == 0) p.part_ml[rec] = make_float2(m, l);
#pragma unroll
      for (int i = 0; i < PER; ++i) p.part_o[rec * D + lane + 32 * i] = acc[i];
    }
  }
}

// ------------------------------------------------------------------ merge kernel
// grid (segments, ceil(rows / 4)); one warp per query row of a segment.
template <int D>
__global__ void __launch_bounds__(128) attn_merge(const __grid_constant__ AttnParams p) {
  constexpr int PER = D / 32;
  const int s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 4 + warp;
  if (r >= p.rows) return;
  const int b = s / p.Hkv, g = s % p.Hkv;
  int64_t total, cum_b;
  warp_scan_lengths(p, b, total, cum_b);
  const int len = seg_len(p, b);
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  if (len > 0) {
    const int64_t per = keys_per_cta(p, total);
    const int64_t start = cum_b + (int64_t)g * len;
    const int c0 = (int)(start / per), c1 = (int)((start + len - 1) / per);
    const int nks = p.nks;
    float M = neg_inf();
    for (int c = c0; c <= c1; ++c)
      for (int ks = 0; ks < nks; ++ks) M = fmaxf(M, p.part_ml[((int64_t)(s + c) * kMaxSlices + ks) * p.rows + r].x);
    float L = 0.f;
    if (M != neg_inf()) {
      for (int c = c0; c <= c1; ++c) {
        for (int ks = 0; ks < nks; ++ks) {
          const int64_t rec = ((int64_t)(s + c) * kMaxSlices + ks) * p.rows + r;
          const float2 ml = p.part_ml[rec];
          if (ml.x == neg_inf()) continue;
          const float wgt = exp2f(ml.x - M);
          L = fmaf(wgt, ml.y, L);
          const float* po = p.part_o + rec * D;
#pragma unroll
          for (int i = 0; i < PER; ++i) acc[i] = fmaf(wgt, po[lane + 32 * i], acc[i]);
        }
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] *= inv;
  } else if (lane == 0 && g == 0 && r == 0) {
    atomicOr(p.status, p.is_window ? (uint32_t)SPEC_STATUS_BAD_POS : (uint32_t)SPEC_STATUS_BAD_KV_LEN);
  }
  const int j = r / p.G, h = g * p.G + r % p.G;
  const int64_t off = (int64_t)b * p.o_sb + (int64_t)j * p.o_st + (int64_t)h * p.o_sh;
  if (p.o_bf16) {
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.o) + off;
#pragma unroll
    for (int i = 0; i < PER; ++i) ob[lane + 32 * i] = __float2bfloat16_rn(acc[i]);
  } else {
    float* of = reinterpret_cast<float*>(p.o) + off;
#pragma unroll
    for (int i = 0; i < PER; ++i) of[lane + 32 * i] = acc[i];
  }
}

// ------------------------------------------------------------------ ring append
__global__ void window_append_kernel(const WindowAppend a) {
  const int b = blockIdx.x / a.Hkv, g = blockIdx.x % a.Hkv;
  const int pos = a.pos[b];
  if (pos < 1) return;
  const int slot = (pos - 1) % a.W;
  const int64_t dst = (int64_t)b * a.ring_sb + (int64_t)g * a.ring_sh + (int64_t)slot * a.D;
  const int64_t src = (int64_t)b * a.new_sb + (int64_t)g * a.new_sh;
  if (a.bf16) {
    const __nv_bfloat16* kn = reinterpret_cast<const __nv_bfloat16*>(a.k_new) + src;
    const __nv_bfloat16* vn = reinterpret_cast<const __nv_bfloat16*>(a.v_new) + src;
    __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(a.k_ring) + dst;
    __nv_bfloat16* vr = reinterpret_cast<__nv_bfloat16*>(a.v_ring) + dst;
    for (int d = threadIdx.x; d < a.D; d += blockDim.x) { kr[d] = kn[d]; vr[d] = vn[d]; }
  } else {
    const float* kn = reinterpret_cast<const float*>(a.k_new) + src;
    const float* vn = reinterpret_cast<const float*>(a.v_new) + src;
    float* kr = reinterpret_cast<float*>(a.k_ring) + dst;
    float* vr = reinterpret_cast<float*>(a.v_ring) + dst;
    for (int d = threadIdx.x; d < a.D; d += blockDim.x) { kr[d] = kn[d]; vr[d] = vn[d]; }
  }
}

// ------------------------------------------------------------------ host side
size_t attn_workspace_bytes(int segments, int rows, int D) {
  const size_t slots = (size_t)segments + kMaxGridX;
  const size_t recs = slots * kMaxSlices * (size_t)rows;
  size_t bytes = 256;                                   // status word + padding
  bytes += (recs * sizeof(float2) + 255) / 256 * 256;   // (m, l)
  bytes += recs * (size_t)D * sizeof(float);            // unnormalised o
  return bytes;
}

void attn_workspace_carve(void* ws, int segments, int rows, int D, AttnParams* p) {
  const size_t slots = (size_t)segments + kMaxGridX;
  const size_t recs = slots * kMaxSlices * (size_t)rows;
  uint8_t* base = reinterpret_cast<uint8_t*>(ws);
  p->status = reinterpret_cast<uint32_t*>(base);
  p->part_ml = reinterpret_cast<float2*>(base + 256);
  p->part_o = reinterpret_cast<float*>(base + 256 + (recs * sizeof(float2) + 255) / 256 * 256);
  (void)D;
}

template <int D, int MASK, int NKS>
static cudaError_t launch_bf16(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV, dim3 grid,
                               cudaStream_t stream) {
  const size_t smem = 1024 + kStages * 2 * (size_t)(kKeyTile * D * 2) + (size_t)kConsumerWarps * 16 * D * 2;
  auto kern = attn_partial_bf16<D, MASK, NKS>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, (kConsumerWarps + 1) * 32, smem, stream>>>(*tmK, *tmV, p);
  return cudaGetLastError();
}

template <int D, int MASK>
static cudaError_t launch_bf16_nks(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV, dim3 grid,
                                   cudaStream_t stream) {
  switch (p.nks) {
    case kConsumerWarps / 4: return launch_bf16<D, MASK, kConsumerWarps / 4>(p, tmK, tmV, grid, stream);
    case kConsumerWarps / 2: return launch_bf16<D, MASK, kConsumerWarps / 2>(p, tmK, tmV, grid, stream);
    default: return launch_bf16<D, MASK, kConsumerWarps>(p, tmK, tmV, grid, stream);
  }
}

template <int D, int MASK>
static cudaError_t launch_f32(const AttnParams& p, dim3 grid, cudaStream_t stream) {
  attn_partial_f32<D, MASK><<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_partial(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV, int kv_bf16,
                                  dim3 grid, cudaStream_t stream) {
  if (kv_bf16) {
    switch (p.mask) {
      case kMaskNone: return launch_bf16_nks<D, kMaskNone>(p, tmK, tmV, grid, stream);
      case kMaskChain: return launch_bf16_nks<D, kMaskChain>(p, tmK, tmV, grid, stream);
      default: return launch_bf16_nks<D, kMaskTree>(p, tmK, tmV, grid, stream);
    }
  }
  switch (p.mask) {
    case kMaskNone: return launch_f32<D, kMaskNone>(p, grid, stream);
    case kMaskChain: return launch_f32<D, kMaskChain>(p, grid, stream);
    default: return launch_f32<D, kMaskTree>(p, grid, stream);
  }
}

cudaError_t launch_attention(const AttnParams& p_in, const CUtensorMap* tmK, const CUtensorMap* tmV, int kv_bf16,
                             cudaStream_t stream) {
  AttnParams p = p_in;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // bf16: one 288-thread CTA per SM (a 3-stage ring of 64 KB K+V stages); fp32: 2 per SM.
  const int per_sm = kv_bf16 ? 1 : 2;
  p.grid_x = sms * per_sm < kMaxGridX ? sms * per_sm : kMaxGridX;
  e = cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  dim3 mgrid(p.B * p.Hkv, (p.rows + 3) / 4);
  if (kv_bf16 && p.D == 128 && p.rows > 32) {
    // dense query blocks: tcgen05 tiles of 128 rows, one CTA per SM (range x row group)
    p.tc_groups = (p.rows + 127) / 128;
    p.rows_per_group = (p.rows + p.tc_groups - 1) / p.tc_groups;
    p.nks = 1;
    p.grid_x = sms / p.tc_groups > 0 ? sms / p.tc_groups : 1;
    if (p.grid_x > kMaxGridX) p.grid_x = kMaxGridX;
    e = launch_partial_tc(p, tmK, tmV, stream);
    if (e != cudaSuccess) return e;
    attn_merge<128><<<mgrid, 128, 0, stream>>>(p);
    return cudaGetLastError();
  }
  // row groups of equal size (a multiple of 16), so one key-slice count serves the launch
  const int row_groups = (p.rows + kRowsPerGroup - 1) / kRowsPerGroup;
  p.rows_per_group = ((p.rows + row_groups - 1) / row_groups + 15) / 16 * 16;
  p.nks = kv_bf16 ? slices_for_rows(p.rows_per_group) : 1;
  dim3 grid(p.grid_x, row_groups);
  e = (p.D == 64) ? launch_partial<64>(p, tmK, tmV, kv_bf16, grid, stream)
                  : launch_partial<128>(p, tmK, tmV, kv_bf16, grid, stream);
  if (e != cudaSuccess) return e;
  if (p.D == 64) attn_merge<64><<<mgrid, 128, 0, stream>>>(p);
  else attn_merge<128><<<mgrid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_window_append(const WindowAppend& a, cudaStream_t stream) {
  window_append_kernel<<<a.B * a.Hkv, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace specv
