// Split-KV ("flash-decode") attention for speculative verify and for the draft ring window.
//
// Work decomposition (one launch, balanced over the whole batch): the 128-key tiles of all
// (sequence b, kv head g) segments are laid end to end, total = Hkv * sum_b ceil(len_b / 128)
// tiles, and CTA c takes the global tile range [c*T, (c+1)*T), T = max(ceil(total / grid_x),
// kMinTilesPerCta), so no tile is split between two CTAs.  A CTA
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
// Window with a new key: the ring slot of token pos - 1 is about to be overwritten, so the partial
// kernels treat it like a slot past the end, and the merge kernel adds the new key's score and
// value to the softmax and then stores the key into the slot (after every partial has read it).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_internal.h"
#include "common.cuh"
#include "launch_cache.h"

namespace specv {

// key slices per row tile for row groups of `rows_per_group` rows: kConsumerWarps / 16-row tiles
static inline int slices_for_rows(int rows_per_group) {
  return rows_per_group <= 16 ? kConsumerWarps : (rows_per_group <= 32 ? kConsumerWarps / 2 : kConsumerWarps / 4);
}

// ------------------------------------------------------------------ bf16 partial kernel

// Named barrier 1 over the consumer warps only (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}
// Same barrier, returning the OR of `pred` over every consumer thread, so that all consumer warps
// take the same decision.
__device__ __forceinline__ int consumers_sync_or(int pred) {
  int r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\tselp.b32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"(pred), "n"(kConsumerWarps * 32)
      : "memory");
  return r;
}

// Column swizzle of the fp32 combine buffers (rows of CW floats): 8-float groups XOR-ed by row, so
// the float2 fragment stores of 8 rows spread over the banks.
template <int CW>
__device__ __forceinline__ int combine_col(int row, int col) {
  return col ^ (((row & 7) << 3) & (CW - 8));
}

// Direct mode, end of a segment (the CTA owns all of it): the NKS warps of each 16-row tile hold
// flash partials (m, l, o) of disjoint key slices of the same rows.  They are combined through
// shared memory (each warp's Q staging region, free once the segment's tiles are consumed) in
// NPASS column passes: every warp stores its o columns, then warp ks combines rows ks, ks + NKS,
// ... of its tile in fixed slice order, adds the window's new key, normalises and writes the
// output row.  Returns nonzero if the CTA must stop (a wait timed out in any warp).
template <int D, int NKS, int NPASS>
__device__ __forceinline__ int combine_part(const AttnParams& p, float (&o)[D / 8][4], float m_lo, float m_hi,
                                            float l_lo, float l_hi, float* regions, float2* sML, int warp,
                                            int lane, int rt, int ks, int row0, int rows_here, int b, int g,
                                            int len, int bad, volatile int* s_abort) {
  constexpr int DT = D / 8, CW = D / NPASS, EPL = CW / 32, RPW = 16 / NKS;
  constexpr int REGION = 8 * D;  // floats in one warp's region (16 rows x D bf16)
  const int q = lane >> 2, t = lane & 3;
  const int rows_tile = min(16, rows_here - rt * 16);
  if (t == 0) {
    sML[warp * 16 + q] = make_float2(m_lo, l_lo);
    sML[warp * 16 + q + 8] = make_float2(m_hi, l_hi);
  }
  const bool add_new = p.has_new && len > 0;
  // direct mode: score of the new key for each row this warp combines
  float s_new[RPW];
#pragma unroll
  for (int i = 0; i < RPW; ++i) s_new[i] = neg_inf();
  if (add_new) {
    const __nv_bfloat16* kn = reinterpret_cast<const __nv_bfloat16*>(p.k_new) + b * p.new_sb + g * p.new_sh;
    const __nv_bfloat16* qb = reinterpret_cast<const __nv_bfloat16*>(p.q);
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int rr = ks + i * NKS;
      if (rr < rows_tile) {
        const int ro = row0 + rt * 16 + rr;
        const __nv_bfloat16* qr = qb + b * p.q_sb + (ro / p.G) * p.q_st + (g * p.G + ro % p.G) * p.q_sh;
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < D / 32; ++e)
          dot = fmaf(__bfloat162float(qr[lane + 32 * e]), __bfloat162float(kn[lane + 32 * e]), dot);
        s_new[i] = warp_sum(dot) * p.scale_log2;
      }
    }
  }
  float* mine = regions + warp * REGION;
  int stop = 0;
#pragma unroll
  for (int h = 0; h < NPASS; ++h) {
    // ---- this warp's o columns [h * CW, (h + 1) * CW) into its region
#pragma unroll
    for (int dt = h * (DT / NPASS); dt < (h + 1) * (DT / NPASS); ++dt) {
      const int col = dt * 8 + 2 * t - h * CW;
      if (q < rows_tile)
        *reinterpret_cast<float2*>(mine + q * CW + combine_col<CW>(q, col)) = make_float2(o[dt][0], o[dt][1]);
      if (NPASS == 2 && q + 8 < rows_tile)
        *reinterpret_cast<float2*>(mine + (q + 8) * CW + combine_col<CW>(q + 8, col)) =
            make_float2(o[dt][2], o[dt][3]);
    }
    consumers_sync();
    if (h == 0) {
      if (add_new && warp == 0) {
        // every warp is past this segment's tiles: store the new key into its ring slot
        const int slot = window_slot(__ldg(p.lens + b) - 1, p.Lmax, p.n_sinks);
        const int64_t src = (int64_t)b * p.new_sb + (int64_t)g * p.new_sh;
        const int64_t dst = (int64_t)b * p.kv_sb + (int64_t)g * p.kv_sh + (int64_t)slot * D;
        const __nv_bfloat16* kn = reinterpret_cast<const __nv_bfloat16*>(p.k_new) + src;
        const __nv_bfloat16* vn = reinterpret_cast<const __nv_bfloat16*>(p.v_new) + src;
        __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.k)) + dst;
        __nv_bfloat16* vr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.v)) + dst;
#pragma unroll
        for (int e = 0; e < D / 32; ++e) {
          kr[lane + 32 * e] = kn[lane + 32 * e];
          vr[lane + 32 * e] = vn[lane + 32 * e];
        }
      }
      if (len == 0 && warp == 0 && lane == 0) status_report(p.status, (uint32_t)SPEC_STATUS_BAD_POS);
    }
    // ---- combine the rows this warp owns (slice weights relative to the row maximum, the new
    // key included; recomputed per pass to keep registers free)
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int rr = ks + i * NKS;
      if (rr >= rows_tile) continue;
      float M = s_new[i];
#pragma unroll
      for (int k = 0; k < NKS; ++k) M = fmaxf(M, sML[(rt * NKS + k) * 16 + rr].x);
      const int c0 = lane * EPL;
      float acc[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
      float L = 0.f;
#pragma unroll
      for (int k = 0; k < NKS; ++k) {
        const float2 ml = sML[(rt * NKS + k) * 16 + rr];
        const float wk = ml.x == neg_inf() ? 0.f : exp2f(ml.x - M);
        L = fmaf(wk, ml.y, L);
        const float* src = regions + (rt * NKS + k) * REGION + rr * CW + combine_col<CW>(rr, c0);
        float v[EPL];
        if constexpr (EPL == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
        } else if constexpr (EPL == 2) {
          const float2 x = *reinterpret_cast<const float2*>(src);
          v[0] = x.x; v[1] = x.y;
        } else {
          v[0] = *src;
        }
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wk, v[e], acc[e]);
      }
      const int ro = row0 + rt * 16 + rr;
      const int col = h * CW + c0;
      {
        const int j = ro / p.G, head = g * p.G + ro % p.G;
        const int64_t off = (int64_t)b * p.o_sb + (int64_t)j * p.o_st + (int64_t)head * p.o_sh + col;
        if (add_new) {
          const float w_new = exp2f(s_new[i] - M);
          L += w_new;
          const __nv_bfloat16* vn = reinterpret_cast<const __nv_bfloat16*>(p.v_new) + b * p.new_sb + g * p.new_sh;
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(w_new, __bfloat162float(vn[col + e]), acc[e]);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        if (p.o_bf16) {
          __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.o) + off;
#pragma unroll
          for (int e = 0; e < EPL; ++e) ob[e] = __float2bfloat16_rn(acc[e] * inv);
        } else {
          float* of = reinterpret_cast<float*>(p.o) + off;
#pragma unroll
          for (int e = 0; e < EPL; ++e) of[e] = acc[e] * inv;
        }
      }
    }
    // regions are reused by the next pass or the next part's Q staging
    if (h + 1 < NPASS) consumers_sync();
    else stop = consumers_sync_or(bad | *s_abort);
  }
  return stop;
}

template <int D, int MASK, int NKS>
__device__ void consumer_loop(const AttnParams& p, uint8_t* stages, uint8_t* sQ, float2* sML, uint64_t* full,
                              uint64_t* empty, int warp, int lane, int row0, int rows_here, volatile int* s_abort) {
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
  uint8_t* sQw = sQ + warp * (16 * D * 2);
  // column passes of the slice combine: one when every row tile has at most 8 rows
  const int npass = (NKS == kConsumerWarps && min(16, rows_here) <= 8) ? 1 : 2;

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
    // window with a new key: the ring slot being replaced (verify masks have none)
    const int skip = (MASK == kMaskNone && p.has_new) ? window_slot(__ldg(p.lens + b) - 1, p.Lmax, p.n_sinks) : -1;

    int bad = 0;
    for (int key0 = kb; key0 < ke; key0 += KT) {
      if (!mbar_wait_bounded(&full[stage], phase, s_abort)) {
        *s_abort = 1;
        if (lane == 0) status_report(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
        bad = 1;
        break;
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
      const bool skip_tile = MASK == kMaskNone && (unsigned)(skip - key0) < (unsigned)KT;
      const bool tail_tile = key0 + KT > ke || skip_tile;
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
            if (!vis || (MASK == kMaskNone && kk == skip)) x = neg_inf();
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
            auto ok = [&](int k) { return k < ke && (MASK != kMaskNone || k != skip); };
            const uint32_t m0 = (ok(kf) ? 0x0000ffffu : 0u) | (ok(kf + 1) ? 0xffff0000u : 0u);
            const uint32_t m1 = (ok(kf + 8) ? 0x0000ffffu : 0u) | (ok(kf + 9) ? 0xffff0000u : 0u);
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
    if constexpr (MASK == kMaskNone) {
      if (p.direct) {
        float* regions = reinterpret_cast<float*>(sQ);
        int stop;
        if constexpr (NKS == kConsumerWarps) {
          stop = npass == 1 ? combine_part<D, NKS, 1>(p, o, m_lo, m_hi, l_lo, l_hi, regions, sML, warp, lane, rt, ks,
                                                      row0, rows_here, b, g, len, bad, s_abort)
                            : combine_part<D, NKS, 2>(p, o, m_lo, m_hi, l_lo, l_hi, regions, sML, warp, lane, rt, ks,
                                                      row0, rows_here, b, g, len, bad, s_abort);
        } else {
          stop = combine_part<D, NKS, 2>(p, o, m_lo, m_hi, l_lo, l_hi, regions, sML, warp, lane, rt, ks, row0,
                                         rows_here, b, g, len, bad, s_abort);
        }
        if (stop) return;
        continue;
      }
    }
    if (bad) return;
    // split mode: one (m, l, o) record per (part, key slice, row) for the merge kernel
    const int64_t slot = (int64_t)(b * p.Hkv + g) + blockIdx.x;
    const int64_t rec_base = (slot * NKS + ks) * p.rows + row0;
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
  pdl_launch_dependents();  // the merge may be scheduled as SMs free up
  // the call's status word is cleared here (no memset node before the call's first kernel)
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) status_clear_for_launch(p.status);
  constexpr int TILE = kKeyTile * D * 2;
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t bars[2 * kStages];
  __shared__ float2 sML[kConsumerWarps * 16];  // (m, l) of every consumer warp's 16 rows
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
      while (ok && !p.debug_no_loads && walker_next(p, w, b, g, kb, ke, len)) {
        for (int key0 = kb; key0 < ke; key0 += kKeyTile) {
          if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, &s_abort)) {
            s_abort = 1;
            status_report(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t* sK = stages + stage * 2 * TILE;
          uint8_t* sV = sK + TILE;
          mbar_arrive_expect_tx(&full[stage], 2u * TILE);
          tma_load_kv(sK, &tmK, &full[stage], key0, g, b);
          tma_load_kv(sV, &tmV, &full[stage], key0, g, b);
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
  consumer_loop<D, MASK, NKS>(p, stages, sQ, sML, full, empty, warp, lane, row0, rows_here, &s_abort);
}

// ------------------------------------------------------------------ draft window kernel
// The draft's single-query attention over its ring, for up to 16 query rows per kv head (the GQA
// group): one CTA per (sequence, kv head) segment, so every segment of the batch is resident at
// once (two CTAs per SM) and no segment waits for another's latency.  The ring streams through a
// 3-stage TMA ring of 64-key K and V tiles; the first tiles are issued by thread 0 right after the
// barriers are set up, before the segment's length is read (every tile lies inside the ring, so
// the copies are in bounds whatever the length; those past it are only waited for).  Two groups
// of four warps take alternate tiles, so two tiles are in compute at once; within a group each
// warp takes 16 keys of its tile (mma.sync m16n8k16, the group's rows padded to 16, Q.K^T as four
// independent accumulator chains) with an fp32 online softmax.  There is no producer warp (its
// registers would cost the second CTA per SM): the last of a group's four warps to finish a tile
// (a shared counter per stage) refills that stage with the tile three ahead.  A stage's tiles
// alternate between the groups, so each (group, stage) pair has its own full barrier: a group
// then waits on consecutive phases of it (on a shared barrier it would skip the other group's
// phases, and a parity wait could pass on an older phase).  The eight partial
// states are combined through shared memory (the stage buffers, once every copy has landed) with
// the new key (the current token, whose slot is masked in the ring), and the output and the ring
// slot are written.
// Launch: K and V of a tile come in one copy when the rings' heads are contiguous over the batch
// (a map over both rings), else one copy each.  The kernel is a programmatic dependent of the
// previous kernel of the stream: before the grid-dependency wait it only sends its first tiles to
// L2, and it clears the call's status word itself, so back-to-back draft calls have no memset node
// between them and each overlaps its launch with the previous call's tail.
constexpr int kWinKeys = 64;
constexpr int kWinStages = 3;
constexpr int kWinGroups = 2;
constexpr int kWinWarps = 4 * kWinGroups;
constexpr int kWinThreads = kWinWarps * 32;

size_t window_smem_bytes(int D) { return 1024 + (size_t)kWinStages * 2 * kWinKeys * D * 2 + 16 * (size_t)D * 2; }

template <int D>
__global__ void __launch_bounds__(kWinThreads, 2)
    attn_window_bf16(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const __grid_constant__ AttnParams p) {
  constexpr int KT = kWinKeys;
  constexpr int TILE = KT * D * 2;   // bytes of one K (or V) tile
  constexpr int KSTEPS = D / 16;
  constexpr int DT = D / 8;
  static_assert((size_t)kWinWarps * 16 * D * 4 <= (size_t)kWinStages * 2 * TILE, "combine scratch fits the stages");
  extern __shared__ uint8_t smem_raw[];
  __shared__ uint64_t full[kWinGroups][kWinStages];  // tile t lands on full[t % 2][t % 3], phase t / 6
  __shared__ int s_done[kWinStages];  // warp-tiles finished in the stage (four per tile, never reset)
  __shared__ int s_last[kWinStages];  // the last tile copied into the stage (-1: none)
  __shared__ float2 sML[kWinWarps][16];
  __shared__ float sNewK[D], sNewV[D], sNewS[16];  // the new key and value, its score per row
  __shared__ int s_abort;
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* stages = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* sQ = stages + kWinStages * 2 * TILE;  // 16 rows x D bf16, 128-byte swizzle
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seg = blockIdx.x, b = seg / p.Hkv, g = seg % p.Hkv;
  // programmatic dependent launch: the next kernel of the stream may be scheduled while this one
  // runs, and this one starts while its predecessor finishes, touching no memory before the wait
  pdl_launch_dependents();
  if (threadIdx.x == kWinThreads - 32 && !p.debug_no_loads) {
    // while the previous kernel of the stream finishes: the segment's first tiles into L2 (a
    // prefetch may see data the previous kernel is still writing; the copies after the wait
    // read L2, which then holds the written values)
    const int pre = min(kWinStages, (p.Lmax + KT - 1) / KT);
    const size_t off = ((size_t)b * p.kv_sb + (size_t)g * p.kv_sh) * 2;
    l2_prefetch_bulk(static_cast<const uint8_t*>(p.k) + off, (uint32_t)(pre * KT * D * 2));
    l2_prefetch_bulk(static_cast<const uint8_t*>(p.v) + off, (uint32_t)(pre * KT * D * 2));
  }
  pdl_wait();
  if (seg == 0 && threadIdx.x == 0) status_clear_for_launch(p.status);  // no memset before this launch
  auto issue = [&](int t) {  // one thread: tile t into stage t % kWinStages
    const int s = t % kWinStages;
    uint8_t* st = stages + s * 2 * TILE;
    uint64_t* bar = &full[t % kWinGroups][s];
    mbar_arrive_expect_tx(bar, 2u * TILE);
    if (p.kv_pair) {
      tma_load_kv_pair(st, &tmK, bar, t * KT, seg);
    } else {
      tma_load_kv(st, &tmK, bar, t * KT, g, b);
      tma_load_kv(st + TILE, &tmV, bar, t * KT, g, b);
    }
    s_last[s] = t;
  };
  // ---------------- every thread: the segment's length, the group's rows (padded to 16) and the
  // new key.  Every global load is issued before any of them is used, so the prologue costs one
  // round trip; the last warp's lane 0 sets up the ring meanwhile.
  constexpr int EPL = D / 32;
  constexpr int RPW = 16 / kWinWarps;
  const int grp = warp >> 2, wk = warp & 3;    // tile parity of this warp's group, key slice in the tile
  const int rows = p.rows;  // query rows of the segment (the GQA group)
  const __nv_bfloat16* qbase = reinterpret_cast<const __nv_bfloat16*>(p.q);
  const int lraw = __ldg(p.lens + b);
  static_assert(16 * (D / 8) <= kWinThreads, "one 16-byte chunk of Q per thread");
  const int qr = threadIdx.x / (D / 8), qc = threadIdx.x % (D / 8);
  uint4 qval = make_uint4(0u, 0u, 0u, 0u);
  if (threadIdx.x < 16 * (D / 8) && qr < rows)
    qval = *reinterpret_cast<const uint4*>(qbase + b * p.q_sb + (int64_t)(g * p.G + qr) * p.q_sh + qc * 8);
  // the new key (the current token), its value (warp 0 keeps both), and the rows this warp scores
  // against it (rows warp, warp + 8)
  __nv_bfloat16 kraw[EPL], vraw[EPL], qraw[RPW][EPL];
  if (p.has_new) {
    const __nv_bfloat16* kn = reinterpret_cast<const __nv_bfloat16*>(p.k_new) + b * p.new_sb + g * p.new_sh;
    const __nv_bfloat16* vn = reinterpret_cast<const __nv_bfloat16*>(p.v_new) + b * p.new_sb + g * p.new_sh;
#pragma unroll
    for (int e = 0; e < EPL; ++e) {
      kraw[e] = kn[lane * EPL + e];
      vraw[e] = warp == 0 ? vn[lane * EPL + e] : __float2bfloat16_rn(0.f);
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int rr = warp + i * kWinWarps;
#pragma unroll
      for (int e = 0; e < EPL; ++e)
        qraw[i][e] = rr < rows ? qbase[b * p.q_sb + (int64_t)(g * p.G + rr) * p.q_sh + lane * EPL + e]
                               : __float2bfloat16_rn(0.f);
    }
  }
  if (threadIdx.x == kWinThreads - 32) {
    for (int i = 0; i < kWinStages; ++i) {
      mbar_init(&full[0][i], 1);
      mbar_init(&full[1][i], 1);
      s_done[i] = 0;
      s_last[i] = -1;
    }
    s_abort = 0;
    fence_mbar_init();
    if (!p.debug_no_loads) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      // the first stages before the length is known: slots [0, W) are all inside the ring
      const int pre = min(kWinStages, (p.Lmax + KT - 1) / KT);
      for (int t = 0; t < pre; ++t) issue(t);
    }
  }
  const int len = lraw >= 1 ? min(lraw, p.Lmax) : 0;  // valid ring slots (0: bad pos)
  const int ntiles = (len + KT - 1) / KT;
  const int skip = (p.has_new && len > 0) ? window_slot(lraw - 1, p.Lmax, p.n_sinks) : -1;
  if (threadIdx.x < 16 * (D / 8)) *reinterpret_cast<uint4*>(sQ + qr * (D * 2) + ((qc ^ (qr & 7)) << 4)) = qval;
  const bool add_new = p.has_new && len > 0;
  if (p.has_new) {
    if (warp == 0) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        sNewK[lane * EPL + e] = __bfloat162float(kraw[e]);
        sNewV[lane * EPL + e] = __bfloat162float(vraw[e]);
      }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
      const int rr = warp + i * kWinWarps;
      if (rr < rows) {
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(__bfloat162float(qraw[i][e]), __bfloat162float(kraw[e]), dot);
        dot = warp_sum(dot);
        if (lane == 0) sNewS[rr] = dot * p.scale_log2;
      }
    }
  }
  __syncthreads();  // barriers initialised, Q and the new key in shared memory
  float o[DT][4];
#pragma unroll
  for (int dt = 0; dt < DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
  float m_lo = neg_inf(), m_hi = neg_inf(), l_lo = 0.f, l_hi = 0.f;
  bool bad = false;
  for (int t = grp; t < ntiles; t += kWinGroups) {
    const int s = t % kWinStages;
    if (!mbar_wait_bounded(&full[grp][s], (t / (kWinGroups * kWinStages)) & 1, &s_abort)) {
      s_abort = 1;
      if (lane == 0) status_report(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
      bad = true;
      break;
    }
    const uint8_t* sK = stages + s * 2 * TILE + (p.kv_swap ? TILE : 0);
    const uint8_t* sV = stages + s * 2 * TILE + (p.kv_swap ? 0 : TILE);
    const int key0 = t * KT;
    // S = Q.K^T for this warp's 16 keys: two 8-key halves x two K-dimension halves, four
    // independent accumulator chains
    float sc4[2][2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) sc4[nt][hh][0] = sc4[nt][hh][1] = sc4[nt][hh][2] = sc4[nt][hh][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; kk += 2) {
      const int hh = kk < KSTEPS / 2 ? 0 : 1;
      uint32_t qa[4], qb[4];
      {
        const int r = ((lane >> 3) & 1) * 8 + (lane & 7);
        const int c0 = kk * 2 + (lane >> 4);
        ldmatrix_x4(smem_u32(sQ + r * (D * 2) + ((c0 ^ (r & 7)) << 4)), qa[0], qa[1], qa[2], qa[3]);
        const int c1 = c0 + 2;
        ldmatrix_x4(smem_u32(sQ + r * (D * 2) + ((c1 ^ (r & 7)) << 4)), qb[0], qb[1], qb[2], qb[3]);
      }
      const int d0 = kk * 16 + (lane >> 3) * 8;
      const int c = (d0 & 63) >> 3;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const int r = wk * 16 + nt * 8 + (lane & 7);
        uint32_t b0, b1, b2, b3;
        ldmatrix_x4(smem_u32(sK + (d0 >> 6) * (KT * 128) + r * 128 + ((c ^ (r & 7)) << 4)), b0, b1, b2, b3);
        mma_bf16_16816(sc4[nt][hh], qa, b0, b1);
        mma_bf16_16816(sc4[nt][hh], qb, b2, b3);
      }
    }
    float sc[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = sc4[nt][0][e] + sc4[nt][1][e];
    // visible: slots below len, except the one the current token is about to take
    const bool edge = key0 + KT > len || (unsigned)(skip - key0) < (unsigned)KT;
    float mx_lo = neg_inf(), mx_hi = neg_inf();
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = sc[nt][e] * p.scale_log2;
        if (edge) {
          const int kk = key0 + wk * 16 + nt * 8 + 2 * (lane & 3) + (e & 1);
          if (kk >= len || kk == skip) x = neg_inf();
        }
        sc[nt][e] = x;
      }
      mx_lo = fmaxf(mx_lo, fmaxf(sc[nt][0], sc[nt][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(sc[nt][2], sc[nt][3]));
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float mu_lo = mn_lo == neg_inf() ? 0.f : mn_lo, mu_hi = mn_hi == neg_inf() ? 0.f : mn_hi;
    const float a_lo = exp2f(m_lo - mu_lo), a_hi = exp2f(m_hi - mu_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float sum_lo = 0.f, sum_hi = 0.f;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      sc[nt][0] = exp2f(sc[nt][0] - mu_lo);
      sc[nt][1] = exp2f(sc[nt][1] - mu_lo);
      sc[nt][2] = exp2f(sc[nt][2] - mu_hi);
      sc[nt][3] = exp2f(sc[nt][3] - mu_hi);
      sum_lo += sc[nt][0] + sc[nt][1];
      sum_hi += sc[nt][2] + sc[nt][3];
    }
    l_lo = l_lo * a_lo + sum_lo;
    l_hi = l_hi * a_hi + sum_hi;
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) {
      o[dt][0] *= a_lo; o[dt][1] *= a_lo;
      o[dt][2] *= a_hi; o[dt][3] *= a_hi;
    }
    uint32_t a[4];
    a[0] = pack_bf16(sc[0][0], sc[0][1]);
    a[1] = pack_bf16(sc[0][2], sc[0][3]);
    a[2] = pack_bf16(sc[1][0], sc[1][1]);
    a[3] = pack_bf16(sc[1][2], sc[1][3]);
    const int r = wk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
    const int kf = key0 + wk * 16 + 2 * (lane & 3);  // keys of this thread's B-fragment halves
#pragma unroll
    for (int dn = 0; dn < DT; dn += 2) {
      const int d0 = (dn + (lane >> 4)) * 8;
      const int c = (d0 & 63) >> 3;
      uint32_t v0, v1, v2, v3;
      ldmatrix_x4_trans(smem_u32(sV + (d0 >> 6) * (KT * 128) + r * 128 + ((c ^ (r & 7)) << 4)), v0, v1, v2, v3);
      if (edge) {  // V rows of hidden slots may hold anything (NaN): zeroed
        auto okk = [&](int k) { return k < len && k != skip; };
        const uint32_t m0 = (okk(kf) ? 0x0000ffffu : 0u) | (okk(kf + 1) ? 0xffff0000u : 0u);
        const uint32_t m1 = (okk(kf + 8) ? 0x0000ffffu : 0u) | (okk(kf + 9) ? 0xffff0000u : 0u);
        v0 &= m0; v1 &= m1; v2 &= m0; v3 &= m1;
      }
      mma_bf16_16816(o[dn], a, v0, v1);
      mma_bf16_16816(o[dn + 1], a, v2, v3);
    }
    // the last of the group's warps to finish the tile refills its stage (its reads of the stage
    // are done: every ldmatrix result was consumed by an MMA issued above)
    __syncwarp();
    if (lane == 0) {
      __threadfence_block();
      if ((atomicAdd(&s_done[s], 1) & 3) == 3) {
        __threadfence_block();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (t + kWinStages < ntiles && !s_abort && !p.debug_no_loads) issue(t + kWinStages);
      }
    }
  }
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  // ---------------- combine the eight warps' partial states (their o columns through the stage
  // buffers, once every warp is past its last tile and every copy issued has landed: tiles past
  // the length, or after an abort, were never waited for), add the new key, normalise, write
  const int q = lane >> 2, tq = lane & 3;
  if (tq == 0) {
    sML[warp][q] = make_float2(m_lo, l_lo);
    sML[warp][q + 8] = make_float2(m_hi, l_hi);
  }
  __syncthreads();  // no copy is issued after this
  if (threadIdx.x == 0) {
    for (int i = 0; i < kWinStages; ++i) {
      // the stage's last tile: the one before it in the stage had been consumed when it was issued
      const int tl = s_last[i];
      if (tl >= 0 && (tl >= ntiles || s_abort) && !mbar_wait_bounded(&full[tl % kWinGroups][i], (tl / (kWinGroups * kWinStages)) & 1, nullptr)) {
        s_abort = 1;
        status_report(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
      }
    }
  }
  const int stop = [&] {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, %2, p;\n\tselp.b32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((int)(bad || s_abort)), "n"(kWinThreads)
        : "memory");
    return r;
  }();
  if (stop) return;
  float* scratch = reinterpret_cast<float*>(stages);  // [warp][16 rows][D] fp32
  if (q < rows) {
#pragma unroll
    for (int dt = 0; dt < DT; ++dt)
      *reinterpret_cast<float2*>(scratch + (warp * 16 + q) * D + dt * 8 + 2 * tq) = make_float2(o[dt][0], o[dt][1]);
  }
  if (q + 8 < rows) {
#pragma unroll
    for (int dt = 0; dt < DT; ++dt)
      *reinterpret_cast<float2*>(scratch + (warp * 16 + q + 8) * D + dt * 8 + 2 * tq) = make_float2(o[dt][2], o[dt][3]);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kWinThreads) : "memory");
  // warp w finalises rows w, w + 8 of the group; lane l owns columns l * D/32 ..
#pragma unroll
  for (int i = 0; i < RPW; ++i) {
    const int rr = warp + i * kWinWarps;
    if (rr >= rows) break;
    const float s_new = add_new ? sNewS[rr] : neg_inf();
    float M = s_new;
#pragma unroll
    for (int w = 0; w < kWinWarps; ++w) M = fmaxf(M, sML[w][rr].x);
    float L = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    if (M != neg_inf()) {
#pragma unroll
      for (int w = 0; w < kWinWarps; ++w) {
        const float2 ml = sML[w][rr];
        const float wk2 = ml.x == neg_inf() ? 0.f : exp2f(ml.x - M);
        L = fmaf(wk2, ml.y, L);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wk2, scratch[(w * 16 + rr) * D + lane * EPL + e], acc[e]);
      }
      if (add_new) {
        const float wn = exp2f(s_new - M);
        L += wn;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(wn, sNewV[lane * EPL + e], acc[e]);
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const int64_t off = (int64_t)b * p.o_sb + (int64_t)(g * p.G + rr) * p.o_sh + lane * EPL;
    if (p.o_bf16) {
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.o) + off;
#pragma unroll
      for (int e = 0; e < EPL; ++e) ob[e] = __float2bfloat16_rn(acc[e] * inv);
    } else {
      float* of = reinterpret_cast<float*>(p.o) + off;
#pragma unroll
      for (int e = 0; e < EPL; ++e) of[e] = acc[e] * inv;
    }
    if (add_new && rr == 0) {
      // every read of the ring in this segment is done: the current token's K/V into its slot
      const int64_t dst = (int64_t)b * p.kv_sb + (int64_t)g * p.kv_sh + (int64_t)skip * D + lane * EPL;
      __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.k)) + dst;
      __nv_bfloat16* vr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.v)) + dst;
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        kr[e] = __float2bfloat16_rn(sNewK[lane * EPL + e]);  // exact: the values came from bf16
        vr[e] = __float2bfloat16_rn(sNewV[lane * EPL + e]);
      }
    }
  }
  if (len == 0 && warp == 0 && lane == 0) status_report(p.status, (uint32_t)SPEC_STATUS_BAD_POS);
}

// ------------------------------------------------------------------ fp32 partial kernel
template <int D, int MASK>
__global__ void __launch_bounds__(128) attn_partial_f32(const __grid_constant__ AttnParams p) {
  pdl_launch_dependents();
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
    const int skip = p.has_new ? window_slot(__ldg(p.lens + b) - 1, p.Lmax, p.n_sinks) : -1;
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
        if (!key_visible<MASK>(kk, ke, tail_start, j, anc) || kk == skip) continue;
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
      const int64_t rec = slot * p.rows + rr;
      if (lane == 0) p.part_ml[rec] = make_float2(m, l);
#pragma unroll
      for (int i = 0; i < PER; ++i) p.part_o[rec * D + lane + 32 * i] = acc[i];
    }
  }
}

// ------------------------------------------------------------------ merge kernel
// Element `i` of a row of q, k_new or v_new as fp32.
__device__ __forceinline__ float load_elem(const void* base, int64_t off, int bf16) {
  return bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[off])
              : reinterpret_cast<const float*>(base)[off];
}

// Vector of PER consecutive fp32 values (PER = 2 or 4), one 8- or 16-byte load.
template <int PER>
__device__ __forceinline__ void load_vec(const float* src, float (&v)[PER]) {
  if constexpr (PER == 4) {
    const float4 t = *reinterpret_cast<const float4*>(src);
    v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
  } else {
    const float2 t = *reinterpret_cast<const float2*>(src);
    v[0] = t.x; v[1] = t.y;
  }
}

// grid (segments, ceil(rows / 4)); one warp per query row of a segment, lane l owning head-dim
// elements [l * D/32, (l + 1) * D/32).  The records of a row (parts x key slices) are read
// lane-parallel: lane i fetches record i's (m, l), and the weighted sum of the o vectors issues
// its loads independently of one another, so the merge costs a few memory latencies, not one
// per record.
template <int D>
__global__ void __launch_bounds__(128) attn_merge(const __grid_constant__ AttnParams p) {
  constexpr int PER = D / 32;
  const int s = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.y * 4 + warp;
  if (r >= p.rows) return;
  const int b = s / p.Hkv, g = s % p.Hkv;
  // where the segment's records are depends on the lengths only (inputs, final before the partial
  // kernel started): worked out while the partial kernel still runs
  int64_t total, cum_b;
  warp_scan_tiles(p, b, total, cum_b);
  const int len = seg_len(p, b);
  const int j = r / p.G, h = g * p.G + r % p.G;
  const int e0 = lane * PER;
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  pdl_wait();  // the partial kernel's records
  if (len > 0) {
    const int ntiles = seg_tiles(len);
    const int64_t per = tiles_per_cta(p, total);
    const int64_t start = cum_b + (int64_t)g * ntiles;
    const int c0 = (int)(start / per), c1 = (int)((start + ntiles - 1) / per);
    const int nks = p.nks;
    const int nrec = (c1 - c0 + 1) * nks;  // per CTA that took part of the segment: one per key slice
    auto rec_of = [&](int i) -> int64_t { return ((int64_t)(s + c0 + i / nks) * nks + i % nks) * p.rows + r; };
    // (m, l) of records lane, lane + 32, ...; the o columns of the first eight records are
    // loaded in the same round trip (most rows have at most eight records)
    const float2 ml0 = lane < nrec ? p.part_ml[rec_of(lane)] : make_float2(neg_inf(), 0.f);
    float v0[8][PER];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      if (u < nrec) {
        load_vec<PER>(p.part_o + rec_of(u) * D + e0, v0[u]);
      } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) v0[u][i] = 0.f;
      }
    }
    float M = ml0.x;
    for (int i = lane + 32; i < nrec; i += 32) M = fmaxf(M, p.part_ml[rec_of(i)].x);
    M = warp_max(M);
    // the window's new key: score q . k_new (log2 units), weight 1 relative to itself
    float s_new = neg_inf(), kn[PER], vn[PER];
    if (p.has_new) {
      const int64_t qo = (int64_t)b * p.q_sb + (int64_t)j * p.q_st + (int64_t)h * p.q_sh + e0;
      const int64_t no = (int64_t)b * p.new_sb + (int64_t)g * p.new_sh + e0;
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        kn[i] = load_elem(p.k_new, no + i, p.kv_bf16);
        vn[i] = load_elem(p.v_new, no + i, p.kv_bf16);
        dot = fmaf(load_elem(p.q, qo + i, p.kv_bf16), kn[i], dot);
      }
      s_new = warp_sum(dot) * p.scale_log2;
      M = fmaxf(M, s_new);
    }
    float L = 0.f;
    if (M != neg_inf()) {
      for (int i0 = 0; i0 < nrec; i0 += 32) {
        float wgt = 0.f, lw = 0.f;
        if (i0 + lane < nrec) {
          const float2 ml = i0 == 0 ? ml0 : p.part_ml[rec_of(i0 + lane)];
          wgt = ml.x == neg_inf() ? 0.f : exp2f(ml.x - M);
          lw = wgt * ml.y;
        }
        L += warp_sum(lw);
        const int n = min(32, nrec - i0);
        // eight records' loads in flight at once, then their weighted sum in record order
        for (int t0 = 0; t0 < n; t0 += 8) {
          float v[8][PER];
          const bool first = i0 == 0 && t0 == 0;  // already in flight with the (m, l) loads
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (first) {
#pragma unroll
              for (int i = 0; i < PER; ++i) v[u][i] = v0[u][i];
            } else if (t0 + u < n) {
              load_vec<PER>(p.part_o + rec_of(i0 + t0 + u) * D + e0, v[u]);
            } else {
#pragma unroll
              for (int i = 0; i < PER; ++i) v[u][i] = 0.f;
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float wt = __shfl_sync(0xffffffffu, wgt, t0 + u);
            if (t0 + u < n) {
#pragma unroll
              for (int i = 0; i < PER; ++i) acc[i] = fmaf(wt, v[u][i], acc[i]);
            }
          }
        }
      }
      if (p.has_new) {
        const float wgt = exp2f(s_new - M);
        L += wgt;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] = fmaf(wgt, vn[i], acc[i]);
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] *= inv;
    if (p.has_new && r == 0) {
      // every partial kernel has finished reading the ring (stream order): store the new key
      const int slot = window_slot(__ldg(p.lens + b) - 1, p.Lmax, p.n_sinks);
      const int64_t dst = (int64_t)b * p.kv_sb + (int64_t)g * p.kv_sh + (int64_t)slot * D + e0;
      if (p.kv_bf16) {
        __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.k)) + dst;
        __nv_bfloat16* vr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.v)) + dst;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          kr[i] = __float2bfloat16_rn(kn[i]);  // exact: the value came from bf16
          vr[i] = __float2bfloat16_rn(vn[i]);
        }
      } else {
        float* kr = reinterpret_cast<float*>(const_cast<void*>(p.k)) + dst;
        float* vr = reinterpret_cast<float*>(const_cast<void*>(p.v)) + dst;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          kr[i] = kn[i];
          vr[i] = vn[i];
        }
      }
    }
  } else if (lane == 0 && g == 0 && r == 0) {
    atomicOr(p.status, p.is_window ? (uint32_t)SPEC_STATUS_BAD_POS : (uint32_t)SPEC_STATUS_BAD_KV_LEN);
  }
  const int64_t off = (int64_t)b * p.o_sb + (int64_t)j * p.o_st + (int64_t)h * p.o_sh + e0;
  if (p.o_bf16) {
    __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.o) + off;
#pragma unroll
    for (int i = 0; i < PER; ++i) ob[i] = __float2bfloat16_rn(acc[i]);
  } else {
    float* of = reinterpret_cast<float*>(p.o) + off;
#pragma unroll
    for (int i = 0; i < PER; ++i) of[i] = acc[i];
  }
}

// ------------------------------------------------------------------ verify append
// The fused append of spec_verify_attn: one warp per (sequence, new token, kv head) row, each lane
// moving one 16-byte chunk of the K row and of the V row into cache position kv_len - nq + j (no
// append for an out-of-range kv_len, which the attention kernels flag).  Every row's loads are
// independent, so the whole append costs about one memory latency.  Runs first in the call, so
// the attention kernels after it read the updated cache.
__global__ void __launch_bounds__(128) verify_append_kernel(const __grid_constant__ AttnParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + warp;  // (b, j, g), g fastest
  if (row >= (int64_t)p.B * p.nq * p.Hkv) return;
  const int g = (int)(row % p.Hkv);
  const int j = (int)((row / p.Hkv) % p.nq);
  const int b = (int)(row / ((int64_t)p.Hkv * p.nq));
  const int L = p.lens[b];
  if (L < p.nq || L > p.Lmax) return;
  const int elem = p.kv_bf16 ? 2 : 4;
  if (lane >= p.D * elem / 16) return;
  const int64_t src = ((int64_t)b * p.new_sb + (int64_t)j * p.new_st + (int64_t)g * p.new_sh) * elem + lane * 16;
  const int64_t dst =
      ((int64_t)b * p.kv_sb + (int64_t)g * p.kv_sh + (int64_t)(L - p.nq + j) * p.D) * elem + lane * 16;
  const uint4 kx = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.k_new) + src);
  const uint4 vx = *reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(p.v_new) + src);
  *reinterpret_cast<uint4*>(reinterpret_cast<char*>(const_cast<void*>(p.k)) + dst) = kx;
  *reinterpret_cast<uint4*>(reinterpret_cast<char*>(const_cast<void*>(p.v)) + dst) = vx;
}

// ------------------------------------------------------------------ ring append
// Separate append, used ahead of the tensor-core partial kernel (which has no replaced-slot mask):
// one CTA per (sequence, kv head) stores k_new / v_new into the ring slot of token pos - 1.
__global__ void window_append_kernel(const __grid_constant__ AttnParams p) {
  const int b = blockIdx.x / p.Hkv, g = blockIdx.x % p.Hkv;
  const int pos = p.lens[b];
  if (pos < 1) return;
  const int slot = window_slot(pos - 1, p.Lmax, p.n_sinks);
  const int64_t dst = (int64_t)b * p.kv_sb + (int64_t)g * p.kv_sh + (int64_t)slot * p.D;
  const int64_t src = (int64_t)b * p.new_sb + (int64_t)g * p.new_sh;
  if (p.kv_bf16) {
    const __nv_bfloat16* kn = reinterpret_cast<const __nv_bfloat16*>(p.k_new) + src;
    const __nv_bfloat16* vn = reinterpret_cast<const __nv_bfloat16*>(p.v_new) + src;
    __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.k)) + dst;
    __nv_bfloat16* vr = reinterpret_cast<__nv_bfloat16*>(const_cast<void*>(p.v)) + dst;
    for (int d = threadIdx.x; d < p.D; d += blockDim.x) { kr[d] = kn[d]; vr[d] = vn[d]; }
  } else {
    const float* kn = reinterpret_cast<const float*>(p.k_new) + src;
    const float* vn = reinterpret_cast<const float*>(p.v_new) + src;
    float* kr = reinterpret_cast<float*>(const_cast<void*>(p.k)) + dst;
    float* vr = reinterpret_cast<float*>(const_cast<void*>(p.v)) + dst;
    for (int d = threadIdx.x; d < p.D; d += blockDim.x) { kr[d] = kn[d]; vr[d] = vn[d]; }
  }
}

// ------------------------------------------------------------------ host side
size_t attn_workspace_bytes(int segments, int rows, int D) {
  const size_t slots = (size_t)segments + kMaxGridX;
  const size_t recs = slots * kConsumerWarps * (size_t)rows;  // up to kConsumerWarps key slices
  size_t bytes = 256;                                   // status word + padding
  bytes += (recs * sizeof(float2) + 255) / 256 * 256;   // (m, l)
  bytes += recs * (size_t)D * sizeof(float);            // unnormalised o
  return bytes;
}

void attn_workspace_carve(void* ws, int segments, int rows, int D, AttnParams* p) {
  const size_t slots = (size_t)segments + kMaxGridX;
  const size_t recs = slots * kConsumerWarps * (size_t)rows;
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
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, (kConsumerWarps + 1) * 32, smem, stream>>>(*tmK, *tmV, p);
  return cudaGetLastError();
}

template <int D, int MASK>
static cudaError_t launch_bf16_nks(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV, dim3 grid,
                                   cudaStream_t stream) {
  switch (p.nks) {
    case kConsumerWarps / 4:
      // D = 128 row groups above 32 rows take the tensor-core kernel
      if constexpr (D == 128) return cudaErrorInvalidValue;
      else return launch_bf16<D, MASK, kConsumerWarps / 4>(p, tmK, tmV, grid, stream);
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

int attn_tile_keys(int rows, int D) { return (D == 128 && rows > 128) ? kPairTileKeys : kKeyTile; }

bool window_uses_small_kernel(int rows, int D, int kv_bf16) { return kv_bf16 && rows <= 16 && (D == 64 || D == 128); }

int window_tile_keys(int rows, int D, int kv_bf16) {
  return window_uses_small_kernel(rows, D, kv_bf16) ? kWinKeys : attn_tile_keys(rows, D);
}

template <int D>
static cudaError_t launch_window_small(const AttnParams& p, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                       cudaStream_t stream) {
  const size_t smem = window_smem_bytes(D);
  auto kern = attn_window_bf16<D>;
  cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3(p.B * p.Hkv), dim3(kWinThreads), smem, stream, 0u, *tmK, *tmV, p);
}

bool q_tma_possible(int D, int G, int nq) {
  return D == 128 && G >= 1 && 128 % G == 0 && (nq * G) % 128 == 0 && nq * G > 128;
}

cudaError_t launch_attention(const AttnParams& p_in, const CUtensorMap* tmK, const CUtensorMap* tmV, int kv_bf16,
                             cudaStream_t stream, const CUtensorMap* tmQ) {
  AttnParams p = p_in;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // bf16: one 288-thread CTA per SM (a 3-stage ring of 64 KB K+V stages); fp32: 2 per SM.
  const int per_sm = kv_bf16 ? 1 : 2;
  p.grid_x = sms * per_sm < kMaxGridX ? sms * per_sm : kMaxGridX;
  // bf16 K/V: the call's first attention kernel clears the status word itself (a memset node
  // before a short call costs it several microseconds); fp32 K/V: a memset
  if (!kv_bf16) {
    e = cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
  }
  if (p.verify_append) {
    const int64_t rows = (int64_t)p.B * p.nq * p.Hkv;
    verify_append_kernel<<<(unsigned)((rows + 3) / 4), 128, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  dim3 mgrid(p.B * p.Hkv, (p.rows + 3) / 4);
  if (p.is_window && window_uses_small_kernel(p.rows, p.D, kv_bf16)) {
    // the draft window with up to 16 rows per kv head: one small CTA per segment
    return p.D == 64 ? launch_window_small<64>(p, tmK, tmV, stream) : launch_window_small<128>(p, tmK, tmV, stream);
  }
  if (kv_bf16 && p.D == 128 && p.rows > 32) {
    // dense query blocks: tcgen05 tiles of 128 rows, one CTA per SM (range x row group)
    if (p.has_new) {
      window_append_kernel<<<p.B * p.Hkv, 128, 0, stream>>>(p);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
      p.has_new = 0;
    }
    p.tc_groups = (p.rows + 127) / 128;
    p.rows_per_group = (p.rows + p.tc_groups - 1) / p.tc_groups;
    if (p.tc_groups >= 2) {
      // pairs of row blocks per CTA (each K/V tile serves up to 256 rows), one record per part
      const int pairs = (p.tc_groups + 1) / 2;
      p.nks = 1;
      p.grid_x = sms / pairs > 0 ? sms / pairs : 1;
      // a whole number of CTAs per segment when every segment gets one: with equal lengths no
      // CTA's range then spans two segments (a part change costs the CTA about five 64-key tiles:
      // its records, the next part's Q rows and the refill), at the price of idle SMs
      const int segs = p.B * p.Hkv;
      if (segs <= p.grid_x) p.grid_x = segs * (p.grid_x / segs);
      if (p.grid_x > kMaxGridX) p.grid_x = kMaxGridX;
      p.q_tma = (tmQ != nullptr && p.rows_per_group == 128 && q_tma_possible(p.D, p.G, p.nq)) ? 1 : 0;
      e = launch_partial_tc_pair(p, tmK, tmV, p.q_tma ? tmQ : tmK, stream);
      if (e != cudaSuccess) return e;
      return launch_merge_pair(p, stream);
    }
    p.nks = kTcSlices;
    p.grid_x = sms / p.tc_groups > 0 ? sms / p.tc_groups : 1;
    if (p.grid_x > kMaxGridX) p.grid_x = kMaxGridX;
    e = launch_partial_tc(p, tmK, tmV, stream);
    if (e != cudaSuccess) return e;
    return launch_dependent(attn_merge<128>, mgrid, dim3(128), 0, stream, 0u, p);
  }
  // row groups of equal size (a multiple of 16), so one key-slice count serves the launch
  const int row_groups = (p.rows + kRowsPerGroup - 1) / kRowsPerGroup;
  p.rows_per_group = ((p.rows + row_groups - 1) / row_groups + 15) / 16 * 16;
  p.nks = kv_bf16 ? slices_for_rows(p.rows_per_group) : 1;
  if (kv_bf16 && p.is_window && row_groups == 1) {
    // short segments (a ring of W keys): whole segments per CTA, no merge pass, as long as that
    // does not put many more tiles on a CTA than the even split would
    const int64_t S = (int64_t)p.B * p.Hkv;
    const int64_t spc = (S + sms - 1) / sms;
    const int64_t seg_tiles = (p.Lmax + kKeyTile - 1) / kKeyTile;
    const int64_t even = (S * seg_tiles + sms - 1) / sms;
    if (spc * seg_tiles <= (2 * even > 16 ? 2 * even : 16)) {
      p.direct = 1;
      p.segs_per_cta = (int)spc;
      p.grid_x = (int)((S + spc - 1) / spc);
    }
  }
  dim3 grid(p.grid_x, row_groups);
  e = (p.D == 64) ? launch_partial<64>(p, tmK, tmV, kv_bf16, grid, stream)
                  : launch_partial<128>(p, tmK, tmV, kv_bf16, grid, stream);
  if (e != cudaSuccess) return e;
  if (p.direct) return cudaSuccess;
  return p.D == 64 ? launch_dependent(attn_merge<64>, mgrid, dim3(128), 0, stream, 0u, p)
                   : launch_dependent(attn_merge<128>, mgrid, dim3(128), 0, stream, 0u, p);
}

}  // namespace specv
