// Segment bookkeeping shared by the attention kernels: the stream-K walk over the (sequence,
// kv head) key segments laid end to end in units of 128-key tiles, and the per-key visibility rule.
#pragma once

#include <stdint.h>

#include "attn_internal.h"
#include "common.cuh"

namespace specv {

// ------------------------------------------------------------------ segment bookkeeping
__device__ __forceinline__ int seg_len(const AttnParams& p, int b) {
  int L = __ldg(p.lens + b);
  if (p.is_window) return L >= 1 ? min(L, p.Lmax) : 0;
  return (L >= p.nq && L <= p.Lmax) ? L : 0;
}

// Ring slot of the window's token t: the first n_sinks tokens keep slots 0..n_sinks-1, later ones
// cycle through the other W - n_sinks slots.
__device__ __forceinline__ int window_slot(int t, int W, int n_sinks) {
  return t < n_sinks ? t : n_sinks + (t - n_sinks) % (W - n_sinks);
}

// 128-key tiles of a segment of `len` keys (the last one may be partial).
__device__ __forceinline__ int seg_tiles(int len) { return (len + kKeyTile - 1) / kKeyTile; }

// Whole-warp: total tiles over all segments, and the exclusive prefix (in tiles) of sequence
// `b_query` (pass -1 to skip).
__device__ __forceinline__ void warp_scan_tiles(const AttnParams& p, int b_query, int64_t& total, int64_t& cum_at) {
  const int lane = threadIdx.x & 31;
  int64_t run = 0;
  cum_at = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int64_t n = (b < p.B) ? (int64_t)seg_tiles(seg_len(p, b)) * p.Hkv : 0;
    int64_t x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const int64_t excl = run + x - n;
    if (b_query >= b0 && b_query < b0 + 32) cum_at = __shfl_sync(0xffffffffu, excl, b_query - b0);
    run += __shfl_sync(0xffffffffu, x, 31);
  }
  total = run;
}

__device__ __forceinline__ int64_t tiles_per_cta(const AttnParams& p, int64_t total) {
  int64_t per = (total + p.grid_x - 1) / p.grid_x;
  return per < kMinTilesPerCta ? (int64_t)kMinTilesPerCta : per;
}

// Walks the parts of a CTA's global tile range.  Every lane of a warp holds the same state.
struct Walker {
  int b, g, len, tile;
  int64_t gpos, gend;
};

// Whole-warp: position the walker at the start of CTA `cta`'s range.  Direct mode: CTA c owns
// the whole segments [c * spc, (c + 1) * spc), spc = p.segs_per_cta, empty ones included.
__device__ __forceinline__ void walker_init(const AttnParams& p, int cta, Walker& w) {
  w.b = 0; w.g = 0; w.len = 0; w.tile = 0;
  if (p.direct) {
    const int64_t S = (int64_t)p.B * p.Hkv;
    w.gpos = min(S, (int64_t)cta * p.segs_per_cta);
    w.gend = min(S, w.gpos + p.segs_per_cta);
    return;
  }
  int64_t total, dummy;
  warp_scan_tiles(p, -1, total, dummy);
  const int64_t per = tiles_per_cta(p, total);
  const int64_t begin = min(total, (int64_t)cta * per);
  w.gpos = begin;
  w.gend = min(total, begin + per);
  if (w.gpos >= w.gend) return;
  // find the sequence whose tile block contains `begin`
  const int lane = threadIdx.x & 31;
  int64_t run = 0;
  int found_b = -1;
  int64_t found_cum = 0;
  for (int b0 = 0; b0 < p.B && found_b < 0; b0 += 32) {
    const int b = b0 + lane;
    const int64_t n = (b < p.B) ? (int64_t)seg_tiles(seg_len(p, b)) * p.Hkv : 0;
    int64_t x = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const int64_t excl = run + x - n;
    const bool hit = n > 0 && begin >= excl && begin < excl + n;
    const unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m) {
      const int src = __ffs(m) - 1;
      found_b = b0 + src;
      found_cum = __shfl_sync(0xffffffffu, excl, src);
    }
    run += __shfl_sync(0xffffffffu, x, 31);
  }
  w.b = found_b;
  w.len = seg_len(p, found_b);
  const int ntiles = seg_tiles(w.len);
  const int64_t rel = begin - found_cum;
  w.g = (int)(rel / ntiles);
  w.tile = (int)(rel % ntiles);
}

// Next part: keys [kb, ke) of segment (b, g), kb a multiple of the tile size.  Direct mode: the
// next whole segment (kb = 0, ke = len, possibly 0).
__device__ __forceinline__ bool walker_next(const AttnParams& p, Walker& w, int& b, int& g, int& kb, int& ke,
                                            int& len) {
  if (w.gpos >= w.gend) return false;
  if (p.direct) {
    const int s = (int)w.gpos++;
    b = s / p.Hkv; g = s % p.Hkv;
    len = seg_len(p, b);
    kb = 0; ke = len;
    return true;
  }
  const int64_t avail = w.gend - w.gpos;
  const int ntiles = seg_tiles(w.len);
  const int take = (int)min((int64_t)(ntiles - w.tile), avail);
  b = w.b; g = w.g; len = w.len;
  kb = w.tile * kKeyTile;
  ke = min(w.len, (w.tile + take) * kKeyTile);
  w.gpos += take;
  w.tile += take;
  if (w.tile == ntiles) {
    w.tile = 0;
    if (++w.g == p.Hkv) {
      w.g = 0;
      do { ++w.b; } while (w.b < p.B && seg_len(p, w.b) == 0);
      w.len = (w.b < p.B) ? seg_len(p, w.b) : 0;
    }
  }
  return true;
}

// Branch-free visibility (bitwise logic only, safe to evaluate for every element of a tile).
template <int MASK>
__device__ __forceinline__ bool key_visible_nb(int kk, int ke, int tail_start, int j, unsigned long long anc) {
  const bool in = kk < ke;
  if (MASK == kMaskNone) return in;
  const int m = kk - tail_start;
  const bool ctx = m < 0;
  const bool tail_ok = (MASK == kMaskChain) ? (m <= j) : (((anc >> (m & 63)) & 1ull) != 0ull);
  return in & (ctx | tail_ok);
}

// Visibility of key index kk (absolute in the segment) for query position j.
template <int MASK>
__device__ __forceinline__ bool key_visible(int kk, int ke, int tail_start, int j, unsigned long long anc) {
  bool vis = kk < ke;
  if (MASK != kMaskNone && kk >= tail_start) {
    const int m = kk - tail_start;
    vis = vis && (MASK == kMaskChain ? (m <= j) : (((anc >> m) & 1ull) != 0ull));
  }
  return vis;
}

}  // namespace specv
