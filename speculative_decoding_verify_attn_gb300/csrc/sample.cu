// The speculative-sampling step over the vocabulary, and greedy chain / tree selection.
//
// Large vocabularies (V > kSmallVocab):
//   K1 sample_stats     grid (chunks, rows, B): every target and draft row is split into
//                       vocabulary chunks; each CTA reads its chunk once with 128-bit loads and
//                       writes the chunk max M_c and S_c = sum exp(x - M_c) (fp32 exp2f of the
//                       scaled difference, compensated fp32 per thread, float-float across the
//                       warp, fp64 across warps) -- or, in greedy modes, the chunk argmax.  The last
//                       CTA of a sequence to finish (atomic ticket, no spinning) merges its rows'
//                       statistics (fp64) and takes every accept decision at once (one lane per
//                       draft, fp64 exponentials of the two selected logits); greedy modes finish
//                       there (argmax merge + chain or tree rule).
//   K2 sample_residual  grid (chunks, B), stochastic chain only: each CTA sums the residual
//                       max(P_{k+1} - Q_{k+1}, 0) (or P_{gamma+1}) over its chunk; the last CTA of
//                       the sequence finds the chunk where the cumulative residual passes u * R,
//                       re-scans that one chunk and writes the emitted tokens.
// Small vocabularies: one warp per sequence runs the whole step (the 16-token chi-square
// workload runs 10^6 sequences at once).
//
// Every sum that decides a token is reproducible: fixed element orders, compensated fp32 per
// thread (Kahan), float-float (Knuth's TwoSum) inside a warp, fp64 above that, no floating-point
// atomics.
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "sample_internal.h"

namespace specv {

struct Kahan {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float x) {
    const float y = __fsub_rn(x, c);
    const float t = __fadd_rn(s, y);
    c = __fsub_rn(__fsub_rn(t, s), y);
    s = t;
  }
  __device__ __forceinline__ double value() const { return (double)s - (double)c; }
};

// exp(x - M) in fp32 through exp2f (2 ulp); x - M <= 0 is formed first so that the dominant
// terms (x near M) carry only the rounding of the final product
__device__ __forceinline__ float exp_shift(float x, float M) {
  return exp2f(__fmul_rn(__fsub_rn(x, M), kLog2e));
}

// residual element: max(P(z) - Q(z), 0), or P(z) when there is no draft row
__device__ __forceinline__ float resid(float t, float d, float Mt, float iZt, float Md, float iZd, bool has_d) {
  const float pt = __fmul_rn(exp_shift(t, Mt), iZt);
  if (!has_d) return pt;
  const float qd = __fmul_rn(exp_shift(d, Md), iZd);
  return fmaxf(__fsub_rn(pt, qd), 0.f);
}

// ------------------------------------------------------------------ block helpers (256 threads)
__device__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < (int)(blockDim.x >> 5) ? red[lane] : neg_inf();
  return warp_max(v);
}
__device__ double block_sum_d(double v, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_d(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];  // fixed order
  return t;
}
__device__ int block_max_i(int v, int* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  int t = INT_MIN;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = max(t, red[w]);
  return t;
}
// (value, index) argmax combine: larger value wins, ties to the smaller index
__device__ __forceinline__ void argmax_combine(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) { v = v2; i = i2; }
}
__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
    argmax_combine(v, i, v2, i2);
  }
}
// Float-float (unevaluated sum hi + lo) addition: Knuth's TwoSum on the high parts, then the low
// parts folded in and renormalised.  About 44 significant bits with fp32 operations only, so warp
// reductions avoid the fp64 pipe.
struct FF {
  float hi, lo;
};
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float v = __fsub_rn(s, a.hi);
  const float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, v)), __fsub_rn(b.hi, v));
  const float t = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s, t);
  return FF{hi, __fsub_rn(t, __fsub_rn(hi, s))};
}
// Block sum of per-thread float-float values: warps reduce in float-float, then thread 0 adds the
// warp results in fp64 in warp order.  The result is valid in thread 0.
__device__ double block_sum_ff(FF v, FF* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF w;
    w.hi = __shfl_down_sync(0xffffffffu, v.hi, o);
    w.lo = __shfl_down_sync(0xffffffffu, v.lo, o);
    if (lane < o) v = ff_add(v, w);
  }
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double t = 0.0;
  if (threadIdx.x == 0)
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += (double)red[w].hi + (double)red[w].lo;
  return t;
}

// ------------------------------------------------------------------ shared decision logic
__device__ __forceinline__ const float* trow(const SampleParams& p, int b, int i) {
  return p.tl + (int64_t)b * p.tl_sb + (int64_t)i * p.V;
}
__device__ __forceinline__ const float* drow(const SampleParams& p, int b, int i) {
  return p.dl + (int64_t)b * p.dl_sb + (int64_t)i * p.V;
}

// k = number of leading drafts passing u_i * Q_i(x_i) < P_i(x_i), or -1 if a token id is invalid.
// sM / sZ hold the row max and normaliser: target row i at i, draft row i at rows_t + i.
// Whole warp: lane i takes draft i (gamma <= 32); the first failing lane is found with a ballot.
// P_i(x_i) and Q_i(x_i) use fp64 exponentials of the two selected logits.  Every lane returns k.
__device__ int chain_decide_warp(const SampleParams& p, int b, const float* sM, const double* sZ) {
  const int i = threadIdx.x & 31;
  bool bad = false, acc = true;
  if (i < p.gamma) {
    const int x = p.tok[(int64_t)b * p.tok_sb + i];
    bad = x < 0 || x >= p.V;
    if (!bad) {
      // u Q(x) < P(x)  <=>  u < P(x) / Q(x) = exp((t_x - M_t) - (d_x - M_d)) * Z_d / Z_t
      // (the differences are exact in fp64; one fp64 exponential per draft)
      const double dt = (double)trow(p, b, i)[x] - (double)sM[i];
      const double dd = (double)drow(p, b, i)[x] - (double)sM[p.rows_t + i];
      const double ratio = exp(dt - dd) * (sZ[p.rows_t + i] / sZ[i]);
      const double uu = (double)p.u[(int64_t)b * p.u_sb + i];
      acc = uu < ratio;
    }
  }
  if (__any_sync(0xffffffffu, bad)) return -1;
  const unsigned rej = __ballot_sync(0xffffffffu, i < p.gamma && !acc);
  return rej ? __ffs(rej) - 1 : p.gamma;
}

__device__ void write_chain_out(const SampleParams& p, int b, int k, int y) {
  int32_t* out = p.out_tok + (int64_t)b * p.out_cols;
  if (k < 0) {
    for (int c = 0; c < p.out_cols; ++c) out[c] = -1;
    p.out_nacc[b] = -1;
    atomicOr(p.status, (uint32_t)SPEC_STATUS_BAD_TOKEN);
    return;
  }
  for (int c = 0; c < p.out_cols; ++c) {
    int v = -1;
    if (c < k) v = p.tok[(int64_t)b * p.tok_sb + c];
    else if (c == k) v = y;
    out[c] = v;
  }
  p.out_nacc[b] = k;
}

// Greedy tree: a[] holds the argmax of every node's row.  Writes the outputs of sequence b.
__device__ void tree_select_write(const SampleParams& p, int b, const int* a) {
  const int32_t* tk = p.tok + (int64_t)b * p.tok_sb;
  int32_t* out = p.out_tok + (int64_t)b * p.out_cols;
  int32_t* nodes = p.out_nodes ? p.out_nodes + (int64_t)b * p.out_cols : nullptr;
  bool bad = false;
  for (int i = 1; i < p.N; ++i) bad |= (tk[i] < 0 || tk[i] >= p.V);
  for (int c = 0; c < p.out_cols; ++c) {
    out[c] = -1;
    if (nodes) nodes[c] = -1;
  }
  if (bad) {
    p.out_nacc[b] = -1;
    atomicOr(p.status, (uint32_t)SPEC_STATUS_BAD_TOKEN);
    return;
  }
  unsigned long long acc = 1ull;
  for (int i = 1; i < p.N; ++i) {
    const int par = p.parent[i];
    if (((acc >> par) & 1ull) && tk[i] == a[par]) acc |= (1ull << i);
  }
  int best = 0;
  for (int i = 1; i < p.N; ++i)
    if (((acc >> i) & 1ull) && p.depth[i] > p.depth[best]) best = i;
  const int d = p.depth[best];
  for (int j = best, lvl = d - 1; j > 0; j = p.parent[j], --lvl) {
    out[lvl] = tk[j];
    if (nodes) nodes[lvl] = j;
  }
  out[d] = a[best];
  p.out_nacc[b] = d;
}

// ------------------------------------------------------------------ large-V kernels
constexpr int kWarps = kSampleThreads / 32;

// Statistics kernel, warp-granular and persistent: global warp w takes the items w, w + W, ...
// (W warps in the grid), an item being kStatChunk = 1024 logits of one row, (b, row, item) in
// row-major order.  Lane l reads elements 4l..4l+3 of each 128-element slab (coalesced 512-byte
// warp loads).  Reductions are warp shuffles only -- no block barriers -- and the next item's
// loads are in flight while the current one is reduced.  Per item: the max and the compensated
// sum of exp(x - max) (float-float across lanes), or the argmax in greedy modes.
template <bool GREEDY>
__global__ void __launch_bounds__(kSampleThreads) sample_stats(const __grid_constant__ SampleParams p) {
  constexpr int PER = kStatChunk / 128;  // float4 loads per lane per item
  const int lane = threadIdx.x & 31;
  const int rows = p.rows_t + p.rows_d;
  const int per_seq = rows * p.schunks;
  const int items = p.B * per_seq;
  const int W = gridDim.x * kWarps;
  auto src_of = [&](int it, int& base) -> const float* {
    const int b = it / per_seq;
    const int rem = it - b * per_seq;
    const int r = rem / p.schunks;
    base = (rem - r * p.schunks) * kStatChunk;
    return (r < p.rows_t) ? trow(p, b, r) : drow(p, b, r - p.rows_t);
  };
  auto load = [&](int it, float4 (&v)[PER]) {
    int base;
    const float* row = src_of(it, base);
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      const int idx = base + i * 128 + lane * 4;
      v[i] = make_float4(neg_inf(), neg_inf(), neg_inf(), neg_inf());
      if (idx < p.V) v[i] = __ldcs(reinterpret_cast<const float4*>(row + idx));
    }
  };
  int it = blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (it >= items) return;
  float4 x[PER], xn[PER];
  load(it, x);
  for (; it < items; it += W) {
    if (it + W < items) load(it + W, xn);
    if (!GREEDY) {
      float m = neg_inf();
#pragma unroll
      for (int i = 0; i < PER; ++i) m = fmaxf(m, fmaxf(fmaxf(x[i].x, x[i].y), fmaxf(x[i].z, x[i].w)));
      m = warp_max(m);
      Kahan k;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        k.add(exp_shift(x[i].x, m)); k.add(exp_shift(x[i].y, m));
        k.add(exp_shift(x[i].z, m)); k.add(exp_shift(x[i].w, m));
      }
      FF v{k.s, -k.c};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        FF w;
        w.hi = __shfl_down_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_down_sync(0xffffffffu, v.lo, o);
        if (lane < o) v = ff_add(v, w);
      }
      if (lane == 0) {
        p.st_m[it] = m;
        p.st_s[it] = (double)v.hi + (double)v.lo;
      }
    } else {
      int base;
      src_of(it, base);
      float bv = neg_inf();
      int bi = INT_MAX;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int idx = base + i * 128 + lane * 4;
        const float e[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (idx + j < p.V && e[j] > bv) { bv = e[j]; bi = idx + j; }
      }
      warp_argmax(bv, bi);
      if (lane == 0) {
        p.st_m[it] = bv;
        p.st_arg[it] = bi;
      }
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) x[i] = xn[i];
  }
}

// One CTA per sequence: merges the chunk statistics of its rows and finishes the sequence --
// accept decisions and the residual row's statistics (stochastic chain), or the argmax merge and
// the greedy chain / tree rule.
template <bool GREEDY>
__global__ void __launch_bounds__(kSampleThreads) sample_finalize(const __grid_constant__ SampleParams p) {
  __shared__ float sM[2 * kMaxGamma + 1];
  __shared__ double sZ[2 * kMaxGamma + 1];
  __shared__ int sa[kMaxTreeNodes > kMaxGamma + 1 ? kMaxTreeNodes : kMaxGamma + 1];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = p.rows_t + p.rows_d;
  if (!GREEDY) {
    for (int rr = warp; rr < rows; rr += kWarps) {
      const int64_t oo = ((int64_t)b * rows + rr) * p.schunks;
      float m = neg_inf();
      for (int cc = lane; cc < p.schunks; cc += 32) m = fmaxf(m, p.st_m[oo + cc]);
      m = warp_max(m);
      // item weights exp(M_c - M) in fp32 (exp2f, 2 ulp; M_c - M is exact or far below 0 where
      // the weight is negligible), products and sums in fp64 in a fixed order
      double z = 0.0;
      for (int cc = lane; cc < p.schunks; cc += 32) z += p.st_s[oo + cc] * (double)exp_shift(p.st_m[oo + cc], m);
      z = warp_sum_d(z);
      if (lane == 0) { sM[rr] = m; sZ[rr] = z; }
    }
    __syncthreads();
    if (warp == 0) {
      const int k = chain_decide_warp(p, b, sM, sZ);
      if (lane == 0) {
        SeqInfo si;
        si.k = k;
        si.pad = 0;
        si.Mt = 0.f; si.Md = 0.f; si.Zt = 1.0; si.Zd = 1.0;
        if (k >= 0) { si.Mt = sM[k]; si.Zt = sZ[k]; }
        if (k >= 0 && k < p.gamma) { si.Md = sM[p.rows_t + k]; si.Zd = sZ[p.rows_t + k]; }
        p.seq[b] = si;
        if (k < 0) write_chain_out(p, b, -1, -1);
      }
    }
  } else {
    for (int rr = warp; rr < rows; rr += kWarps) {
      const int64_t oo = ((int64_t)b * rows + rr) * p.schunks;
      float v = neg_inf();
      int i = INT_MAX;
      for (int cc = lane; cc < p.schunks; cc += 32) argmax_combine(v, i, p.st_m[oo + cc], p.st_arg[oo + cc]);
      warp_argmax(v, i);
      if (lane == 0) sa[rr] = i;
    }
    __syncthreads();
    if (tid == 0) {
      if (p.mode == SPEC_SAMPLE_TREE_GREEDY) {
        tree_select_write(p, b, sa);
      } else {
        int k = p.gamma;
        for (int i = 0; i < p.gamma; ++i) {
          const int xi = p.tok[(int64_t)b * p.tok_sb + i];
          if (xi < 0 || xi >= p.V) { k = -1; break; }
        }
        if (k >= 0)
          for (int i = 0; i < p.gamma; ++i)
            if (p.tok[(int64_t)b * p.tok_sb + i] != sa[i]) { k = i; break; }
        write_chain_out(p, b, k, k >= 0 ? sa[k] : -1);
      }
    }
  }
}

// Residual of four consecutive elements starting at idx (idx < V, V % 4 == 0).
__device__ __forceinline__ float4 resid4(const float* tr, const float* dr, int idx, float Mt, float iZt, float Md,
                                         float iZd, bool has_d) {
  const float4 tv = __ldcs(reinterpret_cast<const float4*>(tr + idx));
  float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (has_d) dv = __ldcs(reinterpret_cast<const float4*>(dr + idx));
  return make_float4(resid(tv.x, dv.x, Mt, iZt, Md, iZd, has_d), resid(tv.y, dv.y, Mt, iZt, Md, iZd, has_d),
                     resid(tv.z, dv.z, Mt, iZt, Md, iZd, has_d), resid(tv.w, dv.w, Mt, iZt, Md, iZd, has_d));
}

// Residual mass of one warp slice of a chunk: warp w of the chunk covers 32 * EPT elements in
// slabs of 128 (lane l takes elements 4l..4l+3 of each slab).  Returns the warp's sum (valid in
// lane 0, float-float reduced) and the last index with positive residual (all lanes).
template <int EPT>
__device__ __forceinline__ double warp_slice_residual(const float* tr, const float* dr, int start, int V, float Mt,
                                                      float iZt, float Md, float iZd, bool has_d, int& last) {
  const int lane = threadIdx.x & 31;
  Kahan ks;
  last = -1;
#pragma unroll
  for (int i = 0; i < EPT / 4; ++i) {
    const int idx = start + i * 128 + lane * 4;
    if (idx < V) {
      const float4 r = resid4(tr, dr, idx, Mt, iZt, Md, iZd, has_d);
      ks.add(r.x); ks.add(r.y); ks.add(r.z); ks.add(r.w);
      last = r.w > 0.f ? idx + 3 : (r.z > 0.f ? idx + 2 : (r.y > 0.f ? idx + 1 : (r.x > 0.f ? idx : last)));
    }
  }
  FF v{ks.s, -ks.c};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF w;
    w.hi = __shfl_down_sync(0xffffffffu, v.hi, o);
    w.lo = __shfl_down_sync(0xffffffffu, v.lo, o);
    if (lane < o) v = ff_add(v, w);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
  return (double)v.hi + (double)v.lo;
}

// Residual pass (stochastic chain): grid (chunks, B).  Each warp sums its slice of the chunk; the
// last CTA of the sequence walks the slice sums in token order to the slice where the cumulative
// residual passes u * R and re-scans that slice (1024 elements for 8192-element chunks) with one
// warp, slab by slab, with an fp64 warp scan.
template <int EPT>
__global__ void __launch_bounds__(kSampleThreads, 4) sample_residual(const __grid_constant__ SampleParams p) {
  __shared__ int s_last;
  __shared__ int s_y;
  const int c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slice = 32 * EPT;                 // elements per warp slice
  const int nslices = p.nchunks * kWarps;
  double* wsum = p.res_sum + (int64_t)b * nslices;
  int32_t* wlast = p.res_last + (int64_t)b * nslices;

  const int k = __ldcg(&p.seq[b].k);
  if (k < 0) return;  // invalid token: the statistics pass already wrote the row
  bool has_d = k < p.gamma;
  const float* tr = trow(p, b, k);
  const float* dr = has_d ? drow(p, b, k) : tr;
  const float Mt = __ldcg(&p.seq[b].Mt);
  const float iZt = (float)(1.0 / __ldcg(&p.seq[b].Zt));
  const float Md = has_d ? __ldcg(&p.seq[b].Md) : 0.f;
  const float iZd = has_d ? (float)(1.0 / __ldcg(&p.seq[b].Zd)) : 0.f;

  {
    int last;
    const double ws = warp_slice_residual<EPT>(tr, dr, c * p.chunk + warp * slice, p.V, Mt, iZt, Md, iZd, has_d, last);
    if (lane == 0) {
      wsum[c * kWarps + warp] = ws;
      wlast[c * kWarps + warp] = last;
    }
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int t = atomicAdd(&p.ticket_b[b], 1);
      s_last = (t == p.nchunks - 1);
    }
    __syncthreads();
    if (!s_last) return;
  }
  __threadfence();
  if (warp != 0) return;

  // ---- last CTA, warp 0.  Lane l owns the consecutive slices [l * per, (l + 1) * per); an fp64
  // exclusive scan over the lanes' sums gives every slice's prefix in token order, and R.
  const int per = (nslices + 31) / 32;
  auto scan_slices = [&](double& pre, double& total) {
    double lsum = 0.0;
    for (int j = 0; j < per; ++j) {
      const int sl = lane * per + j;
      if (sl < nslices) lsum += __ldcg(wsum + sl);
    }
    double incl = lsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    pre = incl - lsum;
    total = __shfl_sync(0xffffffffu, incl, 31);
  };
  double pre, R;
  scan_slices(pre, R);
  if (R == 0.0) {
    // residual identically zero: draw from P_{k+1} itself (recompute every slice with P)
    has_d = false;
    for (int sl = 0; sl < nslices; ++sl) {
      int last;
      const double ws = warp_slice_residual<EPT>(tr, tr, (sl / kWarps) * p.chunk + (sl % kWarps) * slice, p.V, Mt,
                                                 iZt, 0.f, 0.f, false, last);
      if (lane == 0) { wsum[sl] = ws; wlast[sl] = last; }
    }
    __syncwarp();
    __threadfence_block();
    scan_slices(pre, R);
  }
  const double thr = (double)p.u[(int64_t)b * p.u_sb + p.gamma] * R;
  // the first slice whose cumulative sum passes thr: each lane checks its own slices
  int my_sl = -1;
  double my_acc = 0.0;
  {
    double run = pre;
    for (int j = 0; j < per; ++j) {
      const int sl = lane * per + j;
      if (sl >= nslices) break;
      const double ws = __ldcg(wsum + sl);
      if (run + ws > thr) { my_sl = sl; my_acc = run; break; }
      run += ws;
    }
  }
  const unsigned found = __ballot_sync(0xffffffffu, my_sl >= 0);
  int sstar = -1;
  double acc = 0.0;
  if (found) {
    const int src = __ffs(found) - 1;
    sstar = __shfl_sync(0xffffffffu, my_sl, src);
    acc = __shfl_sync(0xffffffffu, my_acc, src);
  }
  int y = -1;
  if (sstar >= 0) {
    const int start = (sstar / kWarps) * p.chunk + (sstar % kWarps) * slice;
    // the whole slice first (all loads in flight together), then the slab-by-slab scan
    float4 rs[EPT / 4];
#pragma unroll
    for (int i = 0; i < EPT / 4; ++i) {
      const int idx = start + i * 128 + lane * 4;
      rs[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (idx < p.V) rs[i] = resid4(tr, dr, idx, Mt, iZt, Md, iZd, has_d);
    }
    double base = acc;
#pragma unroll
    for (int i = 0; i < EPT / 4; ++i) {
      if (y >= 0) break;
      const int idx = start + i * 128 + lane * 4;
      const float4 r = rs[i];
      const double lsum = ((double)r.x + (double)r.y) + ((double)r.z + (double)r.w);
      double incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const unsigned hit = __ballot_sync(0xffffffffu, base + incl > thr);
      if (hit) {
        const int src = __ffs(hit) - 1;
        if (lane == src) {
          const double run0 = base + incl - lsum;
          const double run1 = run0 + (double)r.x, run2 = run1 + (double)r.y, run3 = run2 + (double)r.z;
          const double run4 = run3 + (double)r.w;
          int yy = run1 > thr ? idx : (run2 > thr ? idx + 1 : (run3 > thr ? idx + 2 : (run4 > thr ? idx + 3 : -1)));
          if (yy < 0) yy = r.w > 0.f ? idx + 3 : (r.z > 0.f ? idx + 2 : (r.y > 0.f ? idx + 1 : idx));
          s_y = yy;
        }
        __syncwarp();
        y = s_y;
      }
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (y < 0) y = __ldcg(wlast + sstar);  // rounding left the threshold at the slice end
  }
  if (y < 0) {
    // no slice passed the threshold through rounding: the largest index with positive mass
    int lst = -1;
    for (int i = lane; i < nslices; i += 32) lst = max(lst, __ldcg(wlast + i));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lst = max(lst, __shfl_xor_sync(0xffffffffu, lst, o));
    y = lst;
  }
  if (lane == 0) write_chain_out(p, b, k, y);
}

// ------------------------------------------------------------------ small-V kernel
// One warp per sequence.  Lane l owns the contiguous token range [l*per, (l+1)*per).
__global__ void __launch_bounds__(kSampleThreads) sample_small(const __grid_constant__ SampleParams p) {
  __shared__ float sM_all[kSampleThreads / 32][2 * kMaxGamma + 1];
  __shared__ double sZ_all[kSampleThreads / 32][2 * kMaxGamma + 1];
  __shared__ int a_all[kSampleThreads / 32][kMaxTreeNodes];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x * (kSampleThreads / 32) + warp;
  if (b >= p.B) return;
  float* sM = sM_all[warp];
  double* sZ = sZ_all[warp];
  int* a = a_all[warp];
  const int per = (p.V + 31) / 32;
  const int e0 = min(p.V, lane * per), e1 = min(p.V, e0 + per);
  const bool greedy = p.mode != SPEC_SAMPLE_CHAIN;
  const int rows = p.rows_t + p.rows_d;
  for (int r = 0; r < rows; ++r) {
    const float* row = (r < p.rows_t) ? trow(p, b, r) : drow(p, b, r - p.rows_t);
    if (greedy) {
      float v = neg_inf();
      int i = INT_MAX;
      for (int e = e0; e < e1; ++e)
        if (row[e] > v) { v = row[e]; i = e; }
      warp_argmax(v, i);
      if (lane == 0) a[r] = i;
    } else {
      float m = neg_inf();
      for (int e = e0; e < e1; ++e) m = fmaxf(m, row[e]);
      m = warp_max(m);
      Kahan ks;
      for (int e = e0; e < e1; ++e) ks.add(exp_shift(row[e], m));
      const double z = warp_sum_d(ks.value());
      if (lane == 0) { sM[r] = m; sZ[r] = z; }
    }
  }
  __syncwarp();
  if (greedy) {
    if (lane != 0) return;
    if (p.mode == SPEC_SAMPLE_TREE_GREEDY) {
      tree_select_write(p, b, a);
      return;
    }
    int k = p.gamma;
    for (int i = 0; i < p.gamma; ++i) {
      const int x = p.tok[(int64_t)b * p.tok_sb + i];
      if (x < 0 || x >= p.V) { k = -1; break; }
    }
    if (k >= 0)
      for (int i = 0; i < p.gamma; ++i)
        if (p.tok[(int64_t)b * p.tok_sb + i] != a[i]) { k = i; break; }
    write_chain_out(p, b, k, k >= 0 ? a[k] : -1);
    return;
  }
  const int k = chain_decide_warp(p, b, sM, sZ);
  if (k < 0) {
    if (lane == 0) write_chain_out(p, b, -1, -1);
    return;
  }
  bool has_d = k < p.gamma;
  const float* tr = trow(p, b, k);
  const float* dr = has_d ? drow(p, b, k) : tr;
  const float Mt = sM[k];
  const float iZt = (float)(1.0 / sZ[k]);
  const float Md = has_d ? sM[p.rows_t + k] : 0.f;
  const float iZd = has_d ? (float)(1.0 / sZ[p.rows_t + k]) : 0.f;
  for (int attempt = 0; attempt < 2; ++attempt) {
    Kahan ks;
    int last = -1;
    for (int e = e0; e < e1; ++e) {
      const float r = resid(tr[e], dr[e], Mt, iZt, Md, iZd, has_d);
      ks.add(r);
      if (r > 0.f) last = e;
    }
    const double tsum = ks.value();
    double x = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    const double R = __shfl_sync(0xffffffffu, x, 31);
    int lastall = last;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lastall = max(lastall, __shfl_xor_sync(0xffffffffu, lastall, o));
    if (R == 0.0 && attempt == 0) {
      has_d = false;  // residual identically zero: draw from P_{k+1}
      continue;
    }
    const double thr = (double)p.u[(int64_t)b * p.u_sb + p.gamma] * R;
    const double before = x - tsum;
    const unsigned hit = __ballot_sync(0xffffffffu, x > thr);
    int y = -1;
    if (hit) {
      const int src = __ffs(hit) - 1;
      if (lane == src) {
        Kahan run;
        int lastpos = -1;
        for (int e = e0; e < e1; ++e) {
          const float r = resid(tr[e], dr[e], Mt, iZt, Md, iZd, has_d);
          run.add(r);
          if (r > 0.f) lastpos = e;
          if (before + run.value() > thr) { y = e; break; }
        }
        if (y < 0) y = lastpos;
      }
      y = __shfl_sync(0xffffffffu, y, src);
    }
    if (y < 0) y = lastall;
    if (lane == 0) write_chain_out(p, b, k, y);
    return;
  }
}

// ------------------------------------------------------------------ host side
static int pick_chunk(int V, int rows_total, int B, int num_sms) {
  // the largest chunk that still gives every SM a few CTAs
  const int cands[3] = {8192, 4096, 2048};
  for (int i = 0; i < 3; ++i) {
    const long long ctas = (long long)rows_total * B * ((V + cands[i] - 1) / cands[i]);
    if (ctas >= 4LL * num_sms) return cands[i];
  }
  return 2048;
}

static size_t round256(size_t x) { return (x + 255) / 256 * 256; }

size_t sample_workspace_bytes(int mode, int B, int rows_t, int rows_d, int V) {
  (void)mode;
  const size_t nch = (size_t)(V + kMinChunk - 1) / kMinChunk;
  const size_t sch = (size_t)(V + kStatChunk - 1) / kStatChunk;
  const size_t rows = (size_t)rows_t + rows_d;
  size_t bytes = 256;                                        // status
  bytes += round256(2 * (size_t)B * sizeof(int32_t));        // tickets (zeroed per call)
  bytes += round256((size_t)B * sizeof(SeqInfo));            // accept decisions
  bytes += round256(B * rows * sch * sizeof(float));         // st_m
  bytes += round256(B * rows * sch * sizeof(double));        // st_s / st_arg
  bytes += round256(B * nch * 8 * sizeof(double));           // res_sum (per warp slice)
  bytes += round256(B * nch * 8 * sizeof(int32_t));          // res_last
  return bytes;
}

void sample_workspace_carve(void* ws, SampleParams* p) {
  const size_t nch = (size_t)(p->V + kMinChunk - 1) / kMinChunk;
  const size_t sch = (size_t)(p->V + kStatChunk - 1) / kStatChunk;
  const size_t rows = (size_t)p->rows_t + p->rows_d;
  const size_t B = (size_t)p->B;
  uint8_t* q = reinterpret_cast<uint8_t*>(ws);
  p->status = reinterpret_cast<uint32_t*>(q);
  q += 256;
  p->ticket_a = reinterpret_cast<int32_t*>(q);
  p->ticket_b = p->ticket_a + B;
  q += round256(2 * B * sizeof(int32_t));
  p->seq = reinterpret_cast<SeqInfo*>(q);
  q += round256(B * sizeof(SeqInfo));
  p->st_m = reinterpret_cast<float*>(q);
  q += round256(B * rows * sch * sizeof(float));
  p->st_s = reinterpret_cast<double*>(q);
  p->st_arg = reinterpret_cast<int32_t*>(q);
  q += round256(B * rows * sch * sizeof(double));
  p->res_sum = reinterpret_cast<double*>(q);
  q += round256(B * nch * 8 * sizeof(double));
  p->res_last = reinterpret_cast<int32_t*>(q);
}

template <int EPT>
static cudaError_t launch_large(const SampleParams& p, cudaStream_t stream) {
  const int rows = p.rows_t + p.rows_d;
  // status word and both ticket arrays start at zero for this call
  cudaError_t e = cudaMemsetAsync(p.status, 0, 256 + 2 * (size_t)p.B * sizeof(int32_t), stream);
  if (e != cudaSuccess) return e;
  const int items = p.schunks * rows * p.B;
  // persistent statistics grid: as many CTAs as fit on the GPU at once (warp-granular items)
  int per_sm = 1;
  if (p.mode == SPEC_SAMPLE_CHAIN)
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sample_stats<false>, kSampleThreads, 0);
  else
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sample_stats<true>, kSampleThreads, 0);
  if (per_sm < 1) per_sm = 1;
  const int need = (items + kWarps - 1) / kWarps;
  const int g1 = need < per_sm * p.num_sms ? need : per_sm * p.num_sms;
  if (p.mode == SPEC_SAMPLE_CHAIN) {
    sample_stats<false><<<g1, kSampleThreads, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    sample_finalize<false><<<p.B, kSampleThreads, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    dim3 g2(p.nchunks, p.B);
    sample_residual<EPT><<<g2, kSampleThreads, 0, stream>>>(p);
  } else {
    sample_stats<true><<<g1, kSampleThreads, 0, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    sample_finalize<true><<<p.B, kSampleThreads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_sample(SampleParams& p, int num_sms, cudaStream_t stream) {
  if (p.V <= kSmallVocab) {
    cudaError_t e = cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
    const int per_block = kSampleThreads / 32;
    sample_small<<<(p.B + per_block - 1) / per_block, kSampleThreads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  p.num_sms = num_sms;
  p.chunk = pick_chunk(p.V, p.rows_t + p.rows_d, p.B, num_sms);
  p.nchunks = (p.V + p.chunk - 1) / p.chunk;
  p.schunks = (p.V + kStatChunk - 1) / kStatChunk;
  switch (p.chunk) {
    case 8192: return launch_large<32>(p, stream);
    case 4096: return launch_large<16>(p, stream);
    default: return launch_large<8>(p, stream);
  }
}

}  // namespace specv
