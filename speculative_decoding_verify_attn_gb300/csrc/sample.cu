// The speculative-sampling step over the vocabulary, and greedy chain / tree selection.
//
// Large vocabularies (V > kSmallVocab):
//   sample_stats         persistent, warp-granular: every target and draft row is cut into items of
//                        1024 logits streamed through per-warp shared-memory rings by bulk copies;
//                        per item the max M_c and S_c = sum exp(x - M_c) (MUFU ex2 of the scaled
//                        difference, pairwise fp32 per lane, float-float across the warp) -- or, in
//                        greedy modes, the item argmax -- and the logits of the draft tokens.
//   sample_chain_finish  stochastic chain: one thread-block cluster per sequence.  Every CTA of the
//                        cluster merges the sequence's item statistics (float-float) and takes the
//                        accept decisions (one lane per draft); then CTA c computes the residual
//                        max(P_{k+1} - Q_{k+1}, 0) (or P_{gamma+1}) over its share of the vocabulary
//                        in 512-element slabs, the CTAs exchange their residual masses through
//                        distributed shared memory, and the CTA whose share holds u * R finds its
//                        slab and re-scans it for the emitted token.
//   sample_finalize      greedy modes: argmax merge and the chain or tree rule, one CTA per sequence.
// Small vocabularies: one warp per sequence runs the whole step (the 16-token chi-square
// workload runs 10^6 sequences at once).
//
// Every sum that decides a token is reproducible: fixed element orders, fp32 per lane (pairwise or
// compensated), float-float (Knuth's TwoSum) across lanes, warps, CTAs and the cluster (fp64 in the
// small-vocabulary kernel), no floating-point atomics.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "ff.cuh"
#include "sample_internal.h"
#include "launch_cache.h"

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

// residual element: max(P(z) - Q(z), 0), or P(z) when there is no draft row
__device__ __forceinline__ float resid(float t, float d, float Mt, float iZt, float Md, float iZd, bool has_d) {
  const float pt = __fmul_rn(exp_shift(t, Mt), iZt);
  if (!has_d) return pt;
  const float qd = __fmul_rn(exp_shift(d, Md), iZd);
  return fmaxf(__fsub_rn(pt, qd), 0.f);
}

// The same residual with one MUFU ex2 per exponential (flush-to-zero below 2^-126; relative error
// about 2^-22, inside the decision band), for the large-vocabulary pass.
__device__ __forceinline__ float resid_fast(float t, float d, float Mt, float iZt, float Md, float iZd, bool has_d) {
  const float pt = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(t, Mt), kLog2e)), iZt);
  if (!has_d) return pt;
  const float qd = __fmul_rn(ex2_approx(__fmul_rn(__fsub_rn(d, Md), kLog2e)), iZd);
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
__device__ int chain_decide_warp(const SampleParams& p, int b, const float* sM, const double* sZ,
                                 bool use_sel = false) {
  const int i = threadIdx.x & 31;
  bool bad = false, acc = true;
  if (i < p.gamma) {
    const int x = p.tok[(int64_t)b * p.tok_sb + i];
    // recorded logits are loaded alongside the token (their slots do not depend on it)
    const int rows = p.rows_t + p.rows_d;
    const float tsel = use_sel ? __ldcg(p.sel + (int64_t)b * rows + i) : 0.f;
    const float dsel = use_sel ? __ldcg(p.sel + (int64_t)b * rows + p.rows_t + i) : 0.f;
    bad = x < 0 || x >= p.V;
    if (!bad) {
      // u Q(x) < P(x)  <=>  u < P(x) / Q(x) = exp((t_x - M_t) - (d_x - M_d)) * Z_d / Z_t
      // (the differences are exact in fp64; one fp64 exponential per draft)
      const float tx = use_sel ? tsel : trow(p, b, i)[x];
      const float dx = use_sel ? dsel : drow(p, b, i)[x];
      const double dt = (double)tx - (double)sM[i];
      const double dd = (double)dx - (double)sM[p.rows_t + i];
      const double ratio = exp(dt - dd) * (sZ[p.rows_t + i] / sZ[i]);
      const double uu = (double)p.u[(int64_t)b * p.u_sb + i];
      acc = uu < ratio;
    }
  }
  if (__any_sync(0xffffffffu, bad)) return -1;
  const unsigned rej = __ballot_sync(0xffffffffu, i < p.gamma && !acc);
  return rej ? __ffs(rej) - 1 : p.gamma;
}

// The same decisions from float-float row normalisers and the logits the statistics pass
// recorded, in fp32 arithmetic only: the exponent (t_x - M_t) - (d_x - M_d) is formed exactly as a
// float-float, and the ratio exp(e) * Z_d / Z_t carries a relative error of a few 1e-7, far inside
// the 1e-6 band around each threshold.  u = 0 accepts (P(x) > 0 for every token).
// Lane i < gamma passes draft i's token x, the recorded target and draft logits of x (tx, dx) and
// its uniform uu, loaded by the caller ahead of the row statistics.
__device__ int chain_decide_warp_ff(const SampleParams& p, const float* sM, const FF* sZ, int x, float tx, float dx,
                                    float uu) {
  const int i = threadIdx.x & 31;
  bool bad = false, acc = true;
  if (i < p.gamma) {
    bad = x < 0 || x >= p.V;
    if (!bad) {
      const FF dt = ff_add(FF{tx, 0.f}, FF{-sM[i], 0.f});
      const FF dd = ff_add(FF{dx, 0.f}, FF{-sM[p.rows_t + i], 0.f});
      const FF e = ff_add(dt, ff_neg(dd));
      const FF zt = sZ[i], zd = sZ[p.rows_t + i];
      const float zr = __fdiv_rn(zd.hi, zt.hi) * (1.f + (__fdiv_rn(zd.lo, zd.hi) - __fdiv_rn(zt.lo, zt.hi)));
      const float ratio = expf(e.hi) * (1.f + e.lo) * zr;
      acc = uu == 0.f || uu < ratio;
    }
  }
  if (__any_sync(0xffffffffu, bad)) return -1;
  const unsigned rej = __ballot_sync(0xffffffffu, i < p.gamma && !acc);
  return rej ? __ffs(rej) - 1 : p.gamma;
}

// Outputs of sequence b; the accepted drafts are read from `tok` (its row of draft tokens).
__device__ void write_chain_out(const SampleParams& p, int b, int k, int y, const int32_t* tok) {
  int32_t* out = p.out_tok + (int64_t)b * p.out_cols;
  if (k < 0) {
    for (int c = 0; c < p.out_cols; ++c) out[c] = -1;
    p.out_nacc[b] = -1;
    atomicOr(p.status, (uint32_t)SPEC_STATUS_BAD_TOKEN);
    return;
  }
  for (int c = 0; c < p.out_cols; ++c) {
    int v = -1;
    if (c < k) v = tok[c];
    else if (c == k) v = y;
    out[c] = v;
  }
  p.out_nacc[b] = k;
}

__device__ void write_chain_out(const SampleParams& p, int b, int k, int y) {
  write_chain_out(p, b, k, y, p.tok + (int64_t)b * p.tok_sb);
}

// Greedy tree: a[] holds the argmax of every node's row, tk[] the node tokens of sequence b (in
// global or shared memory).  Writes the outputs of sequence b.
__device__ void tree_select_write(const SampleParams& p, int b, const int* a, const int32_t* tk) {
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
__device__ void tree_select_write(const SampleParams& p, int b, const int* a) {
  tree_select_write(p, b, a, p.tok + (int64_t)b * p.tok_sb);
}

// ------------------------------------------------------------------ large-V kernels
constexpr int kWarps = kSampleThreads / 32;

// Statistics kernel, warp-granular and persistent (one CTA of kStatWarps warps per SM): an item is
// kStatChunk = 1024 logits of one row, items numbered (b, row, c) in row-major order; CTA j takes
// the contiguous items [j * k, (j + 1) * k), k = ceil(items / CTAs), and its warp w the items
// j * k + w + i * kStatWarps, advancing (b, row, c) with carries.  Each warp streams its items through a private ring of kStatSlots
// shared-memory slots filled by bulk copies (lane 0 issues, an mbarrier per slot completes), so
// kStatSlots items per warp are in flight whatever the registers; the warp reads an item from shared memory
// (lane l takes elements 4l..4l+3 of each 128-element slab), refills the slot and reduces it with
// warp shuffles only.  Per item: the max and the sum of exp(x - max) (pairwise per lane,
// float-float across lanes), or the argmax in greedy modes.  In the stochastic chain the warp also records the
// logit of the row's draft token when it falls in the item.
template <bool GREEDY>
__global__ void __launch_bounds__(kStatWarps * 32, 1) sample_stats(const __grid_constant__ SampleParams p) {
  pdl_launch_dependents();  // the finishing kernel may be scheduled as SMs free up
  // the call's status word: cleared here, by CTA 0, unless the caller already cleared it (no memset
  // node before this launch); the finishing kernels report only after waiting for this grid
  if (!p.status_zeroed && blockIdx.x == 0 && threadIdx.x == 0) status_clear_for_launch(p.status);
  constexpr int PER = kStatChunk / 128;  // float4 per lane per item
  extern __shared__ float4 s_ring[];     // [kStatWarps][kStatSlots][kStatChunk / 4]
  __shared__ uint64_t s_bar[kStatWarps][kStatSlots];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = p.rows_t + p.rows_d;
  const long long items = (long long)p.B * rows * p.schunks;
  // the CTA's contiguous range of items; warp w takes items begin + w, begin + w + kStatWarps, ...
  // (one sequential stream of memory per SM)
  const long long per_c = (items + gridDim.x - 1) / gridDim.x;
  const long long c_begin = (long long)blockIdx.x * per_c;
  const long long c_end = min(items, c_begin + per_c);
  long long it = c_begin + warp;
  if (it >= c_end) return;
  const int n_items = (int)((c_end - it + kStatWarps - 1) / kStatWarps);
  float4* ring = s_ring + warp * kStatSlots * (kStatChunk / 4);
  uint64_t* bar = s_bar[warp];
  if (lane == 0) {
    for (int i = 0; i < kStatSlots; ++i) mbar_init(&bar[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  auto row_of = [&](int bb, int rr) -> const float* {
    return (rr < p.rows_t) ? trow(p, bb, rr) : drow(p, bb, rr - p.rows_t);
  };
  // issue side: coordinates of the next item to copy (lane 0 only)
  int ib = 0, ir = 0, ic = 0, issued = 0;
  {
    const long long rowid = it / p.schunks;
    ic = (int)(it % p.schunks);
    ir = (int)(rowid % rows);
    ib = (int)(rowid / rows);
  }
  int b = ib, r = ir, c = ic;  // processing side
  auto issue = [&]() {         // lane 0: copy the next item into its slot, advance
    const int slot = issued % kStatSlots;
    // the warp's reads of the slot (generic proxy) come before the copy's writes (async proxy)
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    const int base = ic * kStatChunk;
    const uint32_t bytes = (uint32_t)(min(kStatChunk, p.V - base) * 4);
    mbar_arrive_expect_tx(&bar[slot], bytes);
    bulk_load(ring + slot * (kStatChunk / 4), row_of(ib, ir) + base, bytes, &bar[slot]);
    ++issued;
    ic += kStatWarps;
    while (ic >= p.schunks) {
      ic -= p.schunks;
      if (++ir == rows) { ir = 0; ++ib; }
    }
  };
  if (lane == 0)
    for (int j = 0; j < kStatSlots && j < n_items; ++j) issue();
  // offset of the row's draft token from the row start (-1: none), refreshed when the row changes
  auto tok_of = [&](int bb, int rr) -> int {
    if (GREEDY || p.mode != SPEC_SAMPLE_CHAIN) return -1;
    const int ti = rr < p.rows_t ? rr : rr - p.rows_t;
    return ti < p.gamma ? __ldg(p.tok + (int64_t)bb * p.tok_sb + ti) : -1;
  };
  int xtok = tok_of(b, r);
  bool ok = true;
  for (int k = 0; k < n_items; ++k, it += kStatWarps) {
    const int slot = k % kStatSlots;
    if (!mbar_wait_bounded(&bar[slot], (uint32_t)((k / kStatSlots) & 1), nullptr)) { ok = false; break; }
    const int base = c * kStatChunk;
    float4 x[PER];
    if (base + kStatChunk <= p.V) {
#pragma unroll
      for (int i = 0; i < PER; ++i) x[i] = ring[slot * (kStatChunk / 4) + i * 32 + lane];
    } else {  // the row's ragged last item
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int idx = base + i * 128 + lane * 4;
        x[i] = idx < p.V ? ring[slot * (kStatChunk / 4) + i * 32 + lane]
                         : make_float4(neg_inf(), neg_inf(), neg_inf(), neg_inf());
      }
    }
    __syncwarp();
    if (lane == 0 && issued < n_items) issue();
    if (!GREEDY) {
      float m = neg_inf();
#pragma unroll
      for (int i = 0; i < PER; ++i) m = fmaxf(m, fmaxf(fmaxf(x[i].x, x[i].y), fmaxf(x[i].z, x[i].w)));
      m = warp_max(m);
      // exp(x - m) = 2^((x - m) log2 e): the difference first (exact for the dominant terms), then one
      // MUFU ex2 (flushing results below 2^-126 to zero, far below any term that counts).  The
      // lane's 32 terms are summed pairwise (relative error at most 5 * 2^-24), the lanes in
      // float-float.
      float e[4 * PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        e[4 * i + 0] = ex2_approx(__fmul_rn(__fsub_rn(x[i].x, m), kLog2e));
        e[4 * i + 1] = ex2_approx(__fmul_rn(__fsub_rn(x[i].y, m), kLog2e));
        e[4 * i + 2] = ex2_approx(__fmul_rn(__fsub_rn(x[i].z, m), kLog2e));
        e[4 * i + 3] = ex2_approx(__fmul_rn(__fsub_rn(x[i].w, m), kLog2e));
      }
#pragma unroll
      for (int w = 4 * PER / 2; w >= 1; w >>= 1)
#pragma unroll
        for (int j = 0; j < w; ++j) e[j] = __fadd_rn(e[j], e[j + w]);
      FF v{e[0], 0.f};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        FF w;
        w.hi = __shfl_down_sync(0xffffffffu, v.hi, o);
        w.lo = __shfl_down_sync(0xffffffffu, v.lo, o);
        if (lane < o) v = ff_add(v, w);
      }
      if (lane == 0) {
        p.st_m[it] = m;
        p.st_s[it] = make_float2(v.hi, v.lo);
      }
      // the row's draft token, if it falls in this item: its logit for the accept test
      const int off = xtok - base;
      if ((unsigned)off < (unsigned)kStatChunk && lane == ((off & 127) >> 2)) {
        const int q = off >> 7, j = off & 3;
        float val = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i)
          if (i == q) val = j == 0 ? x[i].x : (j == 1 ? x[i].y : (j == 2 ? x[i].z : x[i].w));
        p.sel[(int64_t)b * rows + r] = val;
      }
    } else {
      float bv = neg_inf();
      int bi = INT_MAX;
#pragma unroll
      for (int i = 0; i < PER; ++i) {
        const int idx = base + i * 128 + lane * 4;
        const float e[4] = {x[i].x, x[i].y, x[i].z, x[i].w};
#pragma unroll
        for (int j = 0; j < 4; ++j)  // the lane's first -inf seeds it, so an all -inf row gives id 0
          if (idx + j < p.V && (e[j] > bv || (bi == INT_MAX && e[j] == neg_inf()))) { bv = e[j]; bi = idx + j; }
      }
      warp_argmax(bv, bi);
      if (lane == 0) {
        p.st_m[it] = bv;
        p.st_arg[it] = bi;
      }
    }
    const int pb = b, pr = r;
    c += kStatWarps;
    while (c >= p.schunks) {
      c -= p.schunks;
      if (++r == rows) { r = 0; ++b; }
    }
    if (r != pr || b != pb) xtok = tok_of(b, r);
  }
  if (!ok) {
    // a copy never completed: flag it, and wait (bounded) for the copies still in flight into
    // this warp's slots before the CTA can leave
    if (lane == 0) {
      if (p.status_zeroed) atomicOr(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
      else status_report(p.status, (uint32_t)SPEC_STATUS_TIMEOUT);
    }
    const int done = (int)((it - (c_begin + warp)) / kStatWarps);
    for (int k = done; k < issued; ++k)
      mbar_wait_bounded(&bar[k % kStatSlots], (uint32_t)((k / kStatSlots) & 1), nullptr);
  }
}

// Greedy modes, one CTA per sequence: merges the item argmaxes of its rows and applies the greedy
// chain or tree rule.  A warp loads the item records of up to kFinRowBatch rows before it reduces
// any of them (one L2 round trip per 32 items of kFinRowBatch rows, not per row), and the
// sequence's tokens are staged in shared memory by all threads before thread 0 applies the rule.
// The argmax combination (larger value, ties to the smaller id) does not depend on the order in
// which records meet, so the result is that of any merge order.
constexpr int kFinRowBatch = 8;
__global__ void __launch_bounds__(kSampleThreads) sample_finalize(const __grid_constant__ SampleParams p) {
  __shared__ int sa[kMaxTreeNodes > kMaxGamma + 1 ? kMaxTreeNodes : kMaxGamma + 1];
  __shared__ int32_t s_tok[kMaxTreeNodes > kMaxGamma ? kMaxTreeNodes : kMaxGamma];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = p.rows_t + p.rows_d;
  const bool tree = p.mode == SPEC_SAMPLE_TREE_GREEDY;
  const int ntok = tree ? p.N : p.gamma;
  // the tokens are inputs of the call, not of the statistics kernel: loaded before the wait
  if (tid < ntok) s_tok[tid] = p.tok[(int64_t)b * p.tok_sb + tid];
  pdl_wait();  // the statistics kernel's per-item records
  for (int r0 = warp; r0 < rows; r0 += kWarps * kFinRowBatch) {
    float v[kFinRowBatch];
    int ix[kFinRowBatch];
#pragma unroll
    for (int u = 0; u < kFinRowBatch; ++u) {
      v[u] = neg_inf();
      ix[u] = INT_MAX;
    }
    for (int c0 = 0; c0 < p.schunks; c0 += 32) {
      const int cc = c0 + lane;
      float mv[kFinRowBatch];
      int ma[kFinRowBatch];
#pragma unroll
      for (int u = 0; u < kFinRowBatch; ++u) {
        const int rr = r0 + u * kWarps;
        const bool in = rr < rows && cc < p.schunks;
        const int64_t o = ((int64_t)b * rows + rr) * p.schunks + cc;
        mv[u] = in ? __ldcg(p.st_m + o) : neg_inf();
        ma[u] = in ? __ldcg(p.st_arg + o) : INT_MAX;
      }
#pragma unroll
      for (int u = 0; u < kFinRowBatch; ++u) argmax_combine(v[u], ix[u], mv[u], ma[u]);
    }
#pragma unroll
    for (int u = 0; u < kFinRowBatch; ++u) {
      warp_argmax(v[u], ix[u]);
      const int rr = r0 + u * kWarps;
      if (lane == 0 && rr < rows) sa[rr] = ix[u];
    }
  }
  __syncthreads();
  if (tid == 0) {
    if (tree) {
      tree_select_write(p, b, sa, s_tok);
    } else {
      int k = p.gamma;
      for (int i = 0; i < p.gamma; ++i) {
        const int xi = s_tok[i];
        if (xi < 0 || xi >= p.V) { k = -1; break; }
      }
      if (k >= 0)
        for (int i = 0; i < p.gamma; ++i)
          if (s_tok[i] != sa[i]) { k = i; break; }
      write_chain_out(p, b, k, k >= 0 ? sa[k] : -1, s_tok);
    }
  }
}

// ------------------------------------------------------------------ stochastic chain finish
constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kSlab = 512;  // residual slab: lane l takes elements 4l..4l+3 of each 128-element quarter
constexpr int kFinKeepMax = 160 * 1024;  // residual values a CTA keeps in shared memory for the draw

// Dynamic shared memory of the finish kernel for `per` slabs per CTA: the slab masses, then (when
// they fit) every residual value of the CTA's share, so the CTA that holds the threshold scans
// them without re-reading the rows.
__host__ __device__ constexpr bool fin_keeps_resid(int per) { return (size_t)per * kSlab * 4 <= (size_t)kFinKeepMax; }
__host__ __device__ constexpr size_t fin_smem_bytes(int per) {
  return ((size_t)per * sizeof(FF) + 15) / 16 * 16 + (fin_keeps_resid(per) ? (size_t)per * kSlab * 4 : 0);
}
// The largest of them (V <= 2^20: at most 2048 slabs per CTA, residual values kept up to 80): the
// kernel's shared-memory limit is set to this once, whatever the call, so concurrent calls with
// different vocabularies never race on it.
constexpr int kFinKeepSlabs = kFinKeepMax / (kSlab * 4);
constexpr size_t kFinSmemMax = fin_smem_bytes(kFinKeepSlabs) > 2048 * sizeof(FF) ? fin_smem_bytes(kFinKeepSlabs)
                                                                                 : 2048 * sizeof(FF);

// This lane's 16 logits of target and draft row in the slab starting at `base` (0 past V).
struct SlabData {
  float4 tv[4], dv[4];
};
__device__ __forceinline__ void slab_load(const float* tr, const float* dr, int base, int V, bool has_d, SlabData& D) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int idx = base + j * 128 + lane * 4;
    D.tv[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    D.dv[j] = D.tv[j];
    if (idx < V) {
      D.tv[j] = __ldcg(reinterpret_cast<const float4*>(tr + idx));
      if (has_d) D.dv[j] = __ldcg(reinterpret_cast<const float4*>(dr + idx));
    }
  }
}
// Residual of this lane's 16 elements of the slab starting at `base` (0 past V; V % 4 == 0).
__device__ __forceinline__ void slab_compute(const SlabData& D, int base, int V, float Mt, float iZt, float Md,
                                             float iZd, bool has_d, float (&r)[16]) {
  const int lane = threadIdx.x & 31;
  const float4* tv = D.tv;
  const float4* dv = D.dv;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int idx = base + j * 128 + lane * 4;
    const bool in = idx < V;
    r[4 * j + 0] = in ? resid_fast(tv[j].x, dv[j].x, Mt, iZt, Md, iZd, has_d) : 0.f;
    r[4 * j + 1] = in ? resid_fast(tv[j].y, dv[j].y, Mt, iZt, Md, iZd, has_d) : 0.f;
    r[4 * j + 2] = in ? resid_fast(tv[j].z, dv[j].z, Mt, iZt, Md, iZd, has_d) : 0.f;
    r[4 * j + 3] = in ? resid_fast(tv[j].w, dv[j].w, Mt, iZt, Md, iZd, has_d) : 0.f;
  }
}
// Keep this lane's 16 residual values of the CTA's local slab `sl` (4 float4, one per quarter).
__device__ __forceinline__ void keep_slab(float4* s_r, int sl, const float (&r)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 4; ++j) s_r[(sl * 4 + j) * 32 + lane] = make_float4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
}
// The residual values of the slab starting at `base` with lane l holding elements 16 l .. 16 l + 15
// (0 past V; V % 4 == 0).
__device__ __forceinline__ void slab_resid_lanes(const float* tr, const float* dr, int base, int V, float Mt,
                                                 float iZt, float Md, float iZd, bool has_d, float (&r)[16]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const int idx = base + lane * 16 + m * 4;
    float4 tv = make_float4(0.f, 0.f, 0.f, 0.f), dv = tv;
    if (idx < V) {
      tv = __ldcg(reinterpret_cast<const float4*>(tr + idx));
      if (has_d) dv = __ldcg(reinterpret_cast<const float4*>(dr + idx));
    }
    const bool in = idx < V;
    r[4 * m + 0] = in ? resid_fast(tv.x, dv.x, Mt, iZt, Md, iZd, has_d) : 0.f;
    r[4 * m + 1] = in ? resid_fast(tv.y, dv.y, Mt, iZt, Md, iZd, has_d) : 0.f;
    r[4 * m + 2] = in ? resid_fast(tv.z, dv.z, Mt, iZt, Md, iZd, has_d) : 0.f;
    r[4 * m + 3] = in ? resid_fast(tv.w, dv.w, Mt, iZt, Md, iZd, has_d) : 0.f;
  }
}
// One slab's residual mass (compensated fp32 per lane, float-float across the warp; lane 0).  It is
// positive exactly when the slab holds a positive residual.
__device__ __forceinline__ FF slab_mass(const float (&r)[16]) {
  const int lane = threadIdx.x & 31;
  Kahan ks;
#pragma unroll
  for (int e = 0; e < 16; ++e) ks.add(r[e]);
  FF v{ks.s, -ks.c};
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF w;
    w.hi = __shfl_down_sync(0xffffffffu, v.hi, o);
    w.lo = __shfl_down_sync(0xffffffffu, v.lo, o);
    if (lane < o) v = ff_add(v, w);
  }
  return v;
}
// Warp 0: slab masses of this CTA in token order, lane l owning slabs [l * pp, (l + 1) * pp):
// its sequential float-float sum and the inclusive scan over lanes (fixed order, so every call
// with the same masses returns the same values).
__device__ __forceinline__ void slab_scan(const FF* s_slab, int ns, FF& lsum, FF& incl) {
  const int lane = threadIdx.x & 31;
  const int pp = (ns + 31) / 32;
  lsum = FF{0.f, 0.f};
  for (int j = 0; j < pp; ++j) {
    const int sl = lane * pp + j;
    if (sl < ns) lsum = ff_add(lsum, s_slab[sl]);
  }
  incl = warp_scan_ff(lsum);
}

// Stochastic chain: grid B * CS CTAs in clusters of CS (one cluster per sequence).  Every CTA
// merges the item statistics of the sequence's rows and decides k (identical in every CTA: same
// inputs, same order); CTA `rank` then takes slabs [rank * per, (rank + 1) * per) of the residual
// row and records each slab's mass in shared memory (compensated fp32 per lane, float-float across
// the warp) and its own total, which it writes into every CTA of the cluster (distributed shared
// memory) before a cluster barrier; each thread then sums the CS totals in rank order, so every
// CTA agrees on R and on each CTA's prefix.  In the CTA whose [prefix, prefix + total) holds u * R,
// warp 0 finds the slab from the scan of its slab masses, then the element: lane l takes the
// slab's elements 16 l .. 16 l + 15 (kept in shared memory, else recomputed), one warp scan of
// the lanes' sums picks the lane, which searches its four groups of four.  All of it in
// float-float (no fp64).
// Every CTA takes the same cluster barriers (the decisions that steer them are identical across
// the cluster).
__global__ void __launch_bounds__(kFinThreads, 1) sample_chain_finish(const __grid_constant__ SampleParams p) {
  namespace cg = cooperative_groups;
  extern __shared__ __align__(16) uint8_t s_fin[];
  __shared__ float sM[2 * kMaxGamma + 1];
  __shared__ FF sZ[2 * kMaxGamma + 1];
  __shared__ int s_k;
  __shared__ int32_t s_x[kMaxGamma];  // the draft tokens (for the output row)
  __shared__ FF s_tot[8];             // the residual mass of every CTA of the cluster, by rank (each
                                      // CTA writes its own into all of them)
  cg::cluster_group cl = cg::this_cluster();
  const int CS = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int b = blockIdx.x / CS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = p.rows_t + p.rows_d;
  const int nslabs = (p.V + kSlab - 1) / kSlab;
  const int per = (nslabs + CS - 1) / CS;
  FF* s_slab = reinterpret_cast<FF*>(s_fin);   // residual mass of each of this CTA's slabs
  float4* s_r = reinterpret_cast<float4*>(s_fin + ((size_t)per * sizeof(FF) + 15) / 16 * 16);
  const bool keep = fin_keeps_resid(per);      // s_r[(slab * 4 + quarter) * 32 + lane]: a lane's 4 values
  // diagnostic word at byte 4 of the workspace: this launch's CTAs per sequence, and whether the
  // draw re-reads the residual row (bit 8) instead of scanning values kept in shared memory
  if (blockIdx.x == 0 && tid == 0) p.status[1] = (uint32_t)CS | (keep ? 0u : 0x100u);

  // the decision's inputs, loaded ahead of the row statistics so that their latency overlaps:
  // lane i < gamma of warp 0 takes draft i (token, uniform, then the two logits the statistics
  // kernel recorded), lane 0 the final draw's uniform
  int x_i = 0;
  float u_i = 0.f, tx_i = 0.f, dx_i = 0.f, u_draw = 0.f;
  if (warp == 0 && lane < p.gamma) {
    x_i = p.tok[(int64_t)b * p.tok_sb + lane];
    u_i = p.u[(int64_t)b * p.u_sb + lane];
  }
  if (warp == 0 && lane == 0) u_draw = p.u[(int64_t)b * p.u_sb + p.gamma];
  pdl_wait();  // the statistics kernel's per-item records
  if (warp == 0 && lane < p.gamma) {
    tx_i = __ldcg(p.sel + (int64_t)b * rows + lane);
    dx_i = __ldcg(p.sel + (int64_t)b * rows + p.rows_t + lane);
  }

  // ---- row statistics and accept decisions.  A warp merges a row's items 256 at a time, each
  // lane's (M_c, S_c) loaded together before any is used (one L2 round trip per 256 items).
  const float2* st_s = p.st_s;
  for (int rr = warp; rr < rows; rr += kFinWarps) {
    const int64_t oo = ((int64_t)b * rows + rr) * p.schunks;
    float m = neg_inf();
    FF z{0.f, 0.f};
    for (int c0 = 0; c0 < p.schunks; c0 += 256) {
      float mc[8];
      float2 sc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int cc = c0 + j * 32 + lane;
        mc[j] = cc < p.schunks ? __ldcg(p.st_m + oo + cc) : neg_inf();
        sc[j] = cc < p.schunks ? __ldcg(st_s + oo + cc) : make_float2(0.f, 0.f);
      }
      float mb = neg_inf();
#pragma unroll
      for (int j = 0; j < 8; ++j) mb = fmaxf(mb, mc[j]);
      mb = warp_max(mb);
      // item weights exp(M_c - M) in fp32 (exp2f, 2 ulp; M_c - M is exact or far below 0 where the
      // weight is negligible), products and sums in float-float in a fixed order
      const float mn = fmaxf(m, mb);
      FF zb{0.f, 0.f};
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (mc[j] != neg_inf()) zb = ff_add(zb, ff_mul_f(FF{sc[j].x, sc[j].y}, exp_shift(mc[j], mn)));
      zb = warp_sum_ff(zb);
      z = ff_add(m == neg_inf() ? FF{0.f, 0.f} : ff_mul_f(z, exp_shift(m, mn)), zb);
      m = mn;
    }
    if (lane == 0) { sM[rr] = m; sZ[rr] = z; }
  }
  if (warp == 0 && lane < p.gamma) s_x[lane] = x_i;
  __syncthreads();
  if (warp == 0) {
    const int kk = chain_decide_warp_ff(p, sM, sZ, x_i, tx_i, dx_i, u_i);
    if (lane == 0) s_k = kk;
  }
  __syncthreads();
  const int k = s_k;

  const int s0 = min(nslabs, rank * per), s1 = min(nslabs, s0 + per);
  bool has_d = k >= 0 && k < p.gamma;
  const float* tr = trow(p, b, k >= 0 ? k : 0);
  const float* dr = has_d ? drow(p, b, k) : tr;
  const float Mt = k >= 0 ? sM[k] : 0.f;
  const float iZt = k >= 0 ? __fdiv_rn(1.f, sZ[k].hi) : 0.f;
  float Md = has_d ? sM[p.rows_t + k] : 0.f;
  float iZd = has_d ? __fdiv_rn(1.f, sZ[p.rows_t + k].hi) : 0.f;

  FF R{0.f, 0.f}, cum{0.f, 0.f}, mine{0.f, 0.f};
  FF lsum{0.f, 0.f}, incl{0.f, 0.f};  // warp 0: lane-block sums and scan of the slab masses
  for (int attempt = 0; attempt < 2; ++attempt) {
    if (k >= 0) {
      // this warp's slabs s0 + warp + j * kFinWarps, two buffers in a pipeline: the next slab of a
      // buffer is loaded as soon as the buffer's slab has been reduced, while the other buffer's
      // slab is reduced
      SlabData D0, D1;
      const int sa0 = s0 + warp;
      if (sa0 < s1) slab_load(tr, dr, sa0 * kSlab, p.V, has_d, D0);
      if (sa0 + kFinWarps < s1) slab_load(tr, dr, (sa0 + kFinWarps) * kSlab, p.V, has_d, D1);
      for (int s = sa0; s < s1; s += 2 * kFinWarps) {
        const int s2 = s + kFinWarps;
        float r[16];
        slab_compute(D0, s * kSlab, p.V, Mt, iZt, Md, iZd, has_d, r);
        if (s + 2 * kFinWarps < s1) slab_load(tr, dr, (s + 2 * kFinWarps) * kSlab, p.V, has_d, D0);
        if (keep) keep_slab(s_r, s - s0, r);
        const FF m0 = slab_mass(r);
        if (lane == 0) s_slab[s - s0] = m0;
        if (s2 < s1) {
          slab_compute(D1, s2 * kSlab, p.V, Mt, iZt, Md, iZd, has_d, r);
          if (s2 + 2 * kFinWarps < s1) slab_load(tr, dr, (s2 + 2 * kFinWarps) * kSlab, p.V, has_d, D1);
          if (keep) keep_slab(s_r, s2 - s0, r);
          const FF m1 = slab_mass(r);
          if (lane == 0) s_slab[s2 - s0] = m1;
        }
      }
    }
    __syncthreads();
    if (warp == 0) {
      // the CTA's total (lane 31 of the scan), pushed into every CTA of the cluster at this rank
      lsum = FF{0.f, 0.f};
      incl = FF{0.f, 0.f};
      if (k >= 0) slab_scan(s_slab, s1 - s0, lsum, incl);
      const FF tot = shfl_ff(incl, 31);
      if (lane < CS) *cl.map_shared_rank(&s_tot[rank], lane) = tot;
    }
    cl.sync();
    // the cluster's totals in rank order, summed in a fixed order: the same R in every thread of
    // every CTA, and this CTA's prefix
    R = FF{0.f, 0.f};
    for (int c = 0; c < CS; ++c) {
      if (c == rank) cum = R;
      R = ff_add(R, s_tot[c]);
    }
    mine = s_tot[rank];
    if (k >= 0 && R.hi == 0.f && has_d) {
      // residual identically zero: draw from P_{k+1} itself
      has_d = false;
      dr = tr;
      Md = 0.f;
      iZd = 0.f;
      cl.sync();  // every CTA has read the totals before they are rewritten
      continue;
    }
    break;
  }

  if (k >= 0 && R.hi > 0.f && warp == 0) {
    const float uu = __shfl_sync(0xffffffffu, u_draw, 0);
    const FF thr = ff_mul_f(R, uu);
    const FF nxt = ff_add(cum, mine);
    if (!ff_gt(cum, thr) && ff_gt(nxt, thr)) {
      // this CTA holds the threshold: the scan of its slab masses (kept from the total) gives
      // every slab's prefix in token order
      const int ns = s1 - s0;
      const int pp = (ns + 31) / 32;
      int my_sl = -1;
      FF my_acc{0.f, 0.f};
      {
        FF run = ff_add(cum, ff_add(incl, ff_neg(lsum)));
        for (int j = 0; j < pp; ++j) {
          const int sl = lane * pp + j;
          if (sl >= ns) break;
          const FF nx = ff_add(run, s_slab[sl]);
          if (ff_gt(nx, thr)) { my_sl = sl; my_acc = run; break; }
          run = nx;
        }
      }
      unsigned found = __ballot_sync(0xffffffffu, my_sl >= 0);
      bool at_end = false;
      if (!found) {
        // rounding left the threshold past this CTA's last slab: its last slab with positive mass,
        // whose last positive element is then taken
        int lastpos = -1;
        for (int j = 0; j < pp; ++j) {
          const int sl = lane * pp + j;
          if (sl < ns && s_slab[sl].hi > 0.f) lastpos = sl;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
        my_sl = lane == 0 ? lastpos : -1;
        found = __ballot_sync(0xffffffffu, my_sl >= 0);
        at_end = true;
      }
      int y = -1;
      if (found) {
        const int src = __ffs(found) - 1;
        const int sl = __shfl_sync(0xffffffffu, my_sl, src);
        const FF base = shfl_ff(my_acc, src);
        // the slab's residual values in token order, lane l holding elements 16 l .. 16 l + 15
        // (kept from the mass pass, else recomputed from the rows)
        const int sbase = (s0 + sl) * kSlab;
        float r[16];
        if (keep) {
          // kept as quarters of 128: element 16 l + m sits in quarter l / 8 at position (l % 8) * 16 + m
#pragma unroll
          for (int m = 0; m < 4; ++m) {
            const float4 v = s_r[(sl * 4 + (lane >> 3)) * 32 + (lane & 7) * 4 + m];
            r[4 * m] = v.x;
            r[4 * m + 1] = v.y;
            r[4 * m + 2] = v.z;
            r[4 * m + 3] = v.w;
          }
        } else {
          slab_resid_lanes(tr, dr, sbase, p.V, Mt, iZt, Md, iZd, has_d, r);
        }
        int last = -1;  // this lane's last element with positive mass
#pragma unroll
        for (int e = 0; e < 16; ++e)
          if (r[e] > 0.f) last = sbase + lane * 16 + e;
        // the lane's 16 values summed exactly in pairs, then in float-float: groups of 4 kept for
        // the search inside the lane
        FF gsum[4];
#pragma unroll
        for (int q = 0; q < 4; ++q)
          gsum[q] = ff_add(two_sum(r[4 * q], r[4 * q + 1]), two_sum(r[4 * q + 2], r[4 * q + 3]));
        const FF lt = ff_add(ff_add(gsum[0], gsum[1]), ff_add(gsum[2], gsum[3]));
        const FF li = warp_scan_ff(lt);
        const unsigned hit = at_end ? 0u : __ballot_sync(0xffffffffu, ff_gt(ff_add(base, li), thr));
        if (hit) {
          const int hl = __ffs(hit) - 1;
          int yy = -1;
          if (lane == hl) {
            FF run = ff_add(base, ff_add(li, ff_neg(lt)));
            int q = 0;
            for (; q < 3; ++q) {
              const FF nx = ff_add(run, gsum[q]);
              if (ff_gt(nx, thr)) break;
              run = nx;
            }
            for (int e = 0; e < 4 && yy < 0; ++e) {
              run = ff_add(run, FF{r[4 * q + e], 0.f});
              if (ff_gt(run, thr)) yy = sbase + lane * 16 + 4 * q + e;
            }
            if (yy < 0) yy = last;  // rounding: the lane's last positive element
          }
          y = __shfl_sync(0xffffffffu, yy, hl);
        }
        if (y < 0) {  // rounding left the threshold at the slab end: its last positive element
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
          y = last;
        }
      }
      if (lane == 0) write_chain_out(p, b, k, y, s_x);
    }
  }
  if (k < 0 && rank == 0 && tid == 0) write_chain_out(p, b, -1, -1, s_x);
  cl.sync();  // no CTA leaves while the cluster may still read its shared memory
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
      for (int e = e0; e < e1; ++e)  // the lane's first -inf seeds it, so an all -inf row gives id 0
        if (row[e] > v || (i == INT_MAX && row[e] == neg_inf())) { v = row[e]; i = e; }
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
static size_t round256(size_t x) { return (x + 255) / 256 * 256; }

size_t sample_workspace_bytes(int mode, int B, int rows_t, int rows_d, int V) {
  if (mode == SPEC_SAMPLE_TREE) return 256;  // the status word: the tree walk keeps no statistics
  const size_t sch = (size_t)(V + kStatChunk - 1) / kStatChunk;
  const size_t rows = (size_t)rows_t + rows_d;
  size_t bytes = 256;                                        // status
  bytes += round256(B * rows * sch * sizeof(float));         // st_m
  bytes += round256(B * rows * sch * sizeof(float2));        // st_s / st_arg
  bytes += round256(B * rows * sizeof(float));               // sel
  return bytes;
}

void sample_workspace_carve(void* ws, SampleParams* p) {
  const size_t sch = (size_t)(p->V + kStatChunk - 1) / kStatChunk;
  const size_t rows = (size_t)p->rows_t + p->rows_d;
  const size_t B = (size_t)p->B;
  uint8_t* q = reinterpret_cast<uint8_t*>(ws);
  p->status = reinterpret_cast<uint32_t*>(q);
  if (p->mode == SPEC_SAMPLE_TREE) return;
  q += 256;
  p->st_m = reinterpret_cast<float*>(q);
  q += round256(B * rows * sch * sizeof(float));
  p->st_s = reinterpret_cast<float2*>(q);
  p->st_arg = reinterpret_cast<int32_t*>(q);
  q += round256(B * rows * sch * sizeof(float2));
  p->sel = reinterpret_cast<float*>(q);
}

static cudaError_t launch_large(const SampleParams& p, cudaStream_t stream) {
  const int rows = p.rows_t + p.rows_d;
  cudaError_t e = cudaSuccess;   // the statistics kernel clears the status word (no memset node)
  const long long items = (long long)p.schunks * rows * p.B;
  // persistent statistics grid: one CTA per SM (its shared-memory rings fill the SM)
  const long long need = (items + kStatWarps - 1) / kStatWarps;  // CTAs with at least a full set of items
  const int g1 = need < (long long)p.num_sms ? (int)(need > 0 ? need : 1) : p.num_sms;
  const size_t ring = (size_t)kStatWarps * kStatSlots * kStatChunk * sizeof(float);
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(p.mode == SPEC_SAMPLE_CHAIN ? sample_stats<false> : sample_stats<true>), (int)ring);
  if (e != cudaSuccess) return e;
  if (p.mode != SPEC_SAMPLE_CHAIN) {
    sample_stats<true><<<g1, kStatWarps * 32, ring, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return launch_dependent(sample_finalize, dim3(p.B), dim3(kSampleThreads), 0, stream, 0u, p);
  }
  sample_stats<false><<<g1, kStatWarps * 32, ring, stream>>>(p);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // clusters of CS CTAs per sequence: the largest CS for which every cluster of the batch can be
  // resident at once (one wave); CS = 1 when the batch alone fills the GPU
  const int nslabs = (p.V + kSlab - 1) / kSlab;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kFinThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = ensure_dynamic_smem(reinterpret_cast<const void*>(sample_chain_finish), (int)kFinSmemMax);
  if (e != cudaSuccess) return e;
  int cs = 8;
  for (; cs > 1; cs >>= 1) {
    if ((long long)p.B * cs > p.num_sms) continue;
    attr[0].val.clusterDim.x = (unsigned)cs;
    cfg.gridDim = dim3((unsigned)(p.B * cs), 1, 1);
    cfg.dynamicSmemBytes = fin_smem_bytes((nslabs + cs - 1) / cs);
    int active = 0;
    if (max_active_clusters(&active, reinterpret_cast<const void*>(sample_chain_finish), &cfg) == cudaSuccess && active >= p.B) break;
    (void)cudaGetLastError();
  }
  const size_t smem = fin_smem_bytes((nslabs + cs - 1) / cs);
  return launch_dependent(sample_chain_finish, dim3((unsigned)(p.B * cs)), dim3(kFinThreads), smem, stream,
                          (unsigned)cs, p);
}

cudaError_t launch_sample(SampleParams& p, int num_sms, cudaStream_t stream) {
  if (p.mode == SPEC_SAMPLE_TREE) return launch_sample_tree(p, stream);
  if (p.V <= kSmallVocab) {
    cudaError_t e = p.status_zeroed ? cudaSuccess : cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return e;
    const int per_block = kSampleThreads / 32;
    sample_small<<<(p.B + per_block - 1) / per_block, kSampleThreads, 0, stream>>>(p);
    return cudaGetLastError();
  }
  p.num_sms = num_sms;
  p.schunks = (p.V + kStatChunk - 1) / kStatChunk;
  return launch_large(p, stream);
}

}  // namespace specv
