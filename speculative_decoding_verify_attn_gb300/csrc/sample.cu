// The speculative-sampling step over the vocabulary, and greedy chain / tree selection.
//
// Large vocabularies (V > kSmallVocab), stochastic chain:
//   K1 sample_stats     grid (chunks, rows, B): every target and draft row is split into
//                       vocabulary chunks; each CTA reads its chunk once with 128-bit loads and
//                       writes the chunk max M_c and S_c = sum exp(x - M_c) (fp32 exp2f of the
//                       scaled difference, compensated fp32 per thread, fp64 across threads).
//   K2 sample_residual  grid (chunks, B): every CTA of a sequence merges the row statistics
//                       (Z = sum_c S_c exp(M_c - M), fp64), takes the accept decisions for all
//                       gamma drafts at once (one lane per draft, fp64 exponentials of the two
//                       selected logits), and sums the
//                       residual max(P_{k+1} - Q_{k+1}, 0) (or P_{gamma+1}) over its chunk.  The last
//                       CTA of the sequence to finish (atomic ticket, no spinning) finds the chunk
//                       where the cumulative residual passes u * R, re-scans that one chunk and
//                       writes the emitted tokens.
// Greedy modes: K1 computes chunk argmaxes (ties to the smallest id), K2 merges them per row and
// applies the chain or tree acceptance rule.
// Small vocabularies: one warp per sequence runs the whole step (the 16-token chi-square
// workload runs 10^6 sequences at once).
//
// Every sum that decides a token is reproducible: per-thread compensated fp32 sums in a fixed
// element order, fp64 above that, no floating-point atomics.
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "sample_internal.h"

namespace specv {

constexpr int kMaxChunks = 512;

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
// exclusive prefix (fp64) over the block's threads in thread order; also returns the total
__device__ double block_exclusive_scan_d(double v, double* red, double& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) red[warp] = x;
  __syncthreads();
  double before = 0.0, tot = 0.0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    if (w < warp) before += red[w];
    tot += red[w];
  }
  total = tot;
  return before + x - v;
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
      const double pt = exp((double)trow(p, b, i)[x] - (double)sM[i]) / sZ[i];
      const double qd = exp((double)drow(p, b, i)[x] - (double)sM[p.rows_t + i]) / sZ[p.rows_t + i];
      const double uu = (double)p.u[(int64_t)b * p.u_sb + i];
      acc = uu * qd < pt;
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
template <int EPT, bool GREEDY>
__global__ void __launch_bounds__(kSampleThreads) sample_stats(const __grid_constant__ SampleParams p) {
  __shared__ float redf[32];
  __shared__ double redd[32];
  __shared__ int redi[32];
  const int c = blockIdx.x, r = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int rows = p.rows_t + p.rows_d;
  const float* row = (r < p.rows_t) ? trow(p, b, r) : drow(p, b, r - p.rows_t);
  const int base = c * p.chunk;
  float x[EPT];
#pragma unroll
  for (int i = 0; i < EPT / 4; ++i) {
    const int idx = base + (i * kSampleThreads + tid) * 4;
    float4 v = make_float4(neg_inf(), neg_inf(), neg_inf(), neg_inf());
    if (idx < p.V) v = __ldcs(reinterpret_cast<const float4*>(row + idx));
    x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
  }
  const int64_t o = ((int64_t)b * rows + r) * p.nchunks + c;
  if (!GREEDY) {
    float m = neg_inf();
#pragma unroll
    for (int e = 0; e < EPT; ++e) m = fmaxf(m, x[e]);
    const float M = block_max(m, redf);
    Kahan k;
#pragma unroll
    for (int e = 0; e < EPT; ++e) k.add(exp_shift(x[e], M));
    const double S = block_sum_d(k.value(), redd);
    if (tid == 0) {
      p.st_m[o] = M;
      p.st_s[o] = S;
    }
  } else {
    float bv = neg_inf();
    int bi = INT_MAX;
#pragma unroll
    for (int i = 0; i < EPT / 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int idx = base + (i * kSampleThreads + tid) * 4 + j;
        if (idx < p.V && x[4 * i + j] > bv) { bv = x[4 * i + j]; bi = idx; }
      }
    warp_argmax(bv, bi);
    const int lane = tid & 31, warp = tid >> 5;
    __syncthreads();
    if (lane == 0) { redf[warp] = bv; redi[warp] = bi; }
    __syncthreads();
    if (tid == 0) {
      float v = redf[0];
      int i0 = redi[0];
      for (int w = 1; w < kSampleThreads / 32; ++w) argmax_combine(v, i0, redf[w], redi[w]);
      p.st_m[o] = v;
      p.st_arg[o] = i0;
    }
  }
  if (c == 0 && r == 0 && tid == 0) {
    p.ticket[b] = 0;
    if (b == 0) *p.status = 0u;
  }
}

// Residual values of this thread's EPT contiguous elements of chunk `c`, and their compensated
// sum / last positive index.  Called identically by the chunk pass and by the final re-scan.
template <int EPT>
__device__ __forceinline__ void chunk_thread_residual(const float* tr, const float* dr, int start, int V, float Mt,
                                                      float iZt, float Md, float iZd, bool has_d, float (&r)[EPT]) {
#pragma unroll
  for (int i = 0; i < EPT / 4; ++i) {
    const int idx = start + 4 * i;
    if (idx < V) {
      const float4 tv = *reinterpret_cast<const float4*>(tr + idx);
      float4 dv = make_float4(0.f, 0.f, 0.f, 0.f);
      if (has_d) dv = *reinterpret_cast<const float4*>(dr + idx);
      r[4 * i] = resid(tv.x, dv.x, Mt, iZt, Md, iZd, has_d);
      r[4 * i + 1] = resid(tv.y, dv.y, Mt, iZt, Md, iZd, has_d);
      r[4 * i + 2] = resid(tv.z, dv.z, Mt, iZt, Md, iZd, has_d);
      r[4 * i + 3] = resid(tv.w, dv.w, Mt, iZt, Md, iZd, has_d);
    } else {
      r[4 * i] = r[4 * i + 1] = r[4 * i + 2] = r[4 * i + 3] = 0.f;
    }
  }
}

template <int EPT>
__global__ void __launch_bounds__(kSampleThreads) sample_residual(const __grid_constant__ SampleParams p) {
  __shared__ float sM[2 * kMaxGamma + 1];
  __shared__ double sZ[2 * kMaxGamma + 1];
  __shared__ double redd[32];
  __shared__ int redi[32];
  __shared__ double s_tot[kMaxChunks];
  __shared__ int s_k, s_last, s_cstar, s_thread, s_y;
  __shared__ double s_acc, s_R;
  const int c = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int rows = p.rows_t + p.rows_d;

  // 1. row statistics (max, normaliser) of every target and draft row of this sequence
  for (int r = warp; r < rows; r += kSampleThreads / 32) {
    const int64_t o = ((int64_t)b * rows + r) * p.nchunks;
    float m = neg_inf();
    for (int cc = lane; cc < p.nchunks; cc += 32) m = fmaxf(m, p.st_m[o + cc]);
    m = warp_max(m);
    double z = 0.0;
    for (int cc = lane; cc < p.nchunks; cc += 32) z += p.st_s[o + cc] * exp((double)p.st_m[o + cc] - (double)m);
    z = warp_sum_d(z);
    if (lane == 0) { sM[r] = m; sZ[r] = z; }
  }
  __syncthreads();
  // 2. accept decisions (one warp, one lane per draft)
  if (warp == 0) {
    const int kk = chain_decide_warp(p, b, sM, sZ);
    if (lane == 0) s_k = kk;
  }
  __syncthreads();
  const int k = s_k;
  if (k < 0) {
    if (c == 0 && tid == 0) write_chain_out(p, b, -1, -1);
    return;
  }
  bool has_d = k < p.gamma;
  const float* tr = trow(p, b, k);
  const float* dr = has_d ? drow(p, b, k) : tr;
  const float Mt = sM[k];
  const float iZt = (float)(1.0 / sZ[k]);
  const float Md = has_d ? sM[p.rows_t + k] : 0.f;
  const float iZd = has_d ? (float)(1.0 / sZ[p.rows_t + k]) : 0.f;

  // 3. residual mass of this chunk
  {
    float r[EPT];
    const int start = c * p.chunk + tid * EPT;
    chunk_thread_residual<EPT>(tr, dr, start, p.V, Mt, iZt, Md, iZd, has_d, r);
    Kahan ks;
    int last = -1;
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
      ks.add(r[e]);
      if (r[e] > 0.f) last = start + e;
    }
    const double tot = block_sum_d(ks.value(), redd);
    const int lst = block_max_i(last, redi);
    if (tid == 0) {
      p.res_sum[(int64_t)b * p.nchunks + c] = tot;
      p.res_last[(int64_t)b * p.nchunks + c] = lst;
      __threadfence();
      const int t = atomicAdd(&p.ticket[b], 1);
      s_last = (t == p.nchunks - 1);
    }
    __syncthreads();
    if (!s_last) return;
  }
  __threadfence();

  // 4. last CTA of the sequence: locate u * R in the cumulative residual and emit
  for (int cc = tid; cc < p.nchunks; cc += kSampleThreads)
    s_tot[cc] = __ldcg(p.res_sum + (int64_t)b * p.nchunks + cc);
  __syncthreads();
  if (tid == 0) {
    double R = 0.0;
    for (int cc = 0; cc < p.nchunks; ++cc) R += s_tot[cc];
    s_R = R;
  }
  __syncthreads();
  int fallback_last = -1;
  if (s_R == 0.0) {
    // residual identically zero: draw from P_{k+1} itself
    has_d = false;
    for (int cc = 0; cc < p.nchunks; ++cc) {
      float r[EPT];
      const int start = cc * p.chunk + tid * EPT;
      chunk_thread_residual<EPT>(tr, tr, start, p.V, Mt, iZt, 0.f, 0.f, false, r);
      Kahan ks;
      int last = -1;
#pragma unroll
      for (int e = 0; e < EPT; ++e) {
        ks.add(r[e]);
        if (r[e] > 0.f) last = start + e;
      }
      const double tot = block_sum_d(ks.value(), redd);
      const int lst = block_max_i(last, redi);
      if (tid == 0) s_tot[cc] = tot;
      fallback_last = max(fallback_last, lst);
    }
    __syncthreads();
    if (tid == 0) {
      double R = 0.0;
      for (int cc = 0; cc < p.nchunks; ++cc) R += s_tot[cc];
      s_R = R;
    }
    __syncthreads();
  }
  const double thr = (double)p.u[(int64_t)b * p.u_sb + p.gamma] * s_R;
  if (tid == 0) {
    double acc = 0.0;
    int cs = -1;
    for (int cc = 0; cc < p.nchunks; ++cc) {
      if (acc + s_tot[cc] > thr) { cs = cc; break; }
      acc += s_tot[cc];
    }
    s_cstar = cs;
    s_acc = acc;
    s_thread = INT_MAX;
    s_y = -1;
  }
  __syncthreads();
  const int cs = s_cstar;
  if (cs >= 0) {
    float r[EPT];
    const int start = cs * p.chunk + tid * EPT;
    chunk_thread_residual<EPT>(tr, dr, start, p.V, Mt, iZt, Md, iZd, has_d, r);
    Kahan ks;
#pragma unroll
    for (int e = 0; e < EPT; ++e) ks.add(r[e]);
    double total;
    const double excl = block_exclusive_scan_d(ks.value(), redd, total);
    const double before = s_acc + excl;
    if (before + ks.value() > thr) atomicMin(&s_thread, tid);
    __syncthreads();
    if (tid == s_thread) {
      Kahan run;
      int y = -1, lastpos = -1;
      for (int e = 0; e < EPT; ++e) {
        run.add(r[e]);
        if (r[e] > 0.f) lastpos = start + e;
        if (before + run.value() > thr) { y = start + e; break; }
      }
      s_y = (y >= 0) ? y : lastpos;
    }
    __syncthreads();
  }
  if (tid == 0) {
    int y = s_y;
    if (y < 0) {
      // no index passed the threshold through rounding: the largest index with positive mass
      int lst = -1;
      if (s_R != 0.0 && fallback_last < 0)
        for (int cc = 0; cc < p.nchunks; ++cc) lst = max(lst, __ldcg(p.res_last + (int64_t)b * p.nchunks + cc));
      else lst = fallback_last;
      y = lst;
    }
    write_chain_out(p, b, k, y);
  }
}

// greedy: merge chunk argmaxes per row, then the chain or tree rule.  grid (B), 256 threads.
__global__ void __launch_bounds__(kSampleThreads) sample_greedy_decide(const __grid_constant__ SampleParams p) {
  __shared__ int a[kMaxTreeNodes > kMaxGamma + 1 ? kMaxTreeNodes : kMaxGamma + 1];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rows = p.rows_t;
  for (int r = warp; r < rows; r += kSampleThreads / 32) {
    const int64_t o = ((int64_t)b * rows + r) * p.nchunks;
    float v = neg_inf();
    int i = INT_MAX;
    for (int cc = lane; cc < p.nchunks; cc += 32) argmax_combine(v, i, p.st_m[o + cc], p.st_arg[o + cc]);
    warp_argmax(v, i);
    if (lane == 0) a[r] = i;
  }
  __syncthreads();
  if (tid != 0) return;
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

size_t sample_workspace_bytes(int mode, int B, int rows_t, int rows_d, int V) {
  (void)mode;
  const size_t nch = (size_t)(V + kMinChunk - 1) / kMinChunk;
  const size_t rows = (size_t)rows_t + rows_d;
  size_t bytes = 256;
  bytes += (B * rows * nch * sizeof(float) + 255) / 256 * 256;    // st_m
  bytes += (B * rows * nch * sizeof(double) + 255) / 256 * 256;   // st_s / st_arg
  bytes += (B * nch * sizeof(double) + 255) / 256 * 256;          // res_sum
  bytes += (B * nch * sizeof(int32_t) + 255) / 256 * 256;         // res_last
  bytes += ((size_t)B * sizeof(int32_t) + 255) / 256 * 256;       // ticket
  return bytes;
}

void sample_workspace_carve(void* ws, SampleParams* p) {
  const size_t nch = (size_t)(p->V + kMinChunk - 1) / kMinChunk;
  const size_t rows = (size_t)p->rows_t + p->rows_d;
  const size_t B = (size_t)p->B;
  uint8_t* q = reinterpret_cast<uint8_t*>(ws);
  p->status = reinterpret_cast<uint32_t*>(q);
  q += 256;
  p->st_m = reinterpret_cast<float*>(q);
  q += (B * rows * nch * sizeof(float) + 255) / 256 * 256;
  p->st_s = reinterpret_cast<double*>(q);
  p->st_arg = reinterpret_cast<int32_t*>(q);
  q += (B * rows * nch * sizeof(double) + 255) / 256 * 256;
  p->res_sum = reinterpret_cast<double*>(q);
  q += (B * nch * sizeof(double) + 255) / 256 * 256;
  p->res_last = reinterpret_cast<int32_t*>(q);
  q += (B * nch * sizeof(int32_t) + 255) / 256 * 256;
  p->ticket = reinterpret_cast<int32_t*>(q);
}

template <int EPT>
static cudaError_t launch_large(const SampleParams& p, cudaStream_t stream) {
  const int rows = p.rows_t + p.rows_d;
  dim3 g1(p.nchunks, rows, p.B);
  if (p.mode == SPEC_SAMPLE_CHAIN) {
    sample_stats<EPT, false><<<g1, kSampleThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    dim3 g2(p.nchunks, p.B);
    sample_residual<EPT><<<g2, kSampleThreads, 0, stream>>>(p);
  } else {
    sample_stats<EPT, true><<<g1, kSampleThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    sample_greedy_decide<<<p.B, kSampleThreads, 0, stream>>>(p);
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
  p.chunk = pick_chunk(p.V, p.rows_t + p.rows_d, p.B, num_sms);
  p.nchunks = (p.V + p.chunk - 1) / p.chunk;
  switch (p.chunk) {
    case 8192: return launch_large<32>(p, stream);
    case 4096: return launch_large<16>(p, stream);
    default: return launch_large<8>(p, stream);
  }
}

}  // namespace specv
