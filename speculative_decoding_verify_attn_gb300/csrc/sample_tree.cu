// Stochastic acceptance over a token tree (SPEC_SAMPLE_TREE): multi-step speculative sampling.
//
// The pages name tree verification with sampling (SpecInfer, "Speculative Decoding in LLM
// Serving Systems", Tree-based variants) without its rule; the rule used applies the chain test of
// "Speculative Decoding & Medusa" §2 to a node's children in index order: child c with token x_c
// is accepted iff u_c * Q(x_c) < R(x_c), R = P at first and, after each rejection, the normalised
// residual max(R - Q, 0).  Against one draft distribution Q per node that residual is
// max(P - c Q, 0) / N with c_0 = 0, N_0 = 1, c_{i+1} = c_i + N_i and N_{i+1} = sum max(P - c_{i+1} Q, 0),
// so no residual vector is stored: each rejection costs one pass over the node's two rows.  With
// no child accepted, the token is drawn from max(P - c Q, 0) by inverse CDF with u_0 (u_0 * N as
// the threshold on the unnormalised cumulative sum).
//
// One CTA of 512 threads per sequence walks the tree.  Per visited node: the max and normaliser
// of its target row (and of its draft row if it has children) in float-float; the accept tests in
// fp64 on one thread from the two selected logits; a float-float reduction per rejected child;
// the final draw as a chunked float-float scan (thread t owns a contiguous share of the
// vocabulary) followed by a rescan of the one chunk where the cumulative sum crosses the
// threshold, in the same element order.
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "ff.cuh"
#include "sample_internal.h"

namespace specv {

constexpr int kTreeThreads = 512;
constexpr int kTreeWarps = kTreeThreads / 32;

struct TreeRed {
  float f[kTreeWarps];
  FF ff[kTreeWarps];
  int i[kTreeWarps];
};

// Block reductions in a fixed order; every thread returns the result.
__device__ float tree_block_max(float v, TreeRed& r) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) r.f[warp] = v;
  __syncthreads();
  return warp_max(lane < kTreeWarps ? r.f[lane] : neg_inf());
}
__device__ FF tree_block_sum(FF v, TreeRed& r) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_ff(v);
  __syncthreads();
  if (lane == 0) r.ff[warp] = v;
  __syncthreads();
  return warp_sum_ff(lane < kTreeWarps ? r.ff[lane] : FF{0.f, 0.f});
}
__device__ int tree_block_min_i(int v, TreeRed& r) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if (lane == 0) r.i[warp] = v;
  __syncthreads();
  int t = lane < kTreeWarps ? r.i[lane] : INT_MAX;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) t = min(t, __shfl_xor_sync(0xffffffffu, t, o));
  return t;
}

struct TreeRow {
  float M, iZ;  // row max, 1 / normaliser (fp32) for the element passes
  double Z;     // normaliser sum exp(x - M) for the accept tests
};

// Max and normaliser of one row of V logits (V a multiple of 4), coalesced 16-byte loads.
__device__ TreeRow tree_row_stats(const float* row, int V, TreeRed& r) {
  const float4* r4 = reinterpret_cast<const float4*>(row);
  float m = neg_inf();
  for (int i = threadIdx.x; i < V / 4; i += kTreeThreads) {
    const float4 x = __ldg(r4 + i);
    m = fmaxf(m, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
  }
  const float M = tree_block_max(m, r);
  FF z{0.f, 0.f};
  for (int i = threadIdx.x; i < V / 4; i += kTreeThreads) {
    const float4 x = __ldg(r4 + i);
    const float s = __fadd_rn(__fadd_rn(exp_shift(x.x, M), exp_shift(x.y, M)),
                              __fadd_rn(exp_shift(x.z, M), exp_shift(x.w, M)));
    z = ff_add(z, FF{s, 0.f});
  }
  const FF Z = tree_block_sum(z, r);
  TreeRow out;
  out.M = M;
  out.Z = (double)Z.hi + (double)Z.lo;
  out.iZ = 1.0f / Z.hi;
  return out;
}

// One residual element max(P(y) - c Q(y), 0); P(y) when there is no coefficient (c = 0).
__device__ __forceinline__ float tree_resid(float t, float d, const TreeRow& T, const TreeRow& Dr, float c,
                                            bool use_q) {
  const float pt = __fmul_rn(exp_shift(t, T.M), T.iZ);
  if (!use_q) return pt;
  const float qd = __fmul_rn(exp_shift(d, Dr.M), Dr.iZ);
  return fmaxf(__fsub_rn(pt, __fmul_rn(c, qd)), 0.f);
}

// sum_y max(P(y) - c Q(y), 0) over the row pair.
__device__ FF tree_resid_mass(const float* tr, const float* dr, int V, const TreeRow& T, const TreeRow& Dr, float c,
                              TreeRed& r) {
  const float4* t4 = reinterpret_cast<const float4*>(tr);
  const float4* d4 = reinterpret_cast<const float4*>(dr);
  FF z{0.f, 0.f};
  for (int i = threadIdx.x; i < V / 4; i += kTreeThreads) {
    const float4 t = __ldg(t4 + i), d = __ldg(d4 + i);
    const float s = __fadd_rn(__fadd_rn(tree_resid(t.x, d.x, T, Dr, c, true), tree_resid(t.y, d.y, T, Dr, c, true)),
                              __fadd_rn(tree_resid(t.z, d.z, T, Dr, c, true), tree_resid(t.w, d.w, T, Dr, c, true)));
    z = ff_add(z, FF{s, 0.f});
  }
  return tree_block_sum(z, r);
}

// y = min{y : C(y) > thr}, C the cumulative sum of max(P - c Q, 0) (P when use_q is false) in
// token order; if none qualifies (rounding), the largest y with a positive element.  Thread t
// owns the float4 indices [t per4, (t + 1) per4); its chunk sum is accumulated element by element
// in float-float, the chunk offsets come from a block scan, and the first chunk whose inclusive sum
// exceeds thr is rescanned in the same order.
__device__ int tree_final_draw(const float* tr, const float* dr, int V, const TreeRow& T, const TreeRow& Dr, float c,
                               bool use_q, FF thr, TreeRed& r, FF* s_off, int* s_y) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float4* t4 = reinterpret_cast<const float4*>(tr);
  const float4* d4 = reinterpret_cast<const float4*>(dr);
  const int n4 = V / 4;
  const int per4 = (n4 + kTreeThreads - 1) / kTreeThreads;
  const int lo4 = min(tid * per4, n4), hi4 = min(lo4 + per4, n4);
  auto elems = [&](int i, float (&e)[4]) {
    const float4 t = __ldg(t4 + i);
    const float4 d = use_q ? __ldg(d4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    e[0] = tree_resid(t.x, d.x, T, Dr, c, use_q);
    e[1] = tree_resid(t.y, d.y, T, Dr, c, use_q);
    e[2] = tree_resid(t.z, d.z, T, Dr, c, use_q);
    e[3] = tree_resid(t.w, d.w, T, Dr, c, use_q);
  };
  FF s{0.f, 0.f};
  int lastpos = -1;
  for (int i = lo4; i < hi4; ++i) {
    float e[4];
    elems(i, e);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      s = ff_add(s, FF{e[k], 0.f});
      if (e[k] > 0.f) lastpos = 4 * i + k;
    }
  }
  // exclusive scan of the chunk sums over the threads, in thread order
  const FF inc = warp_scan_ff(s);
  FF ex_lane = shfl_up_ff(inc, 1);
  if (lane == 0) ex_lane = FF{0.f, 0.f};
  __syncthreads();
  if (lane == 31) s_off[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const FF wi = warp_scan_ff(lane < kTreeWarps ? s_off[lane] : FF{0.f, 0.f});
    FF we = shfl_up_ff(wi, 1);
    if (lane == 0) we = FF{0.f, 0.f};
    if (lane < kTreeWarps) s_off[kTreeWarps + lane] = we;
  }
  __syncthreads();
  const FF excl = ff_add(s_off[kTreeWarps + warp], ex_lane);
  const FF incl = ff_add(excl, s);
  const int first = tree_block_min_i(ff_gt(incl, thr) ? tid : INT_MAX, r);
  if (first == INT_MAX) return -tree_block_min_i(-lastpos, r);
  if (tid == first) {
    FF run = excl;
    int y = -1, lastp = -1;
    for (int i = lo4; i < hi4 && y < 0; ++i) {
      float e[4];
      elems(i, e);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        run = ff_add(run, FF{e[k], 0.f});
        if (e[k] > 0.f) lastp = 4 * i + k;
        if (y < 0 && ff_gt(run, thr)) y = 4 * i + k;
      }
    }
    *s_y = y >= 0 ? y : lastp;  // a crossing lost to rounding inside the chunk: its last positive
  }
  __syncthreads();
  return *s_y;
}

__global__ void __launch_bounds__(kTreeThreads, 1) sample_tree_stochastic(const __grid_constant__ SampleParams p) {
  __shared__ TreeRed red;
  __shared__ FF s_off[2 * kTreeWarps];
  __shared__ int s_y, s_next;
  __shared__ int s_path[kMaxTreeNodes];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int32_t* tok = p.tok + (int64_t)b * p.tok_sb;
  const float* u = p.u + (int64_t)b * p.u_sb;
  int32_t* out = p.out_tok + (int64_t)b * p.out_cols;
  int32_t* nodes = p.out_nodes ? p.out_nodes + (int64_t)b * p.out_cols : nullptr;

  int bad = 0;
  for (int c = 1 + tid; c < p.N; c += kTreeThreads) {
    const int x = tok[c];
    bad |= x < 0 || x >= p.V;
  }
  if (__syncthreads_or(bad)) {  // a child token outside [0, V): nothing emitted
    if (tid == 0) {
      for (int i = 0; i < p.out_cols; ++i) {
        out[i] = -1;
        if (nodes) nodes[i] = -1;
      }
      p.out_nacc[b] = -1;
      atomicOr(p.status, (uint32_t)SPEC_STATUS_BAD_TOKEN);
    }
    return;
  }
  const float u0 = u[0];
  int n = 0, d = 0;
  for (;;) {
    const float* tr = p.tl + (int64_t)b * p.tl_sb + (int64_t)n * p.V;
    const float* dr = p.dl + (int64_t)b * p.dl_sb + (int64_t)n * p.V;
    bool kids = false;
    for (int ch = n + 1; ch < p.N; ++ch) kids |= p.parent[ch] == n;
    const TreeRow T = tree_row_stats(tr, p.V, red);
    TreeRow Dr{0.f, 0.f, 1.0};
    if (kids) Dr = tree_row_stats(dr, p.V, red);
    double c = 0.0;        // the residual is max(P - c Q, 0) / Nres
    FF Nres{1.f, 0.f};
    int next = -1;
    for (int ch = n + 1; kids && ch < p.N; ++ch) {
      if (p.parent[ch] != n) continue;
      if (tid == 0) {  // u_ch Q(x) < R(x), with R(x) = max(P(x) - c Q(x), 0) / Nres
        const int x = tok[ch];
        const double Px = exp((double)__ldg(tr + x) - (double)T.M) / T.Z;
        const double Qx = exp((double)__ldg(dr + x) - (double)Dr.M) / Dr.Z;
        const double lhs = (double)__ldg(u + ch) * Qx * ((double)Nres.hi + (double)Nres.lo);
        s_next = lhs < fmax(Px - c * Qx, 0.0) ? ch : -1;
      }
      __syncthreads();
      next = s_next;
      if (next >= 0) break;
      c += (double)Nres.hi + (double)Nres.lo;
      Nres = tree_resid_mass(tr, dr, p.V, T, Dr, (float)c, red);
      if (!(Nres.hi > 0.f)) {  // no residual mass left: fall back to P
        c = 0.0;
        Nres = FF{1.f, 0.f};
      }
    }
    if (next >= 0) {
      if (tid == 0) s_path[d] = next;
      ++d;
      n = next;
      continue;
    }
    const int y = tree_final_draw(tr, dr, p.V, T, Dr, (float)c, c > 0.0, ff_mul_f(Nres, u0), red, s_off, &s_y);
    if (tid == 0) {
      for (int i = 0; i < p.out_cols; ++i) {
        out[i] = i < d ? tok[s_path[i]] : (i == d ? y : -1);
        if (nodes) nodes[i] = i < d ? s_path[i] : -1;
      }
      p.out_nacc[b] = d;
    }
    return;
  }
}

cudaError_t launch_sample_tree(const SampleParams& p, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  sample_tree_stochastic<<<p.B, kTreeThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace specv
