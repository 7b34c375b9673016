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
// One thread-block cluster of kTreeCS CTAs per sequence walks the tree; CTA r owns the r-th share
// of the vocabulary and stages its share of the current node's two rows in shared memory (when
// they fit), while one thread bulk-prefetches the children's shares into L2.  Every reduction is
// a block reduction followed by an exchange through distributed shared memory: each CTA's
// thread 0 posts its value to a double-buffered slot, one cluster barrier, then thread 0 reads
// the kTreeCS slots, combines them in rank order and hands the result to its CTA, so all CTAs
// hold bit-identical values and take identical decisions without a broadcast.  Per visited node:
// the two maxima (one exchange) and the two normalisers in float-float (one exchange); the
// accept tests evaluated by every thread in float-float arithmetic (no fp64: GB300's fp64 pipe
// is slow); one reduction per rejected child; the final draw as a chunked float-float scan over
// the cluster (thread t of CTA r owns a contiguous piece of r's share) whose first crossing
// chunk is rescanned in the same element order by its thread, which stores the token.
#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <limits.h>

#include "common.cuh"
#include "ff.cuh"
#include "sample_internal.h"
#include "launch_cache.h"

namespace specv {

namespace cg = cooperative_groups;

constexpr int kTreeThreads = 256;
constexpr int kTreeWarps = kTreeThreads / 32;
constexpr int kTreeCS = 8;  // CTAs per sequence (portable cluster size)
constexpr size_t kTreeSmemMax = 200 * 1024;  // staging of two row shares in shared memory up to this

struct TreeRed {  // block-reduction scratch
  float f[kTreeWarps];
  FF ff[kTreeWarps];
  int i[kTreeWarps];
};
struct TreeXch {  // cluster exchange slots, double-buffered (one barrier per exchange)
  float f[2][kTreeCS];
  FF ff[2][kTreeCS];
  int i[2][kTreeCS];
  float2 f2[2][kTreeCS];
  FF ff2[2][kTreeCS];
  // the combined result, handed from thread 0 to the rest of its CTA
  float2 bf2;
  float bf;
  int bi;
  FF bff[2];
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

// Cluster exchanges of a per-CTA value (the same in every thread of the CTA); every thread of
// every CTA returns the combination over the ranks in rank order.  Thread 0 alone reads the
// other CTAs' slots (remote shared-memory reads are few and slow) and hands the result to its
// CTA through a local slot.  A slot written at exchange k is read only before the barrier of
// exchange k + 1, so two buffers suffice.
struct TreeCluster {
  cg::cluster_group cl;
  TreeXch& x;
  int rank, ph;
  template <typename V>
  __device__ V remote(V* slot, int r) {
    return *cl.map_shared_rank(slot, r);
  }
  __device__ float max(float v) {
    if (threadIdx.x == 0) x.f[ph][rank] = v;
    cl.sync();
    if (threadIdx.x == 0) {
      float m = neg_inf();
#pragma unroll
      for (int r = 0; r < kTreeCS; ++r) m = fmaxf(m, remote(&x.f[ph][r], r));
      x.bf = m;
    }
    __syncthreads();
    ph ^= 1;
    return x.bf;
  }
  __device__ int min_i(int v) {
    if (threadIdx.x == 0) x.i[ph][rank] = v;
    cl.sync();
    if (threadIdx.x == 0) {
      int m = INT_MAX;
#pragma unroll
      for (int r = 0; r < kTreeCS; ++r) m = ::min(m, remote(&x.i[ph][r], r));
      x.bi = m;
    }
    __syncthreads();
    ph ^= 1;
    return x.bi;
  }
  __device__ float2 max2(float2 v) {
    if (threadIdx.x == 0) x.f2[ph][rank] = v;
    cl.sync();
    if (threadIdx.x == 0) {
      float2 m = make_float2(neg_inf(), neg_inf());
#pragma unroll
      for (int r = 0; r < kTreeCS; ++r) {
        const float2 o = remote(&x.f2[ph][r], r);
        m.x = fmaxf(m.x, o.x);
        m.y = fmaxf(m.y, o.y);
      }
      x.bf2 = m;
    }
    __syncthreads();
    ph ^= 1;
    return x.bf2;
  }
  // two sums at once (the second returned through b_out), in rank order
  __device__ FF sum2(FF a, FF b, FF& b_out) {
    if (threadIdx.x == 0) {
      x.ff[ph][rank] = a;
      x.ff2[ph][rank] = b;
    }
    cl.sync();
    if (threadIdx.x == 0) {
      FF ta{0.f, 0.f}, tb{0.f, 0.f};
#pragma unroll
      for (int r = 0; r < kTreeCS; ++r) {
        ta = ff_add(ta, remote(&x.ff[ph][r], r));
        tb = ff_add(tb, remote(&x.ff2[ph][r], r));
      }
      x.bff[0] = ta;
      x.bff[1] = tb;
    }
    __syncthreads();
    ph ^= 1;
    b_out = x.bff[1];
    return x.bff[0];
  }
  // sum over all ranks, and the sum over the ranks below this one (exclusive prefix)
  __device__ FF sum(FF v, FF* below = nullptr) {
    if (threadIdx.x == 0) x.ff[ph][rank] = v;
    cl.sync();
    if (threadIdx.x == 0) {
      FF t{0.f, 0.f}, bl{0.f, 0.f};
#pragma unroll
      for (int r = 0; r < kTreeCS; ++r) {
        if (r == rank) bl = t;
        t = ff_add(t, remote(&x.ff[ph][r], r));
      }
      x.bff[0] = t;
      x.bff[1] = bl;
    }
    __syncthreads();
    ph ^= 1;
    if (below) *below = x.bff[1];
    return x.bff[0];
  }
};

struct TreeRow {
  float M, iZ;  // row max, 1 / normaliser (fp32) for the element passes
  FF Z;         // normaliser sum exp(x - M)
};

// Max and normaliser of the node's target row (and draft row, with kids) over the cluster: one
// pass for the two maxima, one exchange, one pass for sum exp(x - max) of both rows in
// float-float, one exchange.  This CTA's shares are t4[0, len4), d4[0, len4).
__device__ void tree_node_stats(const float4* t4, const float4* d4, int len4, bool kids, TreeRow& T, TreeRow& Dr,
                                TreeRed& r, TreeCluster& C) {
  float mt = neg_inf(), md = neg_inf();
  for (int i = threadIdx.x; i < len4; i += kTreeThreads) {
    const float4 x = t4[i];
    mt = fmaxf(mt, fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w)));
    if (kids) {
      const float4 y = d4[i];
      md = fmaxf(md, fmaxf(fmaxf(y.x, y.y), fmaxf(y.z, y.w)));
    }
  }
  const float2 M = C.max2(make_float2(tree_block_max(mt, r), tree_block_max(md, r)));
  FF zt{0.f, 0.f}, zd{0.f, 0.f};
  for (int i = threadIdx.x; i < len4; i += kTreeThreads) {
    const float4 x = t4[i];
    zt = ff_add(zt, FF{__fadd_rn(__fadd_rn(exp_shift(x.x, M.x), exp_shift(x.y, M.x)),
                                 __fadd_rn(exp_shift(x.z, M.x), exp_shift(x.w, M.x))), 0.f});
    if (kids) {
      const float4 y = d4[i];
      zd = ff_add(zd, FF{__fadd_rn(__fadd_rn(exp_shift(y.x, M.y), exp_shift(y.y, M.y)),
                                   __fadd_rn(exp_shift(y.z, M.y), exp_shift(y.w, M.y))), 0.f});
    }
  }
  FF Zd;
  const FF Zt = C.sum2(tree_block_sum(zt, r), tree_block_sum(zd, r), Zd);
  T.M = M.x;
  T.Z = Zt;
  T.iZ = 1.0f / Zt.hi;
  Dr.M = M.y;
  Dr.Z = Zd;
  Dr.iZ = kids ? 1.0f / Zd.hi : 0.f;
}

// The accept test of a child with token x: u * Q(x) < R(x), R = max(P - c Q, 0) / N, i.e.
// u N + c < P(x) / Q(x); the ratio's exponent is formed in float-float before one expf, the
// normaliser ratio with its first-order correction (the same evaluation in every thread).
__device__ __forceinline__ bool tree_accept(float tx, float dx, const TreeRow& T, const TreeRow& Dr, FF c, FF N,
                                            float u) {
  const FF e = ff_add(ff_add(FF{tx, 0.f}, FF{-T.M, 0.f}), ff_neg(ff_add(FF{dx, 0.f}, FF{-Dr.M, 0.f})));
  const float zr = __fdiv_rn(Dr.Z.hi, T.Z.hi) * (1.f + (__fdiv_rn(Dr.Z.lo, Dr.Z.hi) - __fdiv_rn(T.Z.lo, T.Z.hi)));
  const float ratio = expf(e.hi) * (1.f + e.lo) * zr;
  return ff_gt(FF{ratio, 0.f}, ff_add(ff_mul_f(N, u), c));
}

// One residual element max(P(y) - c Q(y), 0); P(y) when there is no coefficient (c = 0).
__device__ __forceinline__ float tree_resid(float t, float d, const TreeRow& T, const TreeRow& Dr, float c,
                                            bool use_q) {
  const float pt = __fmul_rn(exp_shift(t, T.M), T.iZ);
  if (!use_q) return pt;
  const float qd = __fmul_rn(exp_shift(d, Dr.M), Dr.iZ);
  return fmaxf(__fsub_rn(pt, __fmul_rn(c, qd)), 0.f);
}

// sum_y max(P(y) - c Q(y), 0) over the row pair and the cluster.
__device__ FF tree_resid_mass(const float4* t4, const float4* d4, int len4, const TreeRow& T, const TreeRow& Dr,
                              float c, TreeRed& r, TreeCluster& C) {
  FF z{0.f, 0.f};
  for (int i = threadIdx.x; i < len4; i += kTreeThreads) {
    const float4 t = t4[i], d = d4[i];
    const float s = __fadd_rn(__fadd_rn(tree_resid(t.x, d.x, T, Dr, c, true), tree_resid(t.y, d.y, T, Dr, c, true)),
                              __fadd_rn(tree_resid(t.z, d.z, T, Dr, c, true), tree_resid(t.w, d.w, T, Dr, c, true)));
    z = ff_add(z, FF{s, 0.f});
  }
  return C.sum(tree_block_sum(z, r));
}

// y = min{y : C(y) > thr}, C the cumulative sum of max(P - c Q, 0) (P when use_q is false) in
// token order over the whole vocabulary; if none qualifies (rounding), the largest y with a
// positive element.  Thread t of this CTA owns a contiguous piece of the CTA's share [lo4, hi4);
// its chunk sum is accumulated element by element in float-float; the offsets come from a block
// scan and the exclusive prefix of the CTA totals over the cluster; the first chunk (in token
// order) whose inclusive sum exceeds thr is rescanned in the same order by its thread, which
// stores y to y_out; the function then returns -2.  With no crossing (rounding) every CTA returns
// the fallback y.
__device__ int tree_final_draw(const float4* t4, const float4* d4, int lo4, int len4, const TreeRow& T,
                               const TreeRow& Dr, float c, bool use_q, FF thr, TreeRed& r, FF* s_off, int32_t* y_out,
                               TreeCluster& C) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per4 = (len4 + kTreeThreads - 1) / kTreeThreads;
  const int a4 = min(tid * per4, len4), b4 = min(tid * per4 + per4, len4);
  // element ids are absolute: 4 (lo4 + i) + k for local float4 index i
  auto elems = [&](int i, float (&e)[4]) {
    const float4 t = t4[i];
    const float4 d = use_q ? d4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
    e[0] = tree_resid(t.x, d.x, T, Dr, c, use_q);
    e[1] = tree_resid(t.y, d.y, T, Dr, c, use_q);
    e[2] = tree_resid(t.z, d.z, T, Dr, c, use_q);
    e[3] = tree_resid(t.w, d.w, T, Dr, c, use_q);
  };
  FF s{0.f, 0.f};
  int lastpos = -1;
  for (int i = a4; i < b4; ++i) {
    float e[4];
    elems(i, e);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      s = ff_add(s, FF{e[k], 0.f});
      if (e[k] > 0.f) lastpos = 4 * (lo4 + i) + k;
    }
  }
  // exclusive scan of the chunk sums over the threads of the CTA, in thread order
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
  const FF cta_total = ff_add(s_off[kTreeWarps + kTreeWarps - 1], s_off[kTreeWarps - 1]);
  FF cta_below{0.f, 0.f};
  C.sum(cta_total, &cta_below);
  const FF excl = ff_add(cta_below, ff_add(s_off[kTreeWarps + warp], ex_lane));
  const FF incl = ff_add(excl, s);
  const int first = C.min_i(tree_block_min_i(ff_gt(incl, thr) ? C.rank * kTreeThreads + tid : INT_MAX, r));
  if (first == INT_MAX) return -C.min_i(tree_block_min_i(-lastpos, r));
  if (first / kTreeThreads == C.rank && tid == first % kTreeThreads) {
    FF run = excl;
    int y = -1, lastp = -1;
    for (int i = a4; i < b4 && y < 0; ++i) {
      float e[4];
      elems(i, e);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        run = ff_add(run, FF{e[k], 0.f});
        if (e[k] > 0.f) lastp = 4 * (lo4 + i) + k;
        if (y < 0 && ff_gt(run, thr)) y = 4 * (lo4 + i) + k;
      }
    }
    *y_out = y >= 0 ? y : lastp;  // a crossing lost to rounding inside the chunk: its last positive
  }
  return -2;  // written by the thread that found it
}

// SM: the CTA's share of the node's two rows is staged in shared memory once per node, so the
// statistics, residual and draw passes after it read shared memory; otherwise they read global.
template <bool SM>
__global__ void __launch_bounds__(kTreeThreads, 1) sample_tree_stochastic(const __grid_constant__ SampleParams p) {
  extern __shared__ float4 s_rows[];  // SM: [2][share4] target share, draft share
  __shared__ TreeRed red;
  __shared__ TreeXch xch;
  __shared__ FF s_off[2 * kTreeWarps];
  __shared__ int s_path[kMaxTreeNodes];
  cg::cluster_group cl = cg::this_cluster();
  TreeCluster C{cl, xch, (int)cl.block_rank(), 0};
  const int b = blockIdx.x / kTreeCS, tid = threadIdx.x;
  const int n4 = p.V / 4, share4 = (n4 + kTreeCS - 1) / kTreeCS;
  const int lo4 = min(C.rank * share4, n4), hi4 = min(lo4 + share4, n4);
  const int32_t* tok = p.tok + (int64_t)b * p.tok_sb;
  const float* u = p.u + (int64_t)b * p.u_sb;
  int32_t* out = p.out_tok + (int64_t)b * p.out_cols;
  int32_t* nodes = p.out_nodes ? p.out_nodes + (int64_t)b * p.out_cols : nullptr;
  const bool writer = C.rank == 0 && tid == 0;

  int bad = 0;
  for (int c = 1 + tid; c < p.N; c += kTreeThreads) {
    const int x = tok[c];
    bad |= x < 0 || x >= p.V;
  }
  if (__syncthreads_or(bad)) {  // a child token outside [0, V): nothing emitted (same in every CTA)
    if (writer) {
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
  int n = 0, d = 0, y = -1;
  for (;;) {
    const float* tr = p.tl + (int64_t)b * p.tl_sb + (int64_t)n * p.V;
    const float* dr = p.dl + (int64_t)b * p.dl_sb + (int64_t)n * p.V;
    bool kids = false;
    for (int ch = n + 1; ch < p.N; ++ch) kids |= p.parent[ch] == n;
    const int len4 = hi4 - lo4;
    const float4* T4 = reinterpret_cast<const float4*>(tr) + lo4;
    const float4* D4 = reinterpret_cast<const float4*>(dr) + lo4;
    if (SM) {
      __syncthreads();  // the previous node's passes are done with the staging buffer
      for (int i = tid; i < len4; i += kTreeThreads) {
        s_rows[i] = __ldg(T4 + i);
        if (kids) s_rows[share4 + i] = __ldg(D4 + i);
      }
      __syncthreads();
      T4 = s_rows;
      D4 = s_rows + share4;
    }
    // the next node is one of the children: their row shares into L2 while this node is decided
    // (one bulk prefetch per share; shares are 16-byte aligned multiples of 16 bytes)
    if (tid == 0 && len4 > 0) {
      for (int ch = n + 1; ch < p.N; ++ch) {
        if (p.parent[ch] != n) continue;
        const float* rows[2] = {p.tl + (int64_t)b * p.tl_sb + (int64_t)ch * p.V, p.dl + (int64_t)b * p.dl_sb + (int64_t)ch * p.V};
        for (int k = 0; k < 2; ++k) l2_prefetch_bulk(rows[k] + 4 * lo4, (uint32_t)len4 * 16u);
      }
    }
    TreeRow T, Dr;
    tree_node_stats(T4, D4, len4, kids, T, Dr, red, C);
    FF c{0.f, 0.f};  // the residual is max(P - c Q, 0) / Nres
    FF Nres{1.f, 0.f};
    int next = -1;
    for (int ch = n + 1; kids && ch < p.N; ++ch) {
      if (p.parent[ch] != n) continue;
      // every thread of every CTA evaluates the same test on the same values
      const int x = tok[ch];
      if (tree_accept(__ldg(tr + x), __ldg(dr + x), T, Dr, c, Nres, __ldg(u + ch))) {
        next = ch;
        break;
      }
      c = ff_add(c, Nres);
      Nres = tree_resid_mass(T4, D4, len4, T, Dr, c.hi, red, C);
      if (!(Nres.hi > 0.f)) {  // no residual mass left: fall back to P
        c = FF{0.f, 0.f};
        Nres = FF{1.f, 0.f};
      }
    }
    if (next >= 0) {
      if (tid == 0) s_path[d] = next;
      ++d;
      n = next;
      continue;
    }
    y = tree_final_draw(T4, D4, lo4, len4, T, Dr, c.hi, c.hi > 0.f, ff_mul_f(Nres, u0), red, s_off, out + d, C);
    break;
  }
  if (writer) {  // out[d] comes from the thread that found the draw (y == -2) or from here
    for (int i = 0; i < p.out_cols; ++i) {
      if (i != d || y != -2) out[i] = i < d ? tok[s_path[i]] : (i == d ? y : -1);
      if (nodes) nodes[i] = i < d ? s_path[i] : -1;
    }
    p.out_nacc[b] = d;
  }
  cl.sync();  // no CTA leaves while another may still read its exchange slots
}

cudaError_t launch_sample_tree(const SampleParams& p, cudaStream_t stream) {
  cudaError_t e = p.status_zeroed ? cudaSuccess : cudaMemsetAsync(p.status, 0, sizeof(uint32_t), stream);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kTreeCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3((unsigned)(p.B * kTreeCS), 1, 1);
  cfg.blockDim = dim3(kTreeThreads, 1, 1);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // stage the two row shares in shared memory when they fit (V up to about 200 000)
  const int share4 = (p.V / 4 + kTreeCS - 1) / kTreeCS;
  const size_t smem = 2 * (size_t)share4 * sizeof(float4);
  if (smem <= kTreeSmemMax) {
    e = ensure_dynamic_smem(reinterpret_cast<const void*>(sample_tree_stochastic<true>), (int)smem);
    if (e != cudaSuccess) return e;
    cfg.dynamicSmemBytes = smem;
    e = cudaLaunchKernelEx(&cfg, sample_tree_stochastic<true>, p);
  } else {
    e = cudaLaunchKernelEx(&cfg, sample_tree_stochastic<false>, p);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace specv
