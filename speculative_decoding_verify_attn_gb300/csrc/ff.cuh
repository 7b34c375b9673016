// Float-float arithmetic (fp32 pairs, about 44 significant bits) and the shifted exponential of
// the sampling kernels: reproducible sums of probabilities without the fp64 pipe.
#pragma once

#include <cuda_runtime.h>

#include "common.cuh"

namespace specv {

// exp(x - M) in fp32 through exp2f (2 ulp); x - M <= 0 is formed first so that the dominant
// terms (x near M) carry only the rounding of the final product
__device__ __forceinline__ float exp_shift(float x, float M) {
  return exp2f(__fmul_rn(__fsub_rn(x, M), kLog2e));
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
__device__ __forceinline__ FF ff_neg(FF a) { return FF{-a.hi, -a.lo}; }
// The exact sum of two floats as a float-float (Knuth's TwoSum).
__device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float v = __fsub_rn(s, a);
  return FF{s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, v)), __fsub_rn(b, v))};
}
// a * b for float-float a and float b: the exact product of the high parts (FMA) plus the low
// part's product, renormalised
__device__ __forceinline__ FF ff_mul_f(FF a, float b) {
  const float p = __fmul_rn(a.hi, b);
  const float e = __fmaf_rn(a.hi, b, -p);
  const float t = __fmaf_rn(a.lo, b, e);
  const float hi = __fadd_rn(p, t);
  return FF{hi, __fsub_rn(t, __fsub_rn(hi, p))};
}
// a > b (the sign of the float-float difference)
__device__ __forceinline__ bool ff_gt(FF a, FF b) {
  const FF d = ff_add(a, ff_neg(b));
  return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}
__device__ __forceinline__ FF shfl_ff(FF v, int src) {
  return FF{__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}
__device__ __forceinline__ FF shfl_up_ff(FF v, int o) {
  return FF{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
}
// Warp sum of float-float values, in a fixed tree order; every lane returns lane 0's result.
__device__ __forceinline__ FF warp_sum_ff(FF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    FF w;
    w.hi = __shfl_down_sync(0xffffffffu, v.hi, o);
    w.lo = __shfl_down_sync(0xffffffffu, v.lo, o);
    if (lane < o) v = ff_add(v, w);
  }
  return shfl_ff(v, 0);
}
// Inclusive warp scan of float-float values in lane order.
__device__ __forceinline__ FF warp_scan_ff(FF v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const FF t = shfl_up_ff(v, o);
    if (lane >= o) v = ff_add(t, v);
  }
  return v;
}

}  // namespace specv
