// dfloat.cuh -- compensated ("double-float") accumulation on the fp32 pipe.
//
// B300's fp64 rate is a small fraction of its fp32 rate, so the reductions
// of the fused update pass and the sink cosines accumulate in pairs of
// floats (hi + lo, the error-free transformations of Knuth's TwoSum and of
// the FMA-based exact product) and convert to double only once per block.
// The pair carries about 44 significant bits; every operation below is a
// fixed sequence of round-to-nearest fp32 operations, so results are
// deterministic for a fixed order of additions.
#pragma once

namespace sds {

struct dfloat {
  float hi, lo;
};

__device__ __forceinline__ dfloat df_make(float x) { return dfloat{x, 0.f}; }

// Exact product a*b as hi + lo (the FMA computes the rounding error exactly).
__device__ __forceinline__ dfloat df_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return dfloat{p, __fmaf_rn(a, b, -p)};
}

// a + b with TwoSum on the high parts and the low parts folded in.
__device__ __forceinline__ dfloat df_add(dfloat a, dfloat b) {
  const float s = __fadd_rn(a.hi, b.hi);
  const float bb = __fsub_rn(s, a.hi);
  float e = __fadd_rn(__fsub_rn(a.hi, __fsub_rn(s, bb)), __fsub_rn(b.hi, bb));
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  const float hi = __fadd_rn(s, e);
  return dfloat{hi, __fsub_rn(e, __fsub_rn(hi, s))};
}

__device__ __forceinline__ double df_to_double(dfloat a) { return (double)a.hi + (double)a.lo; }

// Butterfly over the warp: every lane ends with the same bits.
__device__ __forceinline__ dfloat df_warp_sum(dfloat v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const dfloat w{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
    v = df_add(v, w);
  }
  return v;
}

}  // namespace sds
