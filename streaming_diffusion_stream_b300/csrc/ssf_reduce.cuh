// ssf_reduce.cuh -- the similarity filter's reduction and decision, one
// definition for every kernel that takes it (K4's filter segment and the
// allocation-free entry point), so that they return bit-identical cosines,
// probabilities and skip decisions for the same frame and reference.
//
// StreamDiffusion notes, "Stochastic Similarity Filter": S_C is the cosine
// of the incoming frame I and the reference frame R, and P(skip) =
// max{0, (S_C - eta) / (1 - eta)}, sampled against a uniform draw; the
// overview page caps consecutive skips at max_skip_frame.
//
// Order of the sums (fixed, so results are deterministic): a work block of
// kRedBlockElems elements gives each of its kStepThreads threads kRedVec
// float4 of I and of R, consecutive threads on consecutive float4; a
// thread sums fp32 products over two float4 (8 elements) at a time and
// adds each such 8-element sum to a compensated fp32 pair; the block adds
// the pairs by a butterfly in each warp and then the warps in index order,
// and converts to double once per block.  The per-block partials of one
// quantity are then summed in double by one warp, lane-strided, and a
// butterfly.  dot, |I|^2 and |R|^2 follow one operation sequence, so I == R
// gives three bitwise-equal sums, cosine 1.0 and P 1.0.
#pragma once

#include "dfloat.cuh"
#include "sds_internal.h"

namespace sds {

constexpr int kRedVec = kRedBlockElems / (kStepThreads * 4);  // float4 per thread per array
constexpr int kRedWarps = kStepThreads / 32;

// The thread's share of dot, |I|^2 and |R|^2 over its kRedVec float4 of I (a)
// and R (r); elements past the frame's end must be loaded as zeros.
__device__ __forceinline__ void ssf_accumulate(const float4 (&a)[kRedVec], const float4 (&r)[kRedVec],
                                               dfloat& sd, dfloat& si, dfloat& sr) {
  sd = df_make(0.f);
  si = df_make(0.f);
  sr = df_make(0.f);
#pragma unroll
  for (int k = 0; k < kRedVec; k += 2) {
    float dot = 0.f, ni = 0.f, nr = 0.f;
#pragma unroll
    for (int k2 = k; k2 < k + 2; ++k2) {
      const float4 x = a[k2], y = r[k2];
      dot = __fmaf_rn(x.x, y.x, dot); ni = __fmaf_rn(x.x, x.x, ni); nr = __fmaf_rn(y.x, y.x, nr);
      dot = __fmaf_rn(x.y, y.y, dot); ni = __fmaf_rn(x.y, x.y, ni); nr = __fmaf_rn(y.y, y.y, nr);
      dot = __fmaf_rn(x.z, y.z, dot); ni = __fmaf_rn(x.z, x.z, ni); nr = __fmaf_rn(y.z, y.z, nr);
      dot = __fmaf_rn(x.w, y.w, dot); ni = __fmaf_rn(x.w, x.w, ni); nr = __fmaf_rn(y.w, y.w, nr);
    }
    sd = df_add(sd, df_make(dot));
    si = df_add(si, df_make(ni));
    sr = df_add(sr, df_make(nr));
  }
}

// Block-wide fixed-order sums of three compensated values per thread
// (butterfly within each warp, then the warps in index order); the results
// are valid in thread 0.  red: 3 * kRedWarps entries of shared memory.
__device__ __forceinline__ void block_sum3(dfloat& a, dfloat& b, dfloat& c, dfloat* red) {
  a = df_warp_sum(a);
  b = df_warp_sum(b);
  c = df_warp_sum(c);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    red[warp] = a;
    red[kRedWarps + warp] = b;
    red[2 * kRedWarps + warp] = c;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a = red[0];
    b = red[kRedWarps];
    c = red[2 * kRedWarps];
    for (int w = 1; w < kRedWarps; ++w) {
      a = df_add(a, red[w]);
      b = df_add(b, red[kRedWarps + w]);
      c = df_add(c, red[2 * kRedWarps + w]);
    }
  }
  __syncthreads();
}

__device__ __forceinline__ double warp_sum_f64(double v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// One warp's fixed-order double sum of n partials base[0], base[stride], ...:
// lane-strided, then a butterfly (every lane ends with the same bits).
__device__ __forceinline__ double partials_sum(const double* base, int64_t n, int64_t stride, int lane) {
  double v = 0.0;
  for (int64_t i = lane; i < n; i += 32) v += __ldcg(base + i * stride);
  return warp_sum_f64(v);
}

// The filter's decision from the reduced sums: cosine (0 if a norm is 0),
// skip probability and skip = (u < P) and (count < max_skip).
__device__ __forceinline__ int64_t ssf_decision(double dot, double ni, double nr, double eta, double u,
                                                int64_t count, int64_t max_skip, double& cosv,
                                                double& P) {
  cosv = (ni > 0.0 && nr > 0.0) ? dot / sqrt(ni * nr) : 0.0;
  P = fmin(1.0, fmax(0.0, (cosv - eta) / (1.0 - eta)));
  return (u < P && count < max_skip) ? 1 : 0;
}

}  // namespace sds
