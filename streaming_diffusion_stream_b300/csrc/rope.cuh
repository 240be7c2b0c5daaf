// rope.cuh -- 3-axis rotary position embedding on 8 packed bf16 values.
//
// StreamDiffusionV2 summary, "Adaptive sink and RoPE refresh": keys are
// cached with the rotation of their position and the phase is reset once the
// position exceeds a threshold.  The head dim is split into temporal, row
// and column segments (widths seg[0..2]); pair (2i, 2i+1) of a segment turns
// by pos * base^(-2i/width).  The cos/sin values come from a host-built
// table: tab[off[a] + pos * (seg[a]/2) + i] = (cos, sin).
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

namespace sds {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t rope_pair(uint32_t w, int pair, const int pos[3],
                                              const int seg[3], const float2* tab,
                                              const int off[3]) {
  const int h0 = seg[0] >> 1, h1 = (seg[0] + seg[1]) >> 1;
  // select the axis without indexing the small arrays dynamically (keeps
  // them in registers)
  const bool a0 = pair < h0, a1 = !a0 && pair < h1;
  const int i = a0 ? pair : (a1 ? pair - h0 : pair - h1);
  const int base = a0 ? off[0] + pos[0] * h0
                      : (a1 ? off[1] + pos[1] * (seg[1] >> 1) : off[2] + pos[2] * (seg[2] >> 1));
  const float2 cs = tab[base + i];
  const float u = bf16_lo(w), v = bf16_hi(w);
  const float r0 = __fmaf_rn(u, cs.x, -v * cs.y);
  const float r1 = __fmaf_rn(u, cs.y, v * cs.x);
  __nv_bfloat162 out = __floats2bfloat162_rn(r0, r1);  // .x -> low half
  return *reinterpret_cast<uint32_t*>(&out);
}

// Rotate 8 consecutive head-dim elements e0..e0+7 (e0 even) held in v.
__device__ __forceinline__ uint4 rope8(uint4 v, int e0, const int pos[3], const int seg[3],
                                       const float2* tab, const int off[3]) {
  const int p = e0 >> 1;
  v.x = rope_pair(v.x, p + 0, pos, seg, tab, off);
  v.y = rope_pair(v.y, p + 1, pos, seg, tab, off);
  v.z = rope_pair(v.z, p + 2, pos, seg, tab, off);
  v.w = rope_pair(v.w, p + 3, pos, seg, tab, off);
  return v;
}

// Rotate 8 consecutive elements (4 pairs) with the pairs' (cos, sin) given.
__device__ __forceinline__ uint32_t rope_pair_cs(uint32_t w, float2 cs) {
  const float u = bf16_lo(w), v = bf16_hi(w);
  const float r0 = __fmaf_rn(u, cs.x, -v * cs.y);
  const float r1 = __fmaf_rn(u, cs.y, v * cs.x);
  __nv_bfloat162 out = __floats2bfloat162_rn(r0, r1);
  return *reinterpret_cast<uint32_t*>(&out);
}

__device__ __forceinline__ uint4 rope8_cs(uint4 v, const float2 (&cs)[4]) {
  v.x = rope_pair_cs(v.x, cs[0]);
  v.y = rope_pair_cs(v.y, cs[1]);
  v.z = rope_pair_cs(v.z, cs[2]);
  v.w = rope_pair_cs(v.w, cs[3]);
  return v;
}

}  // namespace sds
