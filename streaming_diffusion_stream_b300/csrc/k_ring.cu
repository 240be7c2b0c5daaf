// k_ring.cu -- K2 (ring append with RoPE) and K3 (adaptive sink refresh).
//
// StreamDiffusionV2 summary, "Adaptive sink and RoPE refresh" and its
// rolling KV cache: the newest chunk's keys are rotated at their positions
// and written over the oldest ring frames; the least similar sink is
// replaced when its cosine to the new chunk embedding falls below s_th.
//
// Both kernels stream 16-byte vectors with consecutive threads on
// consecutive addresses; there is no shared-memory staging because every
// byte is read once and written once.
#include "dfloat.cuh"
#include "rope.cuh"
#include "sds_internal.h"

namespace sds {
namespace {

constexpr int kRingThreads = 256;
constexpr int kDecideThreads = 512;  // one block per stream takes the sink decision
constexpr int kPushX = 64;  // threads along a token row (a multiple of head_dim / 8)
constexpr int kPushY = 4;   // token rows per block

// One block of kPushX x kPushY threads moves kPushY token rows at a time
// (grid-stride over the S*T*L rows of the chunk).  Thread x of a row handles
// vectors x, x + 64, x + 128, ... of the row; since 64 is a multiple of the
// eight-element vectors per head, all of them sit at the same offset inside
// their heads and share one set of RoPE (cos, sin) pairs, which the thread
// fetches once per row.  Index arithmetic is 32-bit per row.
__global__ void __launch_bounds__(kPushX * kPushY) kv_push_kernel(const PushParams p) {
  const int vpr = (int)(p.HD / 8);  // vectors per token row
  const int TL = (int)(p.T * p.L);
  const int64_t rows = p.S * TL;
  const int64_t kv_rows = (p.M + p.R) * p.L;
  const int x = threadIdx.x;
  for (int64_t row = (int64_t)blockIdx.x * kPushY + threadIdx.y; row < rows;
       row += (int64_t)gridDim.x * kPushY) {
    const int s = (int)(row / TL);
    const int tok = (int)(row - (int64_t)s * TL);
    const int j = tok / (int)p.L, l = tok - j * (int)p.L;
    const int64_t slot = (p.F + j) % p.R;
    const uint4* kin = p.k_in + row * vpr;
    const uint4* vin = p.v_in + row * vpr;
    uint4* kout = p.kv_k + ((int64_t)s * kv_rows + (p.M + slot) * p.L + l) * vpr;
    uint4* vout = p.kv_v + ((int64_t)s * kv_rows + (p.M + slot) * p.L + l) * vpr;
    float2 cs[4];
    if (p.rope_on) {
      const int pos[3] = {p.p0 + j, l / p.grid_w, l % p.grid_w};
      const int h0 = p.rope_seg[0] >> 1, h1 = (p.rope_seg[0] + p.rope_seg[1]) >> 1;
      const int pair0 = (int)(((int64_t)x * 8 % p.head_dim) >> 1);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int pair = pair0 + q;
        const bool a0 = pair < h0, a1 = !a0 && pair < h1;
        const int i = a0 ? pair : (a1 ? pair - h0 : pair - h1);
        const int base = a0 ? p.tab_off[0] + pos[0] * h0
                            : (a1 ? p.tab_off[1] + pos[1] * (p.rope_seg[1] >> 1)
                                  : p.tab_off[2] + pos[2] * (p.rope_seg[2] >> 1));
        cs[q] = p.rope_tab[base + i];
      }
    }
    int v = x;
    for (; v + kPushX < vpr; v += 2 * kPushX) {
      uint4 k0 = __ldcs(kin + v), k1 = __ldcs(kin + v + kPushX);
      const uint4 v0 = __ldcs(vin + v), v1 = __ldcs(vin + v + kPushX);
      if (p.rope_on) {
        k0 = rope8_cs(k0, cs);
        k1 = rope8_cs(k1, cs);
      }
      kout[v] = k0;
      kout[v + kPushX] = k1;
      vout[v] = v0;
      vout[v + kPushX] = v1;
    }
    if (v < vpr) {
      uint4 k0 = __ldcs(kin + v);
      const uint4 v0 = __ldcs(vin + v);
      if (p.rope_on) k0 = rope8_cs(k0, cs);
      kout[v] = k0;
      vout[v] = v0;
    }
  }
}

// Fixed-order block sum of one compensated value per thread: a butterfly
// in each warp, then thread 0 adds the warps in index order and converts
// to double once; the result is returned to every thread.
__device__ double block_sum_df(dfloat v, dfloat* red, double* out) {
  v = df_warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    dfloat t = red[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) t = df_add(t, red[w]);
    *out = df_to_double(t);
  }
  __syncthreads();
  return *out;
}

// Copy one frame (L tokens of all heads, K and V) between rows of a stream's
// K/V buffer; this block's share of the vectors, four loads in flight per
// thread before the stores.
__device__ void copy_frame(const SinkParams& p, int64_t s, int64_t src_row0, int64_t dst_row0) {
  const int64_t vpr = p.HD / 8;
  const int64_t kv_rows = (p.M + p.R) * p.L;
  const int64_t n = p.L * vpr;
  const int64_t src = (s * kv_rows + src_row0) * vpr, dst = (s * kv_rows + dst_row0) * vpr;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + stride < n; i += 2 * stride) {
    const uint4 k0 = p.kv_k[src + i], k1 = p.kv_k[src + i + stride];
    const uint4 v0 = p.kv_v[src + i], v1 = p.kv_v[src + i + stride];
    p.kv_k[dst + i] = k0;
    p.kv_k[dst + i + stride] = k1;
    p.kv_v[dst + i] = v0;
    p.kv_v[dst + i + stride] = v1;
  }
  if (i < n) {
    const uint4 k0 = p.kv_k[src + i], v0 = p.kv_v[src + i];
    p.kv_k[dst + i] = k0;
    p.kv_v[dst + i] = v0;
  }
}

// K3a, the decision: grid (S), one block per stream.  Fill mode: the
// record says which sinks the chunk fills (the copy kernel copies them).
// Test mode: alpha_j = cos(h, e_j) from exact fp32 products summed as
// compensated fp32 pairs (fp64 is slow on this part) and a block tree
// finished in double, j* = argmin (lowest index on ties), fire iff
// alpha_{j*} < s_th; the record and, on fire, the sink embedding are
// updated here.  The copy kernel reads the record, so only one block per
// stream does this work however many blocks copy.
__global__ void __launch_bounds__(kDecideThreads) sink_decide_kernel(const SinkParams p) {
  __shared__ dfloat red[kDecideThreads / 32];
  __shared__ double bcast;
  __shared__ int64_t dec_j;
  __shared__ int dec_fire;
  const int64_t s = blockIdx.x;
  const float* h = p.h + s * p.D;
  DevState* st = p.state + s;
  if (p.fill_from >= 0) {
    for (int64_t q = 0; q < p.fill_count; ++q)
      for (int64_t t = threadIdx.x; t < p.D; t += blockDim.x)
        p.emb[(s * p.M + p.fill_from + q) * p.D + t] = h[t];
    if (threadIdx.x == 0) {
      st->pub.sink_j = p.fill_from;
      st->pub.sink_fire = 2;
      st->pub.sink_alpha_min = __longlong_as_double(0x7FF0000000000000ll);
      st->pub.sink_alpha_2 = __longlong_as_double(0x7FF0000000000000ll);
    }
    return;
  }
  // One pass per sink over h and e_j: dot_j = h.e_j, en_j = e_j.e_j, and,
  // with the first sink, hn = h.h.  Each thread takes 4 consecutive
  // elements per step and issues the loads of two steps before it uses them,
  // so the memory round trips overlap instead of following each other.
  const bool vec = (p.D % 4 == 0) && ((reinterpret_cast<uintptr_t>(h) & 15u) == 0) &&
                   ((reinterpret_cast<uintptr_t>(p.emb) & 15u) == 0);
  double hn = 0.0;
  int64_t jstar = -1;
  double amin = __longlong_as_double(0x7FF0000000000000ll), a2 = amin;
  for (int64_t j = 0; j < p.M; ++j) {
    const float* e = p.emb + (s * p.M + j) * p.D;
    dfloat dot_t = df_make(0.f), en_t = df_make(0.f), hn_t = df_make(0.f);
    const bool with_hn = j == 0;
    if (vec) {
      const int64_t stride = (int64_t)blockDim.x * 4;
      int64_t t = (int64_t)threadIdx.x * 4;
      for (; t + stride < p.D; t += 2 * stride) {
        const float4 h0 = __ldg(reinterpret_cast<const float4*>(h + t));
        const float4 e0 = __ldcg(reinterpret_cast<const float4*>(e + t));
        const float4 h1 = __ldg(reinterpret_cast<const float4*>(h + t + stride));
        const float4 e1 = __ldcg(reinterpret_cast<const float4*>(e + t + stride));
        const float hv[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
        const float ev[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          dot_t = df_add(dot_t, df_prod(hv[q], ev[q]));
          en_t = df_add(en_t, df_prod(ev[q], ev[q]));
          if (with_hn) hn_t = df_add(hn_t, df_prod(hv[q], hv[q]));
        }
      }
      if (t < p.D) {
        const float4 h0 = __ldg(reinterpret_cast<const float4*>(h + t));
        const float4 e0 = __ldcg(reinterpret_cast<const float4*>(e + t));
        const float hv[4] = {h0.x, h0.y, h0.z, h0.w};
        const float ev[4] = {e0.x, e0.y, e0.z, e0.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dot_t = df_add(dot_t, df_prod(hv[q], ev[q]));
          en_t = df_add(en_t, df_prod(ev[q], ev[q]));
          if (with_hn) hn_t = df_add(hn_t, df_prod(hv[q], hv[q]));
        }
      }
    } else {
      for (int64_t t = threadIdx.x; t < p.D; t += blockDim.x) {
        const float hv = h[t], ev = e[t];
        dot_t = df_add(dot_t, df_prod(hv, ev));
        en_t = df_add(en_t, df_prod(ev, ev));
        if (with_hn) hn_t = df_add(hn_t, df_prod(hv, hv));
      }
    }
    if (with_hn) hn = block_sum_df(hn_t, red, &bcast);
    const double dot = block_sum_df(dot_t, red, &bcast);
    const double en = block_sum_df(en_t, red, &bcast);
    if (threadIdx.x == 0) {
      const double a = (hn > 0.0 && en > 0.0) ? dot / sqrt(hn * en) : 0.0;
      if (a < amin) {
        a2 = amin;
        amin = a;
        jstar = j;
      } else if (a < a2) {
        a2 = a;
      }
    }
  }
  if (threadIdx.x == 0) {
    dec_j = jstar;
    dec_fire = amin < p.s_th ? 1 : 0;
    st->pub.sink_j = jstar;
    st->pub.sink_fire = dec_fire;
    st->pub.sink_alpha_min = amin;
    st->pub.sink_alpha_2 = a2;
  }
  __syncthreads();
  if (dec_fire)
    for (int64_t t = threadIdx.x; t < p.D; t += blockDim.x) p.emb[(s * p.M + dec_j) * p.D + t] = h[t];
}

// K3b, the copy: grid (blocks, S).  Fill mode copies frames 0.. of the chunk
// just pushed into the empty sinks; test mode copies frame 0 into sink j*
// when the decision kernel's record says it fires, and otherwise exits.
__global__ void __launch_bounds__(kRingThreads) sink_copy_kernel(const SinkParams p) {
  const int64_t s = blockIdx.y;
  if (p.fill_from >= 0) {
    for (int64_t q = 0; q < p.fill_count; ++q) {
      const int64_t slot = (p.chunk_first + q) % p.R;
      copy_frame(p, s, (p.M + slot) * p.L, (p.fill_from + q) * p.L);
    }
    return;
  }
  const DevState* st = p.state + s;
  if (__ldcg(&st->pub.sink_fire) != 1) return;
  const int64_t jstar = __ldcg(&st->pub.sink_j);
  if (jstar < 0 || jstar >= p.M) return;
  const int64_t slot = p.chunk_first % p.R;
  copy_frame(p, s, (p.M + slot) * p.L, jstar * p.L);
}

}  // namespace

cudaError_t launch_kv_push(const PushParams& p, int sm_count, cudaStream_t st) {
  // the thread-to-vector mapping needs the row width to be a multiple of a
  // head and a head to divide the 64-thread row stride
  if (p.HD % 8 != 0 || (p.head_dim != 64 && p.head_dim != 128)) return cudaErrorInvalidValue;
  const int64_t rows = p.S * p.T * p.L;
  int64_t blocks = (rows + kPushY - 1) / kPushY;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  kv_push_kernel<<<(int)blocks, dim3(kPushX, kPushY), 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sink_refresh(const SinkParams& p, int sm_count, cudaStream_t st) {
  sink_decide_kernel<<<(unsigned)p.S, kDecideThreads, 0, st>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t vecs = p.L * (p.HD / 8);
  int64_t bx = (vecs + kRingThreads - 1) / kRingThreads;
  int64_t cap = ((int64_t)sm_count * 4 + p.S - 1) / p.S;
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  dim3 grid((unsigned)bx, (unsigned)p.S);
  sink_copy_kernel<<<grid, kRingThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sds
