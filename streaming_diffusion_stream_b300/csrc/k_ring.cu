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
#include "rope.cuh"
#include "sds_internal.h"

namespace sds {
namespace {

constexpr int kRingThreads = 256;

__global__ void __launch_bounds__(kRingThreads) kv_push_kernel(const PushParams p) {
  const int64_t vpr = p.HD / 8;  // vectors per token row
  const int64_t TL = p.T * p.L;
  const int64_t total = p.S * TL * vpr;
  const int64_t kv_rows = (p.M + p.R) * p.L;
  const int seg[3] = {p.rope_seg[0], p.rope_seg[1], p.rope_seg[2]};
  const int off[3] = {p.tab_off[0], p.tab_off[1], p.tab_off[2]};
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t vr = i % vpr;
    const int64_t row = i / vpr;
    const int64_t tok = row % TL, s = row / TL;
    const int64_t j = tok / p.L, l = tok % p.L;
    const int64_t slot = (p.F + j) % p.R;
    const int64_t dst = (s * kv_rows + (p.M + slot) * p.L + l) * vpr + vr;
    uint4 kv = __ldcs(p.k_in + i);
    const uint4 vv = __ldcs(p.v_in + i);
    if (p.rope_on) {
      const int pos[3] = {p.p0 + (int)j, (int)(l / p.grid_w), (int)(l % p.grid_w)};
      const int e0 = (int)((vr * 8) % p.head_dim);
      kv = rope8(kv, e0, pos, seg, p.rope_tab, off);
    }
    p.kv_k[dst] = kv;
    p.kv_v[dst] = vv;
  }
}

__device__ __forceinline__ double warp_sum(double v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Fixed-order block sum (valid in every thread after return).
__device__ double block_sum_all(double v, double* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double r = 0.0;
  for (int w = 0; w < kRingThreads / 32; ++w) r += red[w];
  __syncthreads();
  return r;
}

// Copy one frame (L tokens of all heads, K and V) between rows of a stream's
// K/V buffer; this block's share of the vectors.
__device__ void copy_frame(const SinkParams& p, int64_t s, int64_t src_row0, int64_t dst_row0) {
  const int64_t vpr = p.HD / 8;
  const int64_t kv_rows = (p.M + p.R) * p.L;
  const int64_t n = p.L * vpr;
  const int64_t src = (s * kv_rows + src_row0) * vpr, dst = (s * kv_rows + dst_row0) * vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    p.kv_k[dst + i] = p.kv_k[src + i];
    p.kv_v[dst + i] = p.kv_v[src + i];
  }
}

// grid (blocks, S).  Fill mode copies frames of the chunk into empty sinks.
// Test mode: every block takes the same decision from the same data (fixed
// reduction order), copies its share when it fires, and the block that
// finishes last for the stream updates the embedding and the record -- so
// no block can read an embedding another block already replaced.
__global__ void __launch_bounds__(kRingThreads) sink_kernel(const SinkParams p) {
  __shared__ double red[kRingThreads / 32];
  __shared__ int last;
  const int64_t s = blockIdx.y;
  const float* h = p.h + s * p.D;
  DevState* st = p.state + s;
  if (p.fill_from >= 0) {
    for (int64_t q = 0; q < p.fill_count; ++q) {
      const int64_t slot = (p.chunk_first + q) % p.R;
      copy_frame(p, s, (p.M + slot) * p.L, (p.fill_from + q) * p.L);
    }
    if (blockIdx.x == 0) {
      for (int64_t q = 0; q < p.fill_count; ++q)
        for (int64_t t = threadIdx.x; t < p.D; t += blockDim.x)
          p.emb[(s * p.M + p.fill_from + q) * p.D + t] = h[t];
      if (threadIdx.x == 0) {
        st->pub.sink_j = p.fill_from;
        st->pub.sink_fire = 2;
        st->pub.sink_alpha_min = __longlong_as_double(0x7FF0000000000000ll);
        st->pub.sink_alpha_2 = __longlong_as_double(0x7FF0000000000000ll);
      }
    }
    return;
  }
  double hn = 0.0;
  for (int64_t t = threadIdx.x; t < p.D; t += blockDim.x) hn += (double)h[t] * (double)h[t];
  hn = block_sum_all(hn, red);
  int64_t jstar = -1;
  double amin = __longlong_as_double(0x7FF0000000000000ll), a2 = amin;
  for (int64_t j = 0; j < p.M; ++j) {
    const float* e = p.emb + (s * p.M + j) * p.D;
    double dot = 0.0, en = 0.0;
    for (int64_t t = threadIdx.x; t < p.D; t += blockDim.x) {
      const double ev = (double)e[t];
      dot += (double)h[t] * ev;
      en += ev * ev;
    }
    dot = block_sum_all(dot, red);
    en = block_sum_all(en, red);
    const double a = (hn > 0.0 && en > 0.0) ? dot / sqrt(hn * en) : 0.0;
    if (a < amin) {
      a2 = amin;
      amin = a;
      jstar = j;
    } else if (a < a2) {
      a2 = a;
    }
  }
  const bool fire = amin < p.s_th;
  if (fire) {
    const int64_t slot = p.chunk_first % p.R;
    copy_frame(p, s, (p.M + slot) * p.L, jstar * p.L);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    last = (atomicAdd(p.counters + s, 1u) == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (fire)
    for (int64_t t = threadIdx.x; t < p.D; t += blockDim.x) p.emb[(s * p.M + jstar) * p.D + t] = h[t];
  if (threadIdx.x == 0) {
    st->pub.sink_j = jstar;
    st->pub.sink_fire = fire ? 1 : 0;
    st->pub.sink_alpha_min = amin;
    st->pub.sink_alpha_2 = a2;
    p.counters[s] = 0u;
    __threadfence();
  }
}

}  // namespace

cudaError_t launch_kv_push(const PushParams& p, int sm_count, cudaStream_t st) {
  const int64_t total = p.S * p.T * p.L * (p.HD / 8);
  int64_t blocks = (total + kRingThreads - 1) / kRingThreads;
  const int64_t cap = (int64_t)sm_count * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  kv_push_kernel<<<(int)blocks, kRingThreads, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_sink_refresh(const SinkParams& p, int sm_count, cudaStream_t st) {
  const int64_t vecs = p.L * (p.HD / 8);
  int64_t bx = (vecs + kRingThreads - 1) / kRingThreads;
  int64_t cap = ((int64_t)sm_count * 4 + p.S - 1) / p.S;
  if (bx > cap) bx = cap;
  if (bx < 1) bx = 1;
  dim3 grid((unsigned)bx, (unsigned)p.S);
  sink_kernel<<<grid, kRingThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sds
