// k_step.cu -- K4: one fused, HBM-streaming pass over three disjoint
// segments, finished by the last block of the launch.
//
//  (i)  StreamDiffusion notes, "Residual CFG (R-CFG)": the self-negative
//       virtual noise eps_neg = (x - sqrt(abar) x0) / sqrt(1 - abar) and the
//       combine delta*eps_neg + gamma*(eps_c - delta*eps_neg), evaluated as
//       gamma*eps_c + delta*(1-gamma)*eps_neg; then the stream-batch update
//       (StreamDiffusion notes, "Stream Batch"; blog section 7's ancestral
//       step read as predict-x0-then-re-noise): x0hat, re-noise to the next
//       slot's level with the supplied z, and noise the incoming frame into
//       slot 0.  Slots are visited last-to-first so x_next may alias x.
//  (ii) StreamDiffusion notes, "Stochastic Similarity Filter": dot and norm
//       sums of the incoming frame against the reference frame; the frame is
//       also copied into the spare reference buffer, which becomes current
//       when the frame is processed.
//  (iii) StreamDiffusionV2 summary, "Motion-aware noise scheduler": sums of
//       squared differences of consecutive latent frames.
//
// Reductions are deterministic: every work block (2048 elements) reduces in
// a fixed order (fp32 over the thread's 8 elements, double beyond), writes
// one partial per quantity, and the block that finishes last sums the
// partials in index order in double and takes the decisions.  dot, |I|^2 and
// |R|^2 use the same operation sequence, so identical frames give three
// bitwise-equal sums, cosine exactly 1 and skip probability exactly 1.
#include "sds_internal.h"

namespace sds {
namespace {

__device__ __forceinline__ double warp_sum(double v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

constexpr int kWarps = kStepThreads / 32;

// Block-wide fixed-order sum of one double per thread; result valid in thread 0.
__device__ __forceinline__ double block_sum(double v, double* red) {
  v = warp_sum(v);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = v;
  __syncthreads();
  double r = 0.0;
  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w) r += red[w];
  }
  __syncthreads();
  return r;
}

__device__ __forceinline__ float4 ld4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st4(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

__device__ __forceinline__ float x0hat1(float x, float x0, float ec, float sa, float inv_s1a,
                                        float s1a, float inv_sa, float g, float dg) {
  const float en = __fmaf_rn(-sa, x0, x) * inv_s1a;
  const float ecfg = __fmaf_rn(g, ec, dg * en);
  return __fmaf_rn(-s1a, ecfg, x) * inv_sa;
}

__device__ __forceinline__ float4 x0hat4(float4 x, float4 x0, float4 ec, const StepParams& p,
                                         int i) {
  const float sa = p.c_sa[i], a = p.c_inv_s1a[i], b = p.c_s1a[i], c = p.c_inv_sa[i];
  return make_float4(x0hat1(x.x, x0.x, ec.x, sa, a, b, c, p.c_gamma, p.c_dg),
                     x0hat1(x.y, x0.y, ec.y, sa, a, b, c, p.c_gamma, p.c_dg),
                     x0hat1(x.z, x0.z, ec.z, sa, a, b, c, p.c_gamma, p.c_dg),
                     x0hat1(x.w, x0.w, ec.w, sa, a, b, c, p.c_gamma, p.c_dg));
}

__device__ __forceinline__ float4 noise4(float4 a, float4 b, float ca, float cb) {
  return make_float4(__fmaf_rn(ca, a.x, cb * b.x), __fmaf_rn(ca, a.y, cb * b.y),
                     __fmaf_rn(ca, a.z, cb * b.z), __fmaf_rn(ca, a.w, cb * b.w));
}

__device__ void update_block(const StepParams& p, int64_t w) {
  const int64_t s = w / p.nb_u, b = w % p.nb_u;
  const int64_t sbase = s * p.N_s;
  for (int k = 0; k < 2; ++k) {
    const int64_t el = b * kStepBlockElems + k * (kStepThreads * 4) + threadIdx.x * 4;
    if (el >= p.N_s) continue;
    const int64_t e = sbase + el;
    for (int i = p.n - 1; i >= 0; --i) {
      const float4 xh = x0hat4(ld4(p.x[i] + e), ld4(p.x0[i] + e), ld4(p.eps_c[i] + e), p, i);
      if (i == p.n - 1) {
        st4(p.out + e, xh);
      } else {
        st4(p.x_next[i + 1] + e, noise4(xh, ld4(p.z[i] + e), p.c_sa[i + 1], p.c_s1a[i + 1]));
      }
    }
    st4(p.x_next[0] + e, noise4(ld4(p.x0_new + e), ld4(p.eps_new + e), p.c_sa[0], p.c_s1a[0]));
  }
}

__device__ void ssf_block(const StepParams& p, int64_t w, double* red) {
  const int64_t s = w / p.nb_s, b = w % p.nb_s;
  const int64_t cur = p.state[s].ssf_cur;
  const float* I = p.ssf_frame + s * p.E;
  const float* R = p.ssf_ref + (cur * p.S + s) * p.E;
  float* Rn = p.ssf_ref + ((cur ^ 1) * p.S + s) * p.E;
  float dot = 0.f, ni = 0.f, nr = 0.f;
  for (int k = 0; k < 2; ++k) {
    const int64_t e = b * kStepBlockElems + k * (kStepThreads * 4) + threadIdx.x * 4;
    if (e >= p.E) continue;
    const float4 a = ld4(I + e), r = ld4(R + e);
    st4(Rn + e, a);
    dot = __fmaf_rn(a.x, r.x, dot); ni = __fmaf_rn(a.x, a.x, ni); nr = __fmaf_rn(r.x, r.x, nr);
    dot = __fmaf_rn(a.y, r.y, dot); ni = __fmaf_rn(a.y, a.y, ni); nr = __fmaf_rn(r.y, r.y, nr);
    dot = __fmaf_rn(a.z, r.z, dot); ni = __fmaf_rn(a.z, a.z, ni); nr = __fmaf_rn(r.z, r.z, nr);
    dot = __fmaf_rn(a.w, r.w, dot); ni = __fmaf_rn(a.w, a.w, ni); nr = __fmaf_rn(r.w, r.w, nr);
  }
  const double sd = block_sum((double)dot, red);
  const double si = block_sum((double)ni, red);
  const double sr = block_sum((double)nr, red);
  if (threadIdx.x == 0) {
    double* part = p.partials + (s * p.nb_s + b) * 3;
    part[0] = sd;
    part[1] = si;
    part[2] = sr;
  }
}

__device__ void motion_block(const StepParams& p, int64_t w, double* red) {
  const int64_t per_s = p.T * p.nb_m;
  const int64_t s = w / per_s, rem = w % per_s, j = rem / p.nb_m, b = rem % p.nb_m;
  const float* B = p.mot_chunk + (s * p.T + j) * p.N_f;
  const float* A = nullptr;
  if (j > 0) {
    A = p.mot_chunk + (s * p.T + j - 1) * p.N_f;
  } else if (p.state[s].mot_has_prev) {
    A = p.mot_prev_in + s * p.N_f;
  }
  float acc = 0.f;
  for (int k = 0; k < 2; ++k) {
    const int64_t e = b * kStepBlockElems + k * (kStepThreads * 4) + threadIdx.x * 4;
    if (e >= p.N_f) continue;
    const float4 bv = ld4(B + e);
    if (j == p.T - 1) st4(p.mot_prev_out + s * p.N_f + e, bv);
    if (A) {
      const float4 av = ld4(A + e);
      const float dx = bv.x - av.x, dy = bv.y - av.y, dz = bv.z - av.z, dw = bv.w - av.w;
      acc = __fmaf_rn(dx, dx, acc);
      acc = __fmaf_rn(dy, dy, acc);
      acc = __fmaf_rn(dz, dz, acc);
      acc = __fmaf_rn(dw, dw, acc);
    }
  }
  const double sa = block_sum((double)acc, red);
  if (threadIdx.x == 0) p.partials[p.S * p.nb_s * 3 + (s * p.T + j) * p.nb_m + b] = sa;
}

// Fixed-order sum of n partials at stride `stride` (thread-strided, then block tree).
__device__ double sum_partials(const double* base, int64_t n, int64_t stride, double* red) {
  double v = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += kStepThreads) v += __ldcg(base + i * stride);
  return block_sum(v, red);
}

__device__ void finalize(const StepParams& p, double* red) {
  for (int64_t s = 0; s < p.S; ++s) {
    DevState* st = p.state + s;
    if (p.ssf_frame) {
      const double* base = p.partials + s * p.nb_s * 3;
      const double dot = sum_partials(base + 0, p.nb_s, 3, red);
      const double ni = sum_partials(base + 1, p.nb_s, 3, red);
      const double nr = sum_partials(base + 2, p.nb_s, 3, red);
      if (threadIdx.x == 0) {
        double cosv = 0.0, P = 0.0;
        int64_t skip = 0;
        if (st->pub.ssf_has_ref) {
          cosv = (ni > 0.0 && nr > 0.0) ? dot / sqrt(ni * nr) : 0.0;
          P = fmin(1.0, fmax(0.0, (cosv - p.eta) / (1.0 - p.eta)));
          const double u = (double)__ldcg(p.ssf_u + s);
          skip = (u < P && st->pub.ssf_skip_count < p.max_skip) ? 1 : 0;
        }
        if (skip) {
          st->pub.ssf_skip_count += 1;
        } else {
          st->pub.ssf_skip_count = 0;
          st->ssf_cur ^= 1;
          st->pub.ssf_has_ref = 1;
        }
        st->pub.ssf_skip = skip;
        st->pub.ssf_cos = cosv;
        st->pub.ssf_p = P;
        st->pub.ssf_evals += 1;
      }
    }
    if (p.mot_chunk) {
      const double* base = p.partials + p.S * p.nb_s * 3 + s * p.T * p.nb_m;
      for (int64_t j = 0; j < p.T; ++j) {
        const double sq = sum_partials(base + j * p.nb_m, p.nb_m, 1, red);
        if (threadIdx.x == 0) {
          const bool present = (j > 0) || (st->mot_has_prev != 0);
          double dv = __longlong_as_double(0x7FF8000000000000ll);  // NaN: pair absent
          if (present) {
            dv = sqrt(sq / (double)p.N_f);
            st->mot_window[st->mot_head] = dv;
            st->mot_head = (st->mot_head + 1) % p.mot_k;
            if (st->mot_count < p.mot_k) st->mot_count += 1;
            st->pub.motion_pairs += 1;
          }
          if (j < SDS_MAX_CHUNK_FRAMES) st->pub.motion_d[j] = dv;
        }
      }
      if (threadIdx.x == 0) {
        for (int64_t j = p.T; j < SDS_MAX_CHUNK_FRAMES; ++j)
          st->pub.motion_d[j] = __longlong_as_double(0x7FF8000000000000ll);
        if (st->mot_count > 0) {
          double mx = 0.0;
          for (int64_t q = 0; q < st->mot_count; ++q) mx = fmax(mx, st->mot_window[q]);
          const double dhat = fmin(1.0, mx / p.sigma);
          const double target = p.s_min + (p.s_max - p.s_min) * dhat;
          st->pub.noise_rate = st->pub.noise_rate + (1.0 - p.lam) * (target - st->pub.noise_rate);
          st->pub.motion_dhat = dhat;
        }
        st->mot_has_prev = 1;
      }
    }
  }
}

__global__ void __launch_bounds__(kStepThreads) step_kernel(const StepParams p) {
  __shared__ double red[kWarps];
  __shared__ int is_last;
  const int64_t tot_u = p.n > 0 ? p.S * p.nb_u : 0;
  const int64_t tot_s = p.ssf_frame ? p.S * p.nb_s : 0;
  const int64_t tot_m = p.mot_chunk ? p.S * p.T * p.nb_m : 0;
  const int64_t total = tot_u + tot_s + tot_m;
  for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
    if (w < tot_u) {
      update_block(p, w);
    } else if (w < tot_u + tot_s) {
      ssf_block(p, w - tot_u, red);
    } else {
      motion_block(p, w - tot_u - tot_s, red);
    }
  }
  if (tot_s + tot_m == 0) return;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned int prev = atomicAdd(p.counter, 1u);
    is_last = (prev == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  finalize(p, red);
  if (threadIdx.x == 0) {
    *p.counter = 0u;
    __threadfence();
  }
}

}  // namespace

cudaError_t launch_step(const StepParams& p, int sm_count, cudaStream_t st) {
  const int64_t tot = (p.n > 0 ? p.S * p.nb_u : 0) + (p.ssf_frame ? p.S * p.nb_s : 0) +
                      (p.mot_chunk ? p.S * p.T * p.nb_m : 0);
  if (tot == 0) return cudaSuccess;
  const int64_t cap = (int64_t)sm_count * (2048 / kStepThreads);
  const int grid = (int)(tot < cap ? tot : cap);
  step_kernel<<<grid, kStepThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace sds
