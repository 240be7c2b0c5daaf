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
//       slot 0.  All of an element's inputs are loaded before any of its
//       outputs is written, so x_next may alias x.  Variants: a supplied
//       negative prediction in place of the virtual one (the onetime-negative
//       R-CFG, or CFG with delta = 1); the strided DDPM posterior step in
//       place of the re-noise; bf16 noise predictions, widened exactly;
//       txt2img, where the incoming frame is the noise draw itself; and the
//       motion noise rate choosing the incoming frame's entry timestep
//       (StreamDiffusionV2 summary), with slot 0's coefficients then taken
//       from per-timestep tables.
//  (ii) StreamDiffusion notes, "Stochastic Similarity Filter": dot and norm
//       sums of the incoming frame against the reference frame; the frame is
//       also copied into the spare reference buffer, which becomes current
//       when the frame is processed.
//  (iii) StreamDiffusionV2 summary, "Motion-aware noise scheduler": sums of
//       squared differences of consecutive latent frames.
//
// Reductions are deterministic: every work block (8192 elements) reduces in
// a fixed order (fp32 over 8 elements of a thread, compensated fp32 pairs
// across threads, since fp64 is slow on this part) and writes one partial
// per quantity.  Reduction work blocks are scheduled before update work
// blocks; the one that completes the set of partials (an arrival counter)
// sums them in a fixed order in double (one warp per sum) and takes the
// decisions (one warp per stream) while the update streams on.  dot, |I|^2 and
// |R|^2 use the same operation sequence, so identical frames give three
// bitwise-equal sums, cosine exactly 1 and skip probability exactly 1.
#include "dfloat.cuh"
#include "sds_internal.h"
#include "ssf_reduce.cuh"

namespace sds {
namespace {

constexpr int kWarps = kStepThreads / 32;

// Block-wide fixed-order sum of one compensated value per thread (as
// block_sum3 of ssf_reduce.cuh); the result is valid in thread 0.
__device__ __forceinline__ void block_sum1(dfloat& a, dfloat* red) {
  a = df_warp_sum(a);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) red[warp] = a;
  __syncthreads();
  if (threadIdx.x == 0) {
    a = red[0];
    for (int w = 1; w < kWarps; ++w) a = df_add(a, red[w]);
  }
  __syncthreads();
}

__device__ __forceinline__ float4 ld4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ void st4(float* p, float4 v) { __stcs(reinterpret_cast<float4*>(p), v); }

// Four bf16 values at element offset e of a bf16 array, widened exactly.
__device__ __forceinline__ float4 ld4_bf16(const float* base, int64_t e) {
  const uint2 u = __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const uint16_t*>(base) + e));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
}

// Schedule coefficients of one slot's update (see StepParams).
struct SlotCoef {
  float sa, inv_s1a, s1a, inv_sa;  // sqrt(abar), 1/sqrt(1-abar), sqrt(1-abar), 1/sqrt(abar)
  float px, pe, sig;               // strided DDPM step to the next slot
};

__device__ __forceinline__ SlotCoef slot_coef(const StepParams& p, int i) {
  return SlotCoef{p.c_sa[i], p.c_inv_s1a[i], p.c_s1a[i], p.c_inv_sa[i],
                  p.c_px[i], p.c_pe[i], p.c_sig[i]};
}

// eps_cfg = gamma eps_c + delta (1 - gamma) eps_neg with eps_neg the virtual
// residual (x - sqrt(abar) x0) / sqrt(1 - abar) (cfg_kind 1) or the supplied
// prediction (cfg_kind 2); eps_c alone without guidance.
__device__ __forceinline__ float eps_cfg1(float x, float neg, float ec, float sa, float inv_s1a,
                                          float g, float dg, int kind) {
  const float en = kind == 1 ? __fmaf_rn(-sa, neg, x) * inv_s1a : neg;
  return __fmaf_rn(g, ec, dg * en);
}

__device__ __forceinline__ float4 eps_cfg4(float4 x, float4 neg, float4 ec, const StepParams& p,
                                           const SlotCoef& k) {
  if (p.cfg_kind == 0) return ec;
  return make_float4(eps_cfg1(x.x, neg.x, ec.x, k.sa, k.inv_s1a, p.c_gamma, p.c_dg, p.cfg_kind),
                     eps_cfg1(x.y, neg.y, ec.y, k.sa, k.inv_s1a, p.c_gamma, p.c_dg, p.cfg_kind),
                     eps_cfg1(x.z, neg.z, ec.z, k.sa, k.inv_s1a, p.c_gamma, p.c_dg, p.cfg_kind),
                     eps_cfg1(x.w, neg.w, ec.w, k.sa, k.inv_s1a, p.c_gamma, p.c_dg, p.cfg_kind));
}

// x0hat = (x - sqrt(1 - abar) eps_cfg) / sqrt(abar)
__device__ __forceinline__ float4 x0hat4(float4 x, float4 ecfg, const SlotCoef& k) {
  const float b = k.s1a, c = k.inv_sa;
  return make_float4(__fmaf_rn(-b, ecfg.x, x.x) * c, __fmaf_rn(-b, ecfg.y, x.y) * c,
                     __fmaf_rn(-b, ecfg.z, x.z) * c, __fmaf_rn(-b, ecfg.w, x.w) * c);
}

// the strided DDPM step: x / sqrt(alpha) - c_pe eps_cfg + sigma z
__device__ __forceinline__ float4 ddpm4(float4 x, float4 ecfg, float4 z, const SlotCoef& k) {
  const float cx = k.px, ce = k.pe, sg = k.sig;
  return make_float4(__fmaf_rn(sg, z.x, __fmaf_rn(-ce, ecfg.x, cx * x.x)),
                     __fmaf_rn(sg, z.y, __fmaf_rn(-ce, ecfg.y, cx * x.y)),
                     __fmaf_rn(sg, z.z, __fmaf_rn(-ce, ecfg.z, cx * x.z)),
                     __fmaf_rn(sg, z.w, __fmaf_rn(-ce, ecfg.w, cx * x.w)));
}

__device__ __forceinline__ float4 noise4(float4 a, float4 b, float ca, float cb) {
  return make_float4(__fmaf_rn(ca, a.x, cb * b.x), __fmaf_rn(ca, a.y, cb * b.y),
                     __fmaf_rn(ca, a.z, cb * b.z), __fmaf_rn(ca, a.w, cb * b.w));
}

// Coefficients of a slot at timestep t from the per-timestep tables.
__device__ __forceinline__ SlotCoef tab_coef(const StepParams& p, int64_t t) {
  const float* c = p.coef_tab;
  const int64_t n = p.n_train;
  return SlotCoef{__ldg(c + t), __ldg(c + n + t), __ldg(c + 2 * n + t), __ldg(c + 3 * n + t),
                  __ldg(c + 4 * n + t), __ldg(c + 5 * n + t), __ldg(c + 6 * n + t)};
}

// One float4 column of every slot: all loads are issued before any store,
// so the update may run in place (x_next[i] aliasing x[i]) and up to
// 3N+1 16-byte loads per thread are in flight at once.
template <int N>
__device__ void update_block(const StepParams& p, int64_t w) {
  const int64_t s = w / p.nb_u, b = w - s * p.nb_u;
  SlotCoef k0 = slot_coef(p, 0);
  float new_sa = p.c_sa[0], new_s1a = p.c_s1a[0];
  if (p.rate_on) {
    // the frame in slot 0 sits at the timestep it entered at; the incoming
    // frame enters at the timestep the previous step derived from its rate
    const DevState* st = p.state + s;
    const int64_t t_old = st->slot0_t_buf[p.par], t_new = st->entry_t_buf[p.par];
    k0 = tab_coef(p, t_old);
    new_sa = __ldg(p.coef_tab + t_new);
    new_s1a = __ldg(p.coef_tab + 2 * p.n_train + t_new);
    if (b == 0 && threadIdx.x == 0) {
      p.state[s].slot0_t_buf[p.par ^ 1] = t_new;
      p.state[s].pub.slot0_timestep = t_new;
    }
  }
  const int64_t el = b * kUpdBlockElems + threadIdx.x * 4;
  if (el >= p.N_s) return;
  const int64_t e = s * p.N_s + el;
  // second operand of the negative branch: x0 (self-negative) or the
  // supplied negative prediction; without guidance x itself (unused), so
  // that every load is unconditional and all are in flight together
  float4 x[N], neg[N], ec[N], z[N > 1 ? N - 1 : 1];
#pragma unroll
  for (int i = 0; i < N; ++i) {
    x[i] = ld4(p.x[i] + e);
    neg[i] = ld4((p.cfg_kind == 2 ? p.eps_neg[i] : (p.cfg_kind == 1 ? p.x0[i] : p.x[i])) + e);
    ec[i] = p.ec_bf16 ? ld4_bf16(p.eps_c[i], e) : ld4(p.eps_c[i] + e);
    if (i < N - 1) z[i] = ld4(p.z[i] + e);
  }
  // txt2img: no input frame; the incoming latent is the noise draw itself
  const float4 en = ld4(p.eps_new + e);
  const float4 xn = p.txt2img ? en : ld4(p.x0_new + e);
#pragma unroll
  for (int i = N - 1; i >= 0; --i) {
    const SlotCoef k = i == 0 ? k0 : slot_coef(p, i);
    const float4 ecfg = eps_cfg4(x[i], neg[i], ec[i], p, k);
    const float4 xh = x0hat4(x[i], ecfg, k);
    if (i == N - 1) {
      st4(p.out + e, xh);
    } else if (p.upd_kind == 1) {
      st4(p.x_next[i + 1] + e, ddpm4(x[i], ecfg, z[i], k));
    } else {
      st4(p.x_next[i + 1] + e, noise4(xh, z[i], p.c_sa[i + 1], p.c_s1a[i + 1]));
    }
  }
  st4(p.x_next[0] + e, p.txt2img ? en : noise4(xn, en, new_sa, new_s1a));
}

// SSF and motion work blocks cover kRedBlockElems elements: kRedVec float4
// per array per thread, all loads in flight before any arithmetic.  Each
// thread sums in fp32 over 8 consecutive elements of its own (two float4)
// and in compensated fp32 pairs beyond (ssf_reduce.cuh).

__device__ void ssf_block(const StepParams& p, int64_t w, dfloat* red) {
  const int64_t s = w / p.nb_s, b = w % p.nb_s;
  const int64_t cur = p.state[s].ssf_cur;
  const float* I = p.ssf_frame + s * p.E;
  const float* R = p.ssf_ref + (cur * p.S + s) * p.E;
  float* Rn = p.ssf_ref + ((cur ^ 1) * p.S + s) * p.E;
  const int64_t base = b * kRedBlockElems + threadIdx.x * 4;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 a[kRedVec], r[kRedVec];
#pragma unroll
  for (int k = 0; k < kRedVec; ++k) {
    const int64_t e = base + k * (kStepThreads * 4);
    const bool h = e < p.E;
    a[k] = h ? ld4(I + e) : z4;
    r[k] = h ? ld4(R + e) : z4;
  }
#pragma unroll
  for (int k = 0; k < kRedVec; ++k) {
    const int64_t e = base + k * (kStepThreads * 4);
    if (e < p.E) st4(Rn + e, a[k]);
  }
  dfloat sd, si, sr;
  ssf_accumulate(a, r, sd, si, sr);
  block_sum3(sd, si, sr, red);
  if (threadIdx.x == 0) {
    double* part = p.partials + (s * p.nb_s + b) * 3;
    part[0] = df_to_double(sd);
    part[1] = df_to_double(si);
    part[2] = df_to_double(sr);
  }
}

__device__ void motion_block(const StepParams& p, int64_t w, dfloat* red) {
  const int64_t per_s = p.T * p.nb_m;
  const int64_t s = w / per_s, rem = w % per_s, j = rem / p.nb_m, b = rem % p.nb_m;
  const float* B = p.mot_chunk + (s * p.T + j) * p.N_f;
  const float* A = nullptr;
  if (j > 0) {
    A = p.mot_chunk + (s * p.T + j - 1) * p.N_f;
  } else if (p.state[s].mot_has_prev) {
    A = p.mot_prev_in + s * p.N_f;
  }
  const int64_t base = b * kRedBlockElems + threadIdx.x * 4;
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 bv[kRedVec], av[kRedVec];
#pragma unroll
  for (int k = 0; k < kRedVec; ++k) {
    const int64_t e = base + k * (kStepThreads * 4);
    const bool h = e < p.N_f;
    bv[k] = h ? ld4(B + e) : z4;
    av[k] = (h && A) ? ld4(A + e) : z4;
  }
  if (j == p.T - 1) {
#pragma unroll
    for (int k = 0; k < kRedVec; ++k) {
      const int64_t e = base + k * (kStepThreads * 4);
      if (e < p.N_f) st4(p.mot_prev_out + s * p.N_f + e, bv[k]);
    }
  }
  dfloat sq = df_make(0.f);
  if (A) {
#pragma unroll
    for (int k = 0; k < kRedVec; k += 2) {
      float acc = 0.f;
#pragma unroll
      for (int k2 = k; k2 < k + 2; ++k2) {
        const float dx = bv[k2].x - av[k2].x, dy = bv[k2].y - av[k2].y;
        const float dz = bv[k2].z - av[k2].z, dw = bv[k2].w - av[k2].w;
        acc = __fmaf_rn(dx, dx, acc);
        acc = __fmaf_rn(dy, dy, acc);
        acc = __fmaf_rn(dz, dz, acc);
        acc = __fmaf_rn(dw, dw, acc);
      }
      sq = df_add(sq, df_make(acc));
    }
  }
  block_sum1(sq, red);
  if (threadIdx.x == 0) p.partials[p.S * p.nb_s * 3 + (s * p.T + j) * p.nb_m + b] = df_to_double(sq);
}

constexpr int kFinChunk = 32;  // streams finished per round of the last block
constexpr int kFinPer = 3 + SDS_MAX_CHUNK_FRAMES;  // sums per stream at most

// The SSF decision and the motion / noise-rate update of stream s, taken by
// one warp from the stream's reduced values (dot, |I|^2, |R|^2, then the RMS
// difference d_j of each pair j).  Every lane reads the record's scalar
// fields (broadcast loads) and two slots of the old motion window; the slot
// a lane owns ends with the last of the chunk's d values written to it, so
// the window max needs no read back of what the warp stores.  The results
// equal those of appending the present pairs one by one to the ring.
__device__ void decide(const StepParams& p, int64_t s, const double* vals, int lane) {
  DevState* st = p.state + s;
  if (p.ssf_frame) {
    if (lane == 0) {
      const int64_t has_ref = st->pub.ssf_has_ref, count = st->pub.ssf_skip_count;
      const int64_t cur = st->ssf_cur, evals = st->pub.ssf_evals;
      const double u = (double)__ldcg(p.ssf_u + s);
      const double dot = vals[0], ni = vals[1], nr = vals[2];
      double cosv = 0.0, P = 0.0;
      int64_t skip = 0;
      if (has_ref) skip = ssf_decision(dot, ni, nr, p.eta, u, count, p.max_skip, cosv, P);
      st->pub.ssf_skip_count = skip ? count + 1 : 0;
      st->ssf_cur = skip ? cur : (cur ^ 1);
      st->pub.ssf_has_ref = skip ? has_ref : 1;
      st->pub.ssf_skip = skip;
      st->pub.ssf_cos = cosv;
      st->pub.ssf_p = P;
      st->pub.ssf_evals = evals + 1;
    }
    vals += 3;
  }
  if (p.mot_chunk) {
    const int K = (int)p.mot_k, T = (int)p.T;
    const int has_prev = (int)st->mot_has_prev, head = (int)st->mot_head, count = (int)st->mot_count;
    const int64_t pairs = st->pub.motion_pairs;
    const double rate = st->pub.noise_rate, dhat_old = st->pub.motion_dhat;
    double w_old[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) w_old[h] = (lane + 32 * h < K) ? st->mot_window[lane + 32 * h] : 0.0;
    const int first = has_prev ? 0 : 1;  // pair 0 is absent on the first chunk
    const int n_new = T - first;          // d values appended, in pair order
    const int count_new = min(count + n_new, K);
    const double nan = __longlong_as_double(0x7FF8000000000000ll);
    double mx = 0.0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int q = lane + 32 * h;
      if (q >= K) continue;
      const int r = (q - head + K) % K;  // appended value r lands on slot q first
      double v = w_old[h];
      if (r < n_new) {
        v = vals[first + r + K * ((n_new - 1 - r) / K)];  // the last one to land there
        st->mot_window[q] = v;
      }
      if (q < count_new) mx = fmax(mx, v);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmax(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane < SDS_MAX_CHUNK_FRAMES)
      st->pub.motion_d[lane] = (lane >= first && lane < T) ? vals[lane] : nan;
    if (lane == 0) {
      double new_rate = rate, dhat = dhat_old;
      if (count_new > 0) {
        dhat = fmin(1.0, mx / p.sigma);
        const double target = p.s_min + (p.s_max - p.s_min) * dhat;
        new_rate = rate + (1.0 - p.lam) * (target - rate);
      }
      st->mot_head = (head + n_new) % K;
      st->mot_count = count_new;
      st->pub.motion_pairs = pairs + n_new;
      st->pub.noise_rate = new_rate;
      // the next step's incoming frame enters the fraction `rate` of the way
      // from slot 1's timestep up to N - 1
      const int64_t t1 = p.t_floor;
      int64_t t_entry = t1 + (int64_t)floor(new_rate * (double)(p.n_train - 1 - t1) + 0.5);
      t_entry = t_entry < t1 ? t1 : (t_entry > p.n_train - 1 ? p.n_train - 1 : t_entry);
      st->entry_t_buf[p.par ^ 1] = t_entry;
      st->pub.motion_dhat = dhat;
      st->mot_has_prev = 1;
    }
  }
}

// Run by the last block: every sum of the launch is reduced by one warp in
// a fixed order (lane-strided over the partials, then a butterfly, which
// leaves the same bits in every lane); a motion sum becomes the pair's RMS
// difference in the same warp, so the square roots of a chunk run in
// parallel.  Then one warp per stream takes the stream's decisions.  The
// three SSF sums of a stream follow one order, so identical frames still
// give dot == |I|^2 == |R|^2 bitwise.
__device__ void finalize(const StepParams& p, double* fin) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_ssf = p.ssf_frame ? 3 : 0;
  const int per_s = n_ssf + (p.mot_chunk ? (int)p.T : 0);
  for (int64_t s0 = 0; s0 < p.S; s0 += kFinChunk) {
    const int ns = (int)min((int64_t)kFinChunk, p.S - s0);
    for (int k = warp; k < ns * per_s; k += kWarps) {
      const int64_t s = s0 + k / per_s;
      const int q = k % per_s;
      const double* base;
      int64_t n, stride;
      if (q < n_ssf) {
        base = p.partials + s * p.nb_s * 3 + q;
        n = p.nb_s;
        stride = 3;
      } else {
        base = p.partials + p.S * p.nb_s * 3 + (s * p.T + (q - n_ssf)) * p.nb_m;
        n = p.nb_m;
        stride = 1;
      }
      const double v = partials_sum(base, n, stride, lane);
      if (lane == 0) fin[k] = q < n_ssf ? v : sqrt(v / (double)p.N_f);
    }
    __syncthreads();
    for (int i = warp; i < ns; i += kWarps) decide(p, s0 + i, fin + i * per_s, lane);
    __syncthreads();
  }
}

template <int N>
__global__ void __launch_bounds__(kStepThreads, 2) step_kernel(const StepParams p) {
  __shared__ dfloat red[3 * kWarps];
  __shared__ double fin[kFinChunk * kFinPer];
  __shared__ int is_last;
  const int64_t tot_u = p.n > 0 ? p.S * p.nb_u : 0;
  const int64_t tot_s = p.ssf_frame ? p.S * p.nb_s : 0;
  const int64_t tot_m = p.mot_chunk ? p.S * p.T * p.nb_m : 0;
  const int64_t tot_r = tot_s + tot_m;  // reduction units come first
  const int64_t total = tot_u + tot_r;
  for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
    if (w < tot_r) {
      if (w < tot_s) {
        ssf_block(p, w, red);
      } else {
        motion_block(p, w - tot_s, red);
      }
      // Count the finished reduction unit (thread 0 wrote its partials);
      // the unit that completes the set finishes the launch's decisions
      // while other blocks go on streaming the update.
      if (threadIdx.x == 0) {
        __threadfence();
        const unsigned int prev = atomicAdd(p.counter, 1u);
        is_last = (prev == (unsigned int)(tot_r - 1)) ? 1 : 0;
      }
      __syncthreads();
      if (is_last) {
        __threadfence();
        finalize(p, fin);
        if (threadIdx.x == 0) {
          *p.counter = 0u;
          __threadfence();
        }
      }
    } else {
      update_block<N>(p, w - tot_r);
    }
  }
}

}  // namespace

cudaError_t launch_step(const StepParams& p, int sm_count, cudaStream_t st) {
  const int64_t tot = (p.n > 0 ? p.S * p.nb_u : 0) + (p.ssf_frame ? p.S * p.nb_s : 0) +
                      (p.mot_chunk ? p.S * p.T * p.nb_m : 0);
  if (tot == 0) return cudaSuccess;
#ifndef SDS_K4_BLOCKS_PER_SM
#define SDS_K4_BLOCKS_PER_SM 8
#endif
  // A resident grid (SDS_K4_BLOCKS_PER_SM blocks per SM) strides over the
  // work units.
  const int64_t cap = (int64_t)sm_count * SDS_K4_BLOCKS_PER_SM;
  const int grid = (int)(tot < cap ? tot : cap);
  switch (p.n) {
    case 0:
    case 1: step_kernel<1><<<grid, kStepThreads, 0, st>>>(p); break;
    case 2: step_kernel<2><<<grid, kStepThreads, 0, st>>>(p); break;
    case 3: step_kernel<3><<<grid, kStepThreads, 0, st>>>(p); break;
    case 4: step_kernel<4><<<grid, kStepThreads, 0, st>>>(p); break;
    case 5: step_kernel<5><<<grid, kStepThreads, 0, st>>>(p); break;
    case 6: step_kernel<6><<<grid, kStepThreads, 0, st>>>(p); break;
    case 7: step_kernel<7><<<grid, kStepThreads, 0, st>>>(p); break;
    case 8: step_kernel<8><<<grid, kStepThreads, 0, st>>>(p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace sds
