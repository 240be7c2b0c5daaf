// sds_oracle.cpp -- plain CPU oracle of the stream-batch diffusion hot path.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file; only the tests, the package's smoke check and the
// benchmark's CPU-baseline leg use it.  It shares no code, header, table or
// constant generator with the CUDA library: every quantity here (bf16
// rounding, RoPE angles, the noise schedule, the key list) is computed by
// this file alone, in double precision, straight from the definitions.
//
// Sources (page title, section / equation):
//  * StreamDiffusion (ICCV 2025 paper notes), "Stream Batch" and its
//    cross-frame attention equation Attn(Q_{t,i}, K_Batch, V_Batch).
//  * same page, "Residual CFG (R-CFG)": the virtual negative
//    eps_neg = (x_tau - sqrt(alpha) x0) / sqrt(beta) and the combine
//    eps_cfg = delta*eps_neg + gamma*(eps_c - delta*eps_neg).
//  * same page, "Stochastic Similarity Filter": P(skip) =
//    max{0, (S_C(I_t, I_ref) - eta) / (1 - eta)}, sampled, not thresholded.
//  * StreamDiffusion overview page, "Stochastic Similarity Filter":
//    at most max_skip_frame consecutive skipped frames.
//  * StreamDiffusionV2 summary, "Adaptive sink and RoPE refresh": refresh the
//    least similar sink when the cosine of the new chunk embedding falls
//    below a threshold; reset the RoPE phase when the frame index exceeds
//    a threshold.
//  * same page, "Motion-aware noise scheduler": L2 motion between
//    consecutive latent frames, normalised by a scale over a k-frame window,
//    clipped to [0,1], EMA into the noise rate bounded by [s_min, s_max].
//  * StreamDiffusion blog (mpbf.cn), section 7: the DDPM ancestral step
//    x_{t-1} = (x_t - (1-a_t)/sqrt(1-abar_t) eps)/sqrt(a_t) + sigma_t z.
//
// Where the pages leave a step open, the plainest reading is taken; each
// reading is marked "reading:" below.
//
// Parity status: every exported function is pinned by tests that check it
// against closed forms, invariants, brute force or library routines
// (tests/test_oracle_*.py); none is "parity unpinned".

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

#ifdef _OPENMP
#include <omp.h>
#endif

extern "C" {

// Oracle-side description of one stream's workload.  Filled by the Python
// test harness; this struct exists only in the oracle.
struct orc_cfg {
  long long n, T, L, H, d, M, R;          // slots, frames/chunk, tokens/frame, heads, head dim, sinks, ring frames
  long long image_mode;                   // 1: external batch K/V, no ring
  long long rope_on, grid_h, grid_w, rope_tau;
  long long D;                            // embedding dim
  long long n_inf, n_train;
  long long cfg_type;                     // 0 none, 1 self-negative R-CFG
  long long N_s;                          // elements of one slot latent
  long long ssf_E, max_skip;
  long long N_f, mot_k;
  long long update_kind;                  // 0: predict x0 then re-noise, 1: strided DDPM posterior
  long long noise_rate_on;                // 1: the incoming frame enters at round(s (N-1))
  long long t_index[8];
  double rope_base, s_th, beta_start, beta_end, gamma, delta, eta;
  double sigma, lam, s_min, s_max;
};

}  // extern "C"

namespace {

// ---------------------------------------------------------------- bf16
// IEEE-style bfloat16: 1 sign, 8 exponent, 7 stored mantissa bits.

double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return (double)f;
}

// Round a double to the nearest bfloat16, ties to even, in one step (no
// intermediate float rounding).  A bf16 normal number has 8 significant
// bits, so the rounding quantum of |x| in [2^(e-1), 2^e) is 2^(e-8);
// below the normal range the quantum is fixed at 2^-133.
uint16_t double_to_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  if (x == 0.0) return std::signbit(x) ? 0x8000 : 0x0000;
  int e;
  std::frexp(x, &e);
  int q = e - 8;
  if (q < -133) q = -133;
  double r = std::ldexp(std::nearbyint(std::ldexp(x, -q)), q);  // ties-to-even
  float f = (float)r;  // exact: r has at most 8 significant bits (or overflows to inf)
  uint32_t u;
  std::memcpy(&u, &f, 4);
  return (uint16_t)(u >> 16);
}

// ---------------------------------------------------------------- schedule
// reading: "scaled linear" betas, beta_s = (sqrt(b0) + s*(sqrt(b1)-sqrt(b0))/(N-1))^2,
// alphabar_t = prod_{s<=t} (1 - beta_s).
std::vector<double> alpha_bar_table(const orc_cfg& c) {
  std::vector<double> ab((size_t)c.n_train);
  double a = std::sqrt(c.beta_start), b = std::sqrt(c.beta_end);
  double prod = 1.0;
  for (long long s = 0; s < c.n_train; ++s) {
    double r = a + (double)s * (b - a) / (double)(c.n_train - 1);
    double beta = r * r;
    prod *= (1.0 - beta);
    ab[(size_t)s] = prod;
  }
  return ab;
}

// reading: t_index selects from a descending, evenly strided list of n_inf
// timesteps, timestep = (n_train - 1) - t_index * (n_train / n_inf).
long long slot_timestep(const orc_cfg& c, long long i) {
  return (c.n_train - 1) - c.t_index[i] * (c.n_train / c.n_inf);
}

// ---------------------------------------------------------------- RoPE
// reading: 3-axis RoPE over (temporal, row, column) positions.  The head
// dim is split into segments d_t, d_y, d_x with d_y = d_x = 2*floor(d/6),
// d_t = d - 2*d_y; inside a segment of width w, the pair (2i, 2i+1) turns
// by angle pos * base^(-2i/w).
void rope_segments(long long d, long long seg[3]) {
  long long dy = 2 * (d / 6);
  seg[0] = d - 2 * dy;
  seg[1] = dy;
  seg[2] = dy;
}

double rope_angle(double base, long long width, long long pair, long long pos) {
  double w = std::pow(base, -2.0 * (double)pair / (double)width);
  return (double)pos * w;
}

// Rotate one head vector (values in double) at positions pos[3]; out may not alias in.
void rope_rotate(const double* in, double* out, long long d, const long long pos[3], double base) {
  long long seg[3];
  rope_segments(d, seg);
  long long start = 0;
  for (int a = 0; a < 3; ++a) {
    for (long long i = 0; i < seg[a] / 2; ++i) {
      double th = rope_angle(base, seg[a], i, pos[a]);
      double cs = std::cos(th), sn = std::sin(th);
      double u = in[start + 2 * i], v = in[start + 2 * i + 1];
      out[start + 2 * i] = u * cs - v * sn;
      out[start + 2 * i + 1] = u * sn + v * cs;
    }
    start += seg[a];
  }
}

// Brute-force softmax attention of one query (double) against a key list.
// keys / vals: bf16 rows; key r's head-h vector starts at r*H*d + h*d.
void attend_row(const double* q, const uint16_t* keys, const uint16_t* vals,
                const std::vector<long long>& key_rows, long long H, long long h,
                long long d, double* out) {
  size_t nk = key_rows.size();
  std::vector<double> s(nk);
  double scale = 1.0 / std::sqrt((double)d);
  double m = -INFINITY;
  for (size_t j = 0; j < nk; ++j) {
    const uint16_t* kr = keys + (size_t)(key_rows[j] * H * d + h * d);
    double acc = 0.0;
    for (long long t = 0; t < d; ++t) acc += q[t] * bf16_to_double(kr[t]);
    s[j] = acc * scale;
    if (s[j] > m) m = s[j];
  }
  double den = 0.0;
  for (long long t = 0; t < d; ++t) out[t] = 0.0;
  for (size_t j = 0; j < nk; ++j) {
    double w = std::exp(s[j] - m);
    den += w;
    const uint16_t* vr = vals + (size_t)(key_rows[j] * H * d + h * d);
    for (long long t = 0; t < d; ++t) out[t] += w * bf16_to_double(vr[t]);
  }
  for (long long t = 0; t < d; ++t) out[t] /= den;
}

// ---------------------------------------------------------------- stream state
struct Stream {
  orc_cfg c;
  std::vector<double> abar;
  // ring + sink (physical layout: M sink frames then R ring frames, each L tokens of H*d bf16)
  long long F = 0;          // frames pushed so far
  long long o = 0;          // RoPE offset: positions are counted from frame o
  long long p0 = 0;         // start position of the most recent chunk
  long long chunk_first = -1;
  long long pushes = 0, resets = 0;
  std::vector<uint16_t> kbuf, vbuf;
  long long sinks_filled = 0;
  std::vector<double> emb;  // [M][D]
  // SSF
  std::vector<float> ref;
  int has_ref = 0;
  long long skip_count = 0;
  // motion
  std::vector<float> prev;
  int has_prev = 0;
  std::vector<double> window;
  double s_rate = 0.0;
  long long slot0_t = -1;   // timestep of the frame in slot 0 (noise-rate application)
  // lazy mode: pushes record where each key frame came from instead of
  // rotating it; materialize later applies the push arithmetic to the frames
  int lazy = 0;
  std::vector<long long> prov;  // [M+R][3]: source chunk index, frame in chunk, chunk start p0
};

long long key_frames(const orc_cfg& c) { return c.image_mode ? 0 : (c.M + c.R); }

}  // namespace

extern "C" {

// ---------------------------------------------------------------- pure helpers

void orc_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

uint16_t orc_bf16_round(double x) { return double_to_bf16(x); }
double orc_bf16_value(uint16_t b) { return bf16_to_double(b); }

void orc_alpha_bar(const orc_cfg* c, double* out) {
  std::vector<double> ab = alpha_bar_table(*c);
  std::memcpy(out, ab.data(), ab.size() * sizeof(double));
}

long long orc_slot_timestep(const orc_cfg* c, long long i) { return slot_timestep(*c, i); }

double orc_rope_angle(double base, long long width, long long pair, long long pos) {
  return rope_angle(base, width, pair, pos);
}

void orc_rope_segments(long long d, long long* seg3) { rope_segments(d, seg3); }

// Rotate nvec head vectors (double in, double out) at positions pos3[nvec][3].
void orc_rope_rotate(const double* in, double* out, long long nvec, long long d,
                     const long long* pos3, double base) {
  for (long long v = 0; v < nvec; ++v) rope_rotate(in + v * d, out + v * d, d, pos3 + 3 * v, base);
}

// Softmax attention (O1) of selected query rows against a bf16 key/value set.
// q: bf16 [q_rows][H][d] (used as given: no RoPE); k, v: bf16 [n_keys][H][d].
// rows: indices of the query rows to evaluate (all H heads of each);
// out: double [nsel][H][d].
void orc_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, long long H,
                   long long d, long long n_keys, const long long* rows, long long nsel,
                   double* out) {
  std::vector<long long> key_rows((size_t)n_keys);
  for (long long j = 0; j < n_keys; ++j) key_rows[(size_t)j] = j;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (long long r = 0; r < nsel; ++r) {
    for (long long h = 0; h < H; ++h) {
      std::vector<double> qd((size_t)d);
      const uint16_t* qr = q + (size_t)(rows[r] * H * d + h * d);
      for (long long t = 0; t < d; ++t) qd[(size_t)t] = bf16_to_double(qr[t]);
      attend_row(qd.data(), k, v, key_rows, H, h, d, out + (size_t)((r * H + h) * d));
    }
  }
}

// ---------------------------------------------------------------- stateful stream

void* orc_create(const orc_cfg* c) {
  Stream* s = new Stream();
  s->c = *c;
  s->abar = alpha_bar_table(*c);
  size_t kv = (size_t)(key_frames(*c) * c->L * c->H * c->d);
  s->kbuf.assign(kv, 0);
  s->vbuf.assign(kv, 0);
  s->emb.assign((size_t)(c->M * c->D), 0.0);
  s->ref.assign((size_t)c->ssf_E, 0.0f);
  s->prev.assign((size_t)c->N_f, 0.0f);
  s->s_rate = c->s_min;
  s->prov.assign((size_t)(key_frames(*c) * 3), -1);
  s->slot0_t = slot_timestep(*c, 0);
  return s;
}

void orc_destroy(void* p) { delete (Stream*)p; }

// a1 + a2: positions with reset, RoPE on K, append into the ring (evicting the
// oldest frame by overwrite).  k, v: bf16 [T*L][H][d].  Returns p0.
// reading: "frame index exceeds tau" compares the chunk's start position,
// counted from the last reset, with tau; cached keys keep their rotation.
// One frame of a pushed chunk into key frame `dst_frame` of the buffer:
// each key vector rotated at (pos_t, y, x) in double and rounded to bf16,
// the values copied.  kf, vf: bf16 [L][H][d] of the frame.
static void write_frame(Stream* s, long long dst_frame, const uint16_t* kf, const uint16_t* vf,
                        long long pos_t) {
  const orc_cfg& c = s->c;
  long long HD = c.H * c.d;
  std::vector<double> in((size_t)c.d), out((size_t)c.d);
  for (long long l = 0; l < c.L; ++l) {
    size_t src = (size_t)(l * HD);
    size_t dst = (size_t)((dst_frame * c.L + l) * HD);
    long long pos[3] = {pos_t, l / c.grid_w, l % c.grid_w};
    for (long long h = 0; h < c.H; ++h) {
      const uint16_t* kr = kf + src + h * c.d;
      if (c.rope_on) {
        for (long long t = 0; t < c.d; ++t) in[(size_t)t] = bf16_to_double(kr[t]);
        rope_rotate(in.data(), out.data(), c.d, pos, c.rope_base);
        for (long long t = 0; t < c.d; ++t) s->kbuf[dst + h * c.d + t] = double_to_bf16(out[(size_t)t]);
      } else {
        std::memcpy(&s->kbuf[dst + h * c.d], kr, (size_t)c.d * 2);
      }
    }
    std::memcpy(&s->vbuf[dst], vf + src, (size_t)HD * 2);
  }
}

long long orc_push(void* p, const uint16_t* k, const uint16_t* v) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  long long p0 = s->F - s->o;
  if (p0 > c.rope_tau) {
    s->o = s->F;
    p0 = 0;
    s->resets++;
  }
  s->p0 = p0;
  const size_t fr = (size_t)(c.L * c.H * c.d);
  for (long long j = 0; j < c.T; ++j) {
    long long f = s->F + j;
    long long slot = f % c.R;
    long long* pv = &s->prov[(size_t)((c.M + slot) * 3)];
    pv[0] = s->pushes;
    pv[1] = j;
    pv[2] = p0;
    if (!s->lazy) write_frame(s, c.M + slot, k + j * fr, v + j * fr, p0 + j);
  }
  s->chunk_first = s->F;
  s->F += c.T;
  s->pushes++;
  return p0;
}

// Lazy mode on/off (see Stream::prov).  Only for a stream that has not
// pushed yet.
void orc_set_lazy(void* p, int on) { ((Stream*)p)->lazy = on; }

// Provenance of every key frame: [M+R][3] = (chunk index, frame in chunk,
// chunk start position p0), -1 for a frame never written.
void orc_provenance(void* p, long long* out) {
  Stream* s = (Stream*)p;
  std::memcpy(out, s->prov.data(), s->prov.size() * sizeof(long long));
}

// Fill the K/V buffer from raw (unrotated) frames given for every key frame
// in buffer order, kf, vf: bf16 [M+R][L][H][d]; each frame with a provenance
// is written as its push wrote it (rotated at p0 + frame in chunk).
void orc_materialize(void* p, const uint16_t* kf, const uint16_t* vf) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  const size_t fr = (size_t)(c.L * c.H * c.d);
#pragma omp parallel for schedule(dynamic, 1)
  for (long long f = 0; f < key_frames(c); ++f) {
    const long long* pv = &s->prov[(size_t)(f * 3)];
    if (pv[0] < 0) continue;
    write_frame(s, f, kf + (size_t)f * fr, vf + (size_t)f * fr, pv[2] + pv[1]);
  }
}

// meta: F, o, p0, ring valid frames, sinks filled, resets
void orc_meta(void* p, long long* out6) {
  Stream* s = (Stream*)p;
  out6[0] = s->F;
  out6[1] = s->o;
  out6[2] = s->p0;
  out6[3] = std::min(s->F, s->c.R);
  out6[4] = s->sinks_filled;
  out6[5] = s->resets;
}

static void copy_frame_to_sink(Stream* s, long long sink, long long chunk_frame) {
  const orc_cfg& c = s->c;
  long long slot = (s->chunk_first + chunk_frame) % c.R;
  size_t fr = (size_t)(c.L * c.H * c.d);
  for (int q = 0; q < 3; ++q) s->prov[(size_t)(sink * 3 + q)] = s->prov[(size_t)((c.M + slot) * 3 + q)];
  if (s->lazy) return;
  std::memcpy(&s->kbuf[(size_t)sink * fr], &s->kbuf[(size_t)(c.M + slot) * fr], fr * 2);
  std::memcpy(&s->vbuf[(size_t)sink * fr], &s->vbuf[(size_t)(c.M + slot) * fr], fr * 2);
}

// a3: adaptive sink refresh.  h: float [D].
// Empty sinks are filled in index order from frames 0.. of the chunk just
// pushed (fill = 2).  Otherwise alpha_j = cos(h, e_j); j* = argmin (lowest
// index on ties); when alpha_{j*} < s_th (strict), sink j* takes frame 0 of
// the chunk and e_{j*} = h (fire = 1).  A zero norm gives cosine 0.
// res[0] = j*, res[1] = fire (0/1/2), res[2] = near-tie flag;
// dres[0] = alpha_min, dres[1] = second smallest alpha (or +inf).
void orc_sink_refresh(void* p, const float* h, long long* res, double* dres) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  res[0] = -1; res[1] = 0; res[2] = 0;
  dres[0] = INFINITY; dres[1] = INFINITY;
  if (c.M == 0 || s->chunk_first < 0) return;
  if (s->sinks_filled < c.M) {
    long long nfill = std::min(c.M - s->sinks_filled, c.T);
    res[0] = s->sinks_filled;
    for (long long q = 0; q < nfill; ++q) {
      long long j = s->sinks_filled + q;
      copy_frame_to_sink(s, j, q);
      for (long long t = 0; t < c.D; ++t) s->emb[(size_t)(j * c.D + t)] = (double)h[t];
    }
    s->sinks_filled += nfill;
    res[1] = 2;
    return;
  }
  double hn = 0.0;
  for (long long t = 0; t < c.D; ++t) hn += (double)h[t] * (double)h[t];
  long long jstar = -1;
  double amin = INFINITY, a2 = INFINITY;
  for (long long j = 0; j < c.M; ++j) {
    double dot = 0.0, en = 0.0;
    for (long long t = 0; t < c.D; ++t) {
      double e = s->emb[(size_t)(j * c.D + t)];
      dot += (double)h[t] * e;
      en += e * e;
    }
    double a = (hn > 0.0 && en > 0.0) ? dot / std::sqrt(hn * en) : 0.0;
    if (a < amin) {
      a2 = amin;
      amin = a;
      jstar = j;
    } else if (a < a2) {
      a2 = a;
    }
  }
  res[0] = jstar;
  dres[0] = amin;
  dres[1] = a2;
  if (std::fabs(amin - c.s_th) < 1e-9 || (a2 - amin) < 1e-9) res[2] = 1;
  if (amin < c.s_th) {
    copy_frame_to_sink(s, jstar, 0);
    for (long long t = 0; t < c.D; ++t) s->emb[(size_t)(jstar * c.D + t)] = (double)h[t];
    res[1] = 1;
  }
}

// Copy out the physical K/V buffer (bf16 [(M+R)*L][H][d]) and the sink embeddings.
void orc_get_kv(void* p, uint16_t* k, uint16_t* v) {
  Stream* s = (Stream*)p;
  std::memcpy(k, s->kbuf.data(), s->kbuf.size() * 2);
  std::memcpy(v, s->vbuf.data(), s->vbuf.size() * 2);
}

void orc_get_emb(void* p, double* e) {
  Stream* s = (Stream*)p;
  std::memcpy(e, s->emb.data(), s->emb.size() * sizeof(double));
}

// Number of valid keys the next attend uses, and the key rows (physical
// indices into the K/V buffer) in order: filled sinks, then filled ring slots.
long long orc_key_rows(void* p, long long* rows_out) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  long long n = 0;
  for (long long j = 0; j < s->sinks_filled; ++j)
    for (long long l = 0; l < c.L; ++l) {
      if (rows_out) rows_out[n] = j * c.L + l;
      n++;
    }
  long long valid = std::min(s->F, c.R);
  for (long long r = 0; r < valid; ++r)
    for (long long l = 0; l < c.L; ++l) {
      if (rows_out) rows_out[n] = (c.M + r) * c.L + l;
      n++;
    }
  return n;
}

// a4 (video mode): attention of selected query rows against the stream's
// sink + ring keys.  q: bf16 [n*T*L][H][d] as given (unrotated); each
// selected row is rotated at its chunk position (O2) and rounded to bf16 --
// the operand the tensor cores consume -- before the scores are formed.
void orc_attend(void* p, const uint16_t* q, const long long* rows, long long nsel, double* out) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  long long nk = orc_key_rows(p, nullptr);
  std::vector<long long> key_rows((size_t)nk);
  orc_key_rows(p, key_rows.data());
  long long TL = c.T * c.L;
#pragma omp parallel for schedule(dynamic, 1) collapse(2)
  for (long long r = 0; r < nsel; ++r) {
    for (long long h = 0; h < c.H; ++h) {
      std::vector<double> in((size_t)c.d), qd((size_t)c.d);
      const uint16_t* qr = q + (size_t)(rows[r] * c.H * c.d + h * c.d);
      for (long long t = 0; t < c.d; ++t) in[(size_t)t] = bf16_to_double(qr[t]);
      if (c.rope_on) {
        long long tok = rows[r] % TL;
        long long j = tok / c.L, l = tok % c.L;
        long long pos[3] = {s->p0 + j, l / c.grid_w, l % c.grid_w};
        rope_rotate(in.data(), qd.data(), c.d, pos, c.rope_base);
        for (long long t = 0; t < c.d; ++t) qd[(size_t)t] = bf16_to_double(double_to_bf16(qd[(size_t)t]));
      } else {
        qd = in;
      }
      attend_row(qd.data(), s->kbuf.data(), s->vbuf.data(), key_rows, c.H, h, c.d,
                 out + (size_t)((r * c.H + h) * c.d));
    }
  }
}

// a5: self-negative R-CFG + stream-batch scheduler update, in double.
// x, x0, eps_c: [n][N_s]; z: [n-1][N_s]; x0_new, eps_new: [N_s].
// x_next: [n][N_s]; out: [N_s].
// reading: alpha and beta of the R-CFG virtual negative are alphabar_t and
// 1 - alphabar_t of the slot's own timestep; x0 is the slot's own input
// latent.  reading: the strided update predicts x0hat, then re-noises it to
// the next slot's level with the supplied ancestral noise z.
// a5: R-CFG combine and the stream-batch update of every slot.
// x, x0, eps_c: float [n][N_s]; z: float [n-1][N_s]; eps_neg: float [n][N_s]
// (cfg_type 2 only, else may be NULL); x0_new, eps_new: float [N_s];
// outputs x_next [n][N_s], out [N_s] in double.
// cfg_type 0: eps_cfg = eps_c.  1 (self-negative R-CFG): eps_neg is the
// virtual residual (x - sqrt(abar) x0) / sqrt(1 - abar).  2 (onetime-negative
// R-CFG, or standard CFG with delta = 1): eps_neg is a supplied negative /
// unconditional prediction.  Both combine as delta*eps_neg +
// gamma*(eps_c - delta*eps_neg).
// update_kind 0 (reading: predict x0, re-noise to the next slot's level):
//   x_next[i+1] = sqrt(abar') x0hat + sqrt(1 - abar') z_i.
// update_kind 1 (the blog's DDPM ancestral step taken between the slot's
// timestep t and the next slot's t', reading: alpha = abar_t / abar_t' and
// sigma^2 the posterior variance (1 - abar_t') / (1 - abar_t) (1 - alpha)):
//   x_next[i+1] = (x - (1 - alpha) / sqrt(1 - abar_t) eps_cfg) / sqrt(alpha) + sigma z_i.
// The last slot's x0hat is the completed frame; the incoming frame enters
// slot 0 as sqrt(abar_0) x0_new + sqrt(1 - abar_0) eps_new.
void orc_step_update2(void* p, const float* x, const float* x0, const float* eps_c, const float* z,
                      const float* eps_neg, const float* x0_new, const float* eps_new,
                      double* x_next, double* out) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  long long N = c.N_s;
  // reading of the motion-aware noise scheduler: the noise rate s chooses
  // the timestep at which the incoming frame enters slot 0, as the fraction
  // s of the way from slot 1's timestep t1 up to pure noise (N_train - 1):
  // t1 + round(s (N_train - 1 - t1)), with t1 = 0 when there is no slot 1.
  // So the entering frame is never less noisy than the frame it precedes
  // and the stream batch's timesteps stay in descending order.  The frame
  // then in slot 0 sits at the timestep it entered at.  The rate is the one
  // in force before this step's motion.
  long long t_new = slot_timestep(c, 0);
  if (c.noise_rate_on) {
    const long long t1 = c.n > 1 ? slot_timestep(c, 1) : 0;
    t_new = t1 + (long long)std::floor(s->s_rate * (double)(c.n_train - 1 - t1) + 0.5);
    t_new = std::min(std::max(t_new, t1), c.n_train - 1);
  }
  for (long long i = 0; i < c.n; ++i) {
    long long ti = (i == 0 && c.noise_rate_on) ? s->slot0_t : slot_timestep(c, i);
    double ab = s->abar[(size_t)ti];
    double ab_next = (i + 1 < c.n) ? s->abar[(size_t)slot_timestep(c, i + 1)] : 0.0;
    for (long long e = 0; e < N; ++e) {
      size_t k = (size_t)(i * N + e);
      double xv = x[k], ec = eps_c[k];
      double eps_cfg = ec;
      if (c.cfg_type == 1 || c.cfg_type == 2) {
        double en = (c.cfg_type == 1) ? (xv - std::sqrt(ab) * (double)x0[k]) / std::sqrt(1.0 - ab)
                                       : (double)eps_neg[k];
        // The printed combine delta*eps_neg + gamma*(eps_c - delta*eps_neg),
        // regrouped as gamma*eps_c + delta*(1-gamma)*eps_neg (equal in real
        // arithmetic) so that gamma = 1 returns eps_c exactly.
        eps_cfg = c.gamma * ec + c.delta * (1.0 - c.gamma) * en;
      }
      double x0hat = (xv - std::sqrt(1.0 - ab) * eps_cfg) / std::sqrt(ab);
      if (i + 1 < c.n) {
        double nx;
        if (c.update_kind == 1) {
          double alpha = ab / ab_next;
          double sigma = std::sqrt((1.0 - ab_next) / (1.0 - ab) * (1.0 - alpha));
          nx = (xv - (1.0 - alpha) / std::sqrt(1.0 - ab) * eps_cfg) / std::sqrt(alpha) +
               sigma * (double)z[k];
        } else {
          nx = std::sqrt(ab_next) * x0hat + std::sqrt(1.0 - ab_next) * (double)z[k];
        }
        x_next[(size_t)((i + 1) * N + e)] = nx;
      } else {
        out[e] = x0hat;
      }
    }
  }
  // the incoming frame noised to its entry level; with no input image
  // (txt2img, x0_new absent) the incoming latent is the noise draw itself
  double ab0 = s->abar[(size_t)t_new];
  for (long long e = 0; e < N; ++e)
    x_next[e] = x0_new ? std::sqrt(ab0) * (double)x0_new[e] + std::sqrt(1.0 - ab0) * (double)eps_new[e]
                       : (double)eps_new[e];
  s->slot0_t = t_new;
}

long long orc_slot0_timestep(void* p) { return ((Stream*)p)->slot0_t; }

void orc_step_update(void* p, const float* x, const float* x0, const float* eps_c, const float* z,
                     const float* x0_new, const float* eps_new, double* x_next, double* out) {
  orc_step_update2(p, x, x0, eps_c, z, nullptr, x0_new, eps_new, x_next, out);
}

// a6: stochastic similarity filter on one incoming frame.
// frame: float [ssf_E]; u: the supplied uniform draw in [0,1).
// res[0] = skip, res[1] = consecutive skip count after this frame, res[2] = near flag;
// dres[0] = cosine, dres[1] = P(skip).
// reading: the first frame (no reference yet) is processed; I_ref is the last
// processed frame; a zero-norm frame has cosine 0; skip iff u < P and fewer
// than max_skip consecutive frames were skipped.
void orc_ssf(void* p, const float* frame, float u, long long* res, double* dres) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  double cosv = 0.0, P = 0.0;
  long long skip = 0;
  if (s->has_ref) {
    double dot = 0.0, ni = 0.0, nr = 0.0;
    for (long long e = 0; e < c.ssf_E; ++e) {
      double a = frame[e], b = s->ref[(size_t)e];
      dot += a * b;
      ni += a * a;
      nr += b * b;
    }
    cosv = (ni > 0.0 && nr > 0.0) ? dot / std::sqrt(ni * nr) : 0.0;
    P = std::min(1.0, std::max(0.0, (cosv - c.eta) / (1.0 - c.eta)));
    skip = ((double)u < P && s->skip_count < c.max_skip) ? 1 : 0;
  }
  res[2] = (s->has_ref && std::fabs((double)u - P) < 1e-4) ? 1 : 0;
  if (skip) {
    s->skip_count++;
  } else {
    s->skip_count = 0;
    std::memcpy(s->ref.data(), frame, (size_t)c.ssf_E * sizeof(float));
    s->has_ref = 1;
  }
  res[0] = skip;
  res[1] = s->skip_count;
  dres[0] = cosv;
  dres[1] = P;
}

// a7: motion estimate and EMA noise rate on one incoming chunk.
// chunk: float [T][N_f].  dres[0..T-1] = motion values of this chunk's frame
// pairs (NaN where the pair does not exist), dres[T] = dhat, dres[T+1] = s.
// reading: the L2 motion is the RMS of the frame difference; the window
// statistic is the max of the last mot_k values; a higher dhat moves the
// target noise rate toward s_max; s <- s + (1 - lambda)(target - s); the
// first chunk has no previous frame, so its first pair is absent.
void orc_motion(void* p, const float* chunk, double* dres) {
  Stream* s = (Stream*)p;
  const orc_cfg& c = s->c;
  for (long long j = 0; j < c.T; ++j) {
    const float* b = chunk + (size_t)(j * c.N_f);
    const float* a = (j == 0) ? (s->has_prev ? s->prev.data() : nullptr) : chunk + (size_t)((j - 1) * c.N_f);
    if (!a) {
      dres[j] = NAN;
      continue;
    }
    double acc = 0.0;
    for (long long e = 0; e < c.N_f; ++e) {
      double df = (double)b[e] - (double)a[e];
      acc += df * df;
    }
    double dv = std::sqrt(acc / (double)c.N_f);
    dres[j] = dv;
    s->window.push_back(dv);
    if ((long long)s->window.size() > c.mot_k) s->window.erase(s->window.begin());
  }
  double dhat = 0.0;
  if (!s->window.empty()) {
    double mx = 0.0;
    for (double w : s->window) mx = std::max(mx, w);
    dhat = std::min(1.0, mx / c.sigma);
    double target = c.s_min + (c.s_max - c.s_min) * dhat;
    s->s_rate = s->s_rate + (1.0 - c.lam) * (target - s->s_rate);
  }
  std::memcpy(s->prev.data(), chunk + (size_t)((c.T - 1) * c.N_f), (size_t)c.N_f * sizeof(float));
  s->has_prev = 1;
  dres[c.T] = dhat;
  dres[c.T + 1] = s->s_rate;
}

double orc_noise_rate(void* p) { return ((Stream*)p)->s_rate; }
long long orc_skip_count(void* p) { return ((Stream*)p)->skip_count; }

}  // extern "C"
