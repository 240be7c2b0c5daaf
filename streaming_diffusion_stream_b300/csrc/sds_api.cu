// sds_api.cu -- host side of the C ABI declared in include/sds.h:
// validation, device buffers, host ring metadata, RoPE and schedule tables,
// and kernel launches.  No compute happens here; every step of the path runs
// in the kernels of k_attn.cu, k_ring.cu and k_step.cu.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "sds_internal.h"

using namespace sds;

struct sds_ctx {
  sds_config cfg;
  int device = 0;
  int sm_count = 0;
  bool image_mode = false;
  // device buffers (owned)
  uint16_t* kv_k = nullptr;
  uint16_t* kv_v = nullptr;
  float* sink_emb = nullptr;
  float2* rope_tab = nullptr;
  float* ssf_ref = nullptr;   // [2][S][E]
  float* mot_prev = nullptr;  // [2][S][N_f]
  DevState* state = nullptr;  // [S]
  double* partials = nullptr;
  unsigned int* counters = nullptr;  // [1]: K4's arrival counter
  void* attn_ws = nullptr;           // split-key workspace of the attention kernel
  float* coef_dev = nullptr;         // per-timestep coefficients (noise-rate application)
  int64_t step_calls = 0;            // sds_step_update calls (parity of the rate buffers)
  uint64_t attn_wait_ns = kAttnWaitNs;  // K1's wait limit (shortened only by the test hook)
  int64_t attn_withhold_k = -1;         // K1 test hook: key tile CTA 0 does not load
  std::vector<void*> allocs;
  // tables
  int rope_seg[3] = {0, 0, 0};
  int tab_off[3] = {0, 0, 0};
  int tab_rows_t = 0;
  double abar_slot[SDS_MAX_SLOTS] = {};
  // host ring metadata
  int64_t F = 0, o = 0, p0 = 0, chunk_first = -1, sinks_filled = 0, resets = 0, chunks = 0;
  int64_t motion_calls = 0;
  int64_t nb_u = 0, nb_s = 0, nb_m = 0;
  CUtensorMap tm_kv_k, tm_kv_v;
  std::string err;
};

namespace {

thread_local std::string g_create_err;

sds_status fail(sds_ctx* c, sds_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  if (c) {
    c->err = buf;
  } else {
    g_create_err = buf;
  }
  return st;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// scaled-linear betas; alphabar_t = prod_{s<=t} (1 - beta_s)
void alpha_bar(const sds_config& c, std::vector<double>& out) {
  out.resize((size_t)c.num_train_steps);
  const double a = std::sqrt(c.beta_start), b = std::sqrt(c.beta_end);
  double prod = 1.0;
  for (int64_t t = 0; t < c.num_train_steps; ++t) {
    const double r = a + (b - a) * (double)t / (double)(c.num_train_steps - 1);
    prod *= 1.0 - r * r;
    out[(size_t)t] = prod;
  }
}

sds_status validate(const sds_config* c, std::string& why) {
  auto bad = [&](const char* m) {
    why = m;
    return SDS_ERR_INVALID_ARG;
  };
  if (!c) return bad("config is NULL");
  if (c->abi_version != SDS_ABI_VERSION) return bad("abi_version mismatch");
  if (c->streams < 1 || c->streams > 65535) return bad("streams must be in [1, 65535]");
  if (c->slots_n < 1 || c->slots_n > SDS_MAX_SLOTS) return bad("slots_n must be in [1, 8]");
  if (c->heads_H < 1 || c->heads_H > 65535) return bad("heads_H must be in [1, 65535]");
  if (c->head_dim != 64 && c->head_dim != 128) return bad("head_dim must be 64 or 128");
  if (c->tokens_L < 1) return bad("tokens_L must be >= 1");
  if (c->frames_T < 1 || c->frames_T > SDS_MAX_CHUNK_FRAMES) return bad("frames_T must be in [1, 8]");
  const bool image = c->ring_R == 0;
  if (c->ring_R < 0 || c->sink_M < 0) return bad("ring_R and sink_M must be >= 0");
  if (!image) {
    if (c->ring_R < c->frames_T) return bad("ring_R must hold at least one chunk (ring_R >= frames_T)");
    if (c->rope_on) {
      if (c->grid_h < 1 || c->grid_w < 1 || c->grid_h * c->grid_w != c->tokens_L)
        return bad("grid_h * grid_w must equal tokens_L");
      if (c->rope_tau < 0 || c->rope_tau > (1 << 20)) return bad("rope_tau must be in [0, 2^20]");
      if (!(c->rope_base > 1.0)) return bad("rope_base must be > 1");
    }
    if (c->sink_M > 0 && (c->emb_dim_D < 1 || c->emb_dim_D > (1 << 24)))
      return bad("emb_dim_D must be >= 1 when sink_M > 0");
    int64_t keys = (c->sink_M + c->ring_R) * c->tokens_L;
    if (keys > (1ll << 30)) return bad("key buffer rows exceed 2^30");
  } else {
    if (c->frames_T != 1) return bad("image mode (ring_R == 0) needs frames_T == 1");
    if (c->sink_M != 0) return bad("image mode (ring_R == 0) has no sinks");
  }
  if (c->num_train_steps < 2 || c->num_inference_steps < 1 ||
      c->num_inference_steps > c->num_train_steps)
    return bad("need 2 <= num_train_steps and 1 <= num_inference_steps <= num_train_steps");
  if (!(c->beta_start > 0.0 && c->beta_end > 0.0 && c->beta_start < 1.0 && c->beta_end < 1.0))
    return bad("betas must be in (0, 1)");
  for (int64_t i = 0; i < c->slots_n; ++i) {
    int64_t t = (c->num_train_steps - 1) -
                c->t_index[i] * (c->num_train_steps / c->num_inference_steps);
    if (c->t_index[i] < 0 || t < 0 || t >= c->num_train_steps)
      return bad("t_index entry maps outside the training schedule");
  }
  if (c->cfg_type < 0 || c->cfg_type > 2)
    return bad("cfg_type must be 0 (none), 1 (self-negative) or 2 (supplied negative)");
  if (c->update_kind != 0 && c->update_kind != 1)
    return bad("update_kind must be 0 (re-noise x0hat) or 1 (strided DDPM posterior)");
  if (c->noise_rate_on != 0 && c->noise_rate_on != 1) return bad("noise_rate_on must be 0 or 1");
  if (c->noise_rate_on && !c->motion_on) return bad("noise_rate_on needs motion_on");
  if (c->eps_c_bf16 != 0 && c->eps_c_bf16 != 1) return bad("eps_c_bf16 must be 0 or 1");
  if (c->txt2img != 0 && c->txt2img != 1) return bad("txt2img must be 0 or 1");
  if (c->txt2img && c->cfg_type == 1) return bad("txt2img has no x0: cfg_type must be 0 or 2");
  if (c->txt2img && c->noise_rate_on) return bad("txt2img has no input frame to noise: noise_rate_on must be 0");
  if (c->attn_ctas < 0 || c->attn_ctas > kAttnMaxCtas) return bad("attn_ctas must be in [0, 160]");
  if (c->slot_elems < 4 || c->slot_elems % 4 != 0) return bad("slot_elems must be a positive multiple of 4");
  if (c->ssf_on) {
    if (c->ssf_elems < 4 || c->ssf_elems % 4 != 0) return bad("ssf_elems must be a positive multiple of 4");
    if (!(c->ssf_eta < 1.0)) return bad("ssf_eta must be < 1");
    if (c->max_skip_frame < 0) return bad("max_skip_frame must be >= 0");
  }
  if (c->motion_on) {
    if (c->frame_elems < 4 || c->frame_elems % 4 != 0) return bad("frame_elems must be a positive multiple of 4");
    if (c->mot_k < 1 || c->mot_k > kMaxMotionWindow) return bad("mot_k must be in [1, 64]");
    if (!(c->mot_sigma > 0.0)) return bad("mot_sigma must be > 0");
    if (!(c->s_min <= c->s_max)) return bad("s_min must be <= s_max");
  }
  if (c->noise_rate_on && (!(c->s_min >= 0.0) || !(c->s_max <= 1.0)))
    return bad("noise_rate_on needs 0 <= s_min <= s_max <= 1 (the rate places the incoming frame "
               "between slot 1's timestep and pure noise)");
  return SDS_OK;
}

sds_status dev_alloc(sds_ctx* c, void** p, size_t bytes) {
  if (bytes == 0) bytes = 16;
  cudaError_t e = cudaMalloc(p, bytes);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(nullptr, SDS_ERR_OOM, "cudaMalloc(%zu) failed: %s", bytes, cudaGetErrorString(e));
  }
  c->allocs.push_back(*p);
  e = cudaMemset(*p, 0, bytes);
  if (e != cudaSuccess) return fail(nullptr, SDS_ERR_CUDA, "cudaMemset failed: %s", cudaGetErrorString(e));
  return SDS_OK;
}

void free_all(sds_ctx* c) {
  for (void* p : c->allocs) cudaFree(p);
  c->allocs.clear();
}

sds_status cuda_fail(sds_ctx* c, cudaError_t e, const char* what) {
  return fail(c, SDS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// The noise rate places the incoming frame the fraction s of the way from
// slot 1's timestep t1 (0 with one slot) up to N - 1.
int64_t entry_floor(const sds_config& c) {
  return c.slots_n > 1 ? (c.num_train_steps - 1) - c.t_index[1] * (c.num_train_steps / c.num_inference_steps) : 0;
}

int64_t entry_timestep(const sds_config& c, double s) {
  const int64_t t1 = entry_floor(c);
  const int64_t t = t1 + (int64_t)std::floor(s * (double)(c.num_train_steps - 1 - t1) + 0.5);
  return std::min<int64_t>(std::max<int64_t>(t, t1), c.num_train_steps - 1);
}

void fill_attn_rope(const sds_ctx* c, AttnParams& ap) {
  ap.rope_on = (int)(c->cfg.rope_on && !c->image_mode);
  ap.p0 = (int)c->p0;
  ap.tokens_L = (int)c->cfg.tokens_L;
  ap.grid_w = (int)(c->cfg.grid_w > 0 ? c->cfg.grid_w : 1);
  ap.chunk_tokens = (int)(c->cfg.frames_T * c->cfg.tokens_L);
  for (int a = 0; a < 3; ++a) {
    ap.rope_seg[a] = c->rope_seg[a];
    ap.tab_off[a] = c->tab_off[a];
  }
  ap.rope_tab = c->rope_tab;
}

// ----------------------------------------------------------------- checkpoints

uint64_t fnv1a(const void* data, size_t n, uint64_t h = 14695981039346656037ull) {
  const unsigned char* b = static_cast<const unsigned char*>(data);
  for (size_t i = 0; i < n; ++i) {
    h ^= b[i];
    h *= 1099511628211ull;
  }
  return h;
}

// Section sizes (bytes) of a checkpoint payload for a configuration.
struct StateLayout {
  int64_t meta, records, emb, ssf, mot, kv;  // kv: per tensor (K and V each)
  int64_t emb_elems, ssf_elems, mot_elems, kv_elems;
  bool with_kv;
  int64_t payload() const { return meta + records + emb + ssf + mot + (with_kv ? 2 * kv : 0); }
};

StateLayout state_layout(const sds_config& c, bool with_kv) {
  StateLayout L{};
  const bool image = c.ring_R == 0;
  const int64_t S = c.streams;
  L.with_kv = with_kv;
  L.emb_elems = image ? 0 : S * c.sink_M * (c.emb_dim_D > 0 ? c.emb_dim_D : 0);
  L.ssf_elems = c.ssf_on ? 2 * S * c.ssf_elems : 0;
  L.mot_elems = c.motion_on ? 2 * S * c.frame_elems : 0;
  L.kv_elems = image ? 0 : S * (c.sink_M + c.ring_R) * c.tokens_L * c.heads_H * c.head_dim;
  L.meta = 16 * 8;
  L.records = S * (int64_t)sizeof(DevState);
  L.emb = L.emb_elems * 4;
  L.ssf = L.ssf_elems * 4;
  L.mot = L.mot_elems * 4;
  L.kv = L.kv_elems * 2;
  return L;
}

// Validate a checkpoint against a configuration; on failure `why` says why.
sds_status check_state(const sds_config& c, const void* buf, size_t len, std::string& why) {
  if (!buf) {
    why = "checkpoint buffer is NULL";
    return SDS_ERR_INVALID_ARG;
  }
  if (len < sizeof(sds_state_header)) {
    why = "checkpoint shorter than its header";
    return SDS_ERR_STATE;
  }
  sds_state_header h;
  std::memcpy(&h, buf, sizeof h);
  if (std::memcmp(h.magic, SDS_STATE_MAGIC, 8) != 0) {
    why = "not a checkpoint (bad magic)";
    return SDS_ERR_STATE;
  }
  if (h.abi_version != SDS_ABI_VERSION) {
    why = "checkpoint written by another ABI version";
    return SDS_ERR_STATE;
  }
  if (h.config_hash != fnv1a(&c, sizeof c)) {
    why = "checkpoint belongs to a different configuration";
    return SDS_ERR_STATE;
  }
  const StateLayout L = state_layout(c, (h.flags & 1) != 0);
  if ((h.flags & ~int64_t(1)) != 0 || h.streams != c.streams ||
      h.devstate_bytes != (int64_t)sizeof(DevState) || h.emb_elems != L.emb_elems ||
      h.ssf_ref_elems != L.ssf_elems || h.mot_prev_elems != L.mot_elems ||
      h.kv_elems != L.kv_elems || h.payload_bytes != L.payload()) {
    why = "checkpoint section sizes do not match the configuration";
    return SDS_ERR_STATE;
  }
  if (len < sizeof h + (size_t)h.payload_bytes) {
    why = "checkpoint truncated";
    return SDS_ERR_STATE;
  }
  const unsigned char* payload = static_cast<const unsigned char*>(buf) + sizeof h;
  if (fnv1a(payload, (size_t)h.payload_bytes) != h.payload_hash) {
    why = "checkpoint payload hash mismatch (corrupted)";
    return SDS_ERR_STATE;
  }
  const int64_t* meta = reinterpret_cast<const int64_t*>(payload);
  int64_t m[16];
  std::memcpy(m, meta, sizeof m);
  bool tail_zero = true;
  for (int i = 9; i < 16; ++i) tail_zero = tail_zero && m[i] == 0;
  if (m[0] < 0 || m[1] < 0 || m[1] > m[0] || m[4] < 0 || m[4] > c.sink_M || m[5] < 0 || m[6] < 0 ||
      m[7] < 0 || m[8] < 0 || !tail_zero) {
    why = "checkpoint metadata out of range";
    return SDS_ERR_STATE;
  }
  return SDS_OK;
}

}  // namespace

void sds::set_thread_error(const char* msg) { g_create_err = msg; }

extern "C" {

int sds_abi_version(void) { return SDS_ABI_VERSION; }

const char* sds_last_error(const sds_ctx* ctx) {
  return ctx ? ctx->err.c_str() : g_create_err.c_str();
}

sds_status sds_create(const sds_config* cfg, sds_ctx** out) {
  if (!out) return fail(nullptr, SDS_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  std::string why;
  sds_status st = validate(cfg, why);
  if (st != SDS_OK) return fail(nullptr, st, "invalid config: %s", why.c_str());
  const sds_config& c = *cfg;
  const int64_t S = c.streams, L = c.tokens_L, HD = c.heads_H * c.head_dim;
  const bool image = c.ring_R == 0;

  // sizes
  const int64_t kv_elems = image ? 0 : S * (c.sink_M + c.ring_R) * L * HD;
  const int64_t emb = image ? 0 : S * c.sink_M * (c.emb_dim_D > 0 ? c.emb_dim_D : 0);
  int seg[3] = {0, 0, 0};
  int64_t tab_entries = 0;
  int tab_off[3] = {0, 0, 0};
  int tab_rows_t = 0;
  if (!image && c.rope_on) {
    const int dy = 2 * (int)(c.head_dim / 6);
    seg[0] = (int)c.head_dim - 2 * dy;
    seg[1] = dy;
    seg[2] = dy;
    tab_rows_t = (int)(c.rope_tau + c.frames_T);
    const int rows[3] = {tab_rows_t, (int)c.grid_h, (int)c.grid_w};
    for (int a = 0; a < 3; ++a) {
      tab_off[a] = (int)tab_entries;
      tab_entries += (int64_t)rows[a] * (seg[a] / 2);
    }
  }
  const int64_t nb_u = cdiv(c.slot_elems, kUpdBlockElems);
  const int64_t nb_s = c.ssf_on ? cdiv(c.ssf_elems, kRedBlockElems) : 0;
  const int64_t nb_m = c.motion_on ? cdiv(c.frame_elems, kRedBlockElems) : 0;
  const int64_t ssf_ref = c.ssf_on ? 2 * S * c.ssf_elems : 0;
  const int64_t mot_prev = c.motion_on ? 2 * S * c.frame_elems : 0;
  const int64_t partials = S * nb_s * 3 + S * c.frames_T * nb_m;
  const size_t ws_bytes = attn_ws_bytes((int)c.head_dim);
  const size_t coef_bytes = c.noise_rate_on ? (size_t)c.num_train_steps * 7 * 4 : 0;
  const size_t bytes = coef_bytes + (size_t)kv_elems * 2 * 2 + (size_t)emb * 4 + (size_t)tab_entries * 8 +
                       (size_t)ssf_ref * 4 + (size_t)mot_prev * 4 + (size_t)S * sizeof(DevState) +
                       (size_t)partials * 8 + (size_t)4 + ws_bytes;
  if (c.mem_cap_bytes > 0 && bytes > (size_t)c.mem_cap_bytes)
    return fail(nullptr, SDS_ERR_OOM, "context needs %zu bytes > mem_cap_bytes %lld", bytes,
                (long long)c.mem_cap_bytes);

  sds_ctx* ctx = new sds_ctx();
  ctx->cfg = c;
  ctx->image_mode = image;
  cudaError_t e = cudaGetDevice(&ctx->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device);
  if (e != cudaSuccess) {
    delete ctx;
    cudaGetLastError();
    return fail(nullptr, SDS_ERR_CUDA, "no usable CUDA device: %s", cudaGetErrorString(e));
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, ctx->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, ctx->device);
  if (major != 10 || minor != 3) {
    delete ctx;
    return fail(nullptr, SDS_ERR_UNSUPPORTED, "this build targets sm_103a; device is sm_%d%d", major, minor);
  }
  for (int a = 0; a < 3; ++a) {
    ctx->rope_seg[a] = seg[a];
    ctx->tab_off[a] = tab_off[a];
  }
  ctx->tab_rows_t = tab_rows_t;
  ctx->nb_u = nb_u;
  ctx->nb_s = nb_s;
  ctx->nb_m = nb_m;

#define ALLOC(ptr, n)                                                         \
  do {                                                                        \
    void* tmp_ = nullptr;                                                     \
    sds_status s_ = dev_alloc(ctx, &tmp_, (size_t)(n));                        \
    if (s_ != SDS_OK) {                                                       \
      free_all(ctx);                                                          \
      delete ctx;                                                             \
      return s_;                                                              \
    }                                                                         \
    ptr = reinterpret_cast<decltype(ptr)>(tmp_);                              \
  } while (0)

  ALLOC(ctx->kv_k, kv_elems * 2);
  ALLOC(ctx->kv_v, kv_elems * 2);
  ALLOC(ctx->sink_emb, emb * 4);
  ALLOC(ctx->rope_tab, tab_entries * 8);
  ALLOC(ctx->ssf_ref, ssf_ref * 4);
  ALLOC(ctx->mot_prev, mot_prev * 4);
  ALLOC(ctx->state, S * (int64_t)sizeof(DevState));
  ALLOC(ctx->partials, partials * 8);
  ALLOC(ctx->counters, 4);
  ALLOC(ctx->attn_ws, ws_bytes);
  ALLOC(ctx->coef_dev, coef_bytes);
#undef ALLOC

  // RoPE table: angle pos * base^(-2i/w) in double, stored as fp32 (cos, sin)
  if (tab_entries > 0) {
    std::vector<float2> tab((size_t)tab_entries);
    const int rows[3] = {tab_rows_t, (int)c.grid_h, (int)c.grid_w};
    for (int a = 0; a < 3; ++a) {
      const int half = seg[a] / 2;
      for (int pos = 0; pos < rows[a]; ++pos)
        for (int i = 0; i < half; ++i) {
          const double th = (double)pos * std::pow(c.rope_base, -2.0 * i / (double)seg[a]);
          tab[(size_t)tab_off[a] + (size_t)pos * half + i] = make_float2((float)std::cos(th), (float)std::sin(th));
        }
    }
    e = cudaMemcpy(ctx->rope_tab, tab.data(), tab.size() * sizeof(float2), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      free_all(ctx);
      delete ctx;
      return fail(nullptr, SDS_ERR_CUDA, "table upload failed: %s", cudaGetErrorString(e));
    }
  }
  // initial decision records
  {
    std::vector<DevState> st0((size_t)S);
    for (auto& d : st0) {
      std::memset(&d, 0, sizeof d);
      d.pub.sink_j = -1;
      d.pub.noise_rate = c.s_min;
      const int64_t te = entry_timestep(c, c.s_min);
      d.entry_t_buf[0] = d.entry_t_buf[1] = te;
      const int64_t t0 = (c.num_train_steps - 1) - c.t_index[0] * (c.num_train_steps / c.num_inference_steps);
      d.slot0_t_buf[0] = d.slot0_t_buf[1] = t0;
      d.pub.slot0_timestep = t0;
      d.pub.sink_alpha_min = INFINITY;
      d.pub.sink_alpha_2 = INFINITY;
      for (double& v : d.pub.motion_d) v = NAN;
    }
    e = cudaMemcpy(ctx->state, st0.data(), st0.size() * sizeof(DevState), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
      free_all(ctx);
      delete ctx;
      return fail(nullptr, SDS_ERR_CUDA, "state upload failed: %s", cudaGetErrorString(e));
    }
  }
  // schedule coefficients of the slots
  {
    std::vector<double> ab;
    alpha_bar(c, ab);
    for (int64_t i = 0; i < c.slots_n; ++i) {
      const int64_t t = (c.num_train_steps - 1) - c.t_index[i] * (c.num_train_steps / c.num_inference_steps);
      ctx->abar_slot[i] = ab[(size_t)t];
    }
    if (c.noise_rate_on) {
      // slot 0's coefficients at every timestep it can sit at; the DDPM rows
      // step from that timestep to slot 1's
      const int64_t nt = c.num_train_steps;
      const double an = c.slots_n > 1 ? ctx->abar_slot[1] : 1.0;
      std::vector<float> tab((size_t)nt * 7, 0.0f);
      for (int64_t t = 0; t < nt; ++t) {
        const double a = ab[(size_t)t];
        tab[(size_t)t] = (float)std::sqrt(a);
        tab[(size_t)(nt + t)] = (float)(1.0 / std::sqrt(1.0 - a));
        tab[(size_t)(2 * nt + t)] = (float)std::sqrt(1.0 - a);
        tab[(size_t)(3 * nt + t)] = (float)(1.0 / std::sqrt(a));
        if (c.slots_n > 1) {
          const double al = a / an;
          tab[(size_t)(4 * nt + t)] = (float)(1.0 / std::sqrt(al));
          tab[(size_t)(5 * nt + t)] = (float)((1.0 - al) / (std::sqrt(al) * std::sqrt(1.0 - a)));
          tab[(size_t)(6 * nt + t)] = (float)std::sqrt((1.0 - an) / (1.0 - a) * (1.0 - al));
        }
      }
      e = cudaMemcpy(ctx->coef_dev, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice);
      if (e != cudaSuccess) {
        free_all(ctx);
        delete ctx;
        return fail(nullptr, SDS_ERR_CUDA, "table upload failed: %s", cudaGetErrorString(e));
      }
    }
  }
  if (!image) {
    const int64_t rows = (c.sink_M + c.ring_R) * L;
    if (!make_tmap_bf16(&ctx->tm_kv_k, ctx->kv_k, HD, rows, S) ||
        !make_tmap_bf16(&ctx->tm_kv_v, ctx->kv_v, HD, rows, S)) {
      free_all(ctx);
      delete ctx;
      return fail(nullptr, SDS_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K/V ring");
    }
  }
  *out = ctx;
  return SDS_OK;
}

void sds_destroy(sds_ctx* ctx) {
  if (!ctx) return;
  cudaDeviceSynchronize();
  free_all(ctx);
  delete ctx;
}

sds_status sds_kv_push(sds_ctx* ctx, const void* k, const void* v, sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  if (ctx->image_mode) return fail(ctx, SDS_ERR_STATE, "kv_push: context is in image batch mode");
  if (!k || !v || !aligned16(k) || !aligned16(v))
    return fail(ctx, SDS_ERR_INVALID_ARG, "kv_push: k and v must be non-NULL 16-byte aligned device pointers");
  const sds_config& c = ctx->cfg;
  int64_t p0 = ctx->F - ctx->o;
  int64_t o = ctx->o;
  bool reset = false;
  if (p0 > c.rope_tau) {
    o = ctx->F;
    p0 = 0;
    reset = true;
  }
  PushParams p{};
  p.k_in = reinterpret_cast<const uint4*>(k);
  p.v_in = reinterpret_cast<const uint4*>(v);
  p.kv_k = reinterpret_cast<uint4*>(ctx->kv_k);
  p.kv_v = reinterpret_cast<uint4*>(ctx->kv_v);
  p.S = c.streams;
  p.T = c.frames_T;
  p.L = c.tokens_L;
  p.HD = c.heads_H * c.head_dim;
  p.M = c.sink_M;
  p.R = c.ring_R;
  p.head_dim = c.head_dim;
  p.F = ctx->F;
  p.p0 = (int32_t)p0;
  p.rope_on = (int32_t)c.rope_on;
  p.grid_w = (int32_t)(c.grid_w > 0 ? c.grid_w : 1);
  for (int a = 0; a < 3; ++a) {
    p.rope_seg[a] = ctx->rope_seg[a];
    p.tab_off[a] = ctx->tab_off[a];
  }
  p.rope_tab = ctx->rope_tab;
  cudaError_t e = launch_kv_push(p, ctx->sm_count, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "kv_push launch");
  ctx->o = o;
  ctx->p0 = p0;
  if (reset) ctx->resets++;
  ctx->chunk_first = ctx->F;
  ctx->F += c.frames_T;
  ctx->chunks++;
  return SDS_OK;
}

sds_status sds_sink_refresh(sds_ctx* ctx, const float* chunk_emb, sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  if (ctx->image_mode) return fail(ctx, SDS_ERR_STATE, "sink_refresh: context is in image batch mode");
  const sds_config& c = ctx->cfg;
  if (c.sink_M == 0) return SDS_OK;
  if (ctx->chunk_first < 0) return fail(ctx, SDS_ERR_STATE, "sink_refresh before the first kv_push");
  if (!chunk_emb || !aligned16(chunk_emb))
    return fail(ctx, SDS_ERR_INVALID_ARG, "sink_refresh: chunk_emb must be a 16-byte aligned device pointer");
  SinkParams p{};
  p.h = chunk_emb;
  p.emb = ctx->sink_emb;
  p.kv_k = reinterpret_cast<uint4*>(ctx->kv_k);
  p.kv_v = reinterpret_cast<uint4*>(ctx->kv_v);
  p.state = ctx->state;
  p.S = c.streams;
  p.D = c.emb_dim_D;
  p.M = c.sink_M;
  p.R = c.ring_R;
  p.L = c.tokens_L;
  p.HD = c.heads_H * c.head_dim;
  p.chunk_first = ctx->chunk_first;
  p.s_th = c.s_th;
  int64_t nfill = 0;
  if (ctx->sinks_filled < c.sink_M) {
    nfill = std::min<int64_t>(c.sink_M - ctx->sinks_filled, c.frames_T);
    p.fill_from = ctx->sinks_filled;
    p.fill_count = nfill;
  } else {
    p.fill_from = -1;
    p.fill_count = 0;
  }
  cudaError_t e = launch_sink_refresh(p, ctx->sm_count, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "sink_refresh launch");
  ctx->sinks_filled += nfill;
  return SDS_OK;
}

static sds_status attend_common(sds_ctx* ctx, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, AttnParams& ap, int head_dim, int S,
                                cudaStream_t st) {
  ap.S = S;
  int sm_count = 0;
  if (ctx) {
    sm_count = ctx->sm_count;
    const size_t per_rec = (size_t)kAttnMaxCtas * 2 * 2 * 128;
    ap.ws_o = reinterpret_cast<float*>(ctx->attn_ws);
    ap.ws_ml = reinterpret_cast<float2*>(reinterpret_cast<char*>(ctx->attn_ws) + per_rec * head_dim * 4);
    ap.ws_cnt = reinterpret_cast<unsigned int*>(reinterpret_cast<char*>(ctx->attn_ws) +
                                                per_rec * ((size_t)head_dim * 4 + 8));
    ap.grid = (int32_t)ctx->cfg.attn_ctas;
    ap.wait_ns = ctx->attn_wait_ns;
    ap.withhold_k = ctx->attn_withhold_k;
  } else {
    ap.wait_ns = kAttnWaitNs;
    ap.withhold_k = -1;
  }
  CUtensorMap to;
  if (!make_tmap_bf16(&to, ap.o, (int64_t)ap.H * head_dim, ap.q_rows, S)) {
    if (ctx) return fail(ctx, SDS_ERR_CUDA, "attention: cuTensorMapEncodeTiled failed for o");
    return fail(nullptr, SDS_ERR_CUDA, "attention: cuTensorMapEncodeTiled failed for o");
  }
  cudaError_t e = launch_attention(tq, tk, tv, to, ap, head_dim, S, sm_count, st);
  if (e != cudaSuccess) {
    if (ctx) return cuda_fail(ctx, e, "attention launch");
    return fail(nullptr, SDS_ERR_CUDA, "attention launch: %s", cudaGetErrorString(e));
  }
  return SDS_OK;
}

sds_status sds_attend(sds_ctx* ctx, const void* q, void* o, const void* ext_k, const void* ext_v,
                      sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  const sds_config& c = ctx->cfg;
  if (!q || !o || !aligned16(q) || !aligned16(o))
    return fail(ctx, SDS_ERR_INVALID_ARG, "attend: q and o must be non-NULL 16-byte aligned device pointers");
  const int64_t S = c.streams, HD = c.heads_H * c.head_dim;
  AttnParams ap{};
  ap.o = reinterpret_cast<uint16_t*>(o);
  ap.H = (int32_t)c.heads_H;
  ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)c.head_dim));
  ap.state = ctx->state;
  CUtensorMap tq, tk, tv;
  if (ctx->image_mode) {
    if (!ext_k || !ext_v || !aligned16(ext_k) || !aligned16(ext_v))
      return fail(ctx, SDS_ERR_INVALID_ARG, "attend: image mode needs 16-byte aligned ext_k and ext_v");
    const int64_t rows = c.slots_n * c.tokens_L;
    ap.q_rows = rows;
    ap.seg_start[0] = 0;
    ap.seg_count[0] = (int32_t)rows;
    ap.seg_start[1] = 0;
    ap.seg_count[1] = 0;
    if (!make_tmap_bf16(&tq, q, HD, rows, S) || !make_tmap_bf16(&tk, ext_k, HD, rows, S) ||
        !make_tmap_bf16(&tv, ext_v, HD, rows, S))
      return fail(ctx, SDS_ERR_CUDA, "attend: cuTensorMapEncodeTiled failed");
    fill_attn_rope(ctx, ap);
    ap.rope_on = 0;
    return attend_common(ctx, tq, tk, tv, ap, (int)c.head_dim, (int)S, (cudaStream_t)stream);
  }
  if (ext_k || ext_v) return fail(ctx, SDS_ERR_INVALID_ARG, "attend: ext_k/ext_v must be NULL in video mode");
  if (ctx->chunk_first < 0) return fail(ctx, SDS_ERR_STATE, "attend before the first kv_push");
  const int64_t rows = c.slots_n * c.frames_T * c.tokens_L;
  ap.q_rows = rows;
  const int64_t valid = std::min<int64_t>(ctx->F, c.ring_R);
  ap.seg_start[0] = 0;
  ap.seg_count[0] = (int32_t)(ctx->sinks_filled * c.tokens_L);
  ap.seg_start[1] = (int32_t)(c.sink_M * c.tokens_L);
  ap.seg_count[1] = (int32_t)(valid * c.tokens_L);
  if (ctx->sinks_filled == c.sink_M) {  // one contiguous range: sinks then ring
    ap.seg_count[0] = (int32_t)((c.sink_M + valid) * c.tokens_L);
    ap.seg_start[1] = 0;
    ap.seg_count[1] = 0;
  }
  if (!make_tmap_bf16(&tq, q, HD, rows, S))
    return fail(ctx, SDS_ERR_CUDA, "attend: cuTensorMapEncodeTiled failed");
  fill_attn_rope(ctx, ap);
  return attend_common(ctx, tq, ctx->tm_kv_k, ctx->tm_kv_v, ap, (int)c.head_dim, (int)S,
                       (cudaStream_t)stream);
}

sds_status sds_attention(const void* q, const void* k, const void* v, void* o, int64_t S,
                         int64_t Lq, int64_t Lk, int64_t H, int64_t head_dim, sds_stream_t stream) {
  if (!q || !k || !v || !o || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(nullptr, SDS_ERR_INVALID_ARG, "attention: pointers must be non-NULL and 16-byte aligned");
  if (S < 1 || S > 65535 || H < 1 || H > 65535 || Lq < 1 || Lk < 1 || Lk > (1ll << 30) ||
      Lq > (1ll << 31) - 128)
    return fail(nullptr, SDS_ERR_INVALID_ARG, "attention: sizes out of range");
  if (head_dim != 64 && head_dim != 128)
    return fail(nullptr, SDS_ERR_INVALID_ARG, "attention: head_dim must be 64 or 128");
  const int64_t HD = H * head_dim;
  CUtensorMap tq, tk, tv;
  if (!make_tmap_bf16(&tq, q, HD, Lq, S) || !make_tmap_bf16(&tk, k, HD, Lk, S) ||
      !make_tmap_bf16(&tv, v, HD, Lk, S))
    return fail(nullptr, SDS_ERR_CUDA, "attention: cuTensorMapEncodeTiled failed");
  AttnParams ap{};
  ap.o = reinterpret_cast<uint16_t*>(o);
  ap.q_rows = Lq;
  ap.H = (int32_t)H;
  ap.seg_start[0] = 0;
  ap.seg_count[0] = (int32_t)Lk;
  ap.scale_log2 = (float)(1.4426950408889634 / std::sqrt((double)head_dim));
  ap.rope_on = 0;
  ap.tokens_L = 1;
  ap.grid_w = 1;
  ap.chunk_tokens = 1;
  ap.state = nullptr;
  return attend_common(nullptr, tq, tk, tv, ap, (int)head_dim, (int)S, (cudaStream_t)stream);
}

static sds_status fill_step(sds_ctx* ctx, StepParams& p) {
  const sds_config& c = ctx->cfg;
  p.S = c.streams;
  p.state = ctx->state;
  p.partials = ctx->partials;
  p.counter = ctx->counters;
  p.nb_u = ctx->nb_u;
  p.nb_s = ctx->nb_s;
  p.nb_m = ctx->nb_m;
  p.N_s = c.slot_elems;
  p.E = c.ssf_elems;
  p.eta = c.ssf_eta;
  p.max_skip = c.max_skip_frame;
  p.ssf_ref = ctx->ssf_ref;
  p.T = c.frames_T;
  p.N_f = c.frame_elems;
  p.mot_k = c.mot_k;
  p.sigma = c.mot_sigma;
  p.lam = c.mot_lambda;
  p.s_min = c.s_min;
  p.s_max = c.s_max;
  return SDS_OK;
}

sds_status sds_step_update(sds_ctx* ctx, const sds_step_io* io, sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  if (!io) return fail(ctx, SDS_ERR_INVALID_ARG, "step_update: io is NULL");
  const sds_config& c = ctx->cfg;
  const int n = (int)c.slots_n;
  auto okp = [](const void* p) { return p && aligned16(p); };
  for (int i = 0; i < n; ++i) {
    if (!okp(io->x[i]) || !okp(io->eps_c[i]) || !okp(io->x_next[i]) ||
        (c.cfg_type == 1 && !okp(io->x0[i])) || (c.cfg_type == 2 && !okp(io->eps_neg[i])))
      return fail(ctx, SDS_ERR_INVALID_ARG,
                  "step_update: slot %d arrays (x, eps_c, x_next, and x0 for cfg_type 1 or eps_neg "
                  "for cfg_type 2) must be non-NULL and 16-byte aligned", i);
    if (i < n - 1 && !okp(io->z[i]))
      return fail(ctx, SDS_ERR_INVALID_ARG, "step_update: z[%d] must be non-NULL and 16-byte aligned", i);
  }
  if (!okp(io->out) || (!c.txt2img && !okp(io->x0_new)) || !okp(io->eps_new))
    return fail(ctx, SDS_ERR_INVALID_ARG,
                "step_update: out, eps_new and (unless txt2img) x0_new must be non-NULL and 16-byte aligned");
  if (io->ssf_frame) {
    if (!c.ssf_on) return fail(ctx, SDS_ERR_INVALID_ARG, "step_update: ssf_frame given but ssf_on == 0");
    if (!okp(io->ssf_frame) || !io->ssf_u)
      return fail(ctx, SDS_ERR_INVALID_ARG, "step_update: ssf_frame must be 16-byte aligned and ssf_u non-NULL");
  }
  if (c.noise_rate_on && !io->motion_chunk)
    return fail(ctx, SDS_ERR_INVALID_ARG, "step_update: noise_rate_on needs motion_chunk every step");
  if (io->motion_chunk) {
    if (!c.motion_on) return fail(ctx, SDS_ERR_INVALID_ARG, "step_update: motion_chunk given but motion_on == 0");
    if (!okp(io->motion_chunk)) return fail(ctx, SDS_ERR_INVALID_ARG, "step_update: motion_chunk must be 16-byte aligned");
  }
  StepParams p{};
  fill_step(ctx, p);
  p.n = n;
  for (int i = 0; i < n; ++i) {
    p.x[i] = io->x[i];
    p.x0[i] = io->x0[i];
    p.eps_c[i] = io->eps_c[i];
    p.z[i] = (i < n - 1) ? io->z[i] : nullptr;
    p.x_next[i] = io->x_next[i];
    const double a = ctx->abar_slot[i];
    p.c_sa[i] = (float)std::sqrt(a);
    p.c_inv_s1a[i] = (float)(1.0 / std::sqrt(1.0 - a));
    p.c_s1a[i] = (float)std::sqrt(1.0 - a);
    p.c_inv_sa[i] = (float)(1.0 / std::sqrt(a));
    p.eps_neg[i] = c.cfg_type == 2 ? io->eps_neg[i] : nullptr;
    if (i + 1 < n) {
      // strided DDPM step from this slot's timestep to the next slot's
      const double an = ctx->abar_slot[i + 1];
      const double al = a / an;
      p.c_px[i] = (float)(1.0 / std::sqrt(al));
      p.c_pe[i] = (float)((1.0 - al) / (std::sqrt(al) * std::sqrt(1.0 - a)));
      p.c_sig[i] = (float)std::sqrt((1.0 - an) / (1.0 - a) * (1.0 - al));
    }
  }
  p.cfg_kind = (int32_t)c.cfg_type;
  p.upd_kind = (int32_t)c.update_kind;
  p.rate_on = (int32_t)c.noise_rate_on;
  p.ec_bf16 = (int32_t)c.eps_c_bf16;
  p.txt2img = (int32_t)c.txt2img;
  p.par = (int32_t)(ctx->step_calls & 1);
  p.coef_tab = ctx->coef_dev;
  p.n_train = c.num_train_steps;
  p.t_floor = entry_floor(c);
  if (c.cfg_type != 0) {
    p.c_gamma = (float)c.gamma;
    p.c_dg = (float)(c.delta * (1.0 - c.gamma));
  } else {
    p.c_gamma = 1.0f;
    p.c_dg = 0.0f;
  }
  p.out = io->out;
  p.x0_new = c.txt2img ? nullptr : io->x0_new;
  p.eps_new = io->eps_new;
  p.ssf_frame = io->ssf_frame;
  p.ssf_u = io->ssf_u;
  if (io->motion_chunk) {
    const int64_t par = ctx->motion_calls & 1;
    p.mot_chunk = io->motion_chunk;
    p.mot_prev_in = ctx->mot_prev + par * c.streams * c.frame_elems;
    p.mot_prev_out = ctx->mot_prev + (par ^ 1) * c.streams * c.frame_elems;
  }
  cudaError_t e = launch_step(p, ctx->sm_count, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "step_update launch");
  if (io->motion_chunk) ctx->motion_calls++;
  ctx->step_calls++;
  return SDS_OK;
}

sds_status sds_ssf(sds_ctx* ctx, const float* frame, const float* u, sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  if (!ctx->cfg.ssf_on) return fail(ctx, SDS_ERR_INVALID_ARG, "ssf: ssf_on == 0 in the config");
  if (!frame || !aligned16(frame) || !u)
    return fail(ctx, SDS_ERR_INVALID_ARG, "ssf: frame must be 16-byte aligned and u non-NULL");
  StepParams p{};
  fill_step(ctx, p);
  p.n = 0;
  p.ssf_frame = frame;
  p.ssf_u = u;
  cudaError_t e = launch_step(p, ctx->sm_count, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "ssf launch");
  return SDS_OK;
}

sds_status sds_state_check(const sds_config* cfg, const void* buf, size_t len) {
  if (!cfg) return fail(nullptr, SDS_ERR_INVALID_ARG, "state_check: cfg is NULL");
  std::string why;
  const sds_status st = check_state(*cfg, buf, len, why);
  if (st != SDS_OK) return fail(nullptr, st, "state_check: %s", why.c_str());
  return SDS_OK;
}

sds_status sds_state_export(sds_ctx* ctx, void* buf, size_t* len, int64_t with_kv,
                            sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  if (!len) return fail(ctx, SDS_ERR_INVALID_ARG, "state_export: len is NULL");
  const sds_config& c = ctx->cfg;
  const StateLayout L = state_layout(c, with_kv != 0);
  const size_t need = sizeof(sds_state_header) + (size_t)L.payload();
  if (!buf) {
    *len = need;
    return SDS_OK;
  }
  if (*len < need) {
    *len = need;
    return fail(ctx, SDS_ERR_INVALID_ARG, "state_export: buffer of %zu bytes < %zu needed", *len, need);
  }
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "state_export");
  unsigned char* out = static_cast<unsigned char*>(buf) + sizeof(sds_state_header);
  const int64_t meta[16] = {ctx->F, ctx->o, ctx->p0, ctx->chunk_first,
                            ctx->sinks_filled, ctx->resets, ctx->chunks, ctx->motion_calls,
                            ctx->step_calls};
  std::memcpy(out, meta, sizeof meta);
  unsigned char* q = out + L.meta;
  struct Sec {
    const void* dev;
    int64_t bytes;
  } secs[6] = {{ctx->state, L.records}, {ctx->sink_emb, L.emb}, {ctx->ssf_ref, L.ssf},
               {ctx->mot_prev, L.mot}, {ctx->kv_k, L.with_kv ? L.kv : 0},
               {ctx->kv_v, L.with_kv ? L.kv : 0}};
  for (const Sec& sc : secs) {
    if (sc.bytes > 0) {
      e = cudaMemcpy(q, sc.dev, (size_t)sc.bytes, cudaMemcpyDeviceToHost);
      if (e != cudaSuccess) return cuda_fail(ctx, e, "state_export copy");
    }
    q += sc.bytes;
  }
  sds_state_header h;
  std::memset(&h, 0, sizeof h);
  std::memcpy(h.magic, SDS_STATE_MAGIC, 8);
  h.abi_version = SDS_ABI_VERSION;
  h.config_hash = fnv1a(&c, sizeof c);
  h.flags = L.with_kv ? 1 : 0;
  h.payload_bytes = L.payload();
  h.payload_hash = fnv1a(out, (size_t)L.payload());
  h.streams = c.streams;
  h.devstate_bytes = (int64_t)sizeof(DevState);
  h.emb_elems = L.emb_elems;
  h.ssf_ref_elems = L.ssf_elems;
  h.mot_prev_elems = L.mot_elems;
  h.kv_elems = L.kv_elems;
  std::memcpy(buf, &h, sizeof h);
  *len = need;
  return SDS_OK;
}

sds_status sds_state_import(sds_ctx* ctx, const void* buf, size_t len, sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  std::string why;
  const sds_status st = check_state(ctx->cfg, buf, len, why);
  if (st != SDS_OK) return fail(ctx, st, "state_import: %s", why.c_str());
  sds_state_header h;
  std::memcpy(&h, buf, sizeof h);
  const StateLayout L = state_layout(ctx->cfg, (h.flags & 1) != 0);
  const unsigned char* in = static_cast<const unsigned char*>(buf) + sizeof h;
  int64_t meta[16];
  std::memcpy(meta, in, sizeof meta);
  const unsigned char* q = in + L.meta;
  struct Sec {
    void* dev;
    int64_t bytes;
  } secs[6] = {{ctx->state, L.records}, {ctx->sink_emb, L.emb}, {ctx->ssf_ref, L.ssf},
               {ctx->mot_prev, L.mot}, {ctx->kv_k, L.with_kv ? L.kv : 0},
               {ctx->kv_v, L.with_kv ? L.kv : 0}};
  cudaError_t e = cudaSuccess;
  for (const Sec& sc : secs) {
    if (sc.bytes > 0 && e == cudaSuccess)
      e = cudaMemcpyAsync(sc.dev, q, (size_t)sc.bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream);
    q += sc.bytes;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "state_import copy");
  ctx->F = meta[0];
  ctx->o = meta[1];
  ctx->p0 = meta[2];
  ctx->chunk_first = meta[3];
  ctx->sinks_filled = meta[4];
  ctx->resets = meta[5];
  ctx->chunks = meta[6];
  ctx->motion_calls = meta[7];
  ctx->step_calls = meta[8];
  return SDS_OK;
}

sds_status sds_read_state(sds_ctx* ctx, sds_stream_state* out, sds_stream_t stream) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  if (!out) return fail(ctx, SDS_ERR_INVALID_ARG, "read_state: out is NULL");
  const int64_t S = ctx->cfg.streams;
  std::vector<DevState> tmp((size_t)S);
  cudaError_t e = cudaMemcpyAsync(tmp.data(), ctx->state, (size_t)S * sizeof(DevState),
                                  cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(ctx, e, "read_state");
  for (int64_t s = 0; s < S; ++s) out[s] = tmp[(size_t)s].pub;
  return SDS_OK;
}

sds_status sds_test_attn_timeout(sds_ctx* ctx, int64_t wait_limit_ns, int64_t withhold_k_tile) {
  if (!ctx) return fail(nullptr, SDS_ERR_INVALID_ARG, "ctx is NULL");
  if (wait_limit_ns < 0 || wait_limit_ns > (int64_t)kAttnWaitNs || withhold_k_tile < -1)
    return fail(ctx, SDS_ERR_INVALID_ARG,
                "test_attn_timeout: wait_limit_ns must be in [0, 2e9] (0: default) and "
                "withhold_k_tile >= -1");
  ctx->attn_wait_ns = wait_limit_ns > 0 ? (uint64_t)wait_limit_ns : kAttnWaitNs;
  ctx->attn_withhold_k = withhold_k_tile;
  return SDS_OK;
}

sds_status sds_get_meta(const sds_ctx* ctx, sds_meta* out) {
  if (!ctx || !out) return fail(nullptr, SDS_ERR_INVALID_ARG, "get_meta: NULL argument");
  out->frames_pushed = ctx->F;
  out->rope_offset = ctx->o;
  out->chunk_p0 = ctx->p0;
  out->ring_valid = std::min<int64_t>(ctx->F, ctx->cfg.ring_R);
  out->sinks_filled = ctx->sinks_filled;
  out->rope_resets = ctx->resets;
  out->chunks = ctx->chunks;
  return SDS_OK;
}

sds_status sds_get_buffers(const sds_ctx* ctx, sds_buffers* out) {
  if (!ctx || !out) return fail(nullptr, SDS_ERR_INVALID_ARG, "get_buffers: NULL argument");
  out->kv_k = ctx->kv_k;
  out->kv_v = ctx->kv_v;
  out->sink_emb = ctx->sink_emb;
  out->kv_rows = (ctx->cfg.sink_M + ctx->cfg.ring_R) * ctx->cfg.tokens_L;
  return SDS_OK;
}

}  // extern "C"
