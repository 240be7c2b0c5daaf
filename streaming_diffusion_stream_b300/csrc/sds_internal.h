// sds_internal.h -- declarations shared by the library's translation units
// (host API in sds_api.cu, kernels in k_*.cu).  Not part of the ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/sds.h"

namespace sds {

constexpr int kMaxMotionWindow = 64;

// Device-side per-stream record: the exported decisions plus private state.
struct DevState {
  sds_stream_state pub;
  int64_t ssf_cur;     // which of the two reference buffers holds I_ref
  int64_t mot_count;   // values in the window (<= mot_k)
  int64_t mot_head;    // next write position in the circular window
  int64_t mot_has_prev;
  double mot_window[kMaxMotionWindow];
  // noise-rate application, by update-step parity (a step reads [par] and
  // writes the next step's [par ^ 1]): the timestep at which the step's
  // incoming frame enters slot 0, and the timestep of the frame already there
  int64_t entry_t_buf[2];
  int64_t slot0_t_buf[2];
};

static_assert(sizeof(DevState) == SDS_STATE_RECORD_BYTES,
              "the checkpoint record size is part of the ABI");

// Error bits recorded in DevState::pub.error_word.
enum : int64_t {
  kErrAttnWaitTimeout = 1 << 0,
  kErrAttnBadShape = 1 << 1,
  kErrStepBadArgs = 1 << 2,
  kErrSinkBadArgs = 1 << 3,
};

// ----------------------------------------------------------------- K1 attention
struct AttnParams {
  uint16_t* o;           // bf16 [S][q_rows][H][d]
  int64_t q_rows;        // query rows per stream
  int32_t S;             // independent problems (streams)
  int32_t H;
  int32_t seg_start[2];  // key row ranges inside the K/V tensor of a stream
  int32_t seg_count[2];
  float scale_log2;      // log2(e) / sqrt(d)
  int32_t rope_on;
  int32_t p0;            // temporal position of frame 0 of the chunk
  int32_t tokens_L, grid_w, chunk_tokens;
  int32_t rope_seg[3];   // d_t, d_y, d_x
  const float2* rope_tab;
  int32_t tab_off[3];    // entry offset of each axis table
  DevState* state;       // per stream, for error reporting (may be null)
  // Split-key workspace of the persistent schedule.  Null: one work item
  // (a pair of 128-row query tiles of one stream and head, all keys) per
  // CTA, nothing is split.  Otherwise a grid of at most kAttnMaxCtas CTAs
  // divides the (item, key tile) units evenly; an item whose keys are split
  // between CTAs is finished by the last contributor to arrive.
  float* ws_o;           // [kAttnMaxCtas][2 slots][2 tiles][128 rows][d] partial O, fp32
  float2* ws_ml;         // [kAttnMaxCtas][2][2][128] partial (running max, sum)
  unsigned int* ws_cnt;  // [kAttnMaxCtas][2][128] arrival counters, zero between launches
  int32_t grid;          // CTAs of the persistent schedule (0: the device's SM count)
  uint64_t wait_ns;      // limit of every wait on a barrier (kAttnWaitNs unless a test shortens it)
  int64_t withhold_k;    // test hook: >= 0 makes CTA 0 skip the key copy of that tile (-1: off)
};

constexpr uint64_t kAttnWaitNs = 2000000000ull;  // 2 s

constexpr int kAttnMaxCtas = 160;  // >= the SM count of the target part (148)
// Bytes of the split-key workspace for head_dim d.
inline size_t attn_ws_bytes(int d) {
  return (size_t)kAttnMaxCtas * 2 * 2 * 128 * ((size_t)d * 4 + 8) + (size_t)kAttnMaxCtas * 2 * 128 * 4;
}

// q/k/v/o tensor maps: 3-D {H*d, rows, S}, box {64, 128, 1}, 128-byte swizzle.
// to: the output o as the same kind of map (written by TMA at the end of a
// CTA's last item).
cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& to, const AttnParams& p, int head_dim, int S,
                             int sm_count, cudaStream_t st);

// Build a bf16 3-D tensor map {H*d, rows, S} with a {64, 128, 1} box.
bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t hd, int64_t rows, int64_t S);

// ----------------------------------------------------------------- K2 / K3
struct PushParams {
  const uint4* k_in;  // bf16 [S][T*L][H*d] as 8-element vectors
  const uint4* v_in;
  uint4* kv_k;        // bf16 [S][(M+R)*L][H*d]
  uint4* kv_v;
  int64_t S, T, L, HD, M, R, head_dim;
  int64_t F;          // frames pushed before this chunk
  int32_t p0, rope_on, grid_w;
  int32_t rope_seg[3];
  const float2* rope_tab;
  int32_t tab_off[3];
};
cudaError_t launch_kv_push(const PushParams& p, int sm_count, cudaStream_t st);

struct SinkParams {
  const float* h;       // [S][D]
  float* emb;           // [S][M][D]
  uint4* kv_k;          // bf16 [S][(M+R)*L][H*d]
  uint4* kv_v;
  DevState* state;       // the decision kernel's record, read by the copy kernel
  int64_t S, D, M, R, L, HD;
  int64_t chunk_first;  // global index of frame 0 of the chunk just pushed
  int64_t fill_from;    // >= 0: fill mode, first empty sink; < 0: similarity test
  int64_t fill_count;
  double s_th;
};
// Two launches: the decision (one block per stream), then the copy.
cudaError_t launch_sink_refresh(const SinkParams& p, int sm_count, cudaStream_t st);

// ----------------------------------------------------------------- K4
struct StepParams {
  // update segment
  const float* x[SDS_MAX_SLOTS];
  const float* x0[SDS_MAX_SLOTS];
  const float* eps_c[SDS_MAX_SLOTS];
  const float* z[SDS_MAX_SLOTS];
  float* x_next[SDS_MAX_SLOTS];
  float* out;
  const float* x0_new;
  const float* eps_new;
  float c_sa[SDS_MAX_SLOTS];       // sqrt(abar_i)
  float c_inv_s1a[SDS_MAX_SLOTS];  // 1 / sqrt(1 - abar_i)
  float c_s1a[SDS_MAX_SLOTS];      // sqrt(1 - abar_i)
  float c_inv_sa[SDS_MAX_SLOTS];   // 1 / sqrt(abar_i)
  float c_gamma, c_dg;             // gamma, delta * (1 - gamma)
  const float* eps_neg[SDS_MAX_SLOTS];  // supplied negative predictions (cfg_kind 2)
  int32_t cfg_kind;                // 0 none, 1 self-negative (from x0), 2 supplied eps_neg
  int32_t upd_kind;                // 0 x0hat re-noised, 1 strided DDPM posterior
  float c_px[SDS_MAX_SLOTS];       // DDPM: 1 / sqrt(alpha_i)
  float c_pe[SDS_MAX_SLOTS];       // DDPM: (1 - alpha_i) / (sqrt(alpha_i) sqrt(1 - abar_i))
  float c_sig[SDS_MAX_SLOTS];      // DDPM: sigma_i
  // noise-rate application: slot 0's coefficients come from per-stream
  // timesteps through the abar table
  int32_t rate_on, par;
  int32_t ec_bf16;   // eps_c[i] hold bf16 values
  int32_t txt2img;   // the incoming frame is eps_new itself
  // per-timestep coefficient tables [7][n_train]: sqrt(abar), 1/sqrt(1-abar),
  // sqrt(1-abar), 1/sqrt(abar), and the strided DDPM step to slot 1's
  // timestep: 1/sqrt(alpha), (1-alpha)/(sqrt(alpha) sqrt(1-abar)), sigma
  const float* coef_tab;
  int64_t n_train;
  int64_t t_floor;                 // slot 1's timestep (0 with one slot): the lowest entry timestep
  int32_t n;                       // slots (0: no update segment)
  int64_t N_s;
  // SSF segment
  const float* ssf_frame;          // null: no SSF
  const float* ssf_u;
  float* ssf_ref;                  // [2][S][E]
  int64_t E;
  double eta;
  int64_t max_skip;
  // motion segment
  const float* mot_chunk;          // null: no motion; [S][T][N_f]
  const float* mot_prev_in;        // [S][N_f]
  float* mot_prev_out;             // [S][N_f]
  int64_t T, N_f, mot_k;
  double sigma, lam, s_min, s_max;
  // common
  int64_t S;
  DevState* state;
  double* partials;
  unsigned int* counter;
  int64_t nb_u, nb_s, nb_m;        // work blocks per stream (per pair for motion)
};
// Message for sds_last_error(NULL) from entry points without a context.
void set_thread_error(const char* msg);

constexpr int kStepThreads = 256;
constexpr int kRedBlockElems = 8192;  // elements per SSF / motion work block (32 per thread)
constexpr int kUpdBlockElems = 1024;  // elements per update work block (4 per thread)
cudaError_t launch_step(const StepParams& p, int sm_count, cudaStream_t st);

}  // namespace sds
