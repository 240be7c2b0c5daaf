/*
 * sds.h -- C ABI of the stream-batch diffusion hot path for B300 (sm_103a).
 *
 * One context (sds_ctx) serves S independent streams of one workload shape.
 * Per step a caller typically issues, on one CUDA stream:
 *
 *   sds_kv_push      K2  RoPE the new chunk's keys, append K/V into the ring
 *   sds_sink_refresh K3  fill empty sinks / refresh the least similar sink
 *   sds_attend       K1  cross-frame softmax attention of all n slots' queries
 *   sds_step_update  K4  R-CFG + stream-batch update (+ SSF, + motion EMA)
 *
 * Image batch mode (ring_R == 0) skips the first two: sds_attend then takes
 * the caller's concatenated batch K/V.
 *
 * Common rules for every call below.
 *  - Pointers named "device" are CUDA device (or managed) pointers into
 *    memory the caller owns; the library never frees or retains them past
 *    the call's stream work.  Tensors are dense, row-major, without padding.
 *  - bf16 tensors are IEEE bfloat16 bit patterns; fp32 tensors are float.
 *  - Device pointers must be 16-byte aligned; element counts that feed a
 *    vectorised kernel must be multiples of 4 (checked, see each call).
 *  - Every call enqueues work on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and returns without synchronising, except
 *    sds_read_state.  Host-side metadata (frame counter, RoPE offset, ring
 *    head) advances when a call is enqueued, so calls on one context must
 *    be issued in order on one stream.
 *  - Decisions the kernels take (skip flag, refreshed sink, noise rate) stay
 *    in device memory; sds_read_state copies them out.
 *  - Arguments are validated on the host before any launch.  A failed call
 *    returns a status, changes no state and launches nothing;
 *    sds_last_error() then describes it.  CUDA launch failures map to
 *    SDS_ERR_CUDA.  Nothing aborts the process, traps or waits without bound
 *    on the device: a kernel that meets an impossible condition records it
 *    in the per-stream error word (sds_stream_state.error_word) and returns.
 *  - A context is not thread safe; use one per host thread.
 *
 * Citations name the page and the passage that define each operation:
 *  [SD]  "StreamDiffusion: A Pipeline-level Solution for Real-time
 *        Interactive Generation" (ICCV 2025 paper notes), sections
 *        "Stream Batch", "Residual CFG (R-CFG)", "Stochastic Similarity
 *        Filter (SSF)".
 *  [SDO] "StreamDiffusion complete analysis" (overview page), "Core
 *        features" and "Technical highlights" (cfg_type, max_skip_frame).
 *  [V2]  StreamDiffusionV2 summary page, "Adaptive sink and RoPE refresh",
 *        "Motion-aware noise scheduler", "SLO-aware batching scheduler".
 *  [BLOG] StreamDiffusion blog (mpbf.cn), section 7, the DDPM ancestral step.
 */
#ifndef SDS_H
#define SDS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define SDS_API __attribute__((visibility("default")))
#else
#define SDS_API
#endif

#define SDS_ABI_VERSION 5
#define SDS_MAX_SLOTS 8
#define SDS_MAX_CHUNK_FRAMES 8

typedef struct sds_ctx sds_ctx;
typedef void* sds_stream_t; /* cudaStream_t */

typedef enum {
  SDS_OK = 0,
  SDS_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or config field */
  SDS_ERR_OOM = 2,         /* device allocation failed or exceeds mem_cap_bytes */
  SDS_ERR_CUDA = 3,        /* a CUDA runtime/driver call or launch failed */
  SDS_ERR_STATE = 4,       /* call out of order (e.g. attend before any push) */
  SDS_ERR_UNSUPPORTED = 5  /* valid request this build does not implement */
} sds_status;

/*
 * Workload description, copied at sds_create.  All integers are int64 and
 * all reals double so the struct has no padding.
 *
 * Geometry: streams S; slots_n = n denoise slots of the stream batch
 * ([SD] "Stream Batch": n steps of n different frames form one batch);
 * frames_T frames per chunk; tokens_L tokens per frame; heads_H x head_dim
 * (head_dim 64 or 128); sink_M sink frames and ring_R rolling frames of
 * cached K/V ([V2] sink tokens + rolling KV cache).  ring_R == 0 selects
 * image batch mode: no ring, no RoPE, and sds_attend takes external K/V.
 *
 * RoPE: rope_on, token grid grid_h x grid_w (grid_h*grid_w == tokens_L),
 * rope_base, and rope_tau: when the next chunk's start position, counted
 * from the last reset, exceeds rope_tau the phase is reset ([V2] "reset the
 * RoPE phase when the frame index exceeds a threshold").  The head dim is
 * split into temporal/row/column segments d_t, d_y, d_x with
 * d_y = d_x = 2*floor(head_dim/6), d_t = head_dim - 2*d_y; pair (2i, 2i+1)
 * of a segment of width w turns by pos * rope_base^(-2i/w).
 *
 * Sink refresh ([V2]): emb_dim_D-dimensional chunk embeddings, threshold s_th.
 *
 * Schedule ([SD] R-CFG, [BLOG]): num_train_steps betas, scaled linear from
 * beta_start to beta_end; slot i runs at timestep
 * (num_train_steps-1) - t_index[i]*(num_train_steps/num_inference_steps).
 * cfg_type: 0 = no guidance (eps_cfg = eps_c), 1 = self-negative R-CFG with
 * gamma, delta ([SDO] cfg_type="self"), 2 = R-CFG with a supplied negative
 * prediction per slot (sds_step_io.eps_neg): the onetime-negative variant
 * ([SD] R-CFG, one negative evaluation; [SDO] cfg_type="initialize"), and,
 * with delta = 1 and unconditional predictions, standard CFG.
 * noise_rate_on: 1 applies the motion-aware noise rate s ([V2] "Motion-aware
 * noise scheduler": the rate adapts the denoising path to the motion) to
 * the incoming frame: it enters slot 0 at timestep t_s = t1 + round(s *
 * (num_train_steps - 1 - t1)), the fraction s of the way from slot 1's
 * timestep t1 (0 when slots_n == 1) up to pure noise, instead of slot 0's
 * fixed timestep, so that it is never less noisy than the frame in slot 1
 * ([SD] "Stream Batch": the slots hold descending timesteps).  The rate is
 * the one decided by the previous step, and the next update treats that
 * frame at t_s (needs motion_on and 0 <= s_min <= s_max <= 1;
 * sds_stream_state.slot0_timestep reports t_s).
 * eps_c_bf16: 1 = the eps_c[i] buffers hold bf16 values (the usual output
 * dtype of the noise-prediction network); the update widens them exactly
 * to fp32.  0 = fp32.
 * txt2img: 1 = no input image ([SDO] txt2img): the incoming frame is the
 * noise draw eps_new itself (the initial latent), x0_new is not read and
 * may be NULL; cfg_type must be 0 or 2 (self-negative R-CFG needs x0) and
 * noise_rate_on 0.
 * update_kind: 0 = predict x0 and re-noise it to the next slot's level;
 * 1 = the DDPM ancestral step ([BLOG] section 7) taken between the slot's
 * timestep t and the next slot's t', with alpha = abar_t / abar_t' and
 * sigma^2 = (1 - abar_t') / (1 - abar_t) * (1 - alpha) (posterior variance).
 *
 * slot_elems: fp32 elements of one slot latent (T * frame_elems in video).
 * SSF ([SD] SSF, [SDO]): ssf_elems per frame, ssf_eta, max_skip_frame.
 * Motion ([V2]): frame_elems per latent frame, window mot_k, mot_sigma,
 * mot_lambda, noise-rate bounds s_min <= s_max.
 *
 * mem_cap_bytes: if nonzero, sds_create fails with SDS_ERR_OOM when the
 * context's device memory would exceed it (no allocation is attempted).
 *
 * attn_ctas: 0 lets sds_attend choose its grid (one CTA per pair of 128-row
 * query tiles, or, when that leaves a ragged last wave on a large problem,
 * one persistent CTA per SM with the keys of some tiles split between CTAs).
 * A positive value forces the persistent split schedule on at most that
 * many CTAs (capped at 160), e.g. to leave SMs to concurrent work.
 */
typedef struct {
  int64_t abi_version; /* must equal SDS_ABI_VERSION */
  int64_t streams, slots_n, frames_T, tokens_L, heads_H, head_dim, sink_M, ring_R;
  int64_t rope_on, grid_h, grid_w, rope_tau;
  int64_t emb_dim_D;
  int64_t t_index[SDS_MAX_SLOTS];
  int64_t num_inference_steps, num_train_steps, cfg_type;
  int64_t slot_elems;
  int64_t ssf_on, ssf_elems, max_skip_frame;
  int64_t motion_on, frame_elems, mot_k;
  int64_t mem_cap_bytes;
  int64_t attn_ctas;
  int64_t update_kind;
  int64_t noise_rate_on;
  int64_t eps_c_bf16;
  int64_t txt2img;
  double rope_base, s_th, beta_start, beta_end, gamma, delta, ssf_eta;
  double mot_sigma, mot_lambda, s_min, s_max;
} sds_config;

/*
 * Inputs and outputs of one stream-batch update (sds_step_update).  Every
 * array is fp32, device, [S][slot_elems] (stream-major) unless stated.
 *   x[i]      slot i's current latent x_{t_i}, i < n
 *   x0[i]     slot i's own input-frame latent (the R-CFG x0)
 *   eps_c[i]  the model's conditional noise prediction for slot i (bf16
 *             values when eps_c_bf16; 16-byte aligned either way)
 *   z[i]      ancestral noise that re-noises slot i's prediction to slot
 *             i+1's level, i < n-1
 *   x_next[i] next step's latents: x_next[0] is the incoming frame noised to
 *             slot 0's level; x_next[i+1] comes from slot i.  x_next[i] may
 *             alias x[i] (in-place update is safe).
 *   out       the completed frame: slot n-1's predicted x0
 *   x0_new, eps_new  the incoming frame's latent and its noise (txt2img:
 *             x0_new unused, the incoming frame is eps_new)
 *   ssf_frame [S][ssf_elems] or NULL: run the similarity filter on this
 *             frame in the same pass; ssf_u [S] uniform draws in [0,1)
 *   motion_chunk [S][frames_T][frame_elems] or NULL: update the motion
 *             estimate and noise rate from these latent frames
 *   eps_neg[i] cfg_type 2 only: slot i's negative (or unconditional)
 *             noise prediction; slots may share one buffer
 * x0 shifting between steps (slot i+1's x0 is this step's x0[i]) is left to
 * the caller, which can rotate the pointers at no cost.
 */
typedef struct {
  const float* x[SDS_MAX_SLOTS];
  const float* x0[SDS_MAX_SLOTS];
  const float* eps_c[SDS_MAX_SLOTS];
  const float* z[SDS_MAX_SLOTS];
  float* x_next[SDS_MAX_SLOTS];
  float* out;
  const float* x0_new;
  const float* eps_new;
  const float* ssf_frame;
  const float* ssf_u;
  const float* motion_chunk;
  const float* eps_neg[SDS_MAX_SLOTS];
} sds_step_io;

/* Per-stream decisions, as of the last completed call that made them. */
typedef struct {
  int64_t ssf_evals;      /* frames the filter has seen */
  int64_t ssf_skip;       /* last frame skipped (1) or processed (0) */
  int64_t ssf_skip_count; /* consecutive skips so far */
  int64_t ssf_has_ref;    /* a reference frame exists */
  double ssf_cos;         /* cosine of the last frame vs the reference */
  double ssf_p;           /* its skip probability */
  int64_t sink_j;         /* last refresh: chosen sink (-1 if none) */
  int64_t sink_fire;      /* 0 kept, 1 replaced, 2 filled an empty sink */
  double sink_alpha_min;  /* smallest cosine of the last refresh test */
  double sink_alpha_2;    /* second smallest (+inf if M == 1) */
  int64_t motion_pairs;   /* motion values measured so far */
  double motion_dhat;     /* last normalised, clipped motion */
  double noise_rate;      /* EMA noise rate s */
  double motion_d[SDS_MAX_CHUNK_FRAMES]; /* last chunk's pair motions (NaN if absent) */
  int64_t error_word;     /* nonzero: a kernel met an impossible condition */
  int64_t slot0_timestep; /* timestep of the frame now in slot 0 */
} sds_stream_state;

/* Host-side ring metadata (identical for all streams of a context). */
typedef struct {
  int64_t frames_pushed; /* F */
  int64_t rope_offset;   /* o: positions count from frame o */
  int64_t chunk_p0;      /* start position of the last pushed chunk */
  int64_t ring_valid;    /* min(F, R) */
  int64_t sinks_filled;
  int64_t rope_resets;
  int64_t chunks;
} sds_meta;

/* Device buffers owned by the context, valid until sds_destroy. */
typedef struct {
  void* kv_k;      /* bf16 [S][(M+R)*L][H][d]: sink frames, then ring frames */
  void* kv_v;      /* same layout */
  float* sink_emb; /* fp32 [S][M][D] */
  int64_t kv_rows; /* (M+R)*L */
} sds_buffers;

/* ABI version the library was built with (SDS_ABI_VERSION). */
SDS_API int sds_abi_version(void);

/*
 * Validate cfg, allocate the context's device buffers (K/V ring and sinks,
 * sink embeddings, RoPE cos/sin table, schedule coefficients, SSF reference
 * frames, motion previous frames, decision state, reduction scratch) on the
 * current CUDA device, zero them, and return the context in *out.
 * No allocation happens after this call.
 * Errors: SDS_ERR_INVALID_ARG (cfg), SDS_ERR_OOM, SDS_ERR_CUDA.  On error
 * *out is NULL and sds_last_error(NULL) describes the failure.
 */
SDS_API sds_status sds_create(const sds_config* cfg, sds_ctx** out);

/* Free the context and its device buffers (synchronises the device). */
SDS_API void sds_destroy(sds_ctx* ctx);

/* Description of the last error on ctx (ctx == NULL: the last failed create
 * on this thread).  The string is owned by the library. */
SDS_API const char* sds_last_error(const sds_ctx* ctx);

/*
 * K2 -- ring append with RoPE ([V2] rolling KV cache; "Adaptive sink and
 * RoPE refresh").  k, v: device bf16 [S][T*L][H][d], the new chunk's keys
 * and values.  Computes the chunk start position p0 = F - o (reset: if
 * p0 > rope_tau then o = F, p0 = 0), rotates each key of frame j, token
 * (y, x) at positions (p0 + j, y, x) in fp32 and stores it as bf16; copies
 * the values; frame F + j goes to ring slot (F + j) mod R, overwriting the
 * oldest frame.  Then F += T.
 * Errors: SDS_ERR_STATE in image mode; SDS_ERR_INVALID_ARG for NULL or
 * misaligned pointers.
 */
SDS_API sds_status sds_kv_push(sds_ctx* ctx, const void* k, const void* v, sds_stream_t stream);

/*
 * K3 -- adaptive sink refresh ([V2] "Adaptive sink and RoPE refresh": the
 * least similar sink is refreshed when the cosine of the new chunk embedding
 * to it falls below s_th).  chunk_emb: device fp32 [S][D].
 * While sinks are empty, they are filled in index order from frames 0, 1, ..
 * of the chunk just pushed, and take chunk_emb as their embedding.  Once
 * full: alpha_j = cos(h, e_j) in double, j* = argmin (lowest index on
 * ties); if alpha_{j*} < s_th, sink j*'s K/V become frame 0 of the chunk
 * just pushed (already rotated) and e_{j*} = h.  The decision is taken on
 * the device; nothing is read back.  No-op when sink_M == 0.
 * Errors: SDS_ERR_STATE before the first push or in image mode.
 */
SDS_API sds_status sds_sink_refresh(sds_ctx* ctx, const float* chunk_emb, sds_stream_t stream);

/*
 * K1 -- cross-frame attention ([SD] "Stream Batch": Attn(Q_{t,i}, K_Batch,
 * V_Batch) = Softmax(Q K_Batch^T / sqrt(d)) V_Batch).
 * q: device bf16 [S][n*T*L][H][d] (video) or [S][n*L][H][d] (image): the
 * queries of all n slots, stacked.  o: device bf16, same shape as q.
 * Video mode (ext_k == ext_v == NULL): every query row of the last pushed
 * chunk is rotated at (p0 + j, y, x) (all slots share the chunk's
 * positions), then attends to all valid keys: the filled sinks and the
 * filled ring frames (including the chunk just pushed); no causal mask.
 * Image mode: ext_k, ext_v device bf16 [S][n*L][H][d], the batch K/V; no
 * RoPE.  Softmax in fp32 with bf16 tensor-core products, output rounded
 * to bf16.
 * Errors: SDS_ERR_STATE (video mode before any push); SDS_ERR_INVALID_ARG.
 */
SDS_API sds_status sds_attend(sds_ctx* ctx, const void* q, void* o, const void* ext_k,
                      const void* ext_v, sds_stream_t stream);

/*
 * Context-free attention: o = Softmax(q k^T / sqrt(d)) v for each of S
 * independent problems, q/o device bf16 [S][Lq][H][d], k/v device bf16
 * [S][Lk][H][d], head_dim 64 or 128, no RoPE ([SD] cross-frame attention
 * equation).  Lq >= 1, Lk >= 1.
 */
SDS_API sds_status sds_attention(const void* q, const void* k, const void* v, void* o, int64_t S,
                         int64_t Lq, int64_t Lk, int64_t H, int64_t head_dim,
                         sds_stream_t stream);

/*
 * K4 -- one fused pass ([SD] "Residual CFG", [BLOG] update, [SD] "SSF",
 * [V2] "Motion-aware noise scheduler").  Per slot i, with a = alphabar of
 * slot i's timestep, in fp32 with host-double coefficients:
 *   eps_neg = (x_i - sqrt(a) x0_i) / sqrt(1 - a)   (cfg_type 1; cfg_type 2:
 *             the supplied io->eps_neg[i])
 *   eps_cfg = gamma eps_c + delta (1 - gamma) eps_neg   (= the printed
 *             delta eps_neg + gamma (eps_c - delta eps_neg))
 *   x0hat   = (x_i - sqrt(1 - a) eps_cfg) / sqrt(a)
 *   x_next[i+1] = sqrt(a_{i+1}) x0hat + sqrt(1 - a_{i+1}) z_i  (i < n-1;
 *             update_kind 1: (x_i - (1 - al) / sqrt(1 - a) eps_cfg) / sqrt(al)
 *             + sigma z_i with al = a / a_{i+1})
 *   out = x0hat of slot n-1;  x_next[0] = sqrt(a_0) x0_new + sqrt(1-a_0) eps_new.
 * With io->ssf_frame: the similarity filter of sds_ssf on that frame.
 * With io->motion_chunk: per frame pair the RMS difference d (the previous
 * chunk's last frame pairs with frame 0); dhat = min(1, max of the last
 * mot_k values / mot_sigma); target = s_min + (s_max - s_min) dhat;
 * s <- s + (1 - mot_lambda)(target - s); s starts at s_min.
 * Reductions are deterministic (fixed order, fp32 within a thread, double
 * beyond), finished by the last block of the launch.
 * Errors: SDS_ERR_INVALID_ARG (NULL/misaligned arrays, ssf/motion requested
 * but disabled in the config, sizes not multiples of 4).
 */
SDS_API sds_status sds_step_update(sds_ctx* ctx, const sds_step_io* io, sds_stream_t stream);

/*
 * K4, filter only ([SD] "SSF": P(skip) = max{0, (S_C(I_t, I_ref) - eta) /
 * (1 - eta)} with the cosine S_C, sampled not thresholded; [SDO] at most
 * max_skip_frame consecutive skips).  frame: device fp32 [S][ssf_elems];
 * u: device fp32 [S], uniform draws in [0,1).  Per stream: the first frame
 * is processed; then c = cos(I, I_ref) (0 if a norm is 0), P = min(1,
 * max(0, (c - eta)/(1 - eta))), skip = (u < P) and (skip_count <
 * max_skip_frame).  A processed frame becomes the reference.
 */
SDS_API sds_status sds_ssf(sds_ctx* ctx, const float* frame, const float* u, sds_stream_t stream);

/*
 * Allocation-free similarity filter.  The pages have no counterpart: it is
 * a service of this library for callers that cannot allocate device memory
 * -- code working inside a fixed device-memory budget owned by another
 * allocator, or in a latency-critical loop where cudaMalloc/cudaFree (which
 * may synchronise the device) are not allowed -- and so cannot create a
 * context.  It computes what sds_ssf computes, on a reference frame the
 * caller supplies instead of the context's stored one, with K4's reduction
 * and decision unchanged (the same work blocks of SDS_NOALLOC_BLOCK_ELEMS
 * elements, the same per-thread and per-block sums, the same finish): for
 * the same frame, reference, draw and skip count it returns bit for bit the
 * cosine, probability and decision that sds_ssf records.  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *   frame, ref  device fp32 [S][E]: incoming frame and reference frame
 *   u           device fp32 [S]: uniform draws in [0,1)
 *   skip_count  device int64 [S] consecutive skips so far, or NULL (all 0)
 *   cos_out, p_out  device double [S]; skip_out device int64 [S]
 *   skip = (u < P) and (skip_count < max_skip)
 *
 * Scratch: a static device array of SDS_NOALLOC_SCRATCH_BYTES (256 KiB) in
 * the library, present on every GPU that loads the library until the process
 * exits.  Its reduction partials limit the size: S * ceil(E / 8192) * 3 must
 * not exceed SDS_NOALLOC_MAX_PARTIALS (32736; e.g. S <= 113 streams of
 * 3x512x512 frames); larger requests fail with SDS_ERR_INVALID_ARG and a
 * message in sds_last_error(NULL).  The first call in a device context looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.  A context that
 * is destroyed and created again (cudaDeviceReset) gets a fresh lookup on
 * its first call.  Every call shares the one array and clears its counter on
 * `stream` before use, so calls whose work overlaps on the GPU (other
 * streams, other host threads) race on it: order them.
 */
#define SDS_NOALLOC_BLOCK_ELEMS 8192
#define SDS_NOALLOC_SCRATCH_BYTES 262144
#define SDS_NOALLOC_MAX_PARTIALS 32736
SDS_API sds_status sds_ssf_noalloc(const float* frame, const float* ref, const float* u,
                                   const int64_t* skip_count, int64_t S, int64_t E, double eta,
                                   int64_t max_skip, double* cos_out, double* p_out,
                                   int64_t* skip_out, sds_stream_t stream);

/*
 * Checkpoints.  A checkpoint is an sds_state_header followed by a payload of
 * 8-byte aligned sections, in this order:
 *   meta      int64[16]: frames pushed F, RoPE offset o, last chunk start
 *             p0, first frame of the last chunk, sinks filled, RoPE resets,
 *             chunks pushed, motion updates done, update steps done, then
 *             zeros
 *   records   S per-stream device records (devstate_bytes each; the public
 *             sds_stream_state first, then private SSF / motion fields)
 *   sink_emb  fp32 [S][M][D]
 *   ssf_ref   fp32 [2][S][ssf_elems]      (when ssf_on)
 *   mot_prev  fp32 [2][S][frame_elems]    (when motion_on)
 *   kv_k, kv_v bf16 [S][(M+R)*L][H][d]    (when flags bit 0: with K/V)
 * payload_hash and config_hash are 64-bit FNV-1a hashes of the payload bytes
 * and of the sds_config bytes.  A checkpoint restores only into a context
 * created with a byte-identical sds_config.
 */
#define SDS_STATE_MAGIC "SDSSTAT1"
#define SDS_STATE_RECORD_BYTES 760 /* devstate_bytes of this ABI version */
typedef struct {
  char magic[8];           /* SDS_STATE_MAGIC without its terminating NUL */
  int64_t abi_version;     /* SDS_ABI_VERSION of the writer */
  uint64_t config_hash;
  int64_t flags;           /* bit 0: K/V ring and sinks included */
  int64_t payload_bytes;
  uint64_t payload_hash;
  int64_t streams;
  int64_t devstate_bytes;  /* size of one per-stream device record */
  int64_t emb_elems, ssf_ref_elems, mot_prev_elems, kv_elems; /* per tensor */
  int64_t reserved[4];     /* zero */
} sds_state_header;

/*
 * Write a checkpoint of ctx to buf (host memory, *len bytes available).
 * with_kv != 0 includes the K/V ring and sinks (the bulk of the bytes).
 * buf == NULL: only stores the needed size in *len.  Synchronises `stream`
 * first, so the checkpoint reflects all work enqueued before the call.
 * Errors: SDS_ERR_INVALID_ARG (len NULL, or *len too small: *len then holds
 * the needed size), SDS_ERR_CUDA.
 */
SDS_API sds_status sds_state_export(sds_ctx* ctx, void* buf, size_t* len, int64_t with_kv,
                                    sds_stream_t stream);

/*
 * Restore a checkpoint written by sds_state_export into ctx.  The buffer is
 * validated first (sds_state_check against ctx's config); a rejected buffer
 * changes nothing.  A checkpoint without K/V leaves the ring and sinks as
 * they are.  Synchronises `stream` before returning (buf may be freed then).
 * Errors: SDS_ERR_STATE (bad magic, version, config, sizes or payload hash),
 * SDS_ERR_CUDA (the copy failed: destroy the context).
 */
SDS_API sds_status sds_state_import(sds_ctx* ctx, const void* buf, size_t len,
                                    sds_stream_t stream);

/*
 * Validate a checkpoint against a configuration without touching any
 * device: magic, ABI version, config hash, section sizes and payload hash.
 * Returns SDS_OK or SDS_ERR_STATE / SDS_ERR_INVALID_ARG with a message in
 * sds_last_error(NULL).
 */
SDS_API sds_status sds_state_check(const sds_config* cfg, const void* buf, size_t len);

/*
 * SLO-aware stream-batch controller (host only, no device work).
 * [V2] "SLO-aware batching scheduler": per iteration the system processes
 * B*T frames (B streams, T frames each) with latency L(T,B); in the
 * memory-bound regime L is affine in the activation volume, which is linear
 * in B*T, so the controller fits L = a + b*B*T to the observed latencies
 * (least squares, older observations down-weighted by `forget`).  A stream
 * meets the SLO when T / L >= target_fps; the aggregate rate is B*T / L.
 * The choice is the largest B in [b_min, b_max] that meets the SLO, capped
 * at the knee: the smallest B whose predicted aggregate rate is within
 * knee_gain of the rate at b_max (more streams beyond it add latency, not
 * throughput).  Until two distinct B have been observed it proposes the
 * next unobserved B from b_min up (exploration).
 */
typedef struct sds_slo sds_slo;
typedef struct {
  double target_fps;  /* per-stream frame-rate objective, frames/s (> 0) */
  double forget;      /* weight of an observation after each newer one, (0, 1] */
  double knee_gain;   /* relative throughput gain below which B stops growing, [0, 1) */
  int64_t frames_T;   /* frames per stream per iteration (>= 1) */
  int64_t b_min, b_max; /* 1 <= b_min <= b_max */
} sds_slo_config;

typedef struct {
  int64_t batch;          /* chosen B */
  int64_t meets_slo;      /* 1 if the model predicts T / L(B) >= target_fps */
  int64_t exploring;      /* 1 while fewer than two distinct B were observed */
  int64_t b_slo, b_knee;  /* largest B meeting the SLO (0: none), knee B */
  double a, b;            /* fitted L = a + b*B*T (seconds, seconds per frame) */
  double latency_s, per_stream_fps, total_fps; /* predicted at the chosen B */
} sds_slo_choice;

SDS_API sds_status sds_slo_create(const sds_slo_config* cfg, sds_slo** out);
SDS_API void sds_slo_destroy(sds_slo* c);
/* Record one iteration: B streams took latency_s seconds (> 0). */
SDS_API sds_status sds_slo_observe(sds_slo* c, int64_t batch, double latency_s);
/* The controller's current choice (see above). */
SDS_API sds_status sds_slo_choose(const sds_slo* c, sds_slo_choice* out);

/* Synchronise `stream` and copy the S per-stream decision records to host
 * memory out[0..S-1]. */
SDS_API sds_status sds_read_state(sds_ctx* ctx, sds_stream_state* out, sds_stream_t stream);

/*
 * Failure-detection test hook for K1's bounded waits (no counterpart on the
 * pages).  Every wait of the attention kernel on a barrier gives up after a
 * time limit (2 s by default); the kernel then records a timeout in the
 * error word of every stream (sds_stream_state.error_word bit 0), waits,
 * again bounded, for its own copies in flight, frees its tensor memory and
 * returns, so the context stays usable.  This call lets a test exercise
 * that path without a fault: wait_limit_ns (> 0) shortens the limit (0
 * restores 2 s), and withhold_k_tile >= 0 makes CTA 0 of the following
 * sds_attend launches skip the copy of that key tile (its counter over the
 * CTA's tiles), so the waits for it run out; -1 turns that off.  Outputs of
 * a launch that timed out are undefined.  With the split-key schedule a
 * timed-out CTA leaves its arrival counters behind, so use it only on
 * problems of one work item per CTA (attn_ctas 0 and a small problem).
 * Errors: SDS_ERR_INVALID_ARG.
 */
SDS_API sds_status sds_test_attn_timeout(sds_ctx* ctx, int64_t wait_limit_ns,
                                         int64_t withhold_k_tile);

/* Host-side ring metadata (no device access). */
SDS_API sds_status sds_get_meta(const sds_ctx* ctx, sds_meta* out);

/* Device buffers owned by the context (for inspection and checkpoints). */
SDS_API sds_status sds_get_buffers(const sds_ctx* ctx, sds_buffers* out);

#ifdef __cplusplus
}
#endif

#endif /* SDS_H */
