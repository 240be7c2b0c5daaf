// k_attn.cu -- K1: cross-frame softmax attention on tcgen05 tensor cores.
//
// StreamDiffusion notes, "Stream Batch": the n denoise slots form one batch
// and every slot's queries attend to the keys of the whole batch,
// Attn(Q_{t,i}, K_Batch, V_Batch) = Softmax(Q K_Batch^T / sqrt(d)) V_Batch.
// In video mode the key set is the sink + rolling ring of cached frames
// (StreamDiffusionV2 summary, sink tokens + rolling KV cache).
//
// Work decomposition.  A work item is a pair of 128-row query tiles (Q0, Q1)
// of one (stream, head) against all of its keys, processed as 128-key
// tiles.  The (item, key tile) units of a launch are divided evenly over a
// persistent grid (one CTA per SM), so a CTA may start or stop inside an
// item.  A CTA that covers only part of an item's keys writes its partial
// result (unnormalised O, running max m, running sum l per row) to a
// workspace and counts itself in per-row arrival counters; the contributor
// that arrives last merges the partials and writes the output.  Nobody
// waits for anybody, so a slow CTA cannot stall another.  Without a
// workspace the grid has one CTA per item and nothing is split.
//
// Warp roles inside a CTA:
//   warps 0-3  softmax group 0 (tile Q0), one query row per thread = one TMEM lane
//   warps 4-7  softmax group 1 (tile Q1)
//   warp  8    TMA producer: K and V tiles of 128 keys through an ST-stage ring, Q per item
//   warps 9-10 MMA issuers (one thread each): issuer t serves query tile t
//              (d = 128: its S products only)
//   warp  11   d = 128 only: the PV products of both query tiles
// d = 64.  Tensor memory (512 columns): S0, S1 (128 each, fp32 scores),
// P0, P1 (64 each, packed bf16), O0, O1 (64 each).  Issuer t issues S_t(g+1)
// as soon as group t has read S_t(g) into registers (s_free), then PV_t(g)
// once P_t(g) is written, so the next scores are ready when the softmax
// finishes the current tile.  Group t writes P_t(g) only after PV_t(g-1)
// has completed; it waits for that three quarters of the way through its
// exponentials, holding those parts of P in registers.  Issuer t releases the K stage
// of tile g together with its V stage, after PV_t(g) (see the overflow case
// below).  At an item boundary PV_t(g) is issued before S_t(g+1), because
// the next item's queries are rotated by the softmax only once it has
// finished the current item.
// d = 128.  Each loaded key tile is consumed as two 64-key compute tiles.
// Tensor memory per group t: two score buffers [t*256, +64), [t*256 + 64,
// +64) and O_t [t*256 + 128, +128).  P_t(g) is written over the first 32
// columns of its score buffer.  The MMA stream bounds d = 128 (an issuing
// thread needs 72-78 cycles per MMA, and the S products run at N = 64), so
// it is spread over three warps: warp 9 + t issues S_t, warp 11 issues PV
// for both tiles.  S_t(g+2) goes into the buffer of S_t(g) once PV_t(g)
// has completed (an o_done barrier per buffer), keeping the scores of the
// next compute tile ready while the softmax works on the current one.
// Each score buffer has its own s_full / p_full / o_done barriers, so that
// no barrier can run two phases ahead of its waiter (a parity wait
// distinguishes only the current and the previous phase).
// In both cases the waits for K/V data, which the producer lands several
// tiles ahead, are taken before the wait for P so they stay off the
// critical path.
// The online softmax keeps a reference m per row (O and the row sum l are
// kept relative to 2^m) and rescales O in tensor memory when m moves.
// d = 128: m is the running maximum; each tile's row maximum is taken
// first (a three-input max) and m moves only when a tile raises it by more
// than 8 (log2 units), so probabilities stay below 2^8, which fp32 sums and
// bf16 P hold without loss.
// d = 64: after an item's first tile (maximum first, m = maximum + 64) the
// exponentials go against m with no tile maximum at all: taking it costs
// as much ALU time as the exponentials leave free.  Probabilities are >= 0,
// so a row sum <= 2^8 bounds every one of them, and in the usual case that
// is all there is to check.  A larger finite sum (a row's scores rose more
// than about 64 above its earlier maximum) moves m up by a whole k: the
// row's largest stored P gives k, and P, the sum and O are multiplied by the
// exact power of two 2^-k.  An infinite sum (a rise of 192 or more: exp2
// overflowed) redoes the tile maximum first from scores recomputed on the
// CUDA cores from Q and K in shared memory; K(g) is still there because its
// stage is released only after PV(g).  Offsetting m by 64 above the
// maximum only drops probabilities below 2^-62 of the row's largest.
// Score scaling and row sums use packed
// f32x2 arithmetic, halving their instruction count.  Every wait has a time
// limit (the launch's wait_ns); on expiry the kernel records
// kErrAttnWaitTimeout in the error word of every stream and leaves.
// The schedule knobs (SDS_K1_*) select measured alternatives of the same
// computation; their defaults are the fastest measured on a B300.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "ptx.cuh"
#include "rope.cuh"
#include "sds_internal.h"

namespace sds {
namespace {

constexpr int BM = 128;         // query rows per tile (two tiles per item)
constexpr int BN = 128;         // keys per tile
constexpr int SUB = 128 * 128;  // bytes of one 128-row x 64-column bf16 sub-tile
constexpr float kRescaleThreshold = 8.0f;
// d = 64: exponentials against the running maximum plus kRefShift (log2
// units); a row sum above kRowSumLimit moves the reference (see the header).
constexpr int kRefShift = 64;
constexpr float kRowSumLimit = 256.0f;

template <int D>
struct Cfg {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * SUB;  // one 128-row tile of Q, K or V
  static constexpr int ST = (D == 64) ? 4 : 2;  // K/V pipeline stages
  static constexpr int QB = (D == 64) ? 2 : 1;  // Q buffers (double-buffered across items if it fits)
  // d = 64 (EARLY): P_t gets tensor-memory columns of its own, so the
  // issuer of tile t can start S_t(g+1) as soon as the softmax has read
  // S_t(g) into registers, and each tile has its own issuing thread (an
  // M128 N64 MMA from one thread takes about 50 cycles against 32 of tensor
  // work; two threads issuing concurrently reach the full rate).
  // Layout S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384)
  // O0 [384,448) O1 [448,512).  d = 128 has no spare columns: P overwrites
  // the first columns of its score buffer.
  static constexpr bool EARLY = (D == 64);
#ifndef SDS_K1_ISS128
#define SDS_K1_ISS128 1
#endif
  // MMA-issuing threads.  One thread issues an MMA about every 100 cycles
  // under load against 64 cycles of tensor work for M128 N128 K16, so a
  // single issuer cannot keep the tensor core busy; with two, issuer t
  // serves query tile t alone.  d = 128 keeps P over the scores, so there
  // issuer t issues PV_t(g) before S_t(g+1) (one thread's MMAs run in issue
  // order, so S_t(g+1) cannot overwrite P_t(g) before PV_t(g) has read it).
#ifndef SDS_K1_SUB64
#define SDS_K1_SUB64 1
#endif
  // d = 128 with 64-key compute tiles (SUBS = 2): each loaded 128-key tile
  // is consumed as two 64-key halves.  Tensor memory then holds two score
  // buffers per group, [t*256, +64) and [t*256 + 64, +64), beside O_t at
  // [t*256 + 128, +128): the S issuer of group t computes S_t(g+2) into
  // the buffer of S_t(g) once PV_t(g), issued by the PV warp, has read the
  // P written over it, so the scores of the next half-tile are ready while
  // the softmax works on the current one.
  static constexpr int SUBS = (D == 128 && SDS_K1_SUB64) ? 2 : 1;
  static constexpr int NCOL = BN / SUBS;  // keys per compute tile
  static constexpr int ISS = (EARLY || SUBS == 2) ? 2 : SDS_K1_ISS128;
  static constexpr bool PV_FIRST = !EARLY;  // always PV_t(g) before S_t(g+1)
  static constexpr uint32_t O_COL = EARLY ? 384u : (SUBS == 2 ? 128u : 256u);  // first column of O0
  static constexpr uint32_t O_STRIDE = EARLY ? 64u : (SUBS == 2 ? 256u : 128u);
  static constexpr uint32_t S_STRIDE = SUBS == 2 ? 256u : 128u;  // S region of group t at t * S_STRIDE
  // Threads per query row (HV, "halves"): with two, each of the two threads
  // of a row takes half of its score columns, P columns and O columns, so
  // that a tile has 8 softmax warps (2 per SM sub-partition and tile) and the
  // exponentials of one warp overlap the score loads and row maxima of
  // others.  The halves combine their row maxima every tile and their row
  // sums at the end of an item through shared memory.
#ifndef SDS_K1_HV64
#define SDS_K1_HV64 1
#endif
#ifndef SDS_K1_PWAIT_FIRST
#define SDS_K1_PWAIT_FIRST 0
#endif
#ifndef SDS_K1_HV128
#define SDS_K1_HV128 1
#endif
#ifndef SDS_K1_CHAINS
#define SDS_K1_CHAINS 4
#endif
  static constexpr int HV = (D == 64) ? SDS_K1_HV64 : SDS_K1_HV128;
  static constexpr int SMW = 8 * HV;              // softmax warps (two tiles)
#ifndef SDS_K1_SPLITV
#define SDS_K1_SPLITV 0
#endif
  // K (with Q) and V tiles come from separate producer warps, so that a
  // producer waiting for a free V stage (held until the PV products of two
  // tiles back are done) does not hold back the next K tile, which the
  // next S product needs earlier.
  static constexpr bool SPLITV = SDS_K1_SPLITV;
  static constexpr int WP = SMW;                  // TMA producer warp (K, Q; and V unless SPLITV)
  static constexpr int WI = SMW + 1;              // MMA issuer warp(s): WI, WI + 1
  static constexpr int WPV = SMW + 3;             // V producer warp (SPLITV)
  // d = 128 (64-key compute tiles): warps WI, WI + 1 issue the S products of
  // tiles 0 and 1, warp WPVI the PV products of both
  static constexpr bool PVW = SUBS == 2;
  static constexpr int WPVI = SMW + 3;
  static_assert(!(PVW && SPLITV), "the PV issuer warp and the V producer warp are the same warp");
  static constexpr int THREADS = (SMW + ((SPLITV || PVW) ? 4 : 3)) * 32;
  static constexpr int Q = 0;
  static constexpr int K = Q + QB * 2 * TILE;
  static constexpr int V = K + ST * TILE;
  static constexpr int BAR = V + ST * TILE;
  static constexpr int XCH = BAR + 640;           // row-max [2 parity][2 tile][2 half][128], row-sum [2][2][128]
  static constexpr int TOTAL = XCH + (HV == 2 ? (8 + 4) * 128 * 4 : 0);
  static constexpr int ALLOC = TOTAL + 1024;  // slack for 1024-byte alignment
};

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled sub-tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

// The two bf16 halves of w as floats (low half first); exact.
__device__ __forceinline__ float2 bf16x2_to_float2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

struct Bars {
  uint64_t* q_full;   // [2]
  uint64_t* q_ready;  // [2][2]: buffer, tile
  uint64_t* q_empty;  // [2]
  uint64_t* k_full;
  uint64_t* v_full;
  uint64_t* k_empty;
  uint64_t* v_empty;
  uint64_t* s_full;  // [2 group][2 buffer]: index t, or t * 2 + buffer with 64-key compute tiles
  uint64_t* p_full;  // [2 group][2 buffer], indexed as s_full
  uint64_t* o_done;  // [2 group][2 buffer]: index t, or t * 2 + buffer with 64-key compute tiles
  uint64_t* mma_final;  // [3]: per issuing thread (warps 9, 10 and, d = 128, 11)
  uint64_t* s_free;     // [2]: the softmax has read S_t (EARLY)
  uint64_t* xb;         // [2 tile][2 parity]: both halves' row maxima are in shared memory (HV 2)
  uint64_t* lb;         // [2 tile]: both halves' row sums are in shared memory (HV 2)
  uint64_t* wb;         // [2 tile]: both halves' partial O rows are written (HV 2, split items)
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  float* xmax;          // [2 parity][2 tile][2 half][128]
  float* xsum;          // [2 tile][2 half][128]
};

template <int D>
__device__ __forceinline__ Bars carve(uint8_t* sm) {
  using C = Cfg<D>;
  uint64_t* b = reinterpret_cast<uint64_t*>(sm + C::BAR);
  Bars r;
  r.q_full = b;
  r.q_ready = b + 2;
  r.q_empty = b + 6;
  r.k_full = b + 8;
  r.v_full = r.k_full + C::ST;
  r.k_empty = r.v_full + C::ST;
  r.v_empty = r.k_empty + C::ST;
  r.s_full = r.v_empty + C::ST;
  r.p_full = r.s_full + 4;
  r.o_done = r.p_full + 4;
  r.mma_final = r.o_done + 4;
  r.s_free = r.mma_final + 3;
  r.xb = r.s_free + 2;
  r.lb = r.xb + 4;
  r.wb = r.lb + 2;
  r.tmem_slot = reinterpret_cast<uint32_t*>(r.wb + 2);
  r.abort_flag = reinterpret_cast<volatile int*>(r.tmem_slot + 1);
  r.xmax = reinterpret_cast<float*>(sm + C::XCH);
  r.xsum = r.xmax + 8 * 128;
  return r;
}

__device__ __forceinline__ void key_tile(const AttnParams& p, int nt0, int j, int& key0, int& nvalid) {
  if (j < nt0) {
    key0 = p.seg_start[0] + j * BN;
    nvalid = min(BN, p.seg_count[0] - j * BN);
  } else {
    key0 = p.seg_start[1] + (j - nt0) * BN;
    nvalid = min(BN, p.seg_count[1] - (j - nt0) * BN);
  }
}

__device__ __forceinline__ void fail_wait(const Bars& B) { *B.abort_flag = 1; }

// A wait on the softmax path, where a whole score row is live in registers:
// a short inline spin, then the bounded wait out of line, so that the
// timer bookkeeping (and the register saves of the call) stay off the
// usual path.
__device__ __noinline__ bool wait_slow(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  return mbar_wait(bar, parity, limit_ns);
}
__device__ __forceinline__ bool wait_spin(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_test_wait(bar, parity)) return true;
  for (int i = 0; i < 1024; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return wait_slow(bar, parity, limit_ns);
}

// d = 64, one thread per query row, the rare case of the running reference:
// the exponentials of a key tile overflowed (the row's scores rose 192 or
// more above its reference).  The tile again, its maximum first, from
// scores recomputed on the CUDA cores from the query row and the 128 keys
// in shared memory (64-column bf16 tiles, 128-byte swizzle); P is stored
// over the overflowed one.  Each score is computed twice (maximum, then
// probability), so that no score row is held in registers.  Returns the
// new reference, the factor that takes O and l to it, and the row sum.
__device__ __noinline__ float3 redo_tile_d64(const uint8_t* qrow, const uint8_t* ks, int r, int nvalid,
                                             uint32_t tP, float sc, float m_run, float shift) {
  auto score = [&](int j) -> float {
    float a = 0.f;
#pragma unroll 4
    for (int cw = 0; cw < 32; ++cw) {
      const uint32_t off = (uint32_t)((cw & 3) * 4);
      const float2 qf = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(qrow + swz(r, cw >> 2) + off));
      const float2 kf = bf16x2_to_float2(*reinterpret_cast<const uint32_t*>(ks + swz(j, cw >> 2) + off));
      a = fmaf(qf.y, kf.y, fmaf(qf.x, kf.x, a));
    }
    return a;
  };
  float mt = -INFINITY;
#pragma unroll 1
  for (int j = 0; j < nvalid; ++j) mt = fmaxf(mt, score(j));
  const float m_new = fmaxf(mt * sc + shift, m_run);
  float ls = 0.f;
#pragma unroll 1
  for (int part = 0; part < 4; ++part) {
    uint32_t w[16];
#pragma unroll 1
    for (int q = 0; q < 16; ++q) {
      const int j = part * 32 + 2 * q;
      const float e0 = j < nvalid ? fast_exp2(score(j) * sc - m_new) : 0.f;
      const float e1 = j + 1 < nvalid ? fast_exp2(score(j + 1) * sc - m_new) : 0.f;
      ls += e0 + e1;
      w[q] = pack_bf16x2(e0, e1);
    }
    tmem_st16u(tP + (uint32_t)(part * 16), w);
  }
  tmem_wait_st();
  return make_float3(m_new, fast_exp2(m_run - m_new), ls);
}

// The even division of U units over G CTAs: CTA c owns [lo(c), lo(c+1)).
struct Split {
  int64_t U, G, nkt;
  __device__ __forceinline__ int64_t lo(int64_t c) const { return c * U / G; }
  // the CTA whose range holds unit u
  __device__ __forceinline__ int64_t owner(int64_t u) const { return ((u + 1) * G - 1) / U; }
};

// Walk over one CTA's units: global tile counter g, segment counter sg
// (one segment per item touched), the item and its key-tile range.
struct SegIter {
  int64_t u, u_hi, seg_lo, seg_hi, item, nkt;
  int64_t g;
  int sg;
  __device__ __forceinline__ void init(int64_t lo, int64_t hi, int64_t nkt_) {
    u = lo;
    u_hi = hi;
    nkt = nkt_;
    g = 0;
    sg = 0;
    start_segment();
  }
  __device__ __forceinline__ void start_segment() {
    item = u / nkt;
    seg_lo = u;
    seg_hi = min(u_hi, (item + 1) * nkt);
  }
  __device__ __forceinline__ bool done() const { return u >= u_hi; }
  __device__ __forceinline__ bool first() const { return u == seg_lo; }
  __device__ __forceinline__ int kt() const { return (int)(u - item * nkt); }
  __device__ __forceinline__ void advance() {
    ++u;
    ++g;
    if (u == seg_hi && u < u_hi) {
      ++sg;
      start_segment();
    }
  }
};

struct ItemPos {
  int s, h;
  int64_t q0;
};
__device__ __forceinline__ ItemPos item_pos(const AttnParams& p, int64_t item, int64_t npairs) {
  ItemPos r;
  const int64_t pair = item % npairs, sh = item / npairs;
  r.h = (int)(sh % p.H);
  r.s = (int)(sh / p.H);
  r.q0 = pair * (2 * BM);
  return r;
}

template <int D>
__global__ void __launch_bounds__(Cfg<D>::THREADS, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const Bars B = carve<D>(sm);
  uint8_t* sQ = sm + C::Q;
  uint8_t* sK = sm + C::K;
  uint8_t* sV = sm + C::V;

  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int nt0 = (p.seg_count[0] + BN - 1) / BN;
  const int64_t nkt = nt0 + (p.seg_count[1] + BN - 1) / BN;
  const int64_t npairs = (p.q_rows + 2 * BM - 1) / (2 * BM);
  Split sp;
  sp.nkt = nkt;
  sp.U = (int64_t)p.S * p.H * npairs * nkt;
  sp.G = gridDim.x;
  const int64_t cta = blockIdx.x;
  const int64_t u_lo = sp.lo(cta), u_hi = sp.lo(cta + 1);
  const bool active = nkt > 0 && u_hi > u_lo;

  // d = 64: a tile recomputed in the overflow case reads its queries from
  // shared memory, until the end of its segment.  The producer refills a Q
  // buffer two segments later, after the K/V copies of the full item in
  // between, each of which waits for the PV product ST tiles back; with
  // items of at most ST - 2 key tiles that can happen before the softmax
  // has finished, so then the softmax threads also arrive on q_empty.
  const bool q_by_softmax = C::EARLY && nkt <= C::ST - 2;
  if (tid == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    if (!C::EARLY) prefetch_tensormap(&tm_o);  // o is written by TMA only at d = 128 (a d = 64 prefetch cost 1.5 %)
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.q_full + i, 1);
      mbar_init(B.q_empty + i, q_by_softmax ? C::ISS + 256 * C::HV : C::ISS);
      mbar_init(B.q_ready + 2 * i + 0, 128 * C::HV);
      mbar_init(B.q_ready + 2 * i + 1, 128 * C::HV);
    }
    for (int i = 0; i < C::ST; ++i) {
      mbar_init(B.k_full + i, 1);
      mbar_init(B.v_full + i, 1);
      mbar_init(B.k_empty + i, C::ISS);
      mbar_init(B.v_empty + i, C::PVW ? 1 : C::ISS);
    }
    for (int i = 0; i < 4; ++i) {
      mbar_init(B.s_full + i, 1);
      mbar_init(B.p_full + i, 128 * C::HV);
      mbar_init(B.o_done + i, 1);
    }
    mbar_init(B.mma_final + 2, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.mma_final + i, 1);
      mbar_init(B.s_free + i, 128 * C::HV);
      mbar_init(B.xb + 2 * i + 0, 128 * C::HV);
      mbar_init(B.xb + 2 * i + 1, 128 * C::HV);
      mbar_init(B.lb + i, 128 * C::HV);
      mbar_init(B.wb + i, 128 * C::HV);
    }
    *B.abort_flag = 0;
    fence_barrier_init();
  }
  if (wid == C::WI) {
    tmem_alloc(B.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *B.tmem_slot;

  if (wid == C::WP || (C::SPLITV && wid == C::WPV)) {
    // ------------------------------------------------------------ TMA producer(s)
    const bool do_k = wid == C::WP;                  // K and Q
    const bool do_v = !C::SPLITV || wid == C::WPV;   // V
    if (lane == 0 && active) {
      SegIter it;
      it.init(u_lo, u_hi, nkt);
      int64_t issued_k = 0, issued_v = 0;  // tiles whose K / V copy was issued
      int issued_q = 0;                    // segments whose Q copy was issued
      bool ok = true;
      while (ok && !it.done()) {
        const int64_t g = it.g;
        const int st = (int)(g % C::ST);
        const uint32_t ph = (uint32_t)(g / C::ST) & 1u;
        const ItemPos ip = item_pos(p, it.item, npairs);
        int key0, nvalid;
        key_tile(p, nt0, it.kt(), key0, nvalid);
        if (do_k) {
          if (!mbar_wait(B.k_empty + st, ph ^ 1u, p.wait_ns)) { ok = false; break; }
          // failure-detection test hook: CTA 0 never loads the keys of tile
          // `withhold_k`, so every wait for them runs out
          const bool withhold = p.withhold_k >= 0 && g == p.withhold_k && cta == 0;
          if (!withhold) {
            mbar_arrive_expect_tx(B.k_full + st, C::TILE);
            for (int b = 0; b < C::NSUB; ++b)
              tma_load_3d(sK + st * C::TILE + b * SUB, &tm_k, ip.h * D + b * 64, key0, ip.s, B.k_full + st);
          }
          issued_k = g + 1;
        }
        if (do_v) {
          // d = 64 releases K(g) and V(g) together, on k_empty alone; d = 128
          // releases V(g) on v_empty (the PV warp, after PV(g))
          if (!mbar_wait((C::EARLY ? B.k_empty : B.v_empty) + st, ph ^ 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(B.v_full + st, C::TILE);
          for (int b = 0; b < C::NSUB; ++b)
            tma_load_3d(sV + st * C::TILE + b * SUB, &tm_v, ip.h * D + b * 64, key0, ip.s, B.v_full + st);
          issued_v = g + 1;
        }
        if (do_k && it.first()) {
          // this item's queries; the buffer is free once the last S MMAs
          // of the item that used it before have completed
          const int qb = it.sg % C::QB;
          if (it.sg >= C::QB && !mbar_wait(B.q_empty + qb, (uint32_t)(it.sg / C::QB - 1) & 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(B.q_full + qb, 2 * C::TILE);
          for (int t = 0; t < 2; ++t)
            for (int b = 0; b < C::NSUB; ++b)
              tma_load_3d(sQ + (qb * 2 + t) * C::TILE + b * SUB, &tm_q, ip.h * D + b * 64,
                          (int32_t)(ip.q0 + t * BM), ip.s, B.q_full + qb);
          issued_q = it.sg + 1;
        }
        it.advance();
      }
      if (!ok) fail_wait(B);
      // leave only after every copy we issued has landed in shared memory
      for (int sgi = (issued_q > C::QB ? issued_q - C::QB : 0); sgi < issued_q; ++sgi)
        mbar_wait(B.q_full + sgi % C::QB, (uint32_t)(sgi / C::QB) & 1u, p.wait_ns);
      for (int64_t j = (issued_k > C::ST ? issued_k - C::ST : 0); j < issued_k; ++j)
        if (!(p.withhold_k == j && cta == 0)) mbar_wait(B.k_full + j % C::ST, (uint32_t)(j / C::ST) & 1u, p.wait_ns);
      for (int64_t j = (issued_v > C::ST ? issued_v - C::ST : 0); j < issued_v; ++j)
        mbar_wait(B.v_full + j % C::ST, (uint32_t)(j / C::ST) & 1u, p.wait_ns);
    }
  } else if (C::SUBS == 2 && (wid == C::WI || wid == C::WI + 1 || wid == C::WPVI)) {
    // ------------------------------------------------------------ MMA issuers (d = 128,
    // 64-key compute tiles).  Warp WI + t issues the S products of query
    // tile t; warp WPVI issues the PV products of both tiles.  (One thread
    // issuing both for its tile spent most of a step issuing, at 72-78
    // cycles per MMA; two lanes of one warp do not issue concurrently.)
    // The two halves h of a loaded key tile have score buffers of their
    // own, and P is written over the scores, so S_t(L + 1, h) waits until
    // PV_t(L, h) has completed (one o_done barrier per buffer).  At an item
    // boundary the next item's S products also wait for its queries, which
    // the softmax rotates once it has finished the item.
    if (lane == 0 && active) {
      const bool s_role = wid != C::WPVI;
      const int ts = wid - C::WI;  // the S issuer's tile
      constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, C::NCOL, false);
      constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, true);
      const uint32_t dhi = (uint32_t)(smem_desc_sw128(0, 0, 1024) >> 32);
      const uint32_t qlo = (uint32_t)smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t klo = (uint32_t)smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint32_t vlo = (uint32_t)smem_desc_sw128(smem_u32(sV), SUB, 1024);
      // S_t of half h of the K tile in stage st: keys [h * NCOL, +NCOL) are
      // rows h * NCOL.. of each 64-column sub-tile (a multiple of the 8-row
      // swizzle atom, so the descriptor only moves its start address); the
      // buffer of group t, half h, is at t * S_STRIDE + h * NCOL
      auto issue_s = [&](int t, int qb, uint32_t st, int h) {
        const uint32_t dS = tmem + (uint32_t)t * C::S_STRIDE + (uint32_t)(h * C::NCOL);
        const uint32_t a0 = qlo + (uint32_t)(((qb * 2 + t) * C::TILE) >> 4);
        const uint32_t b0 = klo + st * (uint32_t)(C::TILE >> 4) + (uint32_t)((h * C::NCOL * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * SUB + (kk & 3) * 32) >> 4);
          mma_bf16_ss_w(dS, a0 + off, dhi, b0 + off, dhi, IDESC_S, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t(half h) V(rows h * NCOL.. of the V tile in stage st)
      auto issue_pv = [&](int t, uint32_t st, int h, bool acc) {
        const uint32_t dO = tmem + C::O_COL + (uint32_t)t * C::O_STRIDE;
        const uint32_t aP = tmem + (uint32_t)t * C::S_STRIDE + (uint32_t)(h * C::NCOL);
        const uint32_t b0 = vlo + st * (uint32_t)(C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < C::NCOL / 16; ++kk)
          mma_bf16_ts_w(dO, aP + (uint32_t)(kk * 8),
                        b0 + (uint32_t)(((h * C::NCOL + kk * 16) * 128) >> 4), dhi, IDESC_O,
                        (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      uint32_t L = 0;  // loaded key tiles consumed (compute tiles 2L, 2L + 1)
      int sg = 0;      // segment counter
      int64_t u = u_lo;
      if (s_role) {
        const int64_t item = u / nkt;
        const int64_t seg_hi = min(u_hi, (item + 1) * nkt);
        ok = mbar_wait(B.q_ready + ts, 0, p.wait_ns) && mbar_wait(B.k_full, 0, p.wait_ns);
        if (ok) {
          tc_fence_after();
          for (int h = 0; h < 2; ++h) {
            issue_s(ts, 0, 0, h);
            mma_commit(B.s_full + 2 * ts + h);
          }
          mma_commit(B.k_empty + 0);
          if (seg_hi - u == 1) mma_commit(B.q_empty + 0);
        }
      }
      while (ok && u < u_hi) {
        const int64_t item = u / nkt;
        const int64_t seg_hi = min(u_hi, (item + 1) * nkt);
        const int n_here = (int)(seg_hi - u);
        const bool final_seg = seg_hi == u_hi;
        const int n_next = final_seg ? 0 : (int)(min(u_hi, seg_hi + nkt) - seg_hi);
        const int qb_n = (sg + 1) % C::QB;
        const uint32_t qp_n = (uint32_t)((sg + 1) / C::QB) & 1u;
        for (int i = 0; i < n_here && ok; ++i, ++L) {
          const uint32_t st = L % C::ST, ph = (L / C::ST) & 1u;
          if (s_role) {
            const bool boundary = i + 1 == n_here;  // tile L + 1 opens the next segment
            if (boundary && final_seg) continue;    // no tile L + 1
            const uint32_t st1 = (L + 1) % C::ST, ph1 = ((L + 1) / C::ST) & 1u;
            // tile L + 1 is the last of its segment: its S products release the Q buffer
            const bool next_last = boundary ? n_next == 1 : i + 2 == n_here;
            const int qb1 = boundary ? qb_n : sg % C::QB;
            if (!mbar_wait(B.k_full + st1, ph1, p.wait_ns) ||
                (boundary && !mbar_wait(B.q_ready + 2 * qb1 + ts, qp_n, p.wait_ns))) {
              ok = false;
              break;
            }
            for (int h = 0; h < 2 && ok; ++h) {
              // S_t(L + 1, h) goes over the P that PV_t(L, h) reads.  PV_t(L - 1, h)
              // completed before S_t(L, h) was issued, so the barrier is in
              // phase L or L + 1 here and the parity wait is exact.
              ok = mbar_wait(B.o_done + 2 * ts + h, L & 1u, p.wait_ns);
              if (!ok) break;
              tc_fence_after();
              issue_s(ts, qb1, st1, h);
              mma_commit(B.s_full + 2 * ts + h);
            }
            if (!ok) break;
            mma_commit(B.k_empty + st1);
            if (next_last) mma_commit(B.q_empty + qb1);
          } else {
            if (!mbar_wait(B.v_full + st, ph, p.wait_ns)) {
              ok = false;
              break;
            }
            for (int h = 0; h < 2 && ok; ++h) {
              for (int t = 0; t < 2 && ok; ++t) {
                ok = mbar_wait(B.p_full + 2 * t + h, L & 1u, p.wait_ns);
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, st, h, i > 0 || h > 0);
                mma_commit(B.o_done + 2 * t + h);
              }
            }
            if (!ok) break;
            mma_commit(B.v_empty + st);
          }
        }
        u = seg_hi;
        ++sg;
      }
      if (!ok) fail_wait(B);
      const int fin = s_role ? ts : 2;
      mma_commit(B.mma_final + fin);
      mbar_wait(B.mma_final + fin, 0, p.wait_ns);
    }
  } else if (C::ISS == 2 && C::SUBS == 1 && (wid == C::WI || wid == C::WI + 1)) {
    // ------------------------------------------------------------ MMA issuers (d = 64):
    // one thread per query tile t, for S_t = Q_t K^T and O_t += P_t V.
    // S_t(g+1) goes out as soon as the softmax has read S_t(g) (s_free) and
    // before P_t(g) exists, so the next scores are ready when the softmax
    // finishes the current tile.
    if (lane == 0 && active) {
      const int t = wid - C::WI;
      constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, true);
      const uint32_t dhi = (uint32_t)(smem_desc_sw128(0, 0, 1024) >> 32);
      const uint32_t qlo = (uint32_t)smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t klo = (uint32_t)smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint32_t vlo = (uint32_t)smem_desc_sw128(smem_u32(sV), SUB, 1024);
      const uint32_t dS = tmem + (uint32_t)(t * 128);
      const uint32_t aP = C::EARLY ? tmem + 256u + (uint32_t)(t * 64) : tmem + (uint32_t)(t * 128);
      const uint32_t dO = tmem + C::O_COL + (uint32_t)t * C::O_STRIDE;
      auto issue_s = [&](int qb, uint32_t st) {
        const uint32_t a0 = qlo + (uint32_t)(((qb * 2 + t) * C::TILE) >> 4);
        const uint32_t b0 = klo + st * (uint32_t)(C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * SUB + (kk & 3) * 32) >> 4);
          mma_bf16_ss_w(dS, a0 + off, dhi, b0 + off, dhi, IDESC_S, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](uint32_t st, bool acc) {
        const uint32_t b0 = vlo + st * (uint32_t)(C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts_w(dO, aP + (uint32_t)(kk * 8), b0 + (uint32_t)((kk * 16 * 128) >> 4), dhi,
                        IDESC_O, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      uint32_t g = 0;  // global tile counter
      int sg = 0;      // segment counter
      int64_t u = u_lo;
      {
        const int64_t item = u / nkt;
        const int64_t seg_hi = min(u_hi, (item + 1) * nkt);
        ok = mbar_wait(B.q_ready + t, 0, p.wait_ns) && mbar_wait(B.k_full, 0, p.wait_ns);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0);
          mma_commit(B.s_full + t);
          if (seg_hi - u == 1) mma_commit(B.q_empty + 0);
        }
      }
      while (ok && u < u_hi) {
        const int64_t item = u / nkt;
        const int64_t seg_hi = min(u_hi, (item + 1) * nkt);
        const int n_here = (int)(seg_hi - u);
        const bool final_seg = seg_hi == u_hi;
        const int n_next = final_seg ? 0 : (int)(min(u_hi, seg_hi + nkt) - seg_hi);
        const int qb_n = (sg + 1) % C::QB;
        const uint32_t qp_n = (uint32_t)((sg + 1) / C::QB) & 1u;
        for (int i = 0; i < n_here; ++i, ++g) {
          const uint32_t st = g % C::ST, ph = (g / C::ST) & 1u;
          const uint32_t st1 = (g + 1) % C::ST, ph1 = ((g + 1) / C::ST) & 1u;
          const bool boundary = i + 1 == n_here;
          const bool more = !(boundary && final_seg);
          const bool next_last = boundary ? n_next == 1 : i + 2 == n_here;
          // S_t(g+1); the next item's queries are rotated by the softmax
          // only after it has finished this item, which needs PV_t(g), so
          // at a boundary S_t(g+1) goes after PV_t(g)
          auto next_s = [&]() -> bool {
            const int qb1 = boundary ? qb_n : sg % C::QB;
            if (!mbar_wait(B.k_full + st1, ph1, p.wait_ns) ||
                (C::EARLY && !mbar_wait(B.s_free + t, g & 1u, p.wait_ns)) ||
                (boundary && !mbar_wait(B.q_ready + 2 * qb1 + t, qp_n, p.wait_ns)))
              return false;
            tc_fence_after();
            issue_s(qb1, st1);
            mma_commit(B.s_full + t);
            if (next_last) mma_commit(B.q_empty + qb1);
            return true;
          };
          if (more && !boundary && !C::PV_FIRST && !next_s()) {
            ok = false;
            break;
          }
          if (!mbar_wait(B.v_full + st, ph, p.wait_ns) || !mbar_wait(B.p_full + t, g & 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(st, i > 0);
          mma_commit(B.o_done + t);
          // K(g) and V(g) are released together (one commit on k_empty),
          // once P_t(g) exists: until then the softmax may recompute the
          // tile's scores from K(g)
          mma_commit(B.k_empty + st);
          if (more && (boundary || C::PV_FIRST) && !next_s()) {
            ok = false;
            break;
          }
        }
        u = seg_hi;
        ++sg;
      }
      if (!ok) fail_wait(B);
      mma_commit(B.mma_final + t);
      mbar_wait(B.mma_final + t, 0, p.wait_ns);
    }
  } else if (C::ISS == 1 && wid == C::WI) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && active) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, true);
      // Descriptor words: the high word (stride 1024 B, fixed 0b001, 128-byte
      // swizzle) is common to every operand; the low word holds the start
      // address >> 4 and the leading-dimension offset, so stepping through a
      // tile is a 32-bit add.
      const uint32_t dhi = (uint32_t)(smem_desc_sw128(0, 0, 1024) >> 32);
      const uint32_t qlo = (uint32_t)smem_desc_sw128(smem_u32(sQ), 16, 1024);
      const uint32_t klo = (uint32_t)smem_desc_sw128(smem_u32(sK), 16, 1024);
      const uint32_t vlo = (uint32_t)smem_desc_sw128(smem_u32(sV), SUB, 1024);
      auto issue_s = [&](int t, int qb, uint32_t st) {
        const uint32_t dS = tmem + (uint32_t)(t * 128);
        const uint32_t a0 = qlo + (uint32_t)(((qb * 2 + t) * C::TILE) >> 4);
        const uint32_t b0 = klo + st * (uint32_t)(C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)(((kk >> 2) * SUB + (kk & 3) * 32) >> 4);
          mma_bf16_ss_w(dS, a0 + off, dhi, b0 + off, dhi, IDESC_S, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, uint32_t st, bool acc) {
        const uint32_t dO = tmem + 256u + (uint32_t)(t * 128);
        const uint32_t aP = tmem + (uint32_t)(t * 128);
        const uint32_t b0 = vlo + st * (uint32_t)(C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts_w(dO, aP + (uint32_t)(kk * 8), b0 + (uint32_t)((kk * 16 * 128) >> 4), dhi,
                        IDESC_O, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = true;
      uint32_t g = 0;  // global tile counter
      int sg = 0;      // segment counter
      int64_t u = u_lo;
      // segment 0: S of its first tile for both groups
      {
        const int64_t item = u / nkt;
        const int64_t seg_hi = min(u_hi, (item + 1) * nkt);
        ok = mbar_wait(B.q_ready + 0, 0, p.wait_ns) && mbar_wait(B.k_full, 0, p.wait_ns);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0, 0);
          mma_commit(B.s_full + 0);
          ok = mbar_wait(B.q_ready + 1, 0, p.wait_ns);
        }
        if (ok) {
          tc_fence_after();
          issue_s(1, 0, 0);
          mma_commit(B.s_full + 1);
          mma_commit(B.k_empty + 0);
          if (seg_hi - u == 1) mma_commit(B.q_empty + 0);
        }
      }
      while (ok && u < u_hi) {
        const int64_t item = u / nkt;
        const int64_t seg_hi = min(u_hi, (item + 1) * nkt);
        const int n_here = (int)(seg_hi - u);
        const bool final_seg = seg_hi == u_hi;
        const int n_next = final_seg ? 0 : (int)(min(u_hi, seg_hi + nkt) - seg_hi);
        const int qb_n = (sg + 1) % C::QB;
        const uint32_t qp_n = (uint32_t)((sg + 1) / C::QB) & 1u;
        for (int i = 0; i < n_here; ++i, ++g) {
          const uint32_t st = g % C::ST, ph = (g / C::ST) & 1u;
          const uint32_t st1 = (g + 1) % C::ST, ph1 = ((g + 1) / C::ST) & 1u;
          const bool acc = i > 0;
          const bool boundary = i + 1 == n_here;  // tile g+1 opens the next segment
          const bool more = !(boundary && final_seg);
          // tile g+1 is the last of its segment: its S MMAs release the Q buffer
          const bool next_last = boundary ? n_next == 1 : i + 2 == n_here;
          // the producer lands K/V tiles well ahead: wait for them first
          if (!mbar_wait(B.v_full + st, ph, p.wait_ns) || (more && !mbar_wait(B.k_full + st1, ph1, p.wait_ns))) {
            ok = false;
            break;
          }
          if (!mbar_wait(B.p_full + 0, g & 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(0, st, acc);
          mma_commit(B.o_done + 0);
          const int qb1 = boundary ? qb_n : sg % C::QB;
          if (more) {
            if (boundary && !mbar_wait(B.q_ready + 2 * qb1 + 0, qp_n, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(0, qb1, st1);
            mma_commit(B.s_full + 0);
          }
          if (!mbar_wait(B.p_full + 1, g & 1u, p.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(1, st, acc);
          mma_commit(B.o_done + 1);
          mma_commit(B.v_empty + st);
          if (more) {
            if (boundary && !mbar_wait(B.q_ready + 2 * qb1 + 1, qp_n, p.wait_ns)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(1, qb1, st1);
            mma_commit(B.s_full + 1);
            mma_commit(B.k_empty + st1);
            if (next_last) mma_commit(B.q_empty + qb1);
          }
        }
        u = seg_hi;
        ++sg;
      }
      if (!ok) fail_wait(B);
      // all our MMAs complete before tensor memory is released
      mma_commit(B.mma_final + 0);
      mbar_wait(B.mma_final + 0, 0, p.wait_ns);
    }
  } else if (wid < C::SMW && active) {
    // ------------------------------------------------------------ softmax groups
    // Warp w: query tile t, half hf of each row's columns, TMEM lanes
    // 32 (w mod 4) .. +31 (a warp reaches only its own quarter of the lanes).
    constexpr int HV = C::HV;
    constexpr int NC = C::NCOL / HV;  // score columns of this thread's row per compute tile
    static_assert(C::SUBS == 1 || HV == 1, "64-key compute tiles take one thread per row");
    constexpr int DC = D / HV;    // O columns of this thread's row
    // d = 64 with one thread per row: after an item's first tile the
    // exponentials go against the running reference, without a tile maximum
    constexpr bool RUNREF = C::EARLY && HV == 1;
    constexpr float kRef = RUNREF ? (float)kRefShift : 0.f;
    const int t = wid / (4 * HV);
    const int hf = (wid / 4) % HV;
    const int r = (wid & 3) * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((wid & 3) * 32) << 16;
    // scores of a compute tile: group t's S region, this half's columns, and
    // with 64-key compute tiles the buffer of the tile's parity
    const uint32_t tS0 = tmem + (uint32_t)t * C::S_STRIDE + (uint32_t)(hf * NC) + lane_base;
    const uint32_t tO = tmem + C::O_COL + (uint32_t)t * C::O_STRIDE + (uint32_t)(hf * DC) + lane_base;
    // packed bf16 probabilities: own columns (EARLY) or over the scores
    const uint32_t tP0 = (C::EARLY ? tmem + 256u + (uint32_t)(t * 64) : tmem + (uint32_t)t * C::S_STRIDE) +
                         (uint32_t)(hf * NC / 2) + lane_base;
    // 32 columns of this row's O
    // PV_t of compute tile gg has landed in O.  With 64-key compute tiles
    // each score buffer has its own o_done barrier, whose phase is the
    // loaded tile; otherwise o_done counts compute tiles.
    auto o_landed = [&](int gg) -> bool {
      const int ob = C::SUBS == 2 ? 2 * t + (gg & 1) : t;
      const uint32_t par = C::SUBS == 2 ? (uint32_t)(gg >> 1) & 1u : (uint32_t)gg & 1u;
      return mbar_wait(B.o_done + ob, par, p.wait_ns);
    };
    auto load_o = [&](int c, float(&tmp)[32]) {
      tmem_ld32(tO + (uint32_t)(c * 32), tmp);
      tmem_wait_ld();
      reg_fence32(tmp);
    };
    const float sc = p.scale_log2;
    const float2 sc2 = make_float2(sc, sc);
    int64_t u = u_lo;
    int sg = 0, g = 0;  // segment and global tile counters (as the other roles count them)
    int nsplit = 0;     // split segments finished (phase counter of wb)
    bool ok = true;
    while (ok && u < u_hi) {
      // ---- start of an item: its queries
      const int64_t item = u / nkt;
      const int64_t seg_hi = min(u_hi, (item + 1) * nkt);
      const int k0 = (int)(u - item * nkt), k1 = (int)(seg_hi - item * nkt);
      const ItemPos ip = item_pos(p, item, npairs);
      const int64_t row = ip.q0 + t * BM + r;
      const int qb = sg % C::QB;
      if (!mbar_wait(B.q_full + qb, (uint32_t)(sg / C::QB) & 1u, p.wait_ns)) {
        ok = false;
        break;
      }
      if (p.rope_on && row < p.q_rows) {
        const int tok = (int)(row % p.chunk_tokens);
        const int jf = tok / p.tokens_L, l = tok % p.tokens_L;
        const int pos[3] = {p.p0 + jf, l / p.grid_w, l % p.grid_w};
        const int seg[3] = {p.rope_seg[0], p.rope_seg[1], p.rope_seg[2]};
        const int off[3] = {p.tab_off[0], p.tab_off[1], p.tab_off[2]};
        uint8_t* qt = sQ + (qb * 2 + t) * C::TILE;
        // this half's share of the row's 16-byte chunks (8 per 64 columns);
        // four chunks at a time keep 16 table loads in flight (1 % of the
        // c4 launch against two at a time)
        constexpr int CH = C::NSUB * 8 / HV;
#pragma unroll 4
        for (int k = hf * CH; k < (hf + 1) * CH; ++k) {
          const int b = k >> 3, c = k & 7;
          uint4* ptr = reinterpret_cast<uint4*>(qt + b * SUB + swz(r, c));
          *ptr = rope8(*ptr, b * 64 + c * 8, pos, seg, p.rope_tab, off);
        }
        fence_proxy_async_smem();
      }
      mbar_arrive(B.q_ready + 2 * qb + t);
      float m_run = -INFINITY, l_run = 0.f;
      // ---- the item's key tiles
      for (int kt = k0; kt < k1 && ok; ++kt) {
       int key0, nvalid_t;
       key_tile(p, nt0, kt, key0, nvalid_t);
       for (int hs = 0; hs < C::SUBS; ++hs, ++g) {
        const uint32_t buf = C::SUBS == 2 ? (uint32_t)((g & 1) * C::NCOL) : 0u;
        const uint32_t tS = tS0 + buf;
        const uint32_t tP = tP0 + (C::EARLY ? 0u : buf);
        const int nvalid = min(max(nvalid_t - hs * C::NCOL, 0), C::NCOL);
        const bool first_tile = kt == k0 && hs == 0;
        // with 64-key compute tiles each score buffer has its own barriers
        const int sb = C::SUBS == 2 ? 2 * t + (g & 1) : t;
        const uint32_t sph = C::SUBS == 2 ? (uint32_t)(g >> 1) & 1u : (uint32_t)g & 1u;
        float sv[NC / 32][32];
        // EARLY: P_t(g) may overwrite P_t(g-1) only once PV_t(g-1) has read it
        auto p_free = [&]() -> bool {
          if (!C::EARLY || g == 0) return true;
          if (!wait_spin(B.o_done + t, (uint32_t)(g - 1) & 1u, p.wait_ns)) return false;
          tc_fence_after();
          return true;
        };
        constexpr int NPART = NC / 32;  // 16 packed columns per part
        // PWAIT_FIRST waits for PV_t(g-1) before the exponentials, so P is
        // stored as it is made; otherwise the first three quarters of P wait
        // in registers and the wait falls late in the pass.
        constexpr bool PWAIT_FIRST = C::EARLY && SDS_K1_PWAIT_FIRST;
        constexpr int HOLD = (C::EARLY && !PWAIT_FIRST) ? 3 * NPART / 4 : 0;  // parts held until P is free
        uint32_t pk[NPART][16];
        bool pwait_ok = true;
        // P = exp2(s*sc - m) as packed bf16, stored as it is made over the
        // first half of this thread's S columns (or, EARLY, P_t's own
        // columns); returns the sum of this thread's probabilities.
        auto exp_pass = [&](float m) -> float {
          const float2 nm2 = make_float2(-m, -m);
          constexpr int NRS = SDS_K1_CHAINS;  // independent row-sum chains
          float2 rs[NRS];
#pragma unroll
          for (int i = 0; i < NRS; ++i) rs[i] = make_float2(0.f, 0.f);
#pragma unroll
          for (int part = 0; part < NPART; ++part) {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float a0 = sv[part][2 * q], a1 = sv[part][2 * q + 1];
              const float2 x = __ffma2_rn(make_float2(a0, a1), sc2, nm2);
              const float e0 = fast_exp2(x.x), e1 = fast_exp2(x.y);
              rs[q % NRS] = __fadd2_rn(rs[q % NRS], make_float2(e0, e1));
              pk[part][q] = pack_bf16x2(e0, e1);
            }
            if (part >= HOLD) tmem_st16u(tP + (uint32_t)(part * 16), pk[part]);
            if (HOLD > 0 && part == HOLD - 1) {
              pwait_ok = p_free();
#pragma unroll
              for (int h = 0; h < HOLD; ++h) tmem_st16u(tP + (uint32_t)(h * 16), pk[h]);
            }
          }
#pragma unroll
          for (int w2 = NRS / 2; w2 > 0; w2 /= 2)
#pragma unroll
            for (int i = 0; i < w2; ++i) rs[i] = __fadd2_rn(rs[i], rs[i + w2]);
          return rs[0].x + rs[0].y;
        };
        // this row's maximum score of the tile, times the scale; with two
        // halves, each publishes its own and takes the larger of the two
        auto row_max = [&](bool& good) -> float {
          // SPL independent chains per 32 columns
          constexpr int SPL = (SDS_K1_CHAINS > 4 && NC == 128) || (SDS_K1_CHAINS > 2 && NC == 64) ? 2 : 1;
          constexpr int LEN = 32 / SPL;
          float mx[NC / 32][SPL];
#pragma unroll
          for (int c = 0; c < NC / 32; ++c)
#pragma unroll
            for (int h = 0; h < SPL; ++h) {
              const int b0 = h * LEN;
              float v = fmax3(sv[c][b0], sv[c][b0 + 1], sv[c][b0 + 2]);
#pragma unroll
              for (int i = b0 + 3; i + 1 < b0 + LEN; i += 2) v = fmax3(v, sv[c][i], sv[c][i + 1]);
              if ((LEN - 3) % 2) v = fmaxf(v, sv[c][b0 + LEN - 1]);
              mx[c][h] = v;
            }
          float m = mx[0][0];
#pragma unroll
          for (int c = 0; c < NC / 32; ++c)
#pragma unroll
            for (int h = 0; h < SPL; ++h)
              if (c + h > 0) m = fmaxf(m, mx[c][h]);
          if (HV == 2) {
            float* xm = B.xmax + ((g & 1) * 2 + t) * 2 * 128;
            xm[hf * 128 + r] = m;
            mbar_arrive(B.xb + 2 * t + (g & 1));
            good = wait_spin(B.xb + 2 * t + (g & 1), (uint32_t)(g >> 1) & 1u, p.wait_ns);
            m = fmaxf(m, xm[(hf ^ 1) * 128 + r]);
          }
          return m * sc;
        };
        // RUNREF, a row sum above 2^8 (finite): the row's largest
        // probability from the stored P (non-negative bf16, so the bit
        // patterns order like the values), then P, the row sum and, through
        // alpha, O scaled by the power of two 2^-k that takes it below
        // 2^-kRefShift again; the reference moves up by k.
        auto rebase = [&](bool big, float& ls, float& al, float& mn) {
          tmem_wait_st();
          uint32_t pmax = 0;
#pragma unroll
          for (int h = 0; h < NPART; ++h) {
            uint32_t w[16];
            tmem_ld16u(tP + (uint32_t)(h * 16), w);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q) pmax = max(pmax, max(w[q] >> 16, w[q] & 0xffffu));
          }
          // pmax < 2^(e - 126) for the biased exponent e; one multiply by a
          // normal power of two goes down at most 126 binary orders
          const int e = (int)(pmax >> 7);
          const int k = big ? min(max(e - 126 + kRefShift, 0), 126) : 0;
          const float scale = __int_as_float((127 - k) << 23);
          const uint32_t s2 = pack_bf16x2(scale, scale);
#pragma unroll
          for (int h = 0; h < NPART; ++h) {
            uint32_t w[16];
            tmem_ld16u(tP + (uint32_t)(h * 16), w);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 16; ++q) w[q] = mul_bf16x2(w[q], s2);
            tmem_st16u(tP + (uint32_t)(h * 16), w);
          }
          ls *= scale;
          al = scale;
          mn = m_run + (float)k;
        };
        float alpha = 1.f, m_new = m_run, lsum = 0.f;
        bool rescale = false, xgood = true;
        if (!mbar_wait(B.s_full + sb, sph, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) tmem_ld32(tS + (uint32_t)(c * 32), sv[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < NC / 32; ++c) reg_fence32(sv[c]);
        if (C::EARLY) {
          // the scores are in registers: the issuer may overwrite them
          tc_fence_before();
          // one arrival per warp (c2 0.5 % faster than 32)
          __syncwarp();
          if (lane == 0) mbar_arrive_count(B.s_free + t, 32);
        }
        if (nvalid < C::NCOL) {
#pragma unroll
          for (int c = 0; c < NC; ++c)
            sv[c >> 5][c & 31] = (hf * NC + c < nvalid) ? sv[c >> 5][c & 31] : -INFINITY;
        }
        if (PWAIT_FIRST && !p_free()) {
          ok = false;
          break;
        }
        // the reference of this pass: RUNREF after an item's first tile,
        // the running one (no tile maximum); otherwise the tile maximum first
        const bool run = RUNREF && !first_tile;
        if (!run) {
          const float mt = row_max(xgood) + kRef;
          if (first_tile) {
            m_new = mt;
          } else {
            const bool need = mt > m_run + kRescaleThreshold;
            m_new = need ? mt : m_run;
            alpha = need ? fast_exp2(m_run - m_new) : 1.f;
            rescale = __any_sync(0xffffffffu, need);
          }
        }
        lsum = exp_pass(m_new);
        if (run) {
          // every probability is >= 0, so a row sum <= 2^8 bounds each of them
          const bool big = !(lsum <= kRowSumLimit);
          if (__any_sync(0xffffffffu, big)) {
            if (__any_sync(0xffffffffu, !(lsum < INFINITY))) {
              // exp2 overflowed: the tile again, maximum first (out of line)
              tmem_wait_st();
              if constexpr (RUNREF) {
                const float3 rr = redo_tile_d64(sQ + (size_t)((sg % C::QB) * 2 + t) * C::TILE,
                                                sK + (size_t)(g % C::ST) * C::TILE, r, nvalid, tP, sc,
                                                m_run, kRef);
                m_new = rr.x;
                alpha = rr.y;
                lsum = rr.z;
              }
            } else {
              rebase(big, lsum, alpha, m_new);
            }
            rescale = __any_sync(0xffffffffu, alpha != 1.f);
          }
        }
        if (!ok) break;
        if (!pwait_ok || !xgood) {
          ok = false;
          break;
        }
        if (rescale) {
          // O may be rescaled only once the previous PV into it has landed
          if (!o_landed(g - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DC / 32; ++c) {
            float tmp[32];
            tmem_ld32(tO + (uint32_t)(c * 32), tmp);
            tmem_wait_ld();
            reg_fence32(tmp);
#pragma unroll
            for (int q = 0; q < 32; ++q) tmp[q] *= alpha;
            tmem_st32(tO + (uint32_t)(c * 32), tmp);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        if (C::EARLY) {
          // one arrival per warp: faster at d = 64, slower at d = 128 (measured)
          __syncwarp();
          if (lane == 0) mbar_arrive_count(B.p_full + sb, 32);
        } else {
          mbar_arrive(B.p_full + sb);
        }
        l_run = l_run * alpha + lsum;
        m_run = m_new;
       }
      }
      const int g_last = g - 1;
      if (!ok) break;
      if (q_by_softmax) {
        // every tile of the segment is done, including any recomputation
        // from the queries in shared memory: the Q buffer may be refilled
        mbar_arrive(B.q_empty + qb);
      }
      // ---- end of the item's segment: O is complete once the last PV lands
      // (with 64-key compute tiles, the last PV of each score buffer)
      if ((C::SUBS == 2 && !o_landed(g_last - 1)) || !o_landed(g_last)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (HV == 2) {
        // the row's sum over both halves' columns
        float* xs = B.xsum + t * 2 * 128;
        xs[hf * 128 + r] = l_run;
        mbar_arrive(B.lb + t);
        if (!mbar_wait(B.lb + t, (uint32_t)sg & 1u, p.wait_ns)) {
          ok = false;
          break;
        }
        l_run += xs[(hf ^ 1) * 128 + r];
      }
      u = seg_hi;
      ++sg;
      if (!C::EARLY && k0 == 0 && k1 == nkt && u >= u_hi) {
        // d = 128, the CTA's last item: nothing will land in shared memory
        // any more, so the tile is staged (bf16, the layout of the item's Q
        // slot) and written by TMA in whole lines; rows past the end are not
        // written.  (Measured: 4.7 us of row-by-row stores per item at c4;
        // at d = 64 the extra code cost more than the rare use saved.)
        const float inv = 1.f / l_run;
        uint8_t* ot = sQ + (qb * 2 + t) * C::TILE;
#pragma unroll
        for (int c = 0; c < DC / 32; ++c) {
          float tmp[32];
          load_o(c, tmp);
#pragma unroll
          for (int q = 0; q < 32; q += 8) {
            uint4 pk;
            pk.x = pack_bf16x2(tmp[q + 0] * inv, tmp[q + 1] * inv);
            pk.y = pack_bf16x2(tmp[q + 2] * inv, tmp[q + 3] * inv);
            pk.z = pack_bf16x2(tmp[q + 4] * inv, tmp[q + 5] * inv);
            pk.w = pack_bf16x2(tmp[q + 6] * inv, tmp[q + 7] * inv);
            const int col = hf * DC + c * 32 + q;
            *reinterpret_cast<uint4*>(ot + (col >> 6) * SUB + swz(r, (col & 63) >> 3)) = pk;
          }
        }
        fence_proxy_async_smem();
        if (t == 0) named_bar_sync<1>(128 * HV);  // the group's threads (barrier 0 is the CTA's)
        else named_bar_sync<2>(128 * HV);
        if (r == 0 && hf == 0) {
#pragma unroll
          for (int b = 0; b < C::NSUB; ++b)
            tma_store_3d(&tm_o, ip.h * D + b * 64, (int32_t)(ip.q0 + t * BM), ip.s, ot + b * SUB);
          bulk_commit_group();
          bulk_wait_group_read0();
        }
      } else if (k0 == 0 && k1 == nkt) {
        const float inv = 1.f / l_run;
        uint16_t* orow = p.o + (((int64_t)ip.s * p.q_rows + row) * p.H + ip.h) * D + hf * DC;
#pragma unroll
        for (int c = 0; c < DC / 32; ++c) {
          float tmp[32];
          load_o(c, tmp);
          if (row < p.q_rows) {
#pragma unroll
            for (int q = 0; q < 32; q += 8) {
              uint4 pk;
              pk.x = pack_bf16x2(tmp[q + 0] * inv, tmp[q + 1] * inv);
              pk.y = pack_bf16x2(tmp[q + 2] * inv, tmp[q + 3] * inv);
              pk.z = pack_bf16x2(tmp[q + 4] * inv, tmp[q + 5] * inv);
              pk.w = pack_bf16x2(tmp[q + 6] * inv, tmp[q + 7] * inv);
              *reinterpret_cast<uint4*>(orow + c * 32 + q) = pk;
            }
          }
        }
      } else {
        // partial: publish (O, m, l) of this row, count in, and merge if last
        const int64_t slot = (item == u_lo / nkt) ? 0 : 1;
        const int64_t rec = ((cta * 2 + slot) * 2 + t) * BM + r;
        const int64_t c_first = sp.owner(item * nkt), c_last = sp.owner((item + 1) * nkt - 1);
        unsigned int* cnt = p.ws_cnt + (c_first * 2 + t) * BM + r;
        const unsigned int others = (unsigned int)(c_last - c_first);
        // One thread per row: when every other contributor has already
        // counted in, this one is the last and merges straight from its
        // tensor memory, without publishing its own partial.
        bool last = HV == 1 && ld_acquire_u32(cnt) == others;
        if (!last) {
          float* wo = p.ws_o + rec * D + hf * DC;
#pragma unroll
          for (int c = 0; c < DC / 32; ++c) {
            float tmp[32];
            load_o(c, tmp);
#pragma unroll
            for (int q = 0; q < 32; q += 4)
              __stcg(reinterpret_cast<float4*>(wo + c * 32 + q),
                     make_float4(tmp[q], tmp[q + 1], tmp[q + 2], tmp[q + 3]));
          }
          if (hf == 0) __stcg(p.ws_ml + rec, make_float2(m_run, l_run));
          if (HV == 2) {
            // the row's other half is written too before it is counted
            __threadfence();
            mbar_arrive(B.wb + t);
            if (!mbar_wait(B.wb + t, (uint32_t)nsplit & 1u, p.wait_ns)) {
              ok = false;
              break;
            }
            ++nsplit;
          }
          // release: this row's partial is visible before the count;
          // acquire: the last arriver sees every other partial
          if (hf == 0) last = atomic_add_acq_rel_u32(cnt, 1u) == others;
        }
        if (last && hf == 0) {
          // the others' records; this CTA's own (m, l) and, with one thread
          // per row, its O come from registers and tensor memory
          const bool own_here = HV == 1;
          float M = m_run, Lsum = l_run;
          for (int64_t cc = c_first; cc <= c_last; ++cc) {
            if (cc == cta) continue;
            const int64_t sl = (item == sp.lo(cc) / nkt) ? 0 : 1;
            const float2 ml = __ldcg(p.ws_ml + ((cc * 2 + sl) * 2 + t) * BM + r);
            const float Mn = fmaxf(M, ml.x);
            Lsum = Lsum * fast_exp2(M - Mn) + ml.y * fast_exp2(ml.x - Mn);
            M = Mn;
          }
          const float inv = 1.f / Lsum;
          const float w_own = fast_exp2(m_run - M) * inv;
          uint16_t* orow = p.o + (((int64_t)ip.s * p.q_rows + row) * p.H + ip.h) * D;
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float acc[32];
            if (own_here) {
              load_o(c, acc);
#pragma unroll
              for (int q = 0; q < 32; ++q) acc[q] *= w_own;
            } else {
#pragma unroll
              for (int q = 0; q < 32; ++q) acc[q] = 0.f;
            }
            for (int64_t cc = c_first; cc <= c_last; ++cc) {
              if (cc == cta && own_here) continue;
              const int64_t sl = (item == sp.lo(cc) / nkt) ? 0 : 1;
              const int64_t rc = ((cc * 2 + sl) * 2 + t) * BM + r;
              const float w = fast_exp2(__ldcg(p.ws_ml + rc).x - M) * inv;
              const float4* src = reinterpret_cast<const float4*>(p.ws_o + rc * D + c * 32);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const float4 v = __ldcg(src + q);
                acc[4 * q + 0] = __fmaf_rn(v.x, w, acc[4 * q + 0]);
                acc[4 * q + 1] = __fmaf_rn(v.y, w, acc[4 * q + 1]);
                acc[4 * q + 2] = __fmaf_rn(v.z, w, acc[4 * q + 2]);
                acc[4 * q + 3] = __fmaf_rn(v.w, w, acc[4 * q + 3]);
              }
            }
            if (row < p.q_rows) {
#pragma unroll
              for (int q = 0; q < 32; q += 8) {
                uint4 pk;
                pk.x = pack_bf16x2(acc[q + 0], acc[q + 1]);
                pk.y = pack_bf16x2(acc[q + 2], acc[q + 3]);
                pk.z = pack_bf16x2(acc[q + 4], acc[q + 5]);
                pk.w = pack_bf16x2(acc[q + 6], acc[q + 7]);
                *reinterpret_cast<uint4*>(orow + c * 32 + q) = pk;
              }
            }
          }
          *cnt = 0u;  // ready for the next launch
        }
      }
    }
    if (!ok) fail_wait(B);
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *B.abort_flag && p.state)
    for (int s = 0; s < p.S; ++s)
      atomicOr(reinterpret_cast<unsigned long long*>(&p.state[s].pub.error_word),
               (unsigned long long)kErrAttnWaitTimeout);
  if (wid == C::WI) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

bool make_tmap_bf16(CUtensorMap* map, const void* base, int64_t hd, int64_t rows, int64_t S) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return false;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  cuuint64_t dims[3] = {(cuuint64_t)hd, (cuuint64_t)rows, (cuuint64_t)S};
  cuuint64_t strides[2] = {(cuuint64_t)(hd * 2), (cuuint64_t)(hd * 2 * rows)};
  cuuint32_t box[3] = {64, 128, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims,
                      strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
static cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                            const AttnParams& p, int sm_count, cudaStream_t st) {
  const int smem = Cfg<D>::ALLOC;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool attr_set[64] = {};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int64_t nkt = (p.seg_count[0] + BN - 1) / BN + (p.seg_count[1] + BN - 1) / BN;
  const int64_t items = (int64_t)p.S * p.H * ((p.q_rows + 2 * BM - 1) / (2 * BM));
  if (nkt <= 0 || items <= 0) return cudaErrorInvalidValue;
  // One CTA per item unless that leaves a poor last wave on a large
  // problem; then the persistent split schedule (needs the workspace).
  const int64_t sms = sm_count > 0 ? sm_count : 1;
  const int64_t waves = (items + sms - 1) / sms;
  const bool ragged = items * 10 < waves * sms * 9;  // last wave < 90 % full
  const bool large = items * nkt >= 16 * sms;        // >= 16 key tiles per CTA
  int64_t grid;
  const bool has_ws = p.ws_o && p.ws_ml && p.ws_cnt;
  if (has_ws && p.grid > 0) {
    grid = p.grid;
  } else if (has_ws && ragged && large) {
    grid = sms;
  } else {
    grid = items;  // one item per CTA: nothing is split
  }
  if (has_ws) {
    if (grid > kAttnMaxCtas && grid != items) grid = kAttnMaxCtas;
    if (grid > items * nkt) grid = items * nkt;
  } else {
    grid = items;
  }
  if (grid < 1 || grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
  attn_kernel<D><<<(unsigned)grid, Cfg<D>::THREADS, smem, st>>>(tq, tk, tv, to, p);
  return cudaGetLastError();
}

cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const CUtensorMap& to, const AttnParams& p, int head_dim, int S,
                             int sm_count, cudaStream_t st) {
  if (p.S != S) return cudaErrorInvalidValue;
  if (head_dim == 64) return launch_d<64>(tq, tk, tv, to, p, sm_count, st);
  if (head_dim == 128) return launch_d<128>(tq, tk, tv, to, p, sm_count, st);
  return cudaErrorInvalidValue;
}

}  // namespace sds
