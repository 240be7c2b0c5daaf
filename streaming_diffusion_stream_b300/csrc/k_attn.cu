// k_attn.cu -- K1: cross-frame softmax attention on tcgen05 tensor cores.
//
// StreamDiffusion notes, "Stream Batch": the n denoise slots form one batch
// and every slot's queries attend to the keys of the whole batch,
// Attn(Q_{t,i}, K_Batch, V_Batch) = Softmax(Q K_Batch^T / sqrt(d)) V_Batch.
// In video mode the key set is the sink + rolling ring of cached frames
// (StreamDiffusionV2 summary, sink tokens + rolling KV cache).
//
// One CTA owns two 128-row query tiles (Q0, Q1) of one (stream, head); both
// share every 128-key K/V tile.  Warp roles:
//   warps 0-3  softmax group 0 (tile Q0), one query row per thread = one TMEM lane
//   warps 4-7  softmax group 1 (tile Q1)
//   warp  8    TMA producer: Q once, then K and V tiles through an ST-stage ring
//   warp  9    MMA issuer (one thread): tcgen05.mma into tensor memory
// Tensor memory (512 columns): S0 [0,128), S1 [128,256) fp32 scores;
// O0 [256, 256+d), O1 [384, 384+d) fp32 accumulators.  Each group writes its
// probabilities P as packed bf16 over the first 64 columns of its own S
// region, and O += P V reads P straight from tensor memory (A operand in
// TMEM), so P never touches shared memory.  The MMA issuer interleaves
//   PV0(j), S0(j+1), PV1(j), S1(j+1), ...
// so the tensor core works on one group's tile while the other group runs
// its softmax (ping-pong).  tcgen05 MMAs run in issue order, so S0(j+1) may
// overwrite the P0(j) columns that PV0(j) reads.
// The online softmax keeps a running max m per row and rescales O (in
// tensor memory) only when a tile raises m by more than 8 (log2 units):
// otherwise probabilities may exceed 1 by up to 2^8, which fp32 sums and bf16
// P hold without loss.  Every wait has a time limit; on expiry the kernel
// records kErrAttnWaitTimeout in the stream's error word and leaves.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "rope.cuh"
#include "sds_internal.h"

namespace sds {
namespace {

constexpr int BM = 128;         // query rows per tile (two tiles per CTA)
constexpr int BN = 128;         // keys per tile
constexpr int SUB = 128 * 128;  // bytes of one 128-row x 64-column bf16 sub-tile
constexpr int kThreads = 320;   // 8 softmax warps + producer + MMA
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct Cfg {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * SUB;  // one 128-row tile of Q, K or V
  static constexpr int ST = (D == 64) ? 4 : 2;
  static constexpr int Q = 0;
  static constexpr int K = Q + 2 * TILE;
  static constexpr int V = K + ST * TILE;
  static constexpr int BAR = V + ST * TILE;
  static constexpr int TOTAL = BAR + 512;
  static constexpr int ALLOC = TOTAL + 1024;  // slack for 1024-byte alignment
};

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled sub-tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

struct Bars {
  uint64_t* q_full;
  uint64_t* q_ready;
  uint64_t* k_full;
  uint64_t* v_full;
  uint64_t* k_empty;
  uint64_t* v_empty;
  uint64_t* s_full;  // [2]
  uint64_t* p_full;  // [2]
  uint64_t* o_done;  // [2]
  uint64_t* mma_final;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
};

template <int D>
__device__ __forceinline__ Bars carve(uint8_t* sm) {
  using C = Cfg<D>;
  uint64_t* b = reinterpret_cast<uint64_t*>(sm + C::BAR);
  Bars r;
  r.q_full = b;
  r.q_ready = b + 1;
  r.k_full = b + 2;
  r.v_full = r.k_full + C::ST;
  r.k_empty = r.v_full + C::ST;
  r.v_empty = r.k_empty + C::ST;
  r.s_full = r.v_empty + C::ST;
  r.p_full = r.s_full + 2;
  r.o_done = r.p_full + 2;
  r.mma_final = r.o_done + 2;
  r.tmem_slot = reinterpret_cast<uint32_t*>(r.mma_final + 1);
  r.abort_flag = reinterpret_cast<volatile int*>(r.tmem_slot + 1);
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const Bars B = carve<D>(sm);
  uint8_t* sQ = sm + C::Q;
  uint8_t* sK = sm + C::K;
  uint8_t* sV = sm + C::V;

  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31;
  const int h = blockIdx.y, s = blockIdx.z;
  const int q0 = blockIdx.x * (2 * BM);
  const int nt0 = (p.seg_count[0] + BN - 1) / BN;
  const int nt = nt0 + (p.seg_count[1] + BN - 1) / BN;

  if (tid == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    mbar_init(B.q_full, 1);
    mbar_init(B.q_ready, 256);
    for (int i = 0; i < C::ST; ++i) {
      mbar_init(B.k_full + i, 1);
      mbar_init(B.v_full + i, 1);
      mbar_init(B.k_empty + i, 1);
      mbar_init(B.v_empty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B.s_full + i, 1);
      mbar_init(B.p_full + i, 128);
      mbar_init(B.o_done + i, 1);
    }
    mbar_init(B.mma_final, 1);
    *B.abort_flag = 0;
    fence_barrier_init();
  }
  if (wid == 9) {
    tmem_alloc(B.tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *B.tmem_slot;

  if (wid == 8) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nt > 0) {
      mbar_arrive_expect_tx(B.q_full, 2 * C::TILE);
      for (int t = 0; t < 2; ++t)
        for (int b = 0; b < C::NSUB; ++b)
          tma_load_3d(sQ + t * C::TILE + b * SUB, &tm_q, h * D + b * 64, q0 + t * BM, s, B.q_full);
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int st = j % C::ST;
        const uint32_t ph = (uint32_t)(j / C::ST) & 1u;
        int key0, nvalid;
        key_tile(p, nt0, j, key0, nvalid);
        if (!mbar_wait(B.k_empty + st, ph ^ 1u)) { fail_wait(B); break; }
        mbar_arrive_expect_tx(B.k_full + st, C::TILE);
        for (int b = 0; b < C::NSUB; ++b)
          tma_load_3d(sK + st * C::TILE + b * SUB, &tm_k, h * D + b * 64, key0, s, B.k_full + st);
        if (!mbar_wait(B.v_empty + st, ph ^ 1u)) {
          issued = j;  // K of tile j is in flight; wait for it below
          mbar_wait(B.k_full + st, ph);
          fail_wait(B);
          break;
        }
        mbar_arrive_expect_tx(B.v_full + st, C::TILE);
        for (int b = 0; b < C::NSUB; ++b)
          tma_load_3d(sV + st * C::TILE + b * SUB, &tm_v, h * D + b * 64, key0, s, B.v_full + st);
        issued = j + 1;
      }
      // leave only after every copy of ours has landed in shared memory
      mbar_wait(B.q_full, 0);
      for (int j = (issued > C::ST ? issued - C::ST : 0); j < issued; ++j) {
        mbar_wait(B.k_full + j % C::ST, (uint32_t)(j / C::ST) & 1u);
        mbar_wait(B.v_full + j % C::ST, (uint32_t)(j / C::ST) & 1u);
      }
    }
  } else if (wid == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nt > 0) {
      constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);
      constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, true);
      const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV);
      auto issue_s = [&](int t, int st) {
        const uint32_t dS = tmem + (uint32_t)(t * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * SUB + (kk & 3) * 32);
          mma_bf16_ss(dS, smem_desc_sw128(aQ + t * C::TILE + off, 16, 1024),
                      smem_desc_sw128(aK + st * C::TILE + off, 16, 1024), IDESC_S,
                      kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int st, bool acc) {
        const uint32_t dO = tmem + 256u + (uint32_t)(t * 128);
        const uint32_t aP = tmem + (uint32_t)(t * 128);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          mma_bf16_ts(dO, aP + (uint32_t)(kk * 8),
                      smem_desc_sw128(aV + st * C::TILE + kk * 16 * 128, SUB, 1024), IDESC_O,
                      (acc || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(B.q_ready, 0) && mbar_wait(B.k_full, 0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        mma_commit(B.s_full + 0);
        issue_s(1, 0);
        mma_commit(B.s_full + 1);
        mma_commit(B.k_empty + 0);
      }
      for (int j = 0; ok && j < nt; ++j) {
        const int st = j % C::ST;
        const uint32_t ph = (uint32_t)(j / C::ST) & 1u;
        const int st1 = (j + 1) % C::ST;
        const uint32_t ph1 = (uint32_t)((j + 1) / C::ST) & 1u;
        if (!mbar_wait(B.v_full + st, ph) || !mbar_wait(B.p_full + 0, (uint32_t)j & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(0, st, j > 0);
        mma_commit(B.o_done + 0);
        if (j + 1 < nt) {
          if (!mbar_wait(B.k_full + st1, ph1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_s(0, st1);
          mma_commit(B.s_full + 0);
        }
        if (!mbar_wait(B.p_full + 1, (uint32_t)j & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        issue_pv(1, st, j > 0);
        mma_commit(B.o_done + 1);
        mma_commit(B.v_empty + st);
        if (j + 1 < nt) {
          issue_s(1, st1);
          mma_commit(B.s_full + 1);
          mma_commit(B.k_empty + st1);
        }
      }
      if (!ok) fail_wait(B);
      // all our MMAs complete before tensor memory is released
      mma_commit(B.mma_final);
      mbar_wait(B.mma_final, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax groups
    const int t = wid >> 2;   // query tile of this group
    const int r = tid & 127;  // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((wid & 3) * 32) << 16;
    const uint32_t tS = tmem + (uint32_t)(t * 128) + lane_base;
    const uint32_t tO = tmem + 256u + (uint32_t)(t * 128) + lane_base;
    const int64_t row = (int64_t)q0 + t * BM + r;
    bool ok = nt > 0 && mbar_wait(B.q_full, 0);
    if (ok && p.rope_on && row < p.q_rows) {
      const int tok = (int)(row % p.chunk_tokens);
      const int jf = tok / p.tokens_L, l = tok % p.tokens_L;
      const int pos[3] = {p.p0 + jf, l / p.grid_w, l % p.grid_w};
      const int seg[3] = {p.rope_seg[0], p.rope_seg[1], p.rope_seg[2]};
      const int off[3] = {p.tab_off[0], p.tab_off[1], p.tab_off[2]};
#pragma unroll
      for (int b = 0; b < C::NSUB; ++b) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4* ptr = reinterpret_cast<uint4*>(sQ + t * C::TILE + b * SUB + swz(r, c));
          *ptr = rope8(*ptr, b * 64 + c * 8, pos, seg, p.rope_tab, off);
        }
      }
      fence_proxy_async_smem();
    }
    if (ok) mbar_arrive(B.q_ready);
    const float sc = p.scale_log2;
    float m_run = -INFINITY, l_run = 0.f;
    for (int j = 0; ok && j < nt; ++j) {
      if (!mbar_wait(B.s_full + t, (uint32_t)j & 1u)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float sv[BN / 32][32];
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld32(tS + (uint32_t)(c * 32), sv[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) reg_fence32(sv[c]);
      int key0, nvalid;
      key_tile(p, nt0, j, key0, nvalid);
      if (nvalid < BN) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          sv[c >> 5][c & 31] = (c < nvalid) ? sv[c >> 5][c & 31] : -INFINITY;
      }
      float mx[4] = {sv[0][0], sv[0][1], sv[0][2], sv[0][3]};
#pragma unroll
      for (int c = 4; c < BN; c += 4) {
        mx[0] = fmaxf(mx[0], sv[c >> 5][c & 31]);
        mx[1] = fmaxf(mx[1], sv[c >> 5][(c + 1) & 31]);
        mx[2] = fmaxf(mx[2], sv[c >> 5][(c + 2) & 31]);
        mx[3] = fmaxf(mx[3], sv[c >> 5][(c + 3) & 31]);
      }
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
      const bool need = mt > m_run + kRescaleThreshold;
      const float m_new = need ? mt : m_run;
      const float alpha = need ? fast_exp2(m_run - m_new) : 1.f;
      // P = exp2(s*sc - m) as packed bf16 over the first 64 columns of S
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int part = 0; part < 4; ++part) {
        uint32_t pk[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const float e0 = fast_exp2(__fmaf_rn(sv[part][2 * q], sc, -m_new));
          const float e1 = fast_exp2(__fmaf_rn(sv[part][2 * q + 1], sc, -m_new));
          rs[(2 * q) & 3] += e0;
          rs[(2 * q + 1) & 3] += e1;
          pk[q] = pack_bf16x2(e0, e1);
        }
        tmem_st16u(tS + (uint32_t)(part * 16), pk);
      }
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O may be rescaled only once the previous PV into it has landed
        if (!mbar_wait(B.o_done + t, (uint32_t)(j - 1) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
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
      mbar_arrive(B.p_full + t);
      l_run = l_run * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));
      m_run = m_new;
    }
    if (ok) ok = mbar_wait(B.o_done + t, (uint32_t)(nt - 1) & 1u);
    if (ok) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      uint16_t* orow = p.o + (((int64_t)s * p.q_rows + row) * p.H + h) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float tmp[32];
        tmem_ld32(tO + (uint32_t)(c * 32), tmp);
        tmem_wait_ld();
        reg_fence32(tmp);
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
    } else if (nt > 0) {
      fail_wait(B);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *B.abort_flag && p.state)
    atomicOr(reinterpret_cast<unsigned long long*>(&p.state[s].pub.error_word),
             (unsigned long long)kErrAttnWaitTimeout);
  if (wid == 9) {
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
static cudaError_t launch_d(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const AttnParams& p, int S, cudaStream_t st) {
  const int smem = Cfg<D>::ALLOC;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((unsigned)((p.q_rows + 2 * BM - 1) / (2 * BM)), (unsigned)p.H, (unsigned)S);
  attn_kernel<D><<<grid, kThreads, smem, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

cudaError_t launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const AttnParams& p, int head_dim, int S, cudaStream_t st) {
  if (head_dim == 64) return launch_d<64>(tq, tk, tv, p, S, st);
  if (head_dim == 128) return launch_d<128>(tq, tk, tv, p, S, st);
  return cudaErrorInvalidValue;
}

}  // namespace sds
