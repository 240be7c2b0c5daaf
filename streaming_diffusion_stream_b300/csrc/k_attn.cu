// k_attn.cu -- K1: cross-frame softmax attention on tcgen05 tensor cores.
//
// StreamDiffusion notes, "Stream Batch": the n denoise slots form one batch
// and every slot's queries attend to the keys of the whole batch,
// Attn(Q_{t,i}, K_Batch, V_Batch) = Softmax(Q K_Batch^T / sqrt(d)) V_Batch.
// In video mode the key set is the sink + rolling ring of cached frames
// (StreamDiffusionV2 summary, sink tokens + rolling KV cache).
//
// One CTA owns 128 query rows of one (stream, head).  Per 128-key tile:
//   S = Q K^T    tcgen05.mma M=128 N=128 K=16 steps, bf16 -> fp32 in TMEM
//   softmax      each thread owns one query row = one TMEM lane; online
//                max/sum in fp32 with exp2, P rounded to bf16 into shared
//                memory in the 128-byte-swizzled K-major layout
//   O += P V     tcgen05.mma M=128 N=d, V read MN-major; O stays in TMEM and
//                is rescaled in place when the running max grows
// Q, K and V arrive by TMA (3-D maps {H*d, rows, S}, 64x128 boxes, 128-byte
// swizzle) with a two-stage K/V ring so the next tile's load overlaps the
// current tile's work.  Video queries are rotated (RoPE) in shared memory
// right after their load.  Every wait has a time limit; on expiry the
// kernel records kErrAttnWaitTimeout in the stream's error word and leaves.
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "ptx.cuh"
#include "rope.cuh"
#include "sds_internal.h"

namespace sds {
namespace {

constexpr int BM = 128;                 // query rows per CTA
constexpr int BN = 128;                 // keys per tile
constexpr int SUB = 128 * 128;          // bytes of one 128-row x 64-column bf16 sub-tile
constexpr int kThreads = 128;

template <int D>
struct Smem {
  static constexpr int NSUB = D / 64;
  static constexpr int TILE = NSUB * SUB;  // one Q, K or V tile (128 rows x D)
  static constexpr int Q = 0;
  static constexpr int K = Q + TILE;       // two stages
  static constexpr int V = K + 2 * TILE;   // two stages
  static constexpr int P = V + 2 * TILE;   // 128 x 128 bf16 = two sub-tiles
  static constexpr int BAR = P + 2 * SUB;  // mbarriers
  static constexpr int TOTAL = BAR + 64;
  static constexpr int ALLOC = TOTAL + 1024;  // slack for 1024-byte alignment
};

// Byte offset of 16-byte chunk c (0..7) of row r inside a 128-byte-swizzled sub-tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = sm + L::Q;
  uint8_t* sK = sm + L::K;
  uint8_t* sV = sm + L::V;
  uint8_t* sP = sm + L::P;
  uint64_t* bar_q = reinterpret_cast<uint64_t*>(sm + L::BAR);
  uint64_t* bar_kv = bar_q + 1;   // [2]
  uint64_t* bar_mma = bar_q + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_q + 4);

  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.y, s = blockIdx.z;
  const int q0 = blockIdx.x * BM;

  const int nt0 = (p.seg_count[0] + BN - 1) / BN;
  const int nt = nt0 + (p.seg_count[1] + BN - 1) / BN;

  if (tid == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    mbar_init(bar_q, 1);
    mbar_init(bar_kv + 0, 1);
    mbar_init(bar_kv + 1, 1);
    mbar_init(bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tS = tmem;          // columns [0, 128): S tile
  const uint32_t tO = tmem + 128;    // columns [128, 128 + D): O accumulator
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;

  auto issue_kv = [&](int j, int stage) {
    int key0;
    if (j < nt0) {
      key0 = p.seg_start[0] + j * BN;
    } else {
      key0 = p.seg_start[1] + (j - nt0) * BN;
    }
    mbar_arrive_expect_tx(bar_kv + stage, 2 * L::TILE);
    for (int b = 0; b < L::NSUB; ++b) {
      tma_load_3d(sK + stage * L::TILE + b * SUB, &tm_k, h * D + b * 64, key0, s, bar_kv + stage);
      tma_load_3d(sV + stage * L::TILE + b * SUB, &tm_v, h * D + b * 64, key0, s, bar_kv + stage);
    }
  };

  if (tid == 0) {
    mbar_arrive_expect_tx(bar_q, L::TILE);
    for (int b = 0; b < L::NSUB; ++b) tma_load_3d(sQ + b * SUB, &tm_q, h * D + b * 64, q0, s, bar_q);
    if (nt > 0) issue_kv(0, 0);
  }

  bool ok = mbar_wait(bar_q, 0);
  // K/V tiles issued and tiles whose arrival thread 0 has seen (abort path)
  int kv_issued = (nt > 0) ? 1 : 0, kv_seen = 0;

  const int r = tid;  // this thread's query row within the tile == TMEM lane
  if (ok && p.rope_on) {
    const int64_t row = (int64_t)q0 + r;
    if (row < p.q_rows) {
      const int tok = (int)(row % p.chunk_tokens);
      const int jf = tok / p.tokens_L, l = tok % p.tokens_L;
      const int pos[3] = {p.p0 + jf, l / p.grid_w, l % p.grid_w};
      const int seg[3] = {p.rope_seg[0], p.rope_seg[1], p.rope_seg[2]};
      const int off[3] = {p.tab_off[0], p.tab_off[1], p.tab_off[2]};
#pragma unroll
      for (int b = 0; b < L::NSUB; ++b) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint4* ptr = reinterpret_cast<uint4*>(sQ + b * SUB + swz(r, c));
          *ptr = rope8(*ptr, b * 64 + c * 8, pos, seg, p.rope_tab, off);
        }
      }
    }
    fence_proxy_async_smem();
  }
  ok = __syncthreads_and(ok) != 0;

  constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, false);
  constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, true);
  const uint32_t aQ = smem_u32(sQ), aK = smem_u32(sK), aV = smem_u32(sV), aP = smem_u32(sP);

  float m_run = -INFINITY, l_run = 0.f;
  uint32_t mma_phase = 0;
  int j = 0;
  for (; ok && j < nt; ++j) {
    const int st = j & 1;
    if (tid == 0 && j + 1 < nt) {
      issue_kv(j + 1, st ^ 1);
      kv_issued++;
    }
    bool wok = mbar_wait(bar_kv + st, (uint32_t)(j >> 1) & 1u);
    if (tid == 0 && wok) {
      kv_seen++;
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (uint32_t)((kk >> 2) * SUB + (kk & 3) * 32);
        mma_bf16_ss(tS, smem_desc_sw128(aQ + off, 16, 1024),
                    smem_desc_sw128(aK + st * L::TILE + off, 16, 1024), IDESC_S, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar_mma);
    }
    if (__syncthreads_or(!wok)) {
      ok = false;
      break;
    }
    wok = mbar_wait(bar_mma, mma_phase);
    mma_phase ^= 1u;
    if (__syncthreads_or(!wok)) {
      ok = false;
      break;
    }
    tc_fence_after();

    // ---- softmax on this thread's row
    float sv[BN];
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      float tmp[32];
      tmem_ld32(tS + lane_base + c * 32, tmp);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 32; ++q) sv[c * 32 + q] = tmp[q];
    }
    const int seg = (j < nt0) ? 0 : 1;
    const int tile_in_seg = (j < nt0) ? j : (j - nt0);
    const int nvalid = min(BN, p.seg_count[seg] - tile_in_seg * BN);
    float mt = -INFINITY;
#pragma unroll
    for (int c = 0; c < BN; ++c) {
      if (c >= nvalid) sv[c] = -INFINITY;
      mt = fmaxf(mt, sv[c]);
    }
    const float m_new = fmaxf(m_run, mt * p.scale_log2);
    const float alpha = fast_exp2(m_run - m_new);
    float rs = 0.f;
#pragma unroll
    for (int c = 0; c < BN; c += 8) {
      float e[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        e[q] = fast_exp2(__fmaf_rn(sv[c + q], p.scale_log2, -m_new));
        rs += e[q];
      }
      uint4 pk;
      pk.x = pack_bf16x2(e[0], e[1]);
      pk.y = pack_bf16x2(e[2], e[3]);
      pk.z = pack_bf16x2(e[4], e[5]);
      pk.w = pack_bf16x2(e[6], e[7]);
      *reinterpret_cast<uint4*>(sP + (c >> 6) * SUB + swz(r, (c & 63) >> 3)) = pk;
    }
    l_run = l_run * alpha + rs;
    m_run = m_new;

    // ---- rescale the O accumulator when any row of the warp saw a larger max
    if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float tmp[32];
        tmem_ld32(tO + lane_base + c * 32, tmp);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 32; ++q) tmp[q] *= alpha;
        tmem_st32(tO + lane_base + c * 32, tmp);
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int kk = 0; kk < BN / 16; ++kk) {
        const uint32_t offp = (uint32_t)((kk >> 2) * SUB + (kk & 3) * 32);
        const uint32_t offv = (uint32_t)(st * L::TILE + kk * 16 * 128);
        mma_bf16_ss(tO, smem_desc_sw128(aP + offp, 16, 1024),
                    smem_desc_sw128(aV + offv, SUB, 1024), IDESC_O,
                    (j > 0 || kk > 0) ? 1u : 0u);
      }
      mma_commit(bar_mma);
    }
    wok = mbar_wait(bar_mma, mma_phase);
    mma_phase ^= 1u;
    if (__syncthreads_or(!wok)) {
      ok = false;
      break;
    }
    tc_fence_after();
  }

  if (ok && nt > 0) {
    // ---- epilogue: O / l -> bf16 -> global (rows past the end are not stored)
    const float inv = 1.f / l_run;
    const int64_t row = (int64_t)q0 + r;
    uint16_t* orow = p.o + (((int64_t)s * p.q_rows + row) * p.H + h) * D;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      float tmp[32];
      tmem_ld32(tO + lane_base + c * 32, tmp);
      tmem_wait_ld();
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
  }
  if (!ok) {
    if (tid == 0) {
      // leave only after our own copies have landed (bounded), so no TMA
      // write targets shared memory of a CTA that has exited
      for (int t = kv_seen; t < kv_issued; ++t) mbar_wait(bar_kv + (t & 1), (uint32_t)(t >> 1) & 1u);
      if (p.state) atomicOr(reinterpret_cast<unsigned long long*>(&p.state[s].pub.error_word),
                            (unsigned long long)kErrAttnWaitTimeout);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
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
  const int smem = Smem<D>::ALLOC;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dim3 grid((unsigned)((p.q_rows + BM - 1) / BM), (unsigned)p.H, (unsigned)S);
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
