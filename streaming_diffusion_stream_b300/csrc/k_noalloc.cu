// k_noalloc.cu -- sds_ssf_noalloc: the similarity filter for callers that
// cannot allocate device memory.
//
// Who needs this: code that runs under a fixed device-memory budget owned by
// another allocator, or inside a latency-critical loop where a cudaMalloc /
// cudaFree (which can synchronise the whole device) is not allowed, cannot
// call sds_create and so cannot use sds_ssf.  This entry point takes the
// frame, the reference frame and the uniform draws from the caller and keeps
// its reduction scratch in a fixed static device array instead of allocating.
//
// The arithmetic is K4's filter segment: the same work blocks of
// kRedBlockElems elements, the same per-thread sums and block tree, the same
// per-quantity finish and decision (all from ssf_reduce.cuh), so for the same
// frame, reference, draw and skip count it returns bit for bit the cosine,
// probability and decision that sds_ssf records.
#include <cudaTypedefs.h>

#include <mutex>

#include "ssf_reduce.cuh"

namespace sds {
namespace {

constexpr int64_t kCounterBytes = 256;  // ticket counter, padded to keep the partials aligned
constexpr int kFinStreams = 32;         // streams decided per round of the last block

// The scratch: a ticket counter followed by 3 double partials per (stream,
// work block).  One array per device, kept until the process exits; every
// call reuses it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SDS_NOALLOC_SCRATCH_BYTES];

static_assert((SDS_NOALLOC_SCRATCH_BYTES - kCounterBytes) / 8 == SDS_NOALLOC_MAX_PARTIALS,
              "the documented partials limit is what the scratch array holds");
static_assert(SDS_NOALLOC_BLOCK_ELEMS == kRedBlockElems, "work block size of the documented limit");

__device__ __forceinline__ float4 ld4(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }

struct NoAllocParams {
  const float* frame;          // [S][E]
  const float* ref;            // [S][E]
  const float* u;              // [S]
  const int64_t* skip_count;   // [S] or null (all zero)
  double* cos_out;             // [S]
  double* p_out;               // [S]
  int64_t* skip_out;           // [S]
  unsigned char* scratch;      // device address of g_noalloc_scratch
  int64_t S, E, nb, max_skip;
  double eta;
};

__global__ void __launch_bounds__(kStepThreads) ssf_noalloc_kernel(const NoAllocParams p) {
  __shared__ dfloat red[3 * kRedWarps];
  __shared__ double fin[kFinStreams * 3];
  __shared__ int is_last;
  unsigned int* counter = reinterpret_cast<unsigned int*>(p.scratch);
  double* partials = reinterpret_cast<double*>(p.scratch + kCounterBytes);
  const float4 z4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t total = p.S * p.nb;
  for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
    const int64_t s = w / p.nb, b = w % p.nb;
    const float* I = p.frame + s * p.E;
    const float* R = p.ref + s * p.E;
    const int64_t base = b * kRedBlockElems + threadIdx.x * 4;
    float4 a[kRedVec], r[kRedVec];
#pragma unroll
    for (int k = 0; k < kRedVec; ++k) {
      const int64_t e = base + k * (kStepThreads * 4);
      const bool h = e < p.E;
      a[k] = h ? ld4(I + e) : z4;
      r[k] = h ? ld4(R + e) : z4;
    }
    dfloat sd, si, sr;
    ssf_accumulate(a, r, sd, si, sr);
    block_sum3(sd, si, sr, red);
    if (threadIdx.x == 0) {
      double* part = partials + (s * p.nb + b) * 3;
      part[0] = df_to_double(sd);
      part[1] = df_to_double(si);
      part[2] = df_to_double(sr);
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    is_last = (atomicAdd(counter, 1u) == gridDim.x - 1) ? 1 : 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int64_t s0 = 0; s0 < p.S; s0 += kFinStreams) {
    const int ns = (int)min((int64_t)kFinStreams, p.S - s0);
    // one warp per sum, as K4's finish does it
    for (int k = warp; k < ns * 3; k += kRedWarps) {
      const int64_t s = s0 + k / 3;
      const double v = partials_sum(partials + s * p.nb * 3 + k % 3, p.nb, 3, lane);
      if (lane == 0) fin[k] = v;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < ns; i += kStepThreads) {
      const int64_t s = s0 + i;
      const int64_t cnt = p.skip_count ? p.skip_count[s] : 0;
      const double u = (double)__ldcg(p.u + s);
      double cosv, P;
      p.skip_out[s] = ssf_decision(fin[3 * i], fin[3 * i + 1], fin[3 * i + 2], p.eta, u, cnt,
                                   p.max_skip, cosv, P);
      p.cos_out[s] = cosv;
      p.p_out[s] = P;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    *counter = 0u;
    __threadfence();
  }
}

// Device address of the scratch array, looked up once per device context:
// the key is the id of the context current when the call is made, so a
// context torn down and created again (cudaDeviceReset) gets a fresh lookup.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_ptr[kMaxDevices] = {};
unsigned long long g_ctx_id[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);
typedef CUresult (*PFN_ctxGetId)(CUcontext, unsigned long long*);

cudaError_t current_context_id(unsigned long long* id) {
  static PFN_ctxGetCurrent get_cur = nullptr;
  static PFN_ctxGetId get_id = nullptr;
  if (!get_cur || !get_id) {
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) !=
            cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) !=
            cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return cudaErrorNotSupported;
    get_cur = reinterpret_cast<PFN_ctxGetCurrent>(f1);
    get_id = reinterpret_cast<PFN_ctxGetId>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  return get_id(ctx, id) == CUDA_SUCCESS ? cudaSuccess : cudaErrorDeviceUninitialized;
}

cudaError_t scratch_for_current_device(unsigned char** ptr, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  // make the device's primary context current (created here if no runtime
  // call has needed it yet; nothing is allocated)
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) return e;
  unsigned long long id = 0;
  e = current_context_id(&id);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev] || g_ctx_id[dev] != id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = static_cast<unsigned char*>(p);
    g_ctx_id[dev] = id;
    g_sms[dev] = n;
  }
  *ptr = g_ptr[dev];
  *sms = g_sms[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace sds

extern "C" sds_status sds_ssf_noalloc(const float* frame, const float* ref, const float* u,
                                      const int64_t* skip_count, int64_t S, int64_t E,
                                      double eta, int64_t max_skip, double* cos_out,
                                      double* p_out, int64_t* skip_out, sds_stream_t stream) {
  using namespace sds;
  auto al16 = [](const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
  auto al8 = [](const void* q) { return q && (reinterpret_cast<uintptr_t>(q) & 7u) == 0; };
  if (!al16(frame) || !al16(ref) || !u || !al8(cos_out) || !al8(p_out) || !al8(skip_out) ||
      (skip_count && !al8(skip_count))) {
    set_thread_error("ssf_noalloc: frame/ref must be 16-byte aligned, outputs 8-byte aligned, u non-NULL");
    return SDS_ERR_INVALID_ARG;
  }
  if (S < 1 || S > 65535 || E < 4 || E % 4 != 0 || !(eta < 1.0) || max_skip < 0) {
    set_thread_error("ssf_noalloc: need S in [1, 65535], E a positive multiple of 4, eta < 1, max_skip >= 0");
    return SDS_ERR_INVALID_ARG;
  }
  const int64_t nb = (E + kRedBlockElems - 1) / kRedBlockElems;
  if (S * nb * 3 > SDS_NOALLOC_MAX_PARTIALS) {
    set_thread_error("ssf_noalloc: S * ceil(E/8192) * 3 exceeds SDS_NOALLOC_MAX_PARTIALS (32736): "
                     "the request does not fit the fixed 256 KiB scratch; split it into smaller calls");
    return SDS_ERR_INVALID_ARG;
  }
  unsigned char* scratch = nullptr;
  int sms = 0;
  if (scratch_for_current_device(&scratch, &sms) != cudaSuccess) {
    cudaGetLastError();
    set_thread_error("ssf_noalloc: looking up the scratch array's device address failed");
    return SDS_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the ticket counter must start at zero whatever an earlier call left there
  if (cudaMemsetAsync(scratch, 0, sizeof(unsigned int), st) != cudaSuccess) {
    set_thread_error("ssf_noalloc: clearing the scratch counter failed");
    return SDS_ERR_CUDA;
  }
  NoAllocParams p{frame, ref, u, skip_count, cos_out, p_out, skip_out, scratch, S, E, nb, max_skip, eta};
  const int64_t total = S * nb, cap = (int64_t)sms * (2048 / kStepThreads);
  const int grid = (int)(total < cap ? total : cap);
  ssf_noalloc_kernel<<<grid, kStepThreads, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) {
    set_thread_error("ssf_noalloc: kernel launch failed");
    return SDS_ERR_CUDA;
  }
  return SDS_OK;
}
