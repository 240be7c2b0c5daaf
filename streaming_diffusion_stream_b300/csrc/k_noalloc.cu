// k_noalloc.cu -- sds_ssf_noalloc: the similarity-filter reduction of K4 for
// callers that cannot allocate device memory.
//
// Who needs this: code that runs under a fixed device-memory budget owned by
// another allocator, or inside a latency-critical loop where a cudaMalloc /
// cudaFree (which can synchronise the whole device) is not allowed, cannot
// call sds_create and so cannot use sds_ssf.  This entry point takes the
// frame, the reference frame and the uniform draws from the caller and keeps
// its reduction scratch in a fixed static device array instead of allocating.
//
// The arithmetic is K4's SSF segment, step for step (fp32 per thread over 8
// elements in the same order, a fixed double shuffle tree, one partial per
// 2048-element work block, the last block summing the partials in index
// order), so for the same frame and reference it returns the same cosine,
// probability and decision as sds_ssf.
#include <mutex>

#include "sds_internal.h"

namespace sds {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int64_t kBlockElems = 2048;
constexpr int64_t kCounterBytes = 256;  // ticket counter, padded to keep the partials aligned

// The scratch: a ticket counter followed by 3 double partials per (stream,
// work block).  One array per device, kept until the process exits; every
// call reuses it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SDS_NOALLOC_SCRATCH_BYTES];

__device__ __forceinline__ double warp_sum(double v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

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

__global__ void __launch_bounds__(kThreads) ssf_noalloc_kernel(const NoAllocParams p) {
  __shared__ double red[kWarps];
  __shared__ int is_last;
  unsigned int* counter = reinterpret_cast<unsigned int*>(p.scratch);
  double* partials = reinterpret_cast<double*>(p.scratch + kCounterBytes);
  const int64_t total = p.S * p.nb;
  for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
    const int64_t s = w / p.nb, b = w % p.nb;
    const float* I = p.frame + s * p.E;
    const float* R = p.ref + s * p.E;
    float dot = 0.f, ni = 0.f, nr = 0.f;
    for (int k = 0; k < 2; ++k) {
      const int64_t e = b * kBlockElems + k * (kThreads * 4) + threadIdx.x * 4;
      if (e >= p.E) continue;
      const float4 a = ld4(I + e), r = ld4(R + e);
      dot = __fmaf_rn(a.x, r.x, dot); ni = __fmaf_rn(a.x, a.x, ni); nr = __fmaf_rn(r.x, r.x, nr);
      dot = __fmaf_rn(a.y, r.y, dot); ni = __fmaf_rn(a.y, a.y, ni); nr = __fmaf_rn(r.y, r.y, nr);
      dot = __fmaf_rn(a.z, r.z, dot); ni = __fmaf_rn(a.z, a.z, ni); nr = __fmaf_rn(r.z, r.z, nr);
      dot = __fmaf_rn(a.w, r.w, dot); ni = __fmaf_rn(a.w, a.w, ni); nr = __fmaf_rn(r.w, r.w, nr);
    }
    const double sd = block_sum((double)dot, red);
    const double si = block_sum((double)ni, red);
    const double sr = block_sum((double)nr, red);
    if (threadIdx.x == 0) {
      double* part = partials + (s * p.nb + b) * 3;
      part[0] = sd;
      part[1] = si;
      part[2] = sr;
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
  for (int64_t s = 0; s < p.S; ++s) {
    double q[3];
    for (int c = 0; c < 3; ++c) {
      double v = 0.0;
      for (int64_t i = threadIdx.x; i < p.nb; i += kThreads) v += __ldcg(partials + (s * p.nb + i) * 3 + c);
      q[c] = block_sum(v, red);
    }
    if (threadIdx.x == 0) {
      const double dot = q[0], ni = q[1], nr = q[2];
      const double cosv = (ni > 0.0 && nr > 0.0) ? dot / sqrt(ni * nr) : 0.0;
      const double P = fmin(1.0, fmax(0.0, (cosv - p.eta) / (1.0 - p.eta)));
      const int64_t cnt = p.skip_count ? p.skip_count[s] : 0;
      const double u = (double)__ldcg(p.u + s);
      p.cos_out[s] = cosv;
      p.p_out[s] = P;
      p.skip_out[s] = (u < P && cnt < p.max_skip) ? 1 : 0;
    }
  }
  if (threadIdx.x == 0) {
    *counter = 0u;
    __threadfence();
  }
}

// Device address of the scratch array, looked up once per device.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_ptr[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};

cudaError_t scratch_for_current_device(unsigned char** ptr, int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = static_cast<unsigned char*>(p);
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
  const int64_t nb = (E + kBlockElems - 1) / kBlockElems;
  if (S * nb * 3 > SDS_NOALLOC_MAX_PARTIALS) {
    set_thread_error("ssf_noalloc: S * ceil(E/2048) * 3 exceeds SDS_NOALLOC_MAX_PARTIALS (32736): "
                     "the request does not fit the fixed 256 KiB scratch; split it into smaller calls");
    return SDS_ERR_INVALID_ARG;
  }
  unsigned char* scratch = nullptr;
  int sms = 0;
  if (scratch_for_current_device(&scratch, &sms) != cudaSuccess) {
    cudaGetLastError();
    set_thread_error("ssf_noalloc: cudaGetSymbolAddress of the scratch array failed");
    return SDS_ERR_CUDA;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the ticket counter must start at zero whatever an earlier call left there
  if (cudaMemsetAsync(scratch, 0, sizeof(unsigned int), st) != cudaSuccess) {
    set_thread_error("ssf_noalloc: clearing the scratch counter failed");
    return SDS_ERR_CUDA;
  }
  NoAllocParams p{frame, ref, u, skip_count, cos_out, p_out, skip_out, scratch, S, E, nb, max_skip, eta};
  const int64_t total = S * nb, cap = (int64_t)sms * 8;
  const int grid = (int)(total < cap ? total : cap);
  ssf_noalloc_kernel<<<grid, kThreads, 0, st>>>(p);
  if (cudaGetLastError() != cudaSuccess) {
    set_thread_error("ssf_noalloc: kernel launch failed");
    return SDS_ERR_CUDA;
  }
  return SDS_OK;
}
