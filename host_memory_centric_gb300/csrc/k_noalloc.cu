// k_noalloc.cu -- RMSNorm backward for callers that cannot allocate device memory.
//
// The regular entry point (mt_rmsnorm_bwd) needs a scratch buffer for the
// per-block partial sums of dgamma, which the caller allocates.  Some callers
// cannot do that: code that runs while a stream is being captured into a
// graph, code living inside another framework whose allocator owns all device
// memory (and forbids foreign cudaMalloc calls), or latency-sensitive callers
// for whom cudaMalloc/cudaFree (which may synchronise the device) is not
// acceptable.  For them, this file keeps the scratch in a fixed device array
// that is part of the loaded library image, so a call allocates nothing.
//
// Limits and sharing rules (also stated in include/mt.h):
//   * the array holds kNoAllocFloats floats (9.5 MiB); every GPU that loads
//     the library holds one copy until the process exits;
//   * sizes whose partial sums exceed it are rejected with MT_ERR_ARG;
//   * all calls share the one array: two calls that overlap on the GPU (for
//     example on two streams without ordering) race and give wrong results;
//   * the array keeps the last call's contents; nothing in it has to start at
//     zero, because the first kernel writes every partial row the second
//     kernel reads;
//   * the first call on each device looks up the array's device address
//     (cudaGetSymbolAddress); make that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mt.h"
#include "mt_kernels.h"

namespace {

// 304 blocks x 8192 columns of FP32 partial sums.
constexpr size_t kNoAllocFloats = 304u * 8192u;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
float* g_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device (host code must not use the symbol itself as an address).
cudaError_t scratch_for_current_device(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" mt_status mt_rmsnorm_bwd_noalloc(const void* dy, const void* x, const void* gamma, const float* rstd,
                                            const void* dres, int64_t T, int32_t H, void* dx, void* dgamma,
                                            void* stream) {
  if (!dy || !x || !gamma || !rstd || !dx || !dgamma || T < 0 || H <= 0) return MT_ERR_ARG;
  const int64_t need = mt::rmsnorm_bwd_partial_floats(T, H);
  if (need < 0 || (size_t)need > kNoAllocFloats) return MT_ERR_ARG;
  float* scratch = nullptr;
  cudaError_t e = scratch_for_current_device(&scratch);
  if (e != cudaSuccess) return MT_ERR_CUDA;
  e = mt::rmsnorm_bwd((const mt::bf16*)dy, (const mt::bf16*)x, (const mt::bf16*)gamma, rstd, (const mt::bf16*)dres,
                      T, H, (mt::bf16*)dx, (mt::bf16*)dgamma, scratch, (cudaStream_t)stream);
  if (e == cudaErrorInvalidValue) return MT_ERR_ARG;
  return e == cudaSuccess ? MT_OK : MT_ERR_CUDA;
}
