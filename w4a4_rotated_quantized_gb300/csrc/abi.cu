// Library-wide entry points of libquarot.so: status strings, version, and
// the device error word shared by all kernels.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace quarot {
__device__ unsigned int g_error_word = 0;

namespace {
PFN_cuCtxGetCurrent_v4000 g_get_ctx = nullptr;
PFN_cuCtxGetId_v12000 g_get_id = nullptr;
std::once_flag g_fn_once;
}  // namespace

// The driver's cuCtxGetCurrent and cuCtxGetId are reached through the
// runtime's entry-point query (the library links no driver library itself).
unsigned long long current_context_id() {
  std::call_once(g_fn_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_get_ctx = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (g_get_ctx == nullptr || g_get_id == nullptr) return 0;
  CUcontext ctx = nullptr;
  if (g_get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  unsigned long long id = 0;
  return g_get_id(ctx, &id) == CUDA_SUCCESS ? id : 0;
}

// One thread waits on a shared-memory barrier that nothing completes: the
// bounded wait every kernel uses gives up after kWaitLimitNs, records
// QUAROT_ERR_TIMEOUT and returns, and the kernel ends normally.
__global__ void selftest_wait_kernel() {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  fence_barrier_init();
  mbar_wait_bounded(&bar, 0u, nullptr);
}
}  // namespace quarot

extern "C" const char* quarot_status_string(int status) {
  switch (status) {
    case QUAROT_OK: return "ok";
    case QUAROT_ERR_INVALID_ARG: return "invalid argument";
    case QUAROT_ERR_UNSUPPORTED: return "unsupported size";
    case QUAROT_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case QUAROT_ERR_LAUNCH: return "kernel launch failed";
    case QUAROT_ERR_TIMEOUT: return "device-side wait timed out";
    case QUAROT_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

extern "C" int quarot_version(void) { return (1 << 16) | 1; }

extern "C" int quarot_check_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QUAROT_ERR_CUDA;
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, quarot::g_error_word, sizeof(word)) != cudaSuccess) return QUAROT_ERR_CUDA;
  if (word != 0 && cudaMemcpyToSymbol(quarot::g_error_word, &zero, sizeof(zero)) != cudaSuccess)
    return QUAROT_ERR_CUDA;
  if (word & (1u << QUAROT_ERR_TIMEOUT)) return QUAROT_ERR_TIMEOUT;
  return word ? QUAROT_ERR_CUDA : QUAROT_OK;
}

extern "C" int quarot_selftest_wait(void* stream) {
  quarot::selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>();
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}
