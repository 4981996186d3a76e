// Library-wide entry points of libquarot.so: status strings, version, and
// the device error word shared by all kernels.
#include "common.cuh"

namespace quarot {
__device__ unsigned int g_error_word = 0;

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

extern "C" int quarot_version(void) { return (1 << 16) | 0; }

extern "C" int quarot_check_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QUAROT_ERR_CUDA;
  unsigned int word = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&word, quarot::g_error_word, sizeof(word)) != cudaSuccess) return QUAROT_ERR_CUDA;
  if (word != 0 && cudaMemcpyToSymbol(quarot::g_error_word, &zero, sizeof(zero)) != cudaSuccess)
    return QUAROT_ERR_CUDA;
  if (word & QUAROT_ERR_TIMEOUT) return QUAROT_ERR_TIMEOUT;
  return word ? QUAROT_ERR_CUDA : QUAROT_OK;
}

extern "C" int quarot_selftest_wait(void* stream) {
  quarot::selftest_wait_kernel<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>();
  return cudaGetLastError() == cudaSuccess ? QUAROT_OK : QUAROT_ERR_LAUNCH;
}
