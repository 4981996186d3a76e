// quarot_decode_attn_static: the decode attention of quarot_decode_attn with
// its split-T scratch held in a fixed device array inside this library, so
// the caller passes inputs and outputs but never provides or allocates
// scratch.
//
// Who needs this: callers that cannot allocate device memory at the point
// where they run decode -- plain C hosts with no allocator of their own,
// serving loops that forbid device allocation after start-up (cudaMalloc and
// cudaFree synchronise the device and can fail under memory pressure), and
// plug-in layers that receive only input and output buffers from their host.
//
// The array below is a file-scope __device__ symbol: every GPU that loads
// the library holds QUAROT_DECODE_STATIC_SCRATCH_BYTES of it until the
// process exits.  In host code the symbol name is only a host-side stand-in,
// never a device address, so its device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and cached.
#include <mutex>

#include "common.cuh"

namespace quarot {
namespace {

__device__ __align__(256) unsigned char g_decode_scratch[QUAROT_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_ptr[kMaxDevices] = {};
cudaError_t g_err[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up on the
// first call per device), or nullptr with the CUDA error in *err.
void* scratch_on_current_device(cudaError_t* err) {
  int dev = -1;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::call_once(g_once[dev], [dev] {
    void* p = nullptr;
    g_err[dev] = cudaGetSymbolAddress(&p, g_decode_scratch);
    g_ptr[dev] = (g_err[dev] == cudaSuccess) ? p : nullptr;
  });
  *err = g_err[dev];
  return g_ptr[dev];
}

}  // namespace
}  // namespace quarot

extern "C" int quarot_decode_attn_static(const void* q, const uint8_t* k_q, const void* k_s,
                                         const uint8_t* v_q, const void* v_s, int64_t B, int64_t Hq,
                                         int64_t Hkv, int64_t d, int64_t T, int64_t T_max,
                                         float sm_scale, int unrotate_out, void* out, void* stream) {
  // Size limit first: nothing touches the device for a rejected request.
  if (B < 0 || Hq <= 0 || T < 0) return QUAROT_ERR_INVALID_ARG;
  if (B > 0 && T > 0) {
    const size_t need = quarot_decode_workspace_bytes(B, Hq, d, T);
    if (need == 0) return QUAROT_ERR_UNSUPPORTED;
    if (need > size_t(QUAROT_DECODE_STATIC_SCRATCH_BYTES)) return QUAROT_ERR_UNSUPPORTED;
  }
  cudaError_t err = cudaSuccess;
  void* scratch = quarot::scratch_on_current_device(&err);
  if (scratch == nullptr) return QUAROT_ERR_CUDA;
  return quarot_decode_attn(q, k_q, k_s, v_q, v_s, B, Hq, Hkv, d, T, T_max, sm_scale, unrotate_out, out,
                            scratch, size_t(QUAROT_DECODE_STATIC_SCRATCH_BYTES), stream);
}
