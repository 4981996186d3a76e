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
// never a device address.  Its device address belongs to the CUDA context in
// which the library's module was loaded, so it is looked up with
// cudaGetSymbolAddress (with that device current) the first time a call runs
// in a context, and cached together with that context's unique id.  After a
// cudaDeviceReset, or any other re-creation of the context, the id differs
// and the address is looked up again: the kernels never receive an address
// from a context that no longer exists.
#include <mutex>

#include "common.cuh"

namespace quarot {
namespace {

__device__ __align__(256) unsigned char g_decode_scratch[QUAROT_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
struct Cached {
  unsigned long long ctx_id = 0;  // cuCtxGetId of the context the address belongs to (0: none yet)
  void* ptr = nullptr;
};
std::mutex g_mu;
Cached g_cache[kMaxDevices];

// Device address of the scratch array in the current device's current
// context, or nullptr with the CUDA error in *err.
void* scratch_on_current_device(cudaError_t* err) {
  int dev = -1;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = current_context_id();
  Cached& c = g_cache[dev];
  if (id != 0 && id == c.ctx_id) return c.ptr;
  // first call in this context (or no context current yet: the lookup makes
  // the device's primary context current)
  void* p = nullptr;
  *err = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (*err != cudaSuccess) return nullptr;
  id = current_context_id();
  if (id == 0) {
    *err = cudaErrorContextIsDestroyed;
    return nullptr;
  }
  c.ctx_id = id;
  c.ptr = p;
  return p;
}

}  // namespace
}  // namespace quarot

extern "C" int quarot_decode_attn_static(const void* q, const uint8_t* k_q, const void* k_s,
                                         const uint8_t* v_q, const void* v_s, int64_t B, int64_t Hq,
                                         int64_t Hkv, int64_t d, int64_t T, int64_t T_max,
                                         float sm_scale, int unrotate_out, void* out, void* stream) {
  // The argument checks of quarot_decode_attn, in its order, then the size
  // limit: nothing touches the device for a rejected request, and a request
  // that quarot_decode_attn rejects gets the same status here.
  if (B < 0 || Hq <= 0 || Hkv <= 0 || T < 0 || T_max < 0 || T > T_max) return QUAROT_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return QUAROT_ERR_INVALID_ARG;
  if (d != quarot::kDecodeHeadDim || Hq / Hkv > quarot::kDecodeMaxGroup) return QUAROT_ERR_UNSUPPORTED;
  if (B == 0 || T == 0)  // nothing to attend over: no scratch is read or written
    return quarot_decode_attn(q, k_q, k_s, v_q, v_s, B, Hq, Hkv, d, T, T_max, sm_scale, unrotate_out, out, nullptr,
                              0, stream);
  const size_t need = quarot_decode_workspace_bytes(B, Hq, d, T);
  if (need == 0 || need > size_t(QUAROT_DECODE_STATIC_SCRATCH_BYTES)) return QUAROT_ERR_UNSUPPORTED;
  cudaError_t err = cudaSuccess;
  void* scratch = quarot::scratch_on_current_device(&err);
  if (scratch == nullptr) return QUAROT_ERR_CUDA;
  return quarot_decode_attn(q, k_q, k_s, v_q, v_s, B, Hq, Hkv, d, T, T_max, sm_scale, unrotate_out, out,
                            scratch, size_t(QUAROT_DECODE_STATIC_SCRATCH_BYTES), stream);
}
