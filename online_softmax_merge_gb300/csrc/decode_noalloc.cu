// ring_attn_decode_noalloc: pass-Q decode for callers that cannot allocate device
// memory. It is ring_attn_decode with the per-shard partials kept in a fixed
// scratch array that belongs to the library image instead of a caller workspace.
//
// Who needs it: code that must not call cudaMalloc (or a caching allocator that
// may fall back to it) at the moment it decodes — a latency-critical serving loop
// where an allocation can synchronise the device or stall on the allocator's
// lock, a plugin whose host application owns every byte of device memory and hands
// it only the tensors it works on, or a runtime that plans all device memory up
// front. Such callers still pass q, k, v, o and lse; only the scratch for the
// partials comes from here, so the call itself allocates nothing.
//
// The price: the array (kScratchBytes) is static device memory, held until the
// process exits by every GPU on which this file's module has been loaded. The CUDA
// runtime loads modules lazily by default, so that happens at the first call of this
// entry point on a device (the lookup of the array's address below): that first
// call reserves the array, can fail with RA_ERR_CUDA if the device has no room for
// it, and should come before any stream capture; later calls allocate nothing.
// Problems whose partials need more than the array are rejected; and because every
// call on a GPU shares the one array, calls whose kernels overlap on that GPU
// (different streams, no ordering between them) race on it.
#include <mutex>

#include "internal.cuh"

namespace ra {
namespace {

constexpr size_t kScratchBytes = static_cast<size_t>(RA_DECODE_SCRATCH_BYTES);

// The scratch the partials go to. Host code must not pass the symbol itself to a
// kernel (on the host it is only a stand-in): the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchAddr {
  unsigned long long ctx = 0;   // context the address belongs to (0: not looked up)
  void* ptr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];

// Device address of the scratch array in the current context, looked up (with the
// device current) the first time and again whenever the context is a new one.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lk(g_mu);
  ScratchAddr& a = g_scratch_addr[dev];
  if (a.ptr == nullptr || id == 0 || a.ctx != id) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();   // leave no error behind for the caller's next CUDA call
      a.ptr = nullptr;
      return e;
    }
    a.ptr = ptr;
    a.ctx = current_context_id();
  }
  *out = a.ptr;
  return cudaSuccess;
}

}  // namespace
}  // namespace ra

extern "C" ra_status ring_attn_decode_noalloc(const ra_problem* p, int32_t n_q, int32_t q_pos0,
                                              const void* q, const void* k, const void* v,
                                              void* o, float* lse, void* stream) {
  const size_t need = ring_attn_decode_workspace_bytes(p, n_q);
  if (need == 0) return RA_ERR_INVALID_ARG;                 // invalid problem or n_q
  if (need > ra::kScratchBytes) return RA_ERR_INVALID_ARG;  // partials do not fit the scratch
  void* scratch = nullptr;
  const cudaError_t e = ra::scratch_address(&scratch);
  if (e != cudaSuccess) return ra::cuda_failed(e);
  // Every partial the decode writes is written before the merge reads it, so the
  // previous call's contents need no clearing.
  return ring_attn_decode(p, n_q, q_pos0, q, k, v, o, lse, scratch, ra::kScratchBytes, stream);
}
