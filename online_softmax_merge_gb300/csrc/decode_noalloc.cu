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
// The price: the array (kScratchBytes) is static device memory, reserved on every
// GPU that loads this library and held until the process exits; problems whose
// partials need more than that are rejected; and because every call on a GPU
// shares the one array, calls whose kernels overlap on that GPU (different
// streams, no ordering between them) race on it.
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
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once per
// device (with that device current) and cached.
cudaError_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = ptr;
  }
  *out = g_scratch_addr[dev];
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
  if (ra::scratch_address(&scratch) != cudaSuccess) return RA_ERR_CUDA;
  // Every partial the decode writes is written before the merge reads it, so the
  // previous call's contents need no clearing.
  return ring_attn_decode(p, n_q, q_pos0, q, k, v, o, lse, scratch, ra::kScratchBytes, stream);
}
