// Copies between host memory and the device done by the SMs instead of the copy
// engines, for ring_attn_fwd_host: rows of page-locked host memory, which the GPU
// reaches through its mapping at the same address, are gathered into (or scattered
// from) a packed device buffer by plain 16- or 4-byte loads and stores.
//
// Why: while kernels run under the power cap, a copy-engine transfer over the host
// link was seen to stall for tens of milliseconds at a time; loads and stores issued
// by the SMs over the same link did not stall. Launched on a high-priority stream,
// these copies take their blocks ahead of the ring kernel's pending ones, so they
// finish in a few milliseconds while the ring kernel keeps the SMs busy.
//
// The caller checks that the whole host range is mapped (api.cu, mapped_host); the
// kernels address only rows [0, rows) x bytes [0, width) of each side.
#include <stdint.h>

#include <atomic>

#include "internal.cuh"

namespace ra {
namespace {

constexpr int kCopyThreads = 256;

// dst[r * dpitch + c] = src[r * spitch + c] for r < rows, c < width (in elements of T)
template <typename T>
__global__ void __launch_bounds__(kCopyThreads)
rows_copy(T* __restrict__ dst, const T* __restrict__ src, long long rows, long long width,
          long long spitch, long long dpitch) {
  const long long n = rows * width;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / width, c = i - r * width;
    dst[r * dpitch + c] = src[r * spitch + c];
  }
}

bool multiple(uintptr_t x, uintptr_t m) { return x % m == 0; }

}  // namespace

// Copies rows x width bytes from src (row pitch spitch) to dst (row pitch dpitch) with
// the SMs, in `blocks` blocks; 16-byte elements when every address and size allows,
// else 4-byte ones. Returns cudaErrorInvalidValue (nothing launched) when not even 4
// bytes divide them.
cudaError_t launch_rows_copy(void* dst, size_t dpitch, const void* src, size_t spitch,
                             size_t width, size_t rows, int blocks, cudaStream_t st) {
  // No shared memory: prefer the split that lets these blocks sit beside others. A
  // preference only (its failure is ignored), set once per device context.
  static OncePerContext carveout;
  (void)carveout.run([] {
    cudaError_t r =
        cudaFuncSetAttribute(rows_copy<uint4>, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(rows_copy<uint32_t>, cudaFuncAttributePreferredSharedMemoryCarveout,
                               100);
    if (r != cudaSuccess) (void)cudaGetLastError();
    return r;
  });
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) |
                      static_cast<uintptr_t>(dpitch) | static_cast<uintptr_t>(spitch) |
                      static_cast<uintptr_t>(width);
  if (rows == 0 || width == 0) return cudaSuccess;
  if (multiple(a, 16)) {
    rows_copy<uint4><<<blocks, kCopyThreads, 0, st>>>(
        static_cast<uint4*>(dst), static_cast<const uint4*>(src), static_cast<long long>(rows),
        static_cast<long long>(width / 16), static_cast<long long>(spitch / 16),
        static_cast<long long>(dpitch / 16));
  } else if (multiple(a, 4)) {
    rows_copy<uint32_t><<<blocks, kCopyThreads, 0, st>>>(
        static_cast<uint32_t*>(dst), static_cast<const uint32_t*>(src),
        static_cast<long long>(rows), static_cast<long long>(width / 4),
        static_cast<long long>(spitch / 4), static_cast<long long>(dpitch / 4));
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace ra
