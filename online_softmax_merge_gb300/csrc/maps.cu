// Index maps on the GPU, computed by the same functions the ring kernels use
// (shardmap.cuh), plus the bounded-wait self test.
//  * shard ownership: owner[t], local[t], token_of[u*S + i] for a layout;
//  * tile classes of a (u, b) shard pair ("Part 4: Ring Attention" (Fofadiya)
//    §4.8.1 "Skipping Fully-Masked Blocks");
//  * the element mask of a (u, b) shard pair from the kernels' per-key visibility.
#include "internal.cuh"
#include "ptx.cuh"
#include "shardmap.cuh"

namespace ra {
namespace {

__global__ void shard_map_kernel(int layout, int N, int P, int32_t* owner, int32_t* local,
                                 int32_t* token_of) {
  const int S = N / P;
  for (long long t = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; t < N;
       t += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int tt = static_cast<int>(t);
    owner[tt] = owner_of(layout, S, P, tt);
    local[tt] = local_of(layout, S, P, tt);
    token_of[tt] = pos_of(layout, S, P, tt / S, tt % S);   // index tt = u*S + i
  }
}

__global__ void tile_class_kernel(int layout, int S, int P, int causal, int u, int b, int nt,
                                  int8_t* classes) {
  const long long n = static_cast<long long>(nt) * nt;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int qi = static_cast<int>(idx / nt), kj = static_cast<int>(idx % nt);
    classes[idx] = static_cast<int8_t>(
        tile_class(layout, S, P, causal, u, b, qi * RA_TILE, RA_TILE, kj * RA_TILE, RA_TILE));
  }
}

__global__ void mask_kernel(int layout, int S, int P, int causal, int u, int b, uint8_t* mask) {
  const long long n = static_cast<long long>(S) * S;
  for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(idx / S), j = static_cast<int>(idx % S);
    const int qpos = pos_of(layout, S, P, u, i);
    mask[idx] = visible_prefix(layout, S, P, causal, b, j, 1, qpos) > 0 ? 1 : 0;
  }
}

// One warp waits on a barrier that nothing will complete, for at most limit_ns,
// then records RA_ERR_TIMEOUT: the time-limit path of every wait in the library,
// exercised without a hang.
__global__ void selftest_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncwarp();
  bool ok = true;
  if (threadIdx.x == 0) ok = bounded_wait(smem_u32(&bar), 0, limit_ns, nullptr);
  if (threadIdx.x == 0 && !ok) atomicCAS(status, 0, static_cast<int>(RA_ERR_TIMEOUT));
}

// One thread checks the range [4, 5) against a 4-element extent (no access is made):
// in a debug build the check fails and records RA_ERR_BOUNDS; in a release build the
// check is compiled away and nothing is recorded.
__global__ void selftest_bounds_kernel(int* status) {
  if (threadIdx.x == 0) (void)in_bounds(4, 1, 4, status);
}

int blocks_for(long long n, int threads) {
  long long b = (n + threads - 1) / threads;
  if (b > 65535 * 16) b = 65535 * 16;
  return static_cast<int>(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_shard_map(int layout, int N, int P, int32_t* owner, int32_t* local,
                             int32_t* token_of, cudaStream_t st) {
  shard_map_kernel<<<blocks_for(N, 256), 256, 0, st>>>(layout, N, P, owner, local, token_of);
  return cudaGetLastError();
}

cudaError_t launch_tile_classes(const RingParams& p, int u, int b, int8_t* classes,
                                cudaStream_t st) {
  const int nt = (p.S + RA_TILE - 1) / RA_TILE;
  tile_class_kernel<<<blocks_for(static_cast<long long>(nt) * nt, 256), 256, 0, st>>>(
      p.layout, p.S, p.P, p.causal, u, b, nt, classes);
  return cudaGetLastError();
}

cudaError_t launch_mask(const RingParams& p, int u, int b, uint8_t* mask, cudaStream_t st) {
  mask_kernel<<<blocks_for(static_cast<long long>(p.S) * p.S, 256), 256, 0, st>>>(
      p.layout, p.S, p.P, p.causal, u, b, mask);
  return cudaGetLastError();
}

cudaError_t launch_selftest_bounds(int* status, cudaStream_t st) {
  selftest_bounds_kernel<<<1, 32, 0, st>>>(status);
  return cudaGetLastError();
}

cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t st) {
  selftest_timeout_kernel<<<1, 32, 0, st>>>(limit_ns, status);
  return cudaGetLastError();
}

}  // namespace ra
