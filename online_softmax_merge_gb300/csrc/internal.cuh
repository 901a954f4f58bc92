// Internal declarations shared by the C ABI (api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/ringattn.h"

namespace ra {

// Id of the CUDA context current on the calling thread (the driver's cuCtxGetId,
// unique within the process), or 0 when no context is current or the driver cannot
// say. What the library looks up once and keeps per device -- the device addresses
// of its static arrays, the kernels' shared-memory limits -- is remembered together
// with this id and looked up again when it changes: an application that destroys a
// device's context and makes a new one (cudaDeviceReset, then further calls) would
// otherwise launch kernels with addresses and limits that belong to the old one.
unsigned long long current_context_id();

// A one-time setting (a kernel attribute), made once in every context of a device
// and again whenever the current context is a new one.
class OncePerContext {
 public:
  template <typename F>
  cudaError_t run(F&& set) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::atomic<unsigned long long>& done = done_[dev & 63];  // a shared slot only costs a redo
    const unsigned long long id = current_context_id();
    if (id != 0 && done.load() == id) return cudaSuccess;
    e = set();
    if (e != cudaSuccess) return e;
    const unsigned long long now = current_context_id();    // setting it made one current
    if (now != 0) done.store(now);
    return cudaSuccess;
  }

 private:
  std::atomic<unsigned long long> done_[64] = {};
};

// Debug builds (compiled with -DRA_DEBUG): every raw global access (one that is not
// a TMA copy, which the hardware bounds by its tensor map) first checks its element
// range against the extent of its buffer. A failed check records RA_ERR_BOUNDS in
// the status word and the access is skipped, so a wrong index shows up as a status
// code rather than a memory fault. Release builds compile the checks away.
#ifdef RA_DEBUG
constexpr bool kDebugChecks = true;
#else
constexpr bool kDebugChecks = false;
#endif

// Is [first, first + count) inside [0, extent)?
__device__ __forceinline__ bool in_bounds(size_t first, size_t count, size_t extent,
                                          int* status) {
  if (!kDebugChecks) return true;
  if (first <= extent && count <= extent - first) return true;
  atomicCAS(status, 0, static_cast<int>(RA_ERR_BOUNDS));
  return false;
}

// Element counts of the public tensors of a problem with fields B, N, H, G, D.
template <typename Params>
__host__ __device__ __forceinline__ size_t q_elems(const Params& p) {   // q, o, dout, dq, y
  return static_cast<size_t>(p.B) * p.N * p.H * p.D;
}
template <typename Params>
__host__ __device__ __forceinline__ size_t kv_elems(const Params& p) {  // k, v, dk, dv
  return static_cast<size_t>(p.B) * p.N * p.G * p.D;
}
template <typename Params>
__host__ __device__ __forceinline__ size_t row_elems(const Params& p) { // lse, m, z
  return static_cast<size_t>(p.B) * p.H * p.N;
}

// Everything a ring kernel needs about one call. Sizes follow the public
// conventions: q/o [B,N,H,d], k/v [B,N,G,d], lse/m/z [B,H,N], y [B,N,H,d].
struct RingParams {
  int32_t B, N, H, G, D, S, P, layout, causal;
  // Work decomposition of the tensor-core kernel: a CTA owns two 128-row query
  // sub-tiles. pair_heads = 1: two query heads of one kv group, same rows;
  // pair_heads = 0: one head, two consecutive 128-row tiles.
  int32_t pair_heads;
  int32_t X, L;           // query rows are tiled per chunk: X chunks of L rows
                          // (contiguous, striped: X = P, L = S; zigzag: X = 2P, L = S/2)
  int32_t nq;             // 128-row query tiles per chunk, ceil(L / 128)
  int32_t nqq;            // query units per chunk and head pair
  int32_t pairs_per_g;    // head pairs (or heads) per kv head
  int32_t units_per_bg;   // CTAs per (batch, kv head)
  // Which ring steps this launch folds: s in [s_begin, s_end).
  int32_t s_begin, s_end;
  int32_t step_mode;      // 0: fold all steps then write O, LSE; 1: read/write (m, z, y)
  int32_t load_state;     // step mode: 1 = start from the HBM state, 0 = from empty
  int32_t o_f32;          // o is fp32 (RA_DTYPE_F32) instead of bf16
  float scale;            // score scale (natural units)
  float scale_log2;       // scale * log2(e)
  uint64_t timeout_ns;    // limit of every device-side wait
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  float* m;
  float* z;
  float* y;
  int* status;            // the device status word
};

// Everything the backward kernels need about one call. q, o, dout, dq
// [B,N,H,d]; k, v, dk, dv [B,N,G,d]; lse [B,H,N]. Tiles are addressed by (chunk,
// 128-row tile) as in the forward: X chunks of L rows, nt = ceil(L / 128) tiles
// per chunk (contiguous, striped: chunk = shard; zigzag: chunk = half-shard).
struct BwdParams {
  int32_t B, N, H, G, D, S, P, layout, causal;
  int32_t X, L, nt;
  int32_t tiles;          // B * H * X * nt query tiles
  int32_t o_f32;          // the saved o is fp32 (RA_DTYPE_F32) instead of bf16
  float scale;            // score scale (natural units)
  float scale_log2;       // scale * log2(e)
  uint64_t timeout_ns;    // limit of every device-side wait
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  // Per (batch, head, chunk, tile), 256 floats: LSE * log2(e) of the tile's 128
  // rows, then D = rowsum(dO * O); rows past the chunk's end hold +inf and 0.
  // After the tiles * 256 floats: the extension rows (16 bf16 per query row) of
  // -LSE/scale for every tile, then of -D, then one key-side tile of ones.
  float* ws;
  void* dq;
  void* dk;
  void* dv;
  int* status;
};

// Records e as the calling thread's last CUDA error (ring_attn_last_cuda_error) and
// returns RA_ERR_CUDA.
ra_status cuda_failed(cudaError_t e);

// Launchers (return a cudaError_t of the launch).
cudaError_t launch_ring_tc(const RingParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t st);
cudaError_t launch_ring_simt(const RingParams& p, cudaStream_t st);
cudaError_t launch_finalize(const RingParams& p, cudaStream_t st);
cudaError_t launch_merge(int n, int B, int N, int H, int D, const float* o_parts,
                         const float* lse_parts, void* o, bool o_f32, float* lse,
                         cudaStream_t st);
cudaError_t launch_shard_map(int layout, int N, int P, int32_t* owner, int32_t* local,
                             int32_t* token_of, cudaStream_t st);
cudaError_t launch_tile_classes(const RingParams& p, int u, int b, int8_t* classes,
                                cudaStream_t st);
cudaError_t launch_mask(const RingParams& p, int u, int b, uint8_t* mask, cudaStream_t st);
cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t st);
cudaError_t launch_selftest_bounds(int* status, cudaStream_t st);

// rows x width bytes from src (row pitch spitch) to dst (row pitch dpitch), copied by
// the SMs in `blocks` blocks (hostcopy.cu); either side may be mapped page-locked host
// memory.
cudaError_t launch_rows_copy(void* dst, size_t dpitch, const void* src, size_t spitch,
                             size_t width, size_t rows, int blocks, cudaStream_t st);
// Pass-Q decode, phase 1: per-(shard segment, key chunk) partials into the
// workspace. tk, tv: [B,N,G,d] views with 32-row boxes. With `clustered` (when
// decode_clustered says so) the partials of a row group are merged inside the
// launch, through a thread-block cluster, and O and LSE (p.o, p.lse) are written
// directly: no merge launch follows.
bool decode_clustered(const RingParams& p, int n_q);
cudaError_t launch_decode_partials(const RingParams& p, const CUtensorMap& tk,
                                   const CUtensorMap& tv, int n_q, int q_pos0, float* o_parts,
                                   float* lse_parts, bool clustered, cudaStream_t st);
// Keys per chunk of a shard segment in the decode partial phase, and the number
// of partials (P x segments x chunks per segment).
int decode_chunk_keys(int S, int P, int layout);
int decode_parts(int S, int P, int layout);

// Backward: statistics pass, then the dK/dV and dQ tensor-core kernels.
// tq, tdo: [B,N,H,d] views; tk, tv: [B,N,G,d] views (as for the forward).
cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t st);
cudaError_t launch_bwd_dkdv(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                            const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& text,
                            cudaStream_t st);
cudaError_t launch_bwd_dq(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                          const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st);

// Bytes of dynamic shared memory the tensor-core kernel uses for head_dim D.
int ring_tc_smem_bytes(int D);

}  // namespace ra
