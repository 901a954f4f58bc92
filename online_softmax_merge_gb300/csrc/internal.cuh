// Internal declarations shared by the C ABI (api.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ringattn.h"

namespace ra {

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

// Launchers (return a cudaError_t of the launch).
cudaError_t launch_ring_tc(const RingParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t st);
cudaError_t launch_ring_simt(const RingParams& p, cudaStream_t st);
cudaError_t launch_finalize(const RingParams& p, cudaStream_t st);
cudaError_t launch_merge(int n, int B, int N, int H, int D, const float* o_parts,
                         const float* lse_parts, void* o, float* lse, cudaStream_t st);
cudaError_t launch_shard_map(int layout, int N, int P, int32_t* owner, int32_t* local,
                             int32_t* token_of, cudaStream_t st);
cudaError_t launch_tile_classes(const RingParams& p, int u, int b, int8_t* classes,
                                cudaStream_t st);
cudaError_t launch_mask(const RingParams& p, int u, int b, uint8_t* mask, cudaStream_t st);
cudaError_t launch_selftest_timeout(uint64_t limit_ns, int* status, cudaStream_t st);
// Pass-Q decode, phase 1: per-(shard, key chunk) partials into the workspace.
cudaError_t launch_decode_partials(const RingParams& p, int n_q, int q_pos0, float* o_parts,
                                   float* lse_parts, cudaStream_t st);
// Keys per chunk of a shard in the decode partial phase.
int decode_chunk_keys(int S);

// Bytes of dynamic shared memory the tensor-core kernel uses for head_dim D.
int ring_tc_smem_bytes(int D);

}  // namespace ra
