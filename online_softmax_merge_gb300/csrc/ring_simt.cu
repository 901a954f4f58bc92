// Plain SIMT (CUDA-core, fp32) ring step: a slow cross-check of the tensor-core
// kernel, with the same contract as ring_attn_step. One warp per query row; a
// block of 8 warps shares 32-key K/V chunks staged in shared memory as fp32.
// Scores, exponentials (expf) and the P·V products stay in fp32 — no tensor
// cores and no bf16 rounding of the probabilities.
//
// The fold is the ring recurrence of "Ring Attention" (aarnphm.xyz): with m the
// running max, z the denominator and y the unnormalised output of a row, a block
// of scores S over keys j updates m' = max(m, max_j S_j),
// z' = z e^{m - m'} + sum_j e^{S_j - m'}, y' = y e^{m - m'} + sum_j e^{S_j - m'} V_j.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.cuh"
#include "shardmap.cuh"

namespace ra {
namespace {

constexpr int kWarps = 8;
constexpr int kChunk = 32;

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
ring_simt_kernel(const RingParams p, int s) {
  __shared__ float ks[kChunk][D + 1];
  __shared__ float vs[kChunk][D];
  __shared__ float qs[kWarps][D];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // grid: x = row block within shard, y = batch * heads + head, z = shard u
  const int u = blockIdx.z;
  const int bat = blockIdx.y / p.H, head = blockIdx.y % p.H;
  const int g = (head * p.G) / p.H;
  const int row = blockIdx.x * kWarps + warp;
  const bool valid = row < p.S;
  const int qpos = valid ? pos_of(p.layout, p.S, p.P, u, row) : -1;
  int b = (u - s) % p.P;
  if (b < 0) b += p.P;

  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(p.v);
  constexpr int E = D / 32;   // output columns per lane: lane + 32*e
  float y[E];
  float m = -INFINITY, z = 0.f;
  const size_t md = valid ? (static_cast<size_t>(bat) * p.H + head) * p.N + qpos : 0;
  const size_t yo = valid ? ((static_cast<size_t>(bat) * p.N + qpos) * p.H + head) * D : 0;
  // this row's q, state and output lie in their tensors
  const bool io_ok = valid && in_bounds(md, 1, row_elems(p), p.status) &&
                     in_bounds(yo, D, q_elems(p), p.status);
  if (io_ok && p.load_state) {
    m = p.m[md];
    z = p.z[md];
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = p.y[yo + lane + 32 * e];
  } else {
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] = 0.f;
  }
  for (int c = lane; c < D; c += 32)
    qs[warp][c] = io_ok ? __bfloat162float(q[yo + c]) : 0.f;

  // keys that may be visible: a prefix of the shard except for zigzag (two runs)
  const int n_vis = !valid ? 0
                    : p.layout == kZigzag ? p.S
                                          : visible_prefix(p.layout, p.S, p.P, p.causal, b, 0, p.S, qpos);
  // The block walks the union of its rows' visible prefixes.
  int n_blk = n_vis;
  n_blk = __reduce_max_sync(0xffffffffu, n_blk);
  __shared__ int warp_max[kWarps];
  if (lane == 0) warp_max[warp] = n_blk;
  __syncthreads();
  n_blk = 0;
  for (int w = 0; w < kWarps; ++w) n_blk = max(n_blk, warp_max[w]);

  for (int j0 = 0; j0 < n_blk; j0 += kChunk) {
    __syncthreads();
    for (int idx = threadIdx.x; idx < kChunk * D; idx += blockDim.x) {
      const int jj = idx / D, c = idx % D;
      const int j = j0 + jj;
      float kv = 0.f, vv = 0.f;
      const int tk = j < p.S ? pos_of(p.layout, p.S, p.P, b, j) : 0;
      const size_t off = ((static_cast<size_t>(bat) * p.N + tk) * p.G + g) * D + c;
      if (j < p.S && in_bounds(off, 1, kv_elems(p), p.status)) {
        kv = __bfloat162float(k[off]);
        vv = __bfloat162float(v[off]);
      }
      ks[jj][c] = kv;
      vs[jj][c] = vv;
    }
    __syncthreads();
    // lane jj scores key j0 + jj
    const int jj = lane;
    float sdot = 0.f;
#pragma unroll 8
    for (int c = 0; c < D; ++c) sdot = fmaf(qs[warp][c], ks[jj][c], sdot);
    const bool vis = (j0 + jj < n_vis) && key_visible(p.layout, p.S, p.P, p.causal, b, j0 + jj, qpos);
    float sc = vis ? sdot * p.scale : -INFINITY;
    float bm = sc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, o));
    const float m_new = fmaxf(m, bm);
    if (m_new == -INFINITY) continue;        // nothing visible yet for this row
    const float alpha = (m == -INFINITY) ? 0.f : expf(m - m_new);
    const float pj = expf(sc - m_new);       // 0 for masked keys
    float ps = pj;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    z = z * alpha + ps;
#pragma unroll
    for (int e = 0; e < E; ++e) y[e] *= alpha;
    for (int j = 0; j < kChunk; ++j) {
      const float pb = __shfl_sync(0xffffffffu, pj, j);
#pragma unroll
      for (int e = 0; e < E; ++e) y[e] = fmaf(pb, vs[j][lane + 32 * e], y[e]);
    }
    m = m_new;
  }
  if (io_ok) {
#pragma unroll
    for (int e = 0; e < E; ++e) p.y[yo + lane + 32 * e] = y[e];
    if (lane == 0) {
      p.m[md] = m;
      p.z[md] = z;
    }
  }
}

}  // namespace

cudaError_t launch_ring_simt(const RingParams& p, cudaStream_t st) {
  const dim3 grid((p.S + kWarps - 1) / kWarps, p.B * p.H, p.P);
  if (p.D == 64)
    ring_simt_kernel<64><<<grid, kWarps * 32, 0, st>>>(p, p.s_begin);
  else
    ring_simt_kernel<128><<<grid, kWarps * 32, 0, st>>>(p, p.s_begin);
  return cudaGetLastError();
}

}  // namespace ra
