// Pass-Q decode over the virtual ring: a few query rows attend to a KV cache that
// stays sharded and stationary. Every virtual device u scores the queries against
// its own shard only and leaves a partial (O_u, LSE_u); the partials are combined
// by the merge kernel (merge.cu).
//  * Transformer Math "Ring Attention" (aicassindra), "The ring is a prefill
//    algorithm": broadcast the single query to all P devices, each computes a
//    partial (m, l, o) against its shard, one small reduction combines them.
//  * "Part 4: Ring Attention" (Fofadiya) §4.9.4.4: pass-Q decode.
//
// The partial phase is HBM-bound: each (batch, kv head) reads its K/V rows once,
// and all query rows of the GQA group (heads of the group x decode tokens) share
// them. A CTA owns up to RB query rows of one kv head and a chunk of keys of one
// shard (a shard is cut into chunks so that a small batch still fills the GPU;
// every chunk is one more partial for the merge). It streams 64-key K/V tiles
// through a double-buffered cp.async pipeline into shared memory and runs the
// online softmax in fp32 on CUDA cores: ~4 FLOP per byte read for 4 rows, well
// within the CUDA cores, so no GEMM reshaping.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.cuh"
#include "shardmap.cuh"

namespace ra {
namespace {

constexpr int kThreads = 256;
constexpr int kKT = 64;                    // keys per shared-memory tile
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(smem))),
               "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_le1() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

template <int D, int RB>
struct DecSmem {
  float q[RB][D];                    // query rows, pre-scaled by scale * log2(e)
  __nv_bfloat16 k[2][kKT][D + 8];    // padded rows: neighbouring keys start in other banks
  __nv_bfloat16 v[2][kKT][D];
  float s[RB][kKT];                  // log2-scaled scores, then probabilities
  float m[RB];                       // running max (log2 units)
  float z[RB];                       // running denominator
  float alpha[RB];                   // rescale factor of the current tile
};

// grid: x = key chunk of the shard, y = shard u, z = (batch * G + g) * n_rowgroups + rowgroup
template <int D, int RB>
__global__ void __launch_bounds__(kThreads)
decode_partial_kernel(const RingParams p, int n_q, int q_pos0, int chunk, int n_rowgroups,
                      float* __restrict__ o_parts, float* __restrict__ lse_parts) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  DecSmem<D, RB>& sm = *reinterpret_cast<DecSmem<D, RB>*>(smem_raw);
  const int tid = threadIdx.x;
  const int c = blockIdx.x, u = blockIdx.y;
  const int rg = blockIdx.z % n_rowgroups;
  const int bg = blockIdx.z / n_rowgroups;
  const int bat = bg / p.G, g = bg % p.G;
  const int hpg = p.H / p.G;
  const int rows_total = hpg * n_q;                 // query rows of this kv head
  const int row0 = rg * RB;
  const int n_rows = min(RB, rows_total - row0);
  const int j_begin = c * chunk;
  const int j_end = min(p.S, j_begin + chunk);
  const int part = u * static_cast<int>(gridDim.x) + c;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(p.v);

  // Row r of the CTA is query row rr = row0 + r of the kv head: head g*hpg + rr / n_q,
  // decode token rr % n_q at global position q_pos0 + rr % n_q.
  int qpos_max = -1;
  for (int r = 0; r < n_rows; ++r) qpos_max = max(qpos_max, q_pos0 + (row0 + r) % n_q);
  // Keys of the chunk some row may see: a prefix of the chunk under the causal mask.
  const int n_vis =
      j_end > j_begin ? visible_prefix(p.layout, p.S, p.P, p.causal, u, j_begin, j_end - j_begin, qpos_max) : 0;

  for (int idx = tid; idx < RB * D; idx += kThreads) {
    const int r = idx / D, col = idx % D;
    float val = 0.f;
    if (r < n_rows) {
      const int rr = row0 + r, h = g * hpg + rr / n_q, t = rr % n_q;
      val = __bfloat162float(q[((static_cast<size_t>(bat) * n_q + t) * p.H + h) * D + col]) *
            p.scale_log2;
    }
    sm.q[r][col] = val;
  }
  for (int r = tid; r < RB; r += kThreads) {
    sm.m[r] = -INFINITY;
    sm.z[r] = 0.f;
  }

  // Thread tid accumulates output column col of rows rsub, rsub + kRowStep, ...
  constexpr int kRowStep = kThreads / D;             // 2 (D = 128) or 4 (D = 64)
  constexpr int kOwn = (RB + kRowStep - 1) / kRowStep;
  const int col = tid % D;
  const int rsub = tid / D;
  float acc[kOwn];
#pragma unroll
  for (int i = 0; i < kOwn; ++i) acc[i] = 0.f;

  auto load_tile = [&](int buf, int j0) {
    constexpr int kPieces = kKT * (D / 8);           // 16-byte pieces of K (and of V)
    for (int idx = tid; idx < kPieces; idx += kThreads) {
      const int jj = idx / (D / 8), pc = idx % (D / 8);
      const int j = j0 + jj;
      if (j < j_end) {
        const int tk = pos_of(p.layout, p.S, p.P, u, j);
        const size_t off = ((static_cast<size_t>(bat) * p.N + tk) * p.G + g) * D + pc * 8;
        cp_async16(&sm.k[buf][jj][pc * 8], k + off);
        cp_async16(&sm.v[buf][jj][pc * 8], v + off);
      } else {
        *reinterpret_cast<uint4*>(&sm.k[buf][jj][pc * 8]) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(&sm.v[buf][jj][pc * 8]) = make_uint4(0, 0, 0, 0);
      }
    }
    cp_async_commit();
  };

  const int n_tiles = (n_vis + kKT - 1) / kKT;
  if (n_tiles > 0) load_tile(0, j_begin);
  for (int it = 0; it < n_tiles; ++it) {
    const int buf = it & 1;
    const int j0 = j_begin + it * kKT;
    if (it + 1 < n_tiles) {
      load_tile(buf ^ 1, j0 + kKT);
      cp_async_wait_le1();
    } else {
      cp_async_wait_all();
    }
    __syncthreads();
    // Scores of (row r, key jj): thread -> key jj = tid % 64, rows tid / 64 + 4 i.
    {
      const int jj = tid % kKT;
      const int j = j0 + jj;
      const uint4* kr = reinterpret_cast<const uint4*>(&sm.k[buf][jj][0]);
      for (int r = tid / kKT; r < RB; r += kThreads / kKT) {
        float sdot = -INFINITY;
        if (r < n_rows && j < j_end) {
          const int qp = q_pos0 + (row0 + r) % n_q;
          if (visible_prefix(p.layout, p.S, p.P, p.causal, u, j, 1, qp) > 0) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
            for (int pc = 0; pc < D / 8; ++pc) {
              const uint4 kv = kr[pc];
              const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kv);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 kf = __bfloat1622float2(k2[e]);
                a0 = fmaf(sm.q[r][pc * 8 + 2 * e], kf.x, a0);
                a1 = fmaf(sm.q[r][pc * 8 + 2 * e + 1], kf.y, a1);
              }
            }
            sdot = a0 + a1;
          }
        }
        sm.s[r][jj] = sdot;
      }
    }
    __syncthreads();
    // Online softmax of each row over the tile: warp w takes rows w, w + 8, ...
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int r = warp; r < RB; r += kThreads / 32) {
        const float s0 = sm.s[r][lane], s1 = sm.s[r][lane + 32];
        float mx = fmaxf(s0, s1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = sm.m[r];
        const float m_new = fmaxf(m_old, mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float p0 = exp2f(s0 - m_use), p1 = exp2f(s1 - m_use);
        float ps = p0 + p1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        // exact rescale exp(m_old - m_new); a row that saw nothing yet has a zero state
        const float a = (m_old == -INFINITY) ? 0.f : exp2f(m_old - m_use);
        sm.s[r][lane] = p0;
        sm.s[r][lane + 32] = p1;
        __syncwarp();
        if (lane == 0) {
          sm.m[r] = m_new;
          sm.z[r] = (m_new == -INFINITY) ? 0.f : sm.z[r] * a + ps;
          sm.alpha[r] = (m_new == -INFINITY) ? 1.f : a;
        }
      }
    }
    __syncthreads();
    // y_r = alpha_r y_r + sum_j p_rj V_j for the owned (row, column) outputs
#pragma unroll
    for (int i = 0; i < kOwn; ++i) {
      const int r = rsub + kRowStep * i;
      if (r < RB) {
        float a = acc[i] * sm.alpha[r];
#pragma unroll 8
        for (int jj = 0; jj < kKT; ++jj)
          a = fmaf(sm.s[r][jj], __bfloat162float(sm.v[buf][jj][col]), a);
        acc[i] = a;
      }
    }
    __syncthreads();   // buffer buf is refilled by the next iteration's prefetch
  }
  __syncthreads();
  // Normalised partial of this (shard, chunk): O = y / z, LSE = (m + log2 z) ln 2.
#pragma unroll
  for (int i = 0; i < kOwn; ++i) {
    const int r = rsub + kRowStep * i;
    if (r < n_rows) {
      const int rr = row0 + r, h = g * hpg + rr / n_q, t = rr % n_q;
      const float z = sm.z[r];
      const size_t oo = ((((static_cast<size_t>(part) * p.B + bat) * n_q + t) * p.H + h) * D) + col;
      o_parts[oo] = z > 0.f ? acc[i] / z : 0.f;
      if (col == 0) {
        const size_t lo = ((static_cast<size_t>(part) * p.B + bat) * p.H + h) * n_q + t;
        lse_parts[lo] = z > 0.f ? (sm.m[r] + log2f(z)) * kLn2 : -INFINITY;
      }
    }
  }
}

template <int D, int RB>
cudaError_t launch_rb(const RingParams& p, int n_q, int q_pos0, int chunk, float* o_parts,
                      float* lse_parts, cudaStream_t st) {
  const int rows_total = (p.H / p.G) * n_q;
  const int n_rowgroups = (rows_total + RB - 1) / RB;
  const int n_chunks = (p.S + chunk - 1) / chunk;
  const int smem = static_cast<int>(sizeof(DecSmem<D, RB>));
  cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D, RB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(n_chunks, p.P, p.B * p.G * n_rowgroups);
  decode_partial_kernel<D, RB><<<grid, kThreads, smem, st>>>(p, n_q, q_pos0, chunk, n_rowgroups,
                                                             o_parts, lse_parts);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const RingParams& p, int n_q, int q_pos0, int chunk, float* o_parts,
                     float* lse_parts, cudaStream_t st) {
  const int rows_total = (p.H / p.G) * n_q;
  if (rows_total <= 4) return launch_rb<D, 4>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
  if (rows_total <= 8) return launch_rb<D, 8>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
  if (rows_total <= 16) return launch_rb<D, 16>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
  return launch_rb<D, 32>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
}

}  // namespace

int decode_chunk_keys(int S) {
  // Enough chunks per shard to fill the GPU with a small batch, none shorter than 512 keys.
  return S <= 2048 ? S : 2048;
}

cudaError_t launch_decode_partials(const RingParams& p, int n_q, int q_pos0, float* o_parts,
                                   float* lse_parts, cudaStream_t st) {
  const int chunk = decode_chunk_keys(p.S);
  return p.D == 64 ? launch_d<64>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st)
                   : launch_d<128>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
}

}  // namespace ra
