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
// them. A CTA owns RB query rows of one kv head and a chunk of keys of one shard
// (a shard is cut into chunks so that a small batch still fills the GPU; every
// chunk is one more partial for the merge).
//
// Inside a CTA every warp streams its own groups of KG keys through a private
// multi-stage cp.async pipeline in shared memory (16 KiB of loads in flight per
// warp); lane l then reads d/32 consecutive columns of each K and V row, and those
// registers serve all RB query rows. The
// RB x KG partial dot products of a group are summed across lanes with a
// butterfly reduce-scatter that leaves lane l with the full score of pair
// (key l / RB, row l % RB). Each warp keeps its own online-softmax state
// (m, z, y) in fp32; the warps of the CTA merge theirs once at the end.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.cuh"
#include "ptx.cuh"
#include "shardmap.cuh"

namespace ra {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr float kLn2 = 0.6931471805599453f;

template <int EPL>
struct RowLoad;
template <>
struct RowLoad<4> {   // d = 128: 4 bf16 per lane, one 8-byte load
  static __device__ __forceinline__ void get(const __nv_bfloat16* row, int lane, float (&f)[4]) {
    const uint2 w = __ldcs(reinterpret_cast<const uint2*>(row) + lane);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  }
};
template <>
struct RowLoad<2> {   // d = 64: 2 bf16 per lane, one 4-byte load
  static __device__ __forceinline__ void get(const __nv_bfloat16* row, int lane, float (&f)[2]) {
    const uint32_t w = __ldcs(reinterpret_cast<const unsigned int*>(row) + lane);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    f[0] = a.x; f[1] = a.y;
  }
};

template <int EPL>
__device__ __forceinline__ void smem_cols(const __nv_bfloat16* row, int lane, float (&f)[EPL]) {
  if constexpr (EPL == 4) {
    const uint2 w = reinterpret_cast<const uint2*>(row)[lane];
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w.y));
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  } else {
    const uint32_t w = reinterpret_cast<const uint32_t*>(row)[lane];
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
    f[0] = a.x; f[1] = a.y;
  }
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Sum over the 32 lanes of 32 values. Slot s of lane l must hold the lane's
// contribution to value (s XOR l); afterwards lane l holds the total of value l
// in v[0]. With that slot order every level keeps the lower half of the slots and
// sends the upper half, so no lane-dependent selects are needed.
__device__ __forceinline__ void reduce_scatter32(float (&v)[32]) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
#pragma unroll
    for (int i = 0; i < o; ++i) v[i] += __shfl_xor_sync(0xffffffffu, v[i + o], o);
  }
}

constexpr int kWarpStageBytes = 8192;    // per-warp pipeline: 8 KiB of K/V in flight

template <int D, int RB>
struct DecCfg {
  static constexpr int KG = 32 / RB;                   // keys per group
  static constexpr int kStage = KG * D * 2 * 2;        // K and V rows of one group, bf16
  static constexpr int kStages = kWarpStageBytes / kStage;
  static constexpr int kPipe = kWarps * kStages * kStage;
  static constexpr int kMerge = kWarps * RB * (D + 2) * 4;
  static constexpr int kXchg = kWarps * (32 + RB) * 4;   // per-warp probabilities, rescales
  static constexpr int kSmem = kPipe + kMerge + kXchg;
};

// grid: x = (g * n_rowgroups + rowgroup), y = key chunk of the shard, z = batch * P + u
template <int D, int RB>
__global__ void __launch_bounds__(kThreads, 2)
decode_partial_kernel(const RingParams p, int n_q, int q_pos0, int chunk, int n_rowgroups,
                      float* __restrict__ o_parts, float* __restrict__ lse_parts) {
  using C = DecCfg<D, RB>;
  constexpr int EPL = D / 32;          // columns per lane
  constexpr int KG = C::KG;            // KG * RB = 32 (key, row) pairs per group
  constexpr int NS = C::kStages;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __nv_bfloat16* pipe = reinterpret_cast<__nv_bfloat16*>(smem_raw + warp * NS * C::kStage);
  float* sm_m = reinterpret_cast<float*>(smem_raw + C::kPipe);       // [kWarps][RB]
  float* sm_z = sm_m + kWarps * RB;                                   // [kWarps][RB]
  float* sm_y = sm_z + kWarps * RB;                                   // [kWarps][RB][D]
  float* sm_p = reinterpret_cast<float*>(smem_raw + C::kPipe + C::kMerge) + warp * (32 + RB);
  const int g = blockIdx.x / n_rowgroups, rg = blockIdx.x % n_rowgroups;
  const int c = blockIdx.y;
  const int bat = blockIdx.z / p.P, u = blockIdx.z % p.P;
  const int hpg = p.H / p.G;
  const int rows_total = hpg * n_q;
  const int row0 = rg * RB;
  const int n_rows = min(RB, rows_total - row0);
  const int j_begin = c * chunk;
  const int j_end = min(p.S, j_begin + chunk);
  const int part = u * static_cast<int>(gridDim.y) + c;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  const __nv_bfloat16* k = static_cast<const __nv_bfloat16*>(p.k);
  const __nv_bfloat16* v = static_cast<const __nv_bfloat16*>(p.v);

  // Rows: row r of the CTA is query row rr = row0 + r of kv head g, i.e. head
  // g*hpg + rr / n_q, decode token rr % n_q at global position q_pos0 + rr % n_q.
  int qpos_max = -1;
#pragma unroll
  for (int r = 0; r < RB; ++r)
    if (r < n_rows) qpos_max = max(qpos_max, q_pos0 + (row0 + r) % n_q);
  // keys of the chunk some row may see: a prefix of the chunk, except for zigzag
  // shards whose chunk may span both halves (then the per-key rule alone decides)
  const int n_vis = j_end <= j_begin ? 0
                    : p.layout == kZigzag ? j_end - j_begin
                                          : visible_prefix(p.layout, p.S, p.P, p.causal, u, j_begin,
                                                           j_end - j_begin, qpos_max);
  const int j_stop = j_begin + n_vis;

  // This lane's query columns of every row, pre-scaled by scale * log2(e), with
  // the rows in slot order: slot row i holds row i XOR (lane mod RB).
  float qv[RB][EPL];
#pragma unroll
  for (int i = 0; i < RB; ++i) {
    const int r = i ^ (lane % RB);
    if (r < n_rows) {
      const int rr = row0 + r, h = g * hpg + rr / n_q, t = rr % n_q;
      float f[EPL];
      RowLoad<EPL>::get(q + ((static_cast<size_t>(bat) * n_q + t) * p.H + h) * D, lane, f);
#pragma unroll
      for (int e = 0; e < EPL; ++e) qv[i][e] = f[e] * p.scale_log2;
    } else {
#pragma unroll
      for (int e = 0; e < EPL; ++e) qv[i][e] = 0.f;
    }
  }
  const int my_r = lane % RB;
  const int my_k = lane / RB;
  const int my_qpos = (my_r < n_rows) ? q_pos0 + (row0 + my_r) % n_q : -1;

  float m_run = -INFINITY, z_run = 0.f;   // state of row my_r (same on all its lanes)
  float acc[RB][EPL];
#pragma unroll
  for (int r = 0; r < RB; ++r)
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[r][e] = 0.f;

  const size_t row_stride = static_cast<size_t>(p.G) * D;   // elements between tokens
  const __nv_bfloat16* kb = k + (static_cast<size_t>(bat) * p.N * p.G + g) * D;
  const __nv_bfloat16* vb = v + (static_cast<size_t>(bat) * p.N * p.G + g) * D;

  // The warp's groups: keys [j_begin + (warp + kWarps * n) * KG, +KG), n = 0, 1, ...
  const int n_groups_total = (n_vis + KG - 1) / KG;
  const int n_mine = n_groups_total > warp ? (n_groups_total - warp + kWarps - 1) / kWarps : 0;
  auto issue = [&](int n) {   // copy group n of this warp into stage n % NS (always commits)
    if (n < n_mine) {
      const int j0 = j_begin + (warp + kWarps * n) * KG;
      __nv_bfloat16* st = pipe + (n % NS) * (C::kStage / 2);
      constexpr int kPieces = 2 * KG * (D / 8);          // 16-byte pieces of K and V rows
#pragma unroll
      for (int i = lane; i < kPieces; i += 32) {
        const int row = i / (D / 8), pc = i % (D / 8);   // rows [0, KG): K, [KG, 2KG): V
        const int kk = row % KG;
        const int j = j0 + kk;
        __nv_bfloat16* dst = st + row * D + pc * 8;
        if (j < j_stop) {
          const size_t tok = static_cast<size_t>(pos_of(p.layout, p.S, p.P, u, j));
          const __nv_bfloat16* src = (row < KG ? kb : vb) + tok * row_stride + pc * 8;
          cp_async16(static_cast<uint32_t>(__cvta_generic_to_shared(dst)), src);
        } else {
          *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    cp_async_commit();
  };
#pragma unroll
  for (int n = 0; n < NS - 1; ++n) issue(n);

  for (int n = 0; n < n_mine; ++n) {
    issue(n + NS - 1);
    cp_async_wait<NS - 1>();   // group n has landed (for this lane)
    __syncwarp();              // ... and for every lane of the warp
    const __nv_bfloat16* st = pipe + (n % NS) * (C::kStage / 2);
    const int j0 = j_begin + (warp + kWarps * n) * KG;
    // partial dot products of the 32 (key, row) pairs over this lane's columns, in
    // slot order: slot kk*RB + i holds pair (key kk XOR lane/RB, row i XOR lane%RB)
    float dots[32];
#pragma unroll
    for (int kk = 0; kk < KG; ++kk) {
      float kf[EPL];
      smem_cols<EPL>(st + (kk ^ my_k) * D, lane, kf);
#pragma unroll
      for (int i = 0; i < RB; i += 2) {
        float2 sacc = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < EPL; ++e)
          sacc = ffma2(make_float2(qv[i][e], qv[i + 1][e]), make_float2(kf[e], kf[e]), sacc);
        dots[kk * RB + i] = sacc.x;
        dots[kk * RB + i + 1] = sacc.y;
      }
    }
    reduce_scatter32(dots);
    // lane owns pair (my_k, my_r): its score, masked when invisible
    const int jj = j0 + my_k;
    const bool vis = jj < j_stop && my_r < n_rows &&
                     key_visible(p.layout, p.S, p.P, p.causal, u, jj, my_qpos);
    const float s_own = vis ? dots[0] : -INFINITY;
    // online softmax of each row over the group's keys (lanes of one row differ by RB)
    float mx = s_own;
#pragma unroll
    for (int o = RB; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    const float m_new = fmaxf(m_run, mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    // exact rescale exp(m_old - m_new); a row that saw nothing yet has a zero state
    const float alpha = (m_run == -INFINITY) ? 0.f : exp2f(m_run - m_use);
    const float pr = exp2f(s_own - m_use);   // 0 when masked
    float ps = pr;
#pragma unroll
    for (int o = RB; o < 32; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    if (m_new != -INFINITY) {
      z_run = z_run * alpha + ps;
      m_run = m_new;
    }
    // y_r = alpha_r y_r + sum_k p(k, r) V_k on this lane's columns; the 32
    // probabilities and the RB rescale factors go through the warp's smem slot
    sm_p[lane] = pr;
    if (lane < RB) sm_p[32 + lane] = (m_new == -INFINITY) ? 1.f : alpha;
    __syncwarp();
    float pk[32];
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      const float4 t4 = *reinterpret_cast<const float4*>(sm_p + i);
      pk[i] = t4.x; pk[i + 1] = t4.y; pk[i + 2] = t4.z; pk[i + 3] = t4.w;
    }
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const float a_r = sm_p[32 + r];
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 t2 = fmul2(make_float2(acc[r][e], acc[r][e + 1]), make_float2(a_r, a_r));
        acc[r][e] = t2.x;
        acc[r][e + 1] = t2.y;
      }
    }
#pragma unroll
    for (int kk = 0; kk < KG; ++kk) {
      float vf[EPL];
      smem_cols<EPL>(st + (KG + kk) * D, lane, vf);
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const float pv = pk[kk * RB + r];
#pragma unroll
        for (int e = 0; e < EPL; e += 2) {
          const float2 t2 = ffma2(make_float2(pv, pv), make_float2(vf[e], vf[e + 1]),
                                  make_float2(acc[r][e], acc[r][e + 1]));
          acc[r][e] = t2.x;
          acc[r][e + 1] = t2.y;
        }
      }
    }
    __syncwarp();   // every lane is done with stage n before it is refilled
  }
  cp_async_wait<0>();

  // Merge the warps' states: rescale each to the CTA-wide max and add.
  if (lane < RB) {
    sm_m[warp * RB + lane] = m_run;
    sm_z[warp * RB + lane] = z_run;
  }
  __syncthreads();
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * RB + r]);
    const float mw = sm_m[warp * RB + r];
    const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
#pragma unroll
    for (int e = 0; e < EPL; ++e) sm_y[(warp * RB + r) * D + lane * EPL + e] = acc[r][e] * f;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < RB * D; idx += kThreads) {
    const int r = idx / D, col = idx % D;
    if (r >= n_rows) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * RB + r]);
    float Z = 0.f, Y = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = sm_m[w * RB + r];
      Z += (mw == -INFINITY) ? 0.f : sm_z[w * RB + r] * exp2f(mw - M);
      Y += sm_y[(w * RB + r) * D + col];
    }
    const int rr = row0 + r, h = g * hpg + rr / n_q, t = rr % n_q;
    const size_t oo = (((static_cast<size_t>(part) * p.B + bat) * n_q + t) * p.H + h) * D + col;
    o_parts[oo] = Z > 0.f ? Y / Z : 0.f;
    if (col == 0) {
      const size_t lo = ((static_cast<size_t>(part) * p.B + bat) * p.H + h) * n_q + t;
      lse_parts[lo] = Z > 0.f ? (M + log2f(Z)) * kLn2 : -INFINITY;
    }
  }
}

template <int D, int RB>
cudaError_t launch_rb(const RingParams& p, int n_q, int q_pos0, int chunk, float* o_parts,
                      float* lse_parts, cudaStream_t st) {
  const int rows_total = (p.H / p.G) * n_q;
  const int n_rowgroups = (rows_total + RB - 1) / RB;
  const int n_chunks = (p.S + chunk - 1) / chunk;
  const int smem = DecCfg<D, RB>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(decode_partial_kernel<D, RB>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const dim3 grid(p.G * n_rowgroups, n_chunks, p.B * p.P);
  decode_partial_kernel<D, RB><<<grid, kThreads, smem, st>>>(p, n_q, q_pos0, chunk, n_rowgroups,
                                                             o_parts, lse_parts);
  return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(const RingParams& p, int n_q, int q_pos0, int chunk, float* o_parts,
                     float* lse_parts, cudaStream_t st) {
  const int rows_total = (p.H / p.G) * n_q;
  if (rows_total <= 4) return launch_rb<D, 4>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
  return launch_rb<D, 8>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
}

}  // namespace

int decode_chunk_keys(int S) { return S <= 4096 ? S : 4096; }

cudaError_t launch_decode_partials(const RingParams& p, int n_q, int q_pos0, float* o_parts,
                                   float* lse_parts, cudaStream_t st) {
  const int chunk = decode_chunk_keys(p.S);
  return p.D == 64 ? launch_d<64>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st)
                   : launch_d<128>(p, n_q, q_pos0, chunk, o_parts, lse_parts, st);
}

}  // namespace ra
