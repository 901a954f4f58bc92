// Bandwidth-bound kernels over per-row results: the merge of n normalised
// partials (O_p, LSE_p) and the finalize of a running state (m, z, y).
//
// Merge — Transformer Math "Ring Attention" (aicassindra), "The ring is a prefill
// algorithm": P partial (m, l, o) triples of the same rows are combined by one
// rescale-and-add reduction. With normalised partials O_p = y_p / z_p and
// LSE_p = m_p + ln z_p:  LSE = M + ln sum_p e^{LSE_p - M} (M = max_p LSE_p) and
// O = sum_p e^{LSE_p - LSE} O_p. Finalize — "Ring Attention" (aarnphm.xyz):
// O = y / z; LSE = m + ln z.
//
// Layout: a block owns 32 consecutive tokens of one (batch, head); warp w takes
// tokens w, w + 8, w + 16, w + 24. A warp first reduces the log-sum-exps of its own
// four tokens (eight lanes per token, each over every eighth part, combined by
// shuffles; no block barrier), then streams whole rows: a row of d fp32 is one
// coalesced 16-byte-per-lane (d = 128) or 8-byte-per-lane (d = 64) load per part,
// four parts in flight per lane.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.cuh"

namespace ra {
namespace {

constexpr int kTok = 32;      // tokens per block
constexpr int kWarps = 8;     // 4 tokens per warp (kTok = 4 * kWarps)

template <int D>
struct Vec;
template <>
struct Vec<128> {
  using T = float4;
  static constexpr int kN = 4;
};
template <>
struct Vec<64> {
  using T = float2;
  static constexpr int kN = 2;
};

__device__ __forceinline__ void load_vec(const float4* p, float (&r)[4]) {
  const float4 v = __ldcs(p);
  r[0] = v.x; r[1] = v.y; r[2] = v.z; r[3] = v.w;
}
__device__ __forceinline__ void load_vec(const float2* p, float (&r)[2]) {
  const float2 v = __ldcs(p);
  r[0] = v.x; r[1] = v.y;
}

// One lane's kN consecutive output values: rounded to bf16 (round to nearest
// even), or kept as fp32.
__device__ __forceinline__ void store_out(__nv_bfloat16* dst, const float (&a)[4]) {
  __nv_bfloat162 x = __floats2bfloat162_rn(a[0], a[1]);
  __nv_bfloat162 y = __floats2bfloat162_rn(a[2], a[3]);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&x);
  pk.y = *reinterpret_cast<uint32_t*>(&y);
  *reinterpret_cast<uint2*>(dst) = pk;
}
__device__ __forceinline__ void store_out(__nv_bfloat16* dst, const float (&a)[2]) {
  *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(a[0], a[1]);
}
__device__ __forceinline__ void store_out(float* dst, const float (&a)[4]) {
  *reinterpret_cast<float4*>(dst) = make_float4(a[0], a[1], a[2], a[3]);
}
__device__ __forceinline__ void store_out(float* dst, const float (&a)[2]) {
  *reinterpret_cast<float2*>(dst) = make_float2(a[0], a[1]);
}

template <int D, typename OutT>
__global__ void __launch_bounds__(kWarps * 32)
merge_kernel(int n, int B, int N, int H, const float* __restrict__ o_parts,
             const float* __restrict__ lse_parts, OutT* __restrict__ o,
             float* __restrict__ lse) {
  using V = Vec<D>;
  constexpr int kN = V::kN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTok;
  const int head = blockIdx.y;
  const int bat = blockIdx.z;
  const size_t part_lse = static_cast<size_t>(B) * H * N;           // stride between parts
  const size_t part_o = static_cast<size_t>(B) * N * H * D;
  const size_t lrow = (static_cast<size_t>(bat) * H + head) * N;    // [B,H,N] row base

  // Each warp reduces the log-sum-exps of its own four tokens (tt = warp + 8 j):
  // lanes 8j .. 8j+7 take parts pl, pl + 8, ... of token slot j and combine by shuffles.
  float Lw;
  {
    const int slot = lane >> 3, pl = lane & 7;
    const int t = t0 + warp + kWarps * slot;
    float M = -INFINITY, acc = 0.f;
    if (t < N) {
      for (int q0 = pl; q0 < n; q0 += 32) {
        float lv[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          lv[k] = (q0 + 8 * k < n) ? __ldg(lse_parts + (q0 + 8 * k) * part_lse + lrow + t)
                                   : -INFINITY;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float l = lv[k];
          if (l == -INFINITY) continue;
          if (l > M) {
            acc = acc * expf(M - l) + 1.f;
            M = l;
          } else {
            acc += expf(l - M);
          }
        }
      }
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
      const float Mo = __shfl_xor_sync(0xffffffffu, M, off);
      const float ao = __shfl_xor_sync(0xffffffffu, acc, off);
      const float Mn = fmaxf(M, Mo);
      float s = 0.f;
      if (M != -INFINITY) s += acc * expf(M - Mn);
      if (Mo != -INFINITY) s += ao * expf(Mo - Mn);
      M = Mn;
      acc = s;
    }
    Lw = (M == -INFINITY) ? -INFINITY : M + logf(acc);
    if (pl == 0 && t < N) lse[lrow + t] = Lw;
  }
#pragma unroll 1
  for (int j = 0; j < 4; ++j) {
    const float L = __shfl_sync(0xffffffffu, Lw, 8 * j);   // all lanes: t is warp-uniform
    const int t = t0 + warp + kWarps * j;
    if (t >= N) break;
    const size_t orow = ((static_cast<size_t>(bat) * N + t) * H + head) * D;
    float acc[kN];
#pragma unroll
    for (int e = 0; e < kN; ++e) acc[e] = 0.f;
    if (L != -INFINITY) {
      const typename V::T* src =
          reinterpret_cast<const typename V::T*>(o_parts + orow) + lane;
      int q = 0;
      for (; q + 4 <= n; q += 4) {
        float r[4][kN];
        float wgt[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          load_vec(src + (q + k) * (part_o / kN), r[k]);
          wgt[k] = expf(__ldg(lse_parts + (q + k) * part_lse + lrow + t) - L);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int e = 0; e < kN; ++e) acc[e] = fmaf(wgt[k], r[k][e], acc[e]);
      }
      for (; q < n; ++q) {
        float r[kN];
        load_vec(src + q * (part_o / kN), r);
        const float wgt = expf(__ldg(lse_parts + q * part_lse + lrow + t) - L);
#pragma unroll
        for (int e = 0; e < kN; ++e) acc[e] = fmaf(wgt, r[e], acc[e]);
      }
    }
    store_out(o + orow + lane * kN, acc);
  }
}

// (m, z, y) -> O = y / z (bf16 or fp32), LSE = m + ln z; z = 0 gives O = 0,
// LSE = -inf.
template <int D, typename OutT>
__global__ void __launch_bounds__(kWarps * 32)
finalize_kernel(int N, int H, const float* __restrict__ m, const float* __restrict__ z,
                const float* __restrict__ y, OutT* __restrict__ o, float* __restrict__ lse) {
  using V = Vec<D>;
  constexpr int kN = V::kN;
  __shared__ float s_inv[kTok];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kTok;
  const int head = blockIdx.y;
  const int bat = blockIdx.z;
  const size_t lrow = (static_cast<size_t>(bat) * H + head) * N;
  if (warp == 0) {
    const int t = t0 + lane;
    float inv = 0.f;
    if (t < N) {
      const float zz = z[lrow + t];
      const float mm = m[lrow + t];
      inv = zz > 0.f ? 1.f / zz : 0.f;
      lse[lrow + t] = zz > 0.f ? mm + logf(zz) : -INFINITY;
    }
    s_inv[lane] = inv;
  }
  __syncthreads();
  for (int tt = warp; tt < kTok; tt += kWarps) {
    const int t = t0 + tt;
    if (t >= N) break;
    const float inv = s_inv[tt];
    const size_t orow = ((static_cast<size_t>(bat) * N + t) * H + head) * D;
    float r[kN];
    load_vec(reinterpret_cast<const typename V::T*>(y + orow) + lane, r);
#pragma unroll
    for (int e = 0; e < kN; ++e) r[e] *= inv;
    store_out(o + orow + lane * kN, r);
  }
}

template <int D, typename OutT>
void merge_d(int n, int B, int N, int H, const float* o_parts, const float* lse_parts, void* o,
             float* lse, cudaStream_t st) {
  const dim3 grid((N + kTok - 1) / kTok, H, B);
  merge_kernel<D, OutT><<<grid, kWarps * 32, 0, st>>>(n, B, N, H, o_parts, lse_parts,
                                                      static_cast<OutT*>(o), lse);
}

template <int D, typename OutT>
void finalize_d(const RingParams& p, cudaStream_t st) {
  const dim3 grid((p.N + kTok - 1) / kTok, p.H, p.B);
  finalize_kernel<D, OutT><<<grid, kWarps * 32, 0, st>>>(p.N, p.H, p.m, p.z, p.y,
                                                         static_cast<OutT*>(p.o), p.lse);
}

}  // namespace

cudaError_t launch_merge(int n, int B, int N, int H, int D, const float* o_parts,
                         const float* lse_parts, void* o, bool o_f32, float* lse,
                         cudaStream_t st) {
  if (D == 64)
    o_f32 ? merge_d<64, float>(n, B, N, H, o_parts, lse_parts, o, lse, st)
          : merge_d<64, __nv_bfloat16>(n, B, N, H, o_parts, lse_parts, o, lse, st);
  else
    o_f32 ? merge_d<128, float>(n, B, N, H, o_parts, lse_parts, o, lse, st)
          : merge_d<128, __nv_bfloat16>(n, B, N, H, o_parts, lse_parts, o, lse, st);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const RingParams& p, cudaStream_t st) {
  if (p.D == 64)
    p.o_f32 ? finalize_d<64, float>(p, st) : finalize_d<64, __nv_bfloat16>(p, st);
  else
    p.o_f32 ? finalize_d<128, float>(p, st) : finalize_d<128, __nv_bfloat16>(p, st);
  return cudaGetLastError();
}

}  // namespace ra
