// Pass-Q decode over the virtual ring: a few query rows attend to a KV cache that
// stays sharded and stationary. Every virtual device u scores the queries against
// its own shard only and leaves partials (O, LSE); the partials are combined by
// the merge kernel (merge.cu).
//  * Transformer Math "Ring Attention" (aicassindra), "The ring is a prefill
//    algorithm": broadcast the single query to all P devices, each computes a
//    partial (m, l, o) against its shard, one small reduction combines them.
//  * "Part 4: Ring Attention" (Fofadiya) §4.9.4.4: pass-Q decode.
//
// The partial phase is HBM-bound: each (batch, kv head) reads its K/V rows once,
// and all query rows of the GQA group (heads of the group x decode tokens, up to
// 16 per CTA) share them. A CTA owns those rows and a chunk of keys of one
// segment of one shard (long shards are cut into chunks of up to 8192 keys;
// every chunk is one more partial for the merge).
//
// The two products are tensor-core MMAs of 16 rows (mma.m16n8k16, bf16 in, fp32
// accumulate): with at most 16 query rows per kv head, a 16-row MMA fits the
// problem, and the kernel issues a few instructions per 16 bytes of K/V instead
// of one FMA per element. Each of the 4 warps owns every 4th 32-key tile of the
// chunk and streams it through its own 3-stage ring of shared memory with TMA
// (128-byte swizzle; ldmatrix reads the swizzled rows, K as it is for S = Q K^T
// and V transposed for O += P V). The S accumulators become the A operand of the
// P V product without leaving registers. Each warp keeps its own online-softmax
// state (running max m, denominator l, output O) in fp32; the warps merge theirs
// once at the end and write the chunk's normalised partial.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "internal.cuh"
#include "ptx.cuh"
#include "shardmap.cuh"
#include "views.cuh"

namespace ra {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 3;                    // per-warp TMA ring
constexpr int kTileKeys = 32;
constexpr int kRows = 16;                     // query rows per CTA: the M of one MMA
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s to let in-flight copies land on abort

template <int D>
struct DecSmem {
  static constexpr int kHalf = kTileKeys * 128;          // 32 rows x 64 bf16 (128 B, swizzled)
  static constexpr int kTile = (D / 64) * kHalf;         // one [32 x D] bf16 tile
  static constexpr int kStage = 2 * kTile;               // K, then V
  static constexpr int kRing = kWarps * kStages * kStage;
  static constexpr int kBar = kRing;                     // mbarriers [warp][stage], abort flag
  static constexpr int kBytes = kBar + 8 * kWarps * kStages + 16;
  static constexpr int kAlloc = kBytes + 1024;
  // after the loop the ring holds the warps' states: O [warp][row][D], m, l [warp][row]
  static constexpr int kMergeO = 0;
  static constexpr int kMergeM = kWarps * kRows * D * 4;
  static constexpr int kMergeL = kMergeM + kWarps * kRows * 4;
  // in a cluster, the CTA's own partial for the peers to read: O [row][D], LSE [row]
  static constexpr int kPartO = kMergeL + kWarps * kRows * 4;
  static constexpr int kPartL = kPartO + kRows * D * 4;
  static_assert(kPartL + kRows * 4 <= kRing, "merge area inside the ring");
};

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Four 8x8 bf16 matrices; lanes 8m .. 8m+7 give the row addresses of matrix m.
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Shared address of the 16-byte unit holding columns [col, col + 8) of row `row`
// in a [32 x D] tile stored as 64-column chunks with the 128-byte swizzle (the
// unit index inside a 128-byte row is XORed with row mod 8).
template <int D>
__device__ __forceinline__ uint32_t swz(uint32_t tile, int row, int col) {
  return tile + (col >> 6) * DecSmem<D>::kHalf + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4);
}


// grid: x = g * n_rowgroups + rowgroup, y = segment * n_chunks + chunk, z = batch * P + u.
// CL: the partials of one (sequence, kv head, row group) are the CTAs of one cluster
// (cluster dims 1 x segments*chunks x P), which merge them through distributed shared
// memory and write O and LSE themselves; otherwise each CTA writes its partial to
// o_parts / lse_parts for the merge kernel.
template <int D, bool CL>
__global__ void __launch_bounds__(kThreads, 1)
decode_mma_kernel(const __grid_constant__ RingParams p, const __grid_constant__ CUtensorMap tk,
                  const __grid_constant__ CUtensorMap tv, int n_q, int q_pos0, int chunk,
                  int n_rowgroups, int n_chunks, float* __restrict__ o_parts,
                  float* __restrict__ lse_parts) {
  using L = DecSmem<D>;
  constexpr int KS = D / 16;   // k-steps of S = Q K^T
  constexpr int NT = D / 8;    // 8-column tiles of O
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * kWarps * kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;   // MMA fragment coordinates

  const int g = blockIdx.x / n_rowgroups, rg = blockIdx.x % n_rowgroups;
  const int sidx = blockIdx.y / n_chunks, c = blockIdx.y % n_chunks;
  const int bat = blockIdx.z / p.P, u = blockIdx.z % p.P;
  const int nseg = num_segs(p.layout);
  const int hpg = p.H / p.G;
  const int rows_total = hpg * n_q;
  const int row0 = rg * kRows;
  const int n_rows = min(kRows, rows_total - row0);
  const Seg sg = seg_of(p.layout, p.S, p.P, u, sidx);
  const int j_begin = c * chunk;                     // segment-local key range of the chunk
  const int j_end = min(sg.len, j_begin + chunk);
  const int part = (u * nseg + sidx) * n_chunks + c;

  // Rows: row r of the CTA is query row rr = row0 + r of kv head g, i.e. head
  // g * hpg + rr / n_q, decode token rr % n_q at global position q_pos0 + rr % n_q.
  // This thread's accumulator rows are gid and gid + 8.
  const bool v_lo = gid < n_rows, v_hi = gid + 8 < n_rows;
  const int qpos_lo = v_lo ? q_pos0 + (row0 + gid) % n_q : -1;
  const int qpos_hi = v_hi ? q_pos0 + (row0 + gid + 8) % n_q : -1;
  int qpos_max = -1;
  for (int r = 0; r < n_rows; ++r) qpos_max = max(qpos_max, q_pos0 + (row0 + r) % n_q);
  // keys of the chunk some row may see: a prefix of it
  const int n_vis = j_end > j_begin ? seg_visible(sg, p.causal, j_begin, j_end - j_begin, qpos_max) : 0;
  const int j_stop = j_begin + n_vis;
  const int n_tiles = (n_vis + kTileKeys - 1) / kTileKeys;
  const int mine = n_tiles > warp ? (n_tiles - warp + kWarps - 1) / kWarps : 0;

  // Q rows as A fragments of the k-steps (rows past the CTA's rows are zero)
  uint32_t qa[KS][4];
  {
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    auto qoff = [&](int r) -> size_t {
      const int rr = row0 + r, h = g * hpg + rr / n_q, t = rr % n_q;
      return ((static_cast<size_t>(bat) * n_q + t) * p.H + h) * D;
    };
    const size_t q_n = static_cast<size_t>(p.B) * n_q * p.H * D;   // q is [B, n_q, H, d]
    const bool q_lo = v_lo && in_bounds(qoff(gid), D, q_n, p.status);
    const bool q_hi = v_hi && in_bounds(qoff(gid + 8), D, q_n, p.status);
    const uint32_t* ql = q_lo ? reinterpret_cast<const uint32_t*>(q + qoff(gid)) : nullptr;
    const uint32_t* qh = q_hi ? reinterpret_cast<const uint32_t*>(q + qoff(gid + 8)) : nullptr;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qa[kk][0] = q_lo ? ql[8 * kk + tig] : 0u;
      qa[kk][1] = q_hi ? qh[8 * kk + tig] : 0u;
      qa[kk][2] = q_lo ? ql[8 * kk + 4 + tig] : 0u;
      qa[kk][3] = q_hi ? qh[8 * kk + 4 + tig] : 0u;
    }
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kWarps * kStages; ++i) mbar_init(sbase + L::kBar + 8 * i, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (threadIdx.x == 32) {
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  __syncthreads();

  auto bar = [&](int st) -> uint32_t { return sbase + L::kBar + 8 * (warp * kStages + st); };
  auto ring = [&](int st) -> uint32_t { return sbase + (warp * kStages + st) * L::kStage; };
  auto issue = [&](int n) {   // lane 0: this warp's n-th tile into stage n % kStages
    const int st = n % kStages;
    const int j0 = j_begin + (warp + kWarps * n) * kTileKeys;
    mbar_arrive_expect_tx(bar(st), L::kStage);
#pragma unroll
    for (int dc = 0; dc < D / 64; ++dc) {
      tma_rows(&tk, ring(st) + dc * L::kHalf, bar(st), p.layout, dc, g, sg.chunk, j0, bat);
      tma_rows(&tv, ring(st) + L::kTile + dc * L::kHalf, bar(st), p.layout, dc, g, sg.chunk, j0, bat);
    }
  };
  if (lane == 0)
    for (int n = 0; n < min(kStages, mine); ++n) issue(n);
  __syncwarp();

  const float c2 = p.scale_log2;
  float m_lo = -INFINITY, m_hi = -INFINITY;   // running max of the scaled scores (log2 units)
  float l_lo = 0.f, l_hi = 0.f;               // this thread's share of the denominators
  float o[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
  const int lm = lane >> 3, li = lane & 7;    // ldmatrix: matrix and row of this lane's address
  bool ok = true;
  int consumed = 0;
  for (int n = 0; n < mine; ++n) {
    const int st = n % kStages;
    if (!__all_sync(0xffffffffu, bounded_wait(bar(st), static_cast<uint32_t>(n / kStages) & 1,
                                              p.timeout_ns, abort_flag))) {
      ok = false;
      break;
    }
    const uint32_t sK = ring(st), sV = sK + L::kTile;
    const int j0 = j_begin + (warp + kWarps * n) * kTileKeys;

    // S = Q K^T over the tile's 32 keys: four 8-key tiles
    float s[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
      for (int np = 0; np < 2; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(swz<D>(sK, 8 * (2 * np + (lm >> 1)) + li, 16 * kk + 8 * (lm & 1)), b0, b1, b2, b3);
        mma_16816(s[2 * np], qa[kk], b0, b1);
        mma_16816(s[2 * np + 1], qa[kk], b2, b3);
      }
    }
    // scale to log2 units and mask: keys past the visible prefix, or after the row
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = j0 + 8 * nt + 2 * tig + e;
        const int kp = sg.base + j * sg.stride;
        const bool in = j < j_stop;
        s[nt][e] = (in && v_lo && (!p.causal || kp <= qpos_lo)) ? s[nt][e] * c2 : -INFINITY;
        s[nt][2 + e] = (in && v_hi && (!p.causal || kp <= qpos_hi)) ? s[nt][2 + e] * c2 : -INFINITY;
        mx_lo = fmaxf(mx_lo, s[nt][e]);
        mx_hi = fmaxf(mx_hi, s[nt][2 + e]);
      }
    }
    // the four lanes of a row hold its 32 scores
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    const float mu_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
    const float mu_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    // exact rescale exp(m_old - m_new); a row that saw nothing yet has a zero state
    const float a_lo = ex2(m_lo - mu_lo), a_hi = ex2(m_hi - mu_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    // probabilities, as the A fragments of the two 16-key steps of O += P V
    uint32_t pa[2][4];
    float pl = 0.f, ph = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = ex2(s[nt][0] - mu_lo), p1 = ex2(s[nt][1] - mu_lo);
      const float p2 = ex2(s[nt][2] - mu_hi), p3 = ex2(s[nt][3] - mu_hi);
      pl += p0 + p1;
      ph += p2 + p3;
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(p0, p1);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(p2, p3);
    }
    l_lo = l_lo * a_lo + pl;
    l_hi = l_hi * a_hi + ph;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      o[nt][0] *= a_lo;
      o[nt][1] *= a_lo;
      o[nt][2] *= a_hi;
      o[nt][3] *= a_hi;
    }
#pragma unroll
    for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(swz<D>(sV, 16 * ks + 8 * (lm & 1) + li, 8 * (2 * np + (lm >> 1))), b0, b1, b2,
                      b3);
        mma_16816(o[2 * np], pa[ks], b0, b1);
        mma_16816(o[2 * np + 1], pa[ks], b2, b3);
      }
    }
    consumed = n + 1;
    __syncwarp();   // every lane has read the stage before it is refilled
    if (lane == 0 && n + kStages < mine) issue(n + kStages);
    __syncwarp();
  }
  if (!ok) {
    if (lane == 0) {
      atomicCAS(p.status, 0, static_cast<int>(RA_ERR_TIMEOUT));
      *abort_flag = 1;
      // let this warp's copies in flight land before the CTA exits
      for (int n = consumed; n < min(mine, consumed + kStages); ++n)
        bounded_wait(bar(n % kStages), static_cast<uint32_t>(n / kStages) & 1, kDrainNs, nullptr);
    }
    __syncwarp();
  }
  // full denominators of the thread's rows (the four lanes of a row)
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);

  // Merge the warps' states through the ring memory: rescale each to the
  // CTA-wide max and add.
  __syncthreads();
  float* sm_o = reinterpret_cast<float*>(smem + L::kMergeO);   // [warp][row][D]
  float* sm_m = reinterpret_cast<float*>(smem + L::kMergeM);   // [warp][row]
  float* sm_l = reinterpret_cast<float*>(smem + L::kMergeL);
  if (tig == 0) {
    sm_m[warp * kRows + gid] = m_lo;
    sm_m[warp * kRows + gid + 8] = m_hi;
    sm_l[warp * kRows + gid] = l_lo;
    sm_l[warp * kRows + gid + 8] = l_hi;
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int col = 8 * nt + 2 * tig;
    *reinterpret_cast<float2*>(sm_o + (warp * kRows + gid) * D + col) = make_float2(o[nt][0], o[nt][1]);
    *reinterpret_cast<float2*>(sm_o + (warp * kRows + gid + 8) * D + col) =
        make_float2(o[nt][2], o[nt][3]);
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < kRows * D; idx += kThreads) {
    const int r = idx / D, col = idx % D;
    if (r >= n_rows) continue;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w * kRows + r]);
    float Z = 0.f, Y = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float mw = sm_m[w * kRows + r];
      const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      Z += f * sm_l[w * kRows + r];
      Y += f * sm_o[(w * kRows + r) * D + col];
    }
    if constexpr (CL) {
      // this CTA's normalised partial, in its own shared memory (LSE in log2 units)
      reinterpret_cast<float*>(smem + L::kPartO)[r * D + col] = Z > 0.f ? Y / Z : 0.f;
      if (col == 0)
        reinterpret_cast<float*>(smem + L::kPartL)[r] = Z > 0.f ? M + log2f(Z) : -INFINITY;
      continue;
    }
    const int rr = row0 + r, h = g * hpg + rr / n_q, t = rr % n_q;
    // partials [parts, B, n_q, H, d] and [parts, B, H, n_q], parts = P * nseg * n_chunks
    const size_t rows_n = static_cast<size_t>(p.P) * nseg * n_chunks * p.B * n_q * p.H;
    const size_t oo = (((static_cast<size_t>(part) * p.B + bat) * n_q + t) * p.H + h) * D + col;
    if (in_bounds(oo, 1, rows_n * D, p.status)) o_parts[oo] = Z > 0.f ? Y / Z : 0.f;
    if (col == 0) {
      const size_t lo = ((static_cast<size_t>(part) * p.B + bat) * p.H + h) * n_q + t;
      if (in_bounds(lo, 1, rows_n, p.status))
        lse_parts[lo] = Z > 0.f ? (M + log2f(Z)) * kLn2 : -INFINITY;
    }
  }
  if constexpr (CL) {
    // Merge of the cluster's partials, the element (row, col) by one thread of the
    // cluster: LSE = M + log2 sum_c 2^(LSE_c - M), O = sum_c 2^(LSE_c - LSE) O_c,
    // over the CTAs in rank order (Transformer Math "Ring Attention", "The ring is a
    // prefill algorithm": one small reduction combines the per-shard partials).
    cluster_sync();
    const uint32_t n_cta = cluster_ctas(), rank = cluster_rank();
    const uint32_t part_o = sbase + L::kPartO, part_l = sbase + L::kPartL;
    for (int e = static_cast<int>(rank) * kThreads + threadIdx.x; e < n_rows * D;
         e += static_cast<int>(n_cta) * kThreads) {
      const int r = e / D, col = e % D;
      float M = -INFINITY;
      for (uint32_t c = 0; c < n_cta; ++c)
        M = fmaxf(M, ld_cluster_f32(map_to_rank(part_l + 4 * r, c)));
      float Z = 0.f, Y = 0.f;
      if (M != -INFINITY) {
        for (uint32_t c = 0; c < n_cta; ++c) {
          const float lc = ld_cluster_f32(map_to_rank(part_l + 4 * r, c));
          const float f = (lc == -INFINITY) ? 0.f : ex2(lc - M);
          Z += f;
          Y += f * ld_cluster_f32(map_to_rank(part_o + 4 * (r * D + col), c));
        }
      }
      const int rr = row0 + r, h = g * hpg + rr / n_q, t = rr % n_q;
      const size_t oo = ((static_cast<size_t>(bat) * n_q + t) * p.H + h) * D + col;
      const size_t q_n = static_cast<size_t>(p.B) * n_q * p.H * D;   // o is [B, n_q, H, d]
      const float ov = Z > 0.f ? Y / Z : 0.f;
      if (in_bounds(oo, 1, q_n, p.status)) {
        if (p.o_f32)
          static_cast<float*>(p.o)[oo] = ov;
        else
          static_cast<__nv_bfloat16*>(p.o)[oo] = __float2bfloat16_rn(ov);
      }
      if (col == 0) {
        const size_t lo = (static_cast<size_t>(bat) * p.H + h) * n_q + t;   // lse [B, H, n_q]
        if (in_bounds(lo, 1, static_cast<size_t>(p.B) * p.H * n_q, p.status))
          p.lse[lo] = Z > 0.f ? (M + log2f(Z)) * kLn2 : -INFINITY;
      }
    }
    cluster_sync();   // the peers' partials stay in place until every CTA has read them
  }
}

// The cluster merge applies when a row group's partials are at most 8 CTAs (the
// portable cluster size) and the grid is one wave or less, where the second launch
// and the partials' round trip through HBM are a visible part of a call's time.
// (Clusters of 16 CTAs measured slower than the two launches.)
constexpr int kMaxClusterParts = 8;

template <int D, bool CL>
cudaError_t set_attrs() {
  static OncePerContext attr;
  return attr.run([] {
    cudaError_t r = cudaFuncSetAttribute(decode_mma_kernel<D, CL>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DecSmem<D>::kAlloc);
    return r;
  });
}

struct DecGrid {
  dim3 grid;
  int n_rowgroups, n_chunks, chunk, parts;
};

DecGrid decode_grid(const RingParams& p, int n_q, int chunk) {
  DecGrid d;
  const int rows_total = (p.H / p.G) * n_q;
  d.n_rowgroups = (rows_total + kRows - 1) / kRows;
  const int nseg = num_segs(p.layout);
  const int seg_len = p.S / nseg;
  d.chunk = chunk;
  d.n_chunks = (seg_len + d.chunk - 1) / d.chunk;
  d.parts = p.P * nseg * d.n_chunks;
  d.grid = dim3(p.G * d.n_rowgroups, nseg * d.n_chunks, p.B * p.P);
  return d;
}

long long ctas_of(const DecGrid& d) {
  return static_cast<long long>(d.grid.x) * d.grid.y * d.grid.z;
}

// Keys per chunk of the one-launch form: the chunking of the two-launch form (which
// sizes the workspace), halved while the row group's partials stay within one
// cluster, the grid within one wave and the chunks at 256 keys or more. The
// one-launch form never touches the workspace, so its chunks may be finer; a
// small-P decode then runs on more CTAs, each streaming fewer keys.
int cluster_chunk(const RingParams& p, int n_q, int sms) {
  int chunk = decode_chunk_keys(p.S, p.P, p.layout);
  for (;;) {
    const int half = ((chunk / 2) + kTileKeys - 1) / kTileKeys * kTileKeys;
    if (half < 256 || half >= chunk) break;
    const DecGrid d = decode_grid(p, n_q, half);
    if (d.parts > kMaxClusterParts || ctas_of(d) > sms) break;
    chunk = half;
  }
  return chunk;
}

int device_sms() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return sms;
}

template <int D>
bool clustered_d(const RingParams& p, int n_q) {
  const int sms = device_sms();
  if (sms <= 0) return false;
  const DecGrid d = decode_grid(p, n_q, cluster_chunk(p, n_q, sms));
  if (d.parts < 2 || d.parts > kMaxClusterParts) return false;
  if (ctas_of(d) > sms) return false;
  if (set_attrs<D, true>() != cudaSuccess) {
    (void)cudaGetLastError();
    return false;
  }
  // whether clusters of this size fit on the device at all (kept per context and size)
  static std::atomic<unsigned long long> fits_ctx[kMaxClusterParts + 1] = {};
  static std::atomic<int> fits[kMaxClusterParts + 1] = {};
  const unsigned long long id = current_context_id();
  if (id == 0 || fits_ctx[d.parts].load() != id) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = d.grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = DecSmem<D>::kAlloc;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = d.grid.y;
    at[0].val.clusterDim.z = p.P;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_mma_kernel<D, true>, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      n = 0;
    }
    fits[d.parts].store(n > 0 ? 1 : 0);
    fits_ctx[d.parts].store(id);
  }
  return fits[d.parts].load() != 0;
}

template <int D>
cudaError_t launch_d(const RingParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int n_q,
                     int q_pos0, float* o_parts, float* lse_parts, bool clustered,
                     cudaStream_t st) {
  const DecGrid d = decode_grid(
      p, n_q,
      clustered ? cluster_chunk(p, n_q, device_sms()) : decode_chunk_keys(p.S, p.P, p.layout));
  const int smem = DecSmem<D>::kAlloc;
  // the attributes are set once per device context (a decode loop calls this per token,
  // possibly inside a CUDA graph capture)
  if (!clustered) {
    const cudaError_t e = set_attrs<D, false>();
    if (e != cudaSuccess) return e;
    decode_mma_kernel<D, false><<<d.grid, kThreads, smem, st>>>(
        p, tk, tv, n_q, q_pos0, d.chunk, d.n_rowgroups, d.n_chunks, o_parts, lse_parts);
    return cudaGetLastError();
  }
  const cudaError_t e = set_attrs<D, true>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = d.grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 1;
  at[0].val.clusterDim.y = d.grid.y;
  at[0].val.clusterDim.z = p.P;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_mma_kernel<D, true>, p, tk, tv, n_q, q_pos0, d.chunk,
                            d.n_rowgroups, d.n_chunks, o_parts, lse_parts);
}

}  // namespace

// Keys per chunk of a shard segment: up to 8192 (a CTA's start-up — barriers, Q
// rows, filling the TMA rings — is a few microseconds, so long chunks pay even
// when the last wave of CTAs is partly empty), or more when that would give more
// than 1024 partials (the merge kernel's limit), rounded up to whole 32-key tiles.
int decode_chunk_keys(int S, int P, int layout) {
  const int nseg = num_segs(layout);
  const int seg_len = S / nseg;
  long long chunk = seg_len < 8192 ? seg_len : 8192;
  const long long min_chunk = (static_cast<long long>(seg_len) * nseg * P + 1023) / 1024;
  if (chunk < min_chunk) chunk = (min_chunk + kTileKeys - 1) / kTileKeys * kTileKeys;
  if (chunk > seg_len) chunk = seg_len;
  return static_cast<int>(chunk < 1 ? 1 : chunk);
}

int decode_parts(int S, int P, int layout) {
  const int nseg = num_segs(layout);
  const int seg_len = S / nseg;
  const int chunk = decode_chunk_keys(S, P, layout);
  return P * nseg * ((seg_len + chunk - 1) / chunk);
}

bool decode_clustered(const RingParams& p, int n_q) {
  return p.D == 64 ? clustered_d<64>(p, n_q) : clustered_d<128>(p, n_q);
}

cudaError_t launch_decode_partials(const RingParams& p, const CUtensorMap& tk,
                                   const CUtensorMap& tv, int n_q, int q_pos0, float* o_parts,
                                   float* lse_parts, bool clustered, cudaStream_t st) {
  return p.D == 64 ? launch_d<64>(p, tk, tv, n_q, q_pos0, o_parts, lse_parts, clustered, st)
                   : launch_d<128>(p, tk, tv, n_q, q_pos0, o_parts, lse_parts, clustered, st);
}

}  // namespace ra
