// Tensor-core ring kernel for sm_103a: the fused forward (all P ring steps, then
// O = y / z and LSE) and the single ring step over an HBM-resident (m, z, y).
//
// What it computes — "Ring Attention" (aarnphm.xyz), the ring recurrence display:
// virtual device u keeps its query shard; at step s it scores the queries against
// shard b = (u - s) mod P, S = Q_u K_b^T / sqrt(d_h), and folds S into the running
// (m, z, y) with the rescale exp(m_old - m_new); O = y / z at the end. The same
// update is §4.4 of "Part 4: Ring Attention" (Fofadiya). Key/value tiles that the
// causal mask leaves empty are never loaded ("Part 4" §4.8.1).
//
// How, on one GB300 SM (one CTA per SM, 10 warps):
//  * a CTA owns two 128-row query sub-tiles that read the same K/V tiles: two
//    query heads of one GQA group at the same rows, or (when a group has an odd
//    number of heads) two consecutive row tiles of one head;
//  * warp 9 (TMA producer) loads both Q sub-tiles once, then streams 128-key K and
//    V tiles of the visited shards through two shared-memory stages each, in the
//    ring order, skipping key tiles that no query of the CTA may see;
//  * warp 8 issues the tcgen05 MMAs (one elected lane of a warp-uniform loop):
//    S_i = Q_i K^T into TMEM
//    (fp32, 128 columns per sub-tile) and O_i += P_i V with P_i read from TMEM;
//  * warps 0-3 / 4-7 are the softmax groups of sub-tile 0 / 1: one thread per
//    query row reads its S row from TMEM, applies the causal / tail mask, updates
//    the running max and denominator in fp32, rescales its O row in TMEM when the
//    max grows, and writes P = exp(S - m) as bf16 back over S for the P·V MMA;
//    P is published in two halves (keys 0-63, then 64-127), so the first four
//    P·V MMAs run while the softmax is still on the second half;
//  * the MMA order PV_0(t), S_0(t+1), PV_1(t), S_1(t+1) lets each softmax group
//    work while the tensor core serves the other group, and the commit that
//    signals S_i(t+1) also proves PV_i(t) finished, so O_i is stable when read.
// All arithmetic of the running state is fp32; exponentials use exp2 with
// log2(e) folded into the score scale; P is rounded to bf16 for the MMA.
#include <cuda_bf16.h>
#include <math.h>

#include <atomic>

#include "internal.cuh"
#include "ptx.cuh"
#include "shardmap.cuh"
#include "views.cuh"

namespace ra {
namespace {

constexpr int kThreads = 320;
constexpr int kMmaWarp = 8;
constexpr int kTmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s to let in-flight copies land on abort

template <int D>
struct Smem {
  static constexpr int kChunk = 128 * 128;          // 128 rows x 64 bf16 (128 B, swizzled)
  static constexpr int kTile = (D / 64) * kChunk;   // one [128 x D] bf16 tile
  static constexpr int kQ = 0;                      // query sub-tiles 0, 1
  static constexpr int kK = 2 * kTile;              // K stages 0, 1
  static constexpr int kV = 4 * kTile;              // V stages 0, 1
  static constexpr int kBar = 6 * kTile;            // mbarriers, TMEM base, abort flag
  static constexpr int kBytes = kBar + 256;
  // Keep one CTA per SM (it owns all 512 TMEM columns) and leave room to align.
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
  static constexpr uint32_t kOcol = 256;            // TMEM: S0 [0,128) S1 [128,256) O0 O1
};

enum : int {
  kBarQ = 0, kBarKF = 1, kBarKE = 3, kBarVF = 5, kBarVE = 7, kBarSF = 9, kBarOF = 11,
  kBarDrain = 13, kBarPF = 14,   // kBarPF + 2*i + h: half h of P_i
  kBarSB = 18,                   // d = 64: scores ready in score buffer b (3 buffers)
  kBarPD = 21,                   // d = 64: P V of sub-tile i done (2)
  kNumBars = 23
};

// d = 64 keeps three 128-column score buffers (TMEM columns [0,128), [128,256) and
// [384,512); O0 and O1 take [256,384)) rotating over the sequence k = 2 t + i of
// (tile t, sub-tile i): scores k go to buffer k mod 3 and are computed three ahead of
// their P V instead of two, so a sub-tile's next scores are ready when its softmax
// publishes P. At d = 128 the two O accumulators leave room for two buffers only.
__device__ __forceinline__ uint32_t score_col(int k) {
  const int b = k % 3;
  return b == 2 ? 384u : 128u * static_cast<uint32_t>(b);
}

struct Unit {
  int bat, g, u;
  int seg;        // segment of shard u the query rows lie in
  int head[2];
  int row0[2];    // first row of each sub-tile, relative to the segment
  int qpos_max;   // latest global query position held by the CTA, -1 if none
};

__device__ __forceinline__ Unit decode_unit(const RingParams& p, int idx) {
  Unit w;
  const int bg = idx / p.units_per_bg;
  int r = idx - bg * p.units_per_bg;
  w.bat = bg / p.G;
  w.g = bg - w.bat * p.G;
  const int hp = r % p.pairs_per_g;
  r /= p.pairs_per_g;
  // Within one (batch, kv head), launch the latest query positions first: under
  // a causal mask they carry the most key tiles. Query tiles are enumerated per
  // chunk of L rows (a shard, or a zigzag half-shard); positions grow with
  // (chunk, tile) for contiguous and zigzag, and with (tile, shard) for striped.
  // Striped tiles are taken in blocks of 4 tile indices per shard, so that the
  // CTAs resident at one time cover few shards: their rings then start at nearby
  // shards and reread the same K/V tiles from L2 (at 1M tokens a kv group's K
  // and V are four times the L2); blocks of 4 keep the order close to latest-first.
  const int key = p.X * p.nqq - 1 - r;
  int qq, c;
  if (p.layout == kStriped) {
    const int QB = (p.nqq % 4 == 0) ? 4 : 1;
    const int blk = key / (QB * p.P), rem = key - blk * QB * p.P;
    c = rem / QB;
    qq = blk * QB + (rem - c * QB);
  } else {
    c = key / p.nqq;
    qq = key - c * p.nqq;
  }
  if (p.layout == kZigzag) {
    w.u = c < p.P ? c : 2 * p.P - 1 - c;
    w.seg = c < p.P ? 0 : 1;
  } else {
    w.u = c;
    w.seg = 0;
  }
  const int hpg = p.H / p.G;
  if (p.pair_heads) {
    w.head[0] = w.g * hpg + 2 * hp;
    w.head[1] = w.head[0] + 1;
    w.row0[0] = w.row0[1] = qq * 128;
  } else {
    w.head[0] = w.head[1] = w.g * hpg + hp;
    w.row0[0] = 2 * qq * 128;
    w.row0[1] = w.row0[0] + 128;
  }
  const Seg sq = seg_of(p.layout, p.S, p.P, w.u, w.seg);
  w.qpos_max = -1;
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    if (w.row0[i] < sq.len) {
      const int last = min(w.row0[i] + 127, sq.len - 1);
      w.qpos_max = max(w.qpos_max, sq.base + last * sq.stride);
    }
  }
  return w;
}

__device__ __forceinline__ int shard_at(const RingParams& p, int u, int s) {
  int b = (u - s) % p.P;
  return b < 0 ? b + p.P : b;
}

// Key tiles of segment g that some query of the CTA may see (a prefix of it).
__device__ __forceinline__ int kv_tiles(const RingParams& p, const Seg& g, int qpos_max) {
  const int n = seg_visible(g, p.causal, 0, g.len, qpos_max);
  return (n + 127) >> 7;
}


__device__ __forceinline__ void record_failure(const RingParams& p, volatile int* abort_flag) {
  atomicCAS(p.status, 0, static_cast<int>(RA_ERR_TIMEOUT));
  *abort_flag = 1;
}

// S = Q K^T for one sub-tile: D/16 MMAs of 128 x 128 x 16, K-major operands in
// 128-byte-swizzled 64-column chunks. q_desc / k_desc describe the tile bases;
// the k-th MMA reads 16 columns further on (+32 B inside a 128-B row, a new
// 64-column chunk every four), i.e. a constant added to the address field.
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * Smem<D>::kChunk + (kk & 3) * 32) >> 4);
    mma_ss(d_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O += P V for one sub-tile: 8 MMAs of 128 x D x 16; P (bf16, two per TMEM
// column) from TMEM, V MN-major from shared memory (16 key rows = 2 KiB per MMA,
// 64-column chunks Smem::kChunk apart, which v_desc carries as its leading
// byte offset).
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                              int h, bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, true);
#pragma unroll
  for (int k4 = 0; k4 < 4; ++k4) {
    const int kk = h * 4 + k4;
    mma_ts(d_tmem, p_tmem + kk * 8, v_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc,
           (kk > 0 || accumulate) ? 1u : 0u);
  }
}

// ZIG: zigzag layout (two key segments per shard); otherwise one segment.
template <int D, bool ZIG>
__global__ void __launch_bounds__(kThreads, 1)
ring_tc_kernel(const __grid_constant__ RingParams p, const __grid_constant__ CUtensorMap tq,
               const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv) {
  using L = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  // d = 128 uses the barriers below kBarSB only
  constexpr int kBars = (D == 64) ? kNumBars : kBarSB;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * kBars + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Unit w = decode_unit(p, blockIdx.x);

  // Number of key tiles this CTA folds (every role walks the same sequence).
  int T = 0;
  for (int s = p.s_begin; s < p.s_end; ++s)
    for (int ks = 0; ks < (ZIG ? 2 : 1); ++ks)
      T += kv_tiles(p, seg_of(p.layout, p.S, p.P, shard_at(p, w.u, s), ks), w.qpos_max);
  const Seg sq = seg_of(p.layout, p.S, p.P, w.u, w.seg);   // segment of the query rows

  if (T == 0) {
    // Only in step mode: this shard is invisible to every row of the CTA, so the
    // state is unchanged — or starts empty.
    if (p.step_mode && !p.load_state && threadIdx.x < 256) {
      const int i = threadIdx.x >> 7;
      const int row = w.row0[i] + (threadIdx.x & 127);
      const int tok = sq.base + row * sq.stride;
      const size_t md = (static_cast<size_t>(w.bat) * p.H + w.head[i]) * p.N + tok;
      const size_t y0 = ((static_cast<size_t>(w.bat) * p.N + tok) * p.H + w.head[i]) * D;
      if (row < sq.len && in_bounds(md, 1, row_elems(p), p.status) &&
          in_bounds(y0, D, q_elems(p), p.status)) {
        p.m[md] = -INFINITY;
        p.z[md] = 0.f;
        float4* yr = reinterpret_cast<float4*>(p.y + y0);
#pragma unroll
        for (int c = 0; c < D / 4; ++c) yr[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBars; ++i) mbar_init(bar(i), 1);
    for (int x = 0; x < 4; ++x) mbar_init(bar(kBarPF + x), 4);   // one arrival per softmax warp
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tensormap(&tq);
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      // loads issued per barrier (for the drain on abort): K/V stages 0 and 1
      uint32_t nk0 = 0, nk1 = 0, nv0 = 0, nv1 = 0;
      bool ok = true;
      mbar_arrive_expect_tx(bar(kBarQ), 2 * L::kTile);
#pragma unroll
      for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_rows(&tq, sbase + L::kQ + i * L::kTile + c * L::kChunk, bar(kBarQ), p.layout, c,
                   w.head[i], sq.chunk, w.row0[i], w.bat);
      int t = 0;
      for (int s = p.s_begin; s < p.s_end && ok; ++s) {
        const int b = shard_at(p, w.u, s);
        for (int ks = 0; ks < (ZIG ? 2 : 1) && ok; ++ks) {
          const Seg sk = seg_of(p.layout, p.S, p.P, b, ks);
          const int nk = kv_tiles(p, sk, w.qpos_max);
          for (int kt = 0; kt < nk; ++kt, ++t) {
            const int st = t & 1;
            const uint32_t n = static_cast<uint32_t>(t >> 1);
            if (t >= 2 && !bounded_wait(bar(kBarKE + st), (n - 1) & 1, p.timeout_ns, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(kBarKF + st), L::kTile);
  #pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_rows(&tk, sbase + L::kK + st * L::kTile + c * L::kChunk, bar(kBarKF + st),
                       p.layout, c, w.g, sk.chunk, kt * 128, w.bat);
            if (st) ++nk1; else ++nk0;
            if (t >= 2 && !bounded_wait(bar(kBarVE + st), (n - 1) & 1, p.timeout_ns, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(bar(kBarVF + st), L::kTile);
  #pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_rows(&tv, sbase + L::kV + st * L::kTile + c * L::kChunk, bar(kBarVF + st),
                       p.layout, c, w.g, sk.chunk, kt * 128, w.bat);
            if (st) ++nv1; else ++nv0;
          }
        }
      }
      if (!ok) {
        record_failure(p, abort_flag);
        bounded_wait(bar(kBarQ), 0, kDrainNs, nullptr);
        if (nk0) bounded_wait(bar(kBarKF), (nk0 - 1) & 1, kDrainNs, nullptr);
        if (nk1) bounded_wait(bar(kBarKF + 1), (nk1 - 1) & 1, kDrainNs, nullptr);
        if (nv0) bounded_wait(bar(kBarVF), (nv0 - 1) & 1, kDrainNs, nullptr);
        if (nv1) bounded_wait(bar(kBarVF + 1), (nv1 - 1) & 1, kDrainNs, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    // The whole warp runs the loop and the waits (warp-uniform control flow and
    // operands); one elected lane issues each group of MMAs and commits. A loop
    // run by a single lane issues MMAs far slower than the tensor core executes
    // them.
    if constexpr (D == 64) {
      // Order: S(0) S(1) S(2), then per tile t: PV(2t), S(2t+3), PV(2t+1), S(2t+4).
      // S(k+3) reuses the buffer PV(k) has just read; the MMAs of one thread run in
      // order, so it never overwrites P before its PV has consumed it.
      const uint32_t tO0 = tmem + L::kOcol, tO1 = tmem + L::kOcol + D;
      const uint64_t dq0 = smem_desc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(sbase + L::kQ + L::kTile, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t dk1 = smem_desc_sw128(sbase + L::kK + L::kTile, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sbase + L::kV, L::kChunk, 1024);
      const uint64_t dv1 = smem_desc_sw128(sbase + L::kV + L::kTile, L::kChunk, 1024);
      bool ok = __all_sync(0xffffffffu, bounded_wait(bar(kBarQ), 0, p.timeout_ns, abort_flag) &&
                                        bounded_wait(bar(kBarKF), 0, p.timeout_ns, abort_flag));
      if (ok) {
        tc_fence_after_sync();
        if (elect_one()) {
          issue_qk<D>(tmem + score_col(0), dq0, dk0);
          mma_commit(bar(kBarSB + 0));
          issue_qk<D>(tmem + score_col(1), dq1, dk0);
          mma_commit(bar(kBarSB + 1));
          mma_commit(bar(kBarKE + 0));
        }
        __syncwarp();
      }
      if (ok && T > 1) {
        ok = __all_sync(0xffffffffu, bounded_wait(bar(kBarKF + 1), 0, p.timeout_ns, abort_flag));
        if (ok) {
          tc_fence_after_sync();
          if (elect_one()) {
            issue_qk<D>(tmem + score_col(2), dq0, dk1);
            mma_commit(bar(kBarSB + 2));
          }
          __syncwarp();
        }
      }
      for (int t = 0; t < T && ok; ++t) {
        const int st = t & 1;
        const uint32_t ph = static_cast<uint32_t>(t >> 1) & 1;
        const uint64_t vs = st ? dv1 : dv0;
        const bool acc = t > 0 || p.load_state;
        const int k0 = 2 * t, k1 = 2 * t + 1;
        // P V of sub-tile 0, tile t
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarVF + st), ph, p.timeout_ns, abort_flag) &&
                                     bounded_wait(bar(kBarPF + 0), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) issue_pv_half<D>(tO0, tmem + score_col(k0), vs, 0, acc);
        __syncwarp();
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarPF + 1), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) {
          issue_pv_half<D>(tO0, tmem + score_col(k0), vs, 1, acc);
          mma_commit(bar(kBarPD + 0));
          if (t + 1 == T) mma_commit(bar(kBarOF + 0));
          // S of sub-tile 1, tile t + 1 (its K tile already waited for S(2t+2))
          if (t + 1 < T) {
            const int st1 = (t + 1) & 1;
            issue_qk<D>(tmem + score_col(k0 + 3), dq1, st1 ? dk1 : dk0);
            mma_commit(bar(kBarSB + (k0 + 3) % 3));
            mma_commit(bar(kBarKE + st1));
          }
        }
        __syncwarp();
        // P V of sub-tile 1, tile t
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarPF + 2), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) issue_pv_half<D>(tO1, tmem + score_col(k1), vs, 0, acc);
        __syncwarp();
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarPF + 3), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) {
          issue_pv_half<D>(tO1, tmem + score_col(k1), vs, 1, acc);
          mma_commit(bar(kBarPD + 1));
          mma_commit(bar(kBarVE + st));
          if (t + 1 == T) mma_commit(bar(kBarOF + 1));
        }
        __syncwarp();
        // S of sub-tile 0, tile t + 2
        if (t + 2 < T) {
          const int st2 = (t + 2) & 1;
          const uint32_t ph2 = static_cast<uint32_t>((t + 2) >> 1) & 1;
          if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarKF + st2), ph2, p.timeout_ns, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (elect_one()) {
            issue_qk<D>(tmem + score_col(k1 + 3), dq0, st2 ? dk1 : dk0);
            mma_commit(bar(kBarSB + (k1 + 3) % 3));
          }
          __syncwarp();
        }
      }
      if (!ok) {
        if (lane == 0) record_failure(p, abort_flag);
        if (elect_one()) mma_commit(bar(kBarDrain));
        __syncwarp();
        bounded_wait(bar(kBarDrain), 0, kDrainNs, nullptr);
      }
    } else {
      const uint32_t tS0 = tmem, tS1 = tmem + 128;
      const uint32_t tO0 = tmem + L::kOcol, tO1 = tmem + L::kOcol + D;
      // Shared-memory descriptors of every tile base, computed once.
      const uint64_t dq0 = smem_desc_sw128(sbase + L::kQ, 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(sbase + L::kQ + L::kTile, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sbase + L::kK, 16, 1024);
      const uint64_t dk1 = smem_desc_sw128(sbase + L::kK + L::kTile, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sbase + L::kV, L::kChunk, 1024);
      const uint64_t dv1 = smem_desc_sw128(sbase + L::kV + L::kTile, L::kChunk, 1024);
      bool ok = __all_sync(0xffffffffu, bounded_wait(bar(kBarQ), 0, p.timeout_ns, abort_flag) &&
                                        bounded_wait(bar(kBarKF), 0, p.timeout_ns, abort_flag));
      if (ok) {
        tc_fence_after_sync();
        if (elect_one()) {
          issue_qk<D>(tS0, dq0, dk0);
          mma_commit(bar(kBarSF + 0));
          issue_qk<D>(tS1, dq1, dk0);
          mma_commit(bar(kBarSF + 1));
          mma_commit(bar(kBarKE + 0));
        }
        __syncwarp();
      }
      for (int t = 0; t < T && ok; ++t) {
        const int st = t & 1;
        const uint32_t ph = static_cast<uint32_t>(t >> 1) & 1;
        const bool has_next = t + 1 < T;
        const int st1 = (t + 1) & 1;
        const uint32_t ph1 = static_cast<uint32_t>((t + 1) >> 1) & 1;
        const uint64_t vs = st ? dv1 : dv0;
        const uint64_t ks1 = st1 ? dk1 : dk0;
        const bool acc = t > 0 || p.load_state;
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarVF + st), ph, p.timeout_ns, abort_flag) &&
                                     bounded_wait(bar(kBarPF + 0), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) issue_pv_half<D>(tO0, tS0, vs, 0, acc);
        __syncwarp();
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarPF + 1), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) {
          issue_pv_half<D>(tO0, tS0, vs, 1, acc);
          if (!has_next) mma_commit(bar(kBarOF + 0));
        }
        __syncwarp();
        if (has_next) {
          if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarKF + st1), ph1, p.timeout_ns, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          if (elect_one()) {
            issue_qk<D>(tS0, dq0, ks1);
            mma_commit(bar(kBarSF + 0));
          }
          __syncwarp();
        }
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarPF + 2), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) issue_pv_half<D>(tO1, tS1, vs, 0, acc);
        __syncwarp();
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarPF + 3), t & 1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) {
          issue_pv_half<D>(tO1, tS1, vs, 1, acc);
          mma_commit(bar(kBarVE + st));
          if (!has_next) mma_commit(bar(kBarOF + 1));
          if (has_next) {
            issue_qk<D>(tS1, dq1, ks1);
            mma_commit(bar(kBarSF + 1));
            mma_commit(bar(kBarKE + st1));
          }
        }
        __syncwarp();
      }
      if (!ok) {
        if (lane == 0) record_failure(p, abort_flag);
        if (elect_one()) mma_commit(bar(kBarDrain));
        __syncwarp();
        bounded_wait(bar(kBarDrain), 0, kDrainNs, nullptr);
      }
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int i = warp >> 2;                 // sub-tile of this group
    const int quarter = warp & 3;            // TMEM lanes [32*quarter, 32*quarter + 32)
    const int row = w.row0[i] + quarter * 32 + lane;   // within the query segment
    const bool valid = row < sq.len;
    const int qpos = valid ? sq.base + row * sq.stride : -1;
    const int head = w.head[i];
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS = tmem + i * 128 + lane_off;
    const uint32_t tO = tmem + L::kOcol + i * D + lane_off;
    const size_t md = valid ? (static_cast<size_t>(w.bat) * p.H + head) * p.N + qpos : 0;
    const size_t yo = valid ? ((static_cast<size_t>(w.bat) * p.N + qpos) * p.H + head) * D : 0;
    // this row's global reads and writes (O, LSE, or the state m, z, y) stay in bounds
    const bool io_ok = valid && in_bounds(md, 1, row_elems(p), p.status) &&
                       in_bounds(yo, D, q_elems(p), p.status);
    const float c2 = p.scale_log2;
    float m_run = -INFINITY;   // running max of the scaled scores, log2 units
    float z_run = 0.f;         // running denominator

    if (p.step_mode && p.load_state) {
      if (io_ok) {
        const float mm = p.m[md];
        m_run = (mm == -INFINITY) ? -INFINITY : mm * kLog2e;
        z_run = p.z[md];
      }
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t buf[32];
        if (io_ok) {
          const float4* src = reinterpret_cast<const float4*>(p.y + yo + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f = src[j];
            buf[4 * j + 0] = __float_as_uint(f.x);
            buf[4 * j + 1] = __float_as_uint(f.y);
            buf[4 * j + 2] = __float_as_uint(f.z);
            buf[4 * j + 3] = __float_as_uint(f.w);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) buf[j] = 0u;
        }
        tmem_st_x32(tO + c * 32, buf);
      }
      tmem_st_wait();
    }

    bool ok = true;
    int t = 0;
    for (int s = p.s_begin; s < p.s_end && ok; ++s) {
      const int b = shard_at(p, w.u, s);
      for (int ks = 0; ks < (ZIG ? 2 : 1) && ok; ++ks) {
        const Seg sk = seg_of(p.layout, p.S, p.P, b, ks);
        const int nk = kv_tiles(p, sk, w.qpos_max);
        // this row's visible keys of the segment, a prefix (one division per segment
        // rather than per tile in the striped layout)
        const int row_vis = seg_visible(sk, p.causal, 0, sk.len, qpos);
        for (int kt = 0; kt < nk; ++kt, ++t) {
          // this tile's scores: buffer i at d = 128; buffer (2t + i) mod 3 at d = 64
          const int kseq = 2 * t + i;
          const uint32_t tSt = (D == 64) ? tmem + score_col(kseq) + lane_off : tS;
          const bool got =
              (D == 64) ? bounded_wait(bar(kBarSB + kseq % 3), (kseq / 3) & 1, p.timeout_ns, abort_flag)
                        : bounded_wait(bar(kBarSF + i), t & 1, p.timeout_ns, abort_flag);
          if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          float sc[128];
          {
            uint32_t r[128];
            tmem_ld_x128(tSt, r);
  #pragma unroll
            for (int j = 0; j < 128; ++j) sc[j] = __uint_as_float(r[j]);
          }
          // Causal and segment-tail mask: the visible keys of this tile are a prefix.
          const int cnt = min(max(row_vis - kt * 128, 0), 128);
          if (__any_sync(0xffffffffu, cnt < 128)) {
  #pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= cnt) sc[c] = -INFINITY;
          }
          float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
  #pragma unroll
          for (int c = 0; c < 128; c += 8) {
            mx0 = fmax3(mx0, sc[c], sc[c + 1]);
            mx1 = fmax3(mx1, sc[c + 2], sc[c + 3]);
            mx2 = fmax3(mx2, sc[c + 4], sc[c + 5]);
            mx3 = fmax3(mx3, sc[c + 6], sc[c + 7]);
          }
          const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c2;
          float alpha = 1.f;
          bool rescale = false;
          if (m_tile > m_run) {
            // exact rescale by alpha = exp(m_old - m_new) whenever the running max grows
            if (m_run == -INFINITY) {
              alpha = 0.f;            // nothing accumulated yet: the state is zero
            } else {
              alpha = ex2(m_run - m_tile);
              rescale = true;
            }
            m_run = m_tile;
          }
          const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
          const float2 cc = make_float2(c2, c2);
          const float2 mneg = make_float2(-m_use, -m_use);
          float z_tile = 0.f;
#pragma unroll
          for (int h2 = 0; h2 < 2; ++h2) {
            // probabilities of keys [64 h2, 64 h2 + 64), stored as P columns [32 h2, 32 h2 + 32)
            float2 za = make_float2(0.f, 0.f), zb = za, zc = za, zd = za;
#pragma unroll
            for (int c = h2 * 64; c < h2 * 64 + 64; c += 8) {
              float2 x0 = ffma2(make_float2(sc[c], sc[c + 1]), cc, mneg);
              float2 x1 = ffma2(make_float2(sc[c + 2], sc[c + 3]), cc, mneg);
              float2 x2 = ffma2(make_float2(sc[c + 4], sc[c + 5]), cc, mneg);
              float2 x3 = ffma2(make_float2(sc[c + 6], sc[c + 7]), cc, mneg);
              x0 = make_float2(ex2(x0.x), ex2(x0.y));
              x1 = make_float2(ex2(x1.x), ex2(x1.y));
              x2 = make_float2(ex2(x2.x), ex2(x2.y));
              x3 = make_float2(ex2(x3.x), ex2(x3.y));
              za = fadd2(za, x0);
              zb = fadd2(zb, x1);
              zc = fadd2(zc, x2);
              zd = fadd2(zd, x3);
              sc[c] = x0.x; sc[c + 1] = x0.y; sc[c + 2] = x1.x; sc[c + 3] = x1.y;
              sc[c + 4] = x2.x; sc[c + 5] = x2.y; sc[c + 6] = x3.x; sc[c + 7] = x3.y;
            }
            const float2 zs = fadd2(fadd2(za, zb), fadd2(zc, zd));
            z_tile += zs.x + zs.y;
            uint32_t pk[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) pk[j] = pack_bf16x2(sc[h2 * 64 + 2 * j], sc[h2 * 64 + 2 * j + 1]);
            tmem_st_x32(tSt + h2 * 32, pk);
            if (h2 == 0) {
              // At d = 64 the commit of these scores does not cover the previous
              // tile's P V of this sub-tile (it was issued after them): wait for it
              // before touching O. At d = 128 the scores' commit already proves it.
              if constexpr (D == 64) {
                if (t > 0) {
                  const bool pv = bounded_wait(bar(kBarPD + i), (t - 1) & 1, p.timeout_ns, abort_flag);
                  if (!__all_sync(0xffffffffu, pv)) {
                    ok = false;
                    break;
                  }
                  tc_fence_after_sync();
                }
              }
              // Rescale this row's O by alpha before any P V MMA of this tile is
              // issued (the MMA that produced O so far has completed).
              if (__any_sync(0xffffffffu, rescale)) {
                const float2 a2 = rescale ? make_float2(alpha, alpha) : make_float2(1.f, 1.f);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                  uint32_t r[32];
                  tmem_ld_x32(tO + c * 32, r);
#pragma unroll
                  for (int j = 0; j < 32; j += 2) {
                    const float2 v = fmul2(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])), a2);
                    r[j] = __float_as_uint(v.x);
                    r[j + 1] = __float_as_uint(v.y);
                  }
                  tmem_st_x32(tO + c * 32, r);
                }
              }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kBarPF + 2 * i + h2));
          }
          if constexpr (D == 64) {
            if (!ok) break;
          }
          z_run = z_run * alpha + z_tile;
        }
      }
    }

    if (ok) {
      const bool got = bounded_wait(bar(kBarOF + i), 0, p.timeout_ns, abort_flag);
      ok = __all_sync(0xffffffffu, got);
    }
    if (!ok) {
      if (lane == 0) record_failure(p, abort_flag);
    } else {
      tc_fence_after_sync();
      if (!p.step_mode) {
        const float inv = z_run > 0.f ? 1.f / z_run : 0.f;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld_x32(tO + c * 32, r);
          if (io_ok && p.o_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.o) + yo + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(r[4 * j]) * inv, __uint_as_float(r[4 * j + 1]) * inv,
                                   __uint_as_float(r[4 * j + 2]) * inv,
                                   __uint_as_float(r[4 * j + 3]) * inv);
          } else if (io_ok) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.o) + yo + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(r[8 * j + 0]) * inv, __uint_as_float(r[8 * j + 1]) * inv);
              v.y = pack_bf16x2(__uint_as_float(r[8 * j + 2]) * inv, __uint_as_float(r[8 * j + 3]) * inv);
              v.z = pack_bf16x2(__uint_as_float(r[8 * j + 4]) * inv, __uint_as_float(r[8 * j + 5]) * inv);
              v.w = pack_bf16x2(__uint_as_float(r[8 * j + 6]) * inv, __uint_as_float(r[8 * j + 7]) * inv);
              dst[j] = v;
            }
          }
        }
        if (io_ok) p.lse[md] = z_run > 0.f ? (m_run + log2f(z_run)) * kLn2 : -INFINITY;
      } else {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t r[32];
          tmem_ld_x32(tO + c * 32, r);
          if (io_ok) {
            float4* dst = reinterpret_cast<float4*>(p.y + yo + c * 32);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(r[4 * j]), __uint_as_float(r[4 * j + 1]),
                                   __uint_as_float(r[4 * j + 2]), __uint_as_float(r[4 * j + 3]));
          }
        }
        if (io_ok) {
          p.m[md] = (m_run == -INFINITY) ? -INFINITY : m_run * kLn2;
          p.z[md] = z_run;
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D>
cudaError_t launch_d(const RingParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                     const CUtensorMap& tv, cudaStream_t st) {
  const int smem = Smem<D>::kAlloc;
  static OncePerContext attr;   // the limit belongs to the device's current context
  cudaError_t e = attr.run([&] {
    cudaError_t r = cudaFuncSetAttribute(ring_tc_kernel<D, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (r == cudaSuccess)
      r = cudaFuncSetAttribute(ring_tc_kernel<D, true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return r;
  });
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.B) * p.G * p.units_per_bg;
  if (grid <= 0) return cudaSuccess;
  if (p.layout == kZigzag)
    ring_tc_kernel<D, true><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(p, tq, tk, tv);
  else
    ring_tc_kernel<D, false><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace

int ring_tc_smem_bytes(int D) { return D == 64 ? Smem<64>::kAlloc : Smem<128>::kAlloc; }

cudaError_t launch_ring_tc(const RingParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t st) {
  return p.D == 64 ? launch_d<64>(p, tq, tk, tv, st) : launch_d<128>(p, tq, tk, tv, st);
}

}  // namespace ra
