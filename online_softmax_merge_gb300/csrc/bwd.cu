// Backward of the ring on sm_103a: dQ, dK, dV of softmax attention over P
// virtual shards, from the forward's saved output O and LSE.
//
// What it computes — Transformer Math "Ring Attention" (aicassindra), "The
// backward pass costs a second ring": the K/V blocks circulate a second time,
// carrying their accumulating dK/dV, and every query shard they pass adds its
// contribution; scores are rebuilt from the saved per-row statistics instead of
// being stored. The gradients flow in the reverse direction ("Ring Attention:
// what the near-infinite context paper actually says", "Production tradeoffs"):
// at backward step s virtual device u holds block (u + s) mod P. With
// S = scale Q K^T (causal mask on global positions), A = exp(S - LSE) and
// D = rowsum(dO * O) of each query row:
//     dV_b += A^T dO_u,   dS = A * (dO_u V_b^T - D_u),
//     dQ_u += scale dS K_b,   dK_b += scale dS^T Q_u.
//
// How, on one GB300 SM. Three launches:
//  * bwd_prep: D and LSE * log2(e) of every query row, written per 128-row tile
//    (1 KiB each, for the dQ kernel), and the same two numbers as extension tiles
//    for the dK/dV kernel's products (below);
//  * bwd_dkdv: a CTA owns one 128-key tile of one kv head — the circulating
//    block — and meets the query tiles of every query head of its group, shard by
//    shard in the reverse ring order u = (b - s) mod P, skipping tiles the causal
//    mask leaves empty. dK and dV stay in TMEM for the whole walk;
//  * bwd_dq: a CTA owns one 128-row query tile of one head and walks the key
//    tiles of blocks b = (u + s) mod P; dQ stays in TMEM, and so do the tile's
//    Q and dO (the workers store their rows there once), so all three products
//    of this kernel read only K or V from shared memory, streamed through three
//    stages.
// Both tensor-core kernels have 10 warps: warp 9 streams two tiles per step
// through two shared-memory stages with TMA, warp 8 issues the tcgen05 MMAs
// (one elected lane of a warp-uniform loop), and warps 0-7 are the element-wise
// workers — warp w reads TMEM lane quarter w % 4 and score columns
// [64 (w / 4), 64 (w / 4) + 64), so no row needs a reduction across threads.
// Per step, the workers turn the score tile into A (phase 1) and dP into dS
// (phase 2), each written back to TMEM as bf16 for the MMAs that take them as
// the TMEM operand.
//
// dK/dV kernel, per query tile t (TMEM: dK [0,D), dV [D,2D), S^T [256,384),
// dP^T [384,512)):  MMA order  dP^T(t) | dV += A^T(t) dO(t) | S^T(t+1) |
// dK += dS^T(t) Q(t) | dP^T(t+1) ...  so the workers' phase 1 overlaps dP^T(t)
// and phase 2 overlaps dV(t) and S^T(t+1). Each query column's LSE and D enter
// these products as one more 16-wide K slice: the key side holds ones in its
// first three columns, the query side the bf16 split hi + mid + lo of -LSE/scale
// (for S^T) or of -D (for dP^T), so the tensor core returns S^T - LSE/scale and
// dP^T - D in fp32 (three bf16 terms carry ~24 significant bits) and the workers
// need no per-column statistics. A stage's Q and dO have their own full and
// empty barriers: dO(t) is last read by dV(t), which completes before dK(t)
// reads Q(t) for the last time, so dO(t + 2) is loaded without waiting for dK(t).
// dQ kernel, per key tile t (TMEM: S [0,128), dP [128,256), dQ [256,256+D),
// Q and dO as bf16 pairs [384,512)): MMA order  dP(t) | S(t+1) | dQ += dS(t) K(t)
// | dP(t+1) ...
// The tensor core runs these in issue order, so an MMA that overwrites a TMEM
// region is always behind the MMAs that read it; the workers signal when they
// have read a region into registers.
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
constexpr int kWorkers = 8;                   // element-wise warps
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainNs = 200000000ull;   // 0.2 s to let in-flight copies land on abort
constexpr int kExtBytes = 128 * 16 * 2;       // one extension tile: 128 rows x 16 bf16

template <int D>
struct BwdSmem {
  static constexpr int kChunk = 128 * 128;          // 128 rows x 64 bf16 (128 B, swizzled)
  static constexpr int kTile = (D / 64) * kChunk;   // one [128 x D] bf16 tile
  // stages of the streamed Q and dO tiles: three where shared memory allows (d = 64)
  static constexpr int kStages = D == 64 ? 3 : 2;
  static constexpr int kFix = 0;                    // two stationary tiles
  static constexpr int kStage = 2 * kTile;          // kStages stages of two streamed tiles
  static constexpr int kAext = (2 + 2 * kStages) * kTile;   // key-side extension (ones)
  static constexpr int kExt = kAext + kExtBytes;    // + stage: query-side extensions of Q, dO
  static constexpr int kBar = kExt + kStages * 2 * kExtBytes;
  static constexpr int kBytes = kBar + 256;
  // One CTA per SM: it owns all 512 TMEM columns.
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

// dQ kernel: K/V stages only (Q and dO live in TMEM).
template <int D>
struct DqSmem {
  static constexpr int kChunk = 128 * 128;
  static constexpr int kTile = (D / 64) * kChunk;
  static constexpr int kStages = 3;
  static constexpr int kStage = 0;                  // stage st: K at kStage + 2 st kTile, V after
  static constexpr int kBar = kStages * 2 * kTile;
  static constexpr int kBytes = kBar + 256;
  static constexpr int kAlloc = (kBytes + 1024) > 120 * 1024 ? (kBytes + 1024) : 120 * 1024;
};

// dK/dV kernel barriers, for NS stages of streamed tiles. A stage's Q and dO tiles
// are tracked apart: dO(t) is last read by dV(t), which runs before dK(t), Q's last
// reader, so dO(t + NS) can start loading before the stage's Q slot is free.
constexpr int kBarFix = 0;   // stationary tiles landed (both backward kernels)
template <int NS>
struct BwdBars {
  static constexpr int kFull = 1;               // + stage: Q tile and its extension landed
  static constexpr int kEmpty = 1 + NS;         // + stage: dK done with the stage's Q
  static constexpr int kSF = 1 + 2 * NS;        // score tile in TMEM (score buffer 0)
  static constexpr int kDPF = kSF + 1;          // dP tile in TMEM
  static constexpr int kW1 = kSF + 2;           // workers: phase 1 done (8 arrivals)
  static constexpr int kW2 = kSF + 3;           // workers: dS written (8 arrivals)
  static constexpr int kDone = kSF + 4;         // every MMA of the CTA completed
  static constexpr int kDrain = kSF + 5;
  static constexpr int kFullO = kSF + 6;        // + stage: dO tile and its extension landed
  static constexpr int kEmptyO = kFullO + NS;   // + stage: dV done with the stage's dO
  static constexpr int kSF1 = kEmptyO + NS;     // d = 64: score tile in score buffer 1
  static constexpr int kNum = kSF1 + 1;
  static_assert(8 * kNum + 8 <= 256, "barrier area");
};

__device__ __forceinline__ void record_failure(const BwdParams& p, volatile int* abort_flag) {
  atomicCAS(p.status, 0, static_cast<int>(RA_ERR_TIMEOUT));
  *abort_flag = 1;
}


// 2-D tiled TMA load (the extension tiles: 16 bf16 x 128 rows, 32-byte swizzle).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :
      : "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// Shared-memory descriptor of a K-major operand whose rows are 32 bytes (one
// 16-element K slice) with the 32-byte swizzle: 8-row groups 256 bytes apart,
// layout code 6 in bits [61,64), descriptor version 1 at bit 46.
__device__ __forceinline__ uint64_t smem_desc_sw32(uint32_t saddr) {
  uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;            // leading offset (unused at this width)
  d |= static_cast<uint64_t>(256 >> 4) << 32;     // stride between 8-row groups
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(6) << 61;
  return d;
}

// D[tmem] = A B^T for two 128 x D tiles in shared memory (K-major, 128-byte
// swizzled 64-column chunks): D/16 MMAs of 128 x 128 x 16.
template <int D>
__device__ __forceinline__ void issue_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off =
        static_cast<uint64_t>(((kk >> 2) * BwdSmem<D>::kChunk + (kk & 3) * 32) >> 4);
    mma_ss(d_tmem, a_desc + off, b_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// D[tmem] (+)= A B with A [128 x 128] bf16 in TMEM — its 16-column K slices at
// a_tmem + (kk / 4) * 64 + (kk % 4) * 8, i.e. two 32-column halves 64 columns
// apart, as the workers write them — and B [128 x D] MN-major in shared memory
// (16 rows = 2 KiB per MMA; the descriptor's leading offset is the chunk stride).
template <int D>
__device__ __forceinline__ void issue_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                         bool accumulate) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, D, true);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk)
    mma_ts(d_tmem, a_tmem + (kk >> 2) * 64 + (kk & 3) * 8,
           b_desc + static_cast<uint64_t>((kk * 2048) >> 4), idesc,
           (kk > 0 || accumulate) ? 1u : 0u);
}

// D[tmem] = A B^T with A [128 x D] bf16 in TMEM (two elements per column, the
// k-th 16-element slice at a_tmem + 8 k) and B a [128 x D] K-major tile in
// shared memory: D/16 MMAs of 128 x 128 x 16.
template <int D>
__device__ __forceinline__ void issue_ts_kmajor(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off =
        static_cast<uint64_t>(((kk >> 2) * BwdSmem<D>::kChunk + (kk & 3) * 32) >> 4);
    mma_ts(d_tmem, a_tmem + kk * 8, b_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

__device__ __forceinline__ int ring_mod(int x, int P) {
  x %= P;
  return x < 0 ? x + P : x;
}

// Statistics tile of (batch, head, chunk, tile).
__device__ __forceinline__ const float* stats_tile(const BwdParams& p, int bat, int h, int chunk,
                                                   int tile) {
  return p.ws + ((((static_cast<size_t>(bat) * p.H + h) * p.X + chunk) * p.nt + tile) << 8);
}

// Workspace extents: tiles x 256 statistics floats, then (2 tiles + 1) extension
// tiles of 128 rows x 16 bf16.
__device__ __forceinline__ size_t stats_elems(const BwdParams& p) {
  return static_cast<size_t>(p.tiles) << 8;
}
__device__ __forceinline__ size_t ext_elems(const BwdParams& p) {
  return (2 * static_cast<size_t>(p.tiles) + 1) << 11;
}

// --------------------------------------------------------------------------- prep
// One row per TPR = D/8 threads (16 bytes of O and of dO each); warps advance
// together so the shuffles always see whole groups.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const BwdParams p) {
  constexpr int TPR = D / 8;
  constexpr int RPW = 32 / TPR;                       // rows per warp
  const int lane = threadIdx.x & 31;
  const int sub = lane % TPR;
  const long long tile_rows = static_cast<long long>(p.nt) * 128;
  const long long rows = static_cast<long long>(p.B) * p.H * p.X * tile_rows;
  const long long warp0 = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  for (long long base = warp0 * RPW; base < rows; base += nwarps * RPW) {
    const long long r = base + lane / TPR;
    const bool in = r < rows;
    long long rest = in ? r : 0;
    const int ii = static_cast<int>(rest % tile_rows);
    rest /= tile_rows;
    const int c = static_cast<int>(rest % p.X);
    rest /= p.X;
    const int h = static_cast<int>(rest % p.H);
    const int bat = static_cast<int>(rest / p.H);
    const bool valid = in && ii < p.L;
    float dsum = 0.f;
    float l2 = INFINITY;
    const int pos = p.layout == kStriped ? ii * p.P + c : c * p.L + ii;
    const size_t off = ((static_cast<size_t>(bat) * p.N + pos) * p.H + h) * D + sub * 8;
    const size_t li = (static_cast<size_t>(bat) * p.H + h) * p.N + pos;
    if (valid && in_bounds(off, 8, q_elems(p), p.status) &&
        in_bounds(li, 1, row_elems(p), p.status)) {
      const uint4 b =
          *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.dout) + off);
      const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
      float ov[8];
      if (p.o_f32) {
        const float4* src = reinterpret_cast<const float4*>(static_cast<const float*>(p.o) + off);
        const float4 a0 = src[0], a1 = src[1];
        ov[0] = a0.x; ov[1] = a0.y; ov[2] = a0.z; ov[3] = a0.w;
        ov[4] = a1.x; ov[5] = a1.y; ov[6] = a1.z; ov[7] = a1.w;
      } else {
        const uint4 a =
            *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.o) + off);
        const uint32_t av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 fa = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&av[e]));
          ov[2 * e] = fa.x;
          ov[2 * e + 1] = fa.y;
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fb = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&bv[e]));
        dsum = fmaf(ov[2 * e], fb.x, dsum);
        dsum = fmaf(ov[2 * e + 1], fb.y, dsum);
      }
      const float l = p.lse[li];
      l2 = (l == -INFINITY) ? INFINITY : l * kLog2e;   // a row with no key contributes 0
    }
#pragma unroll
    for (int o = TPR / 2; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
    const size_t tile = ((static_cast<size_t>(bat) * p.H + h) * p.X + c) * p.nt + (ii >> 7);
    const size_t r7 = ii & 127;
    if (in && sub == 0 && in_bounds((tile << 8) + r7, 129, stats_elems(p), p.status) &&
        in_bounds(((tile << 7) + r7) * 16, 16, ext_elems(p), p.status) &&
        in_bounds((((p.tiles + tile) << 7) + r7) * 16, 16, ext_elems(p), p.status)) {
      float* dst = p.ws + (tile << 8) + (ii & 127);
      dst[0] = l2;
      dst[128] = dsum;
      // extension rows: [-beta_hi, -beta_mid, -beta_lo, 0 ...] with beta = LSE / scale
      // (a huge finite value for rows that contribute nothing) and the same for D
      const float beta = (l2 == INFINITY) ? 1e30f : l2 / p.scale_log2;
      __nv_bfloat16* ext = reinterpret_cast<__nv_bfloat16*>(p.ws + (static_cast<size_t>(p.tiles) << 8));
      uint4* eq = reinterpret_cast<uint4*>(ext + ((tile << 7) + (ii & 127)) * 16);
      uint4* ed = reinterpret_cast<uint4*>(ext + (((static_cast<size_t>(p.tiles) + tile) << 7) + (ii & 127)) * 16);
      auto split3 = [](float x, uint32_t& w0, uint32_t& w1) {
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        const float r1 = x - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        w0 = static_cast<uint32_t>(__bfloat16_as_ushort(hi)) |
             (static_cast<uint32_t>(__bfloat16_as_ushort(mid)) << 16);
        w1 = static_cast<uint32_t>(__bfloat16_as_ushort(lo));
      };
      uint32_t a0, a1, b0, b1;
      split3(-beta, a0, a1);
      split3(-dsum, b0, b1);
      eq[0] = make_uint4(a0, a1, 0u, 0u);
      eq[1] = make_uint4(0u, 0u, 0u, 0u);
      ed[0] = make_uint4(b0, b1, 0u, 0u);
      ed[1] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // key-side extension tile: ones in columns 0-2 of all 128 rows
  if (blockIdx.x == 0 && threadIdx.x < 128 &&
      in_bounds(((2 * static_cast<size_t>(p.tiles)) << 11) + threadIdx.x * 16, 16, ext_elems(p),
                p.status)) {
    const uint32_t one2 = 0x3F803F80u;   // two bf16 ones
    __nv_bfloat16* ext = reinterpret_cast<__nv_bfloat16*>(p.ws + (static_cast<size_t>(p.tiles) << 8));
    uint4* ea = reinterpret_cast<uint4*>(ext + ((2 * static_cast<size_t>(p.tiles)) << 7) * 16 +
                                         threadIdx.x * 16);
    ea[0] = make_uint4(one2, 0x3F80u, 0u, 0u);
    ea[1] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// --------------------------------------------------------------------------- dK/dV
struct KUnit {
  int bat, g, b, kt;
  Seg sk;       // segment of shard b that holds the key rows
  int kpos0;    // global position of the tile's first key
};

__device__ __forceinline__ KUnit decode_kunit(const BwdParams& p, int idx) {
  const int per_bg = p.X * p.nt;
  const int bg = idx / per_bg;
  const int r = idx - bg * per_bg;
  // Earliest key positions first: under a causal mask they meet the most queries.
  // Striped tiles go in blocks of 4 tile indices per shard, so that the CTAs
  // resident at one time cover few shards and reread the same Q/dO tiles from L2.
  int c, kt;
  if (p.layout == kStriped) {
    const int QB = (p.nt % 4 == 0) ? 4 : 1;
    const int blk = r / (QB * p.P), rem = r - blk * QB * p.P;
    c = rem / QB;
    kt = blk * QB + (rem - c * QB);
  } else {
    c = r / p.nt;
    kt = r - c * p.nt;
  }
  KUnit w;
  w.bat = bg / p.G;
  w.g = bg - w.bat * p.G;
  w.kt = kt;
  int seg = 0;
  if (p.layout == kZigzag) {
    w.b = c < p.P ? c : 2 * p.P - 1 - c;
    seg = c < p.P ? 0 : 1;
  } else {
    w.b = c;
  }
  w.sk = seg_of(p.layout, p.S, p.P, w.b, seg);
  w.kpos0 = w.sk.base + kt * 128 * w.sk.stride;
  return w;
}

// First 128-row tile of query segment sq holding a query at or after position
// kpos0 (every tile without the causal mask); p.nt if none.
__device__ __forceinline__ int first_qtile(const BwdParams& p, const Seg& sq, int kpos0) {
  if (!p.causal || kpos0 <= sq.base) return 0;
  const int i = (kpos0 - sq.base + sq.stride - 1) / sq.stride;
  return i >= sq.len ? p.nt : (i >> 7);
}

// Calls f(t, h, sq, qt) for every query tile the key tile meets, in the order
// every role of the CTA walks: query heads of the group, then the reverse ring
// u = (b - s) mod P, then segments and tiles. Stops when f returns false.
template <bool ZIG, typename F>
__device__ __forceinline__ void walk_qtiles(const BwdParams& p, const KUnit& w, F&& f) {
  const int hpg = p.H / p.G;
  int t = 0;
  for (int hh = 0; hh < hpg; ++hh) {
    const int h = w.g * hpg + hh;
    for (int s = 0; s < p.P; ++s) {
      const int u = ring_mod(w.b - s, p.P);
      for (int qs = 0; qs < (ZIG ? 2 : 1); ++qs) {
        const Seg sq = seg_of(p.layout, p.S, p.P, u, qs);
        for (int qt = first_qtile(p, sq, w.kpos0); qt < p.nt; ++qt, ++t)
          if (!f(t, h, sq, qt)) return;
      }
    }
  }
}

template <int D, bool ZIG>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tq,
                const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap text) {
  using L = BwdSmem<D>;
  constexpr int NS = L::kStages;
  using Bars = BwdBars<NS>;
  constexpr int kBarFull = Bars::kFull, kBarEmpty = Bars::kEmpty, kBarSF = Bars::kSF,
                kBarDPF = Bars::kDPF, kBarW1 = Bars::kW1, kBarW2 = Bars::kW2,
                kBarDone = Bars::kDone, kBarDrain = Bars::kDrain, kBarFullO = Bars::kFullO,
                kBarEmptyO = Bars::kEmptyO, kBarSF1 = Bars::kSF1, kNumBars = Bars::kNum;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * kNumBars + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const KUnit w = decode_kunit(p, blockIdx.x);

  int T = 0;
  walk_qtiles<ZIG>(p, w, [&](int, int, const Seg&, int) { ++T; return true; });

  if (T == 0) {
    // No query sees these keys: their gradients are zero.
    if (threadIdx.x < 128) {
      const int j = w.kt * 128 + threadIdx.x;
      const int kpos = w.sk.base + j * w.sk.stride;
      const size_t off = ((static_cast<size_t>(w.bat) * p.N + kpos) * p.G + w.g) * D;
      if (j < w.sk.len && in_bounds(off, D, kv_elems(p), p.status)) {
        uint4* a = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dk) + off);
        uint4* b = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dv) + off);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) a[c] = b[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(kBarW1), kWorkers);
    mbar_init(bar(kBarW2), kWorkers);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tensormap(&tq);
    prefetch_tensormap(&tdo);
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
    prefetch_tensormap(&text);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // TMEM: dK, dV (fp32), the score tile S^T and dP^T (fp32, overwritten by A^T and dS^T
  // as bf16). At d = 64 the free columns [128, 256) hold a second score buffer: tile t's
  // scores go to buffer t % 2, so the next tile's scores need not wait for dV to have
  // read this tile's A^T.
  constexpr bool kTwoS = (D == 64);
  constexpr uint32_t kColDK = 0, kColDV = D, kColS = 256, kColS1 = 128, kColDP = 384;

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      uint32_t nfq[NS] = {}, nfo[NS] = {};   // loads issued per barrier (for the drain on abort)
      bool ok = true;
      mbar_arrive_expect_tx(bar(kBarFix), 2 * L::kTile + kExtBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_rows(&tk, sbase + L::kFix + c * L::kChunk, bar(kBarFix), p.layout, c, w.g,
                 w.sk.chunk, w.kt * 128, w.bat);
        tma_rows(&tv, sbase + L::kFix + L::kTile + c * L::kChunk, bar(kBarFix), p.layout, c, w.g,
                 w.sk.chunk, w.kt * 128, w.bat);
      }
      tma_load_2d(sbase + L::kAext, &text, bar(kBarFix), 0, 2 * p.tiles * 128);
      walk_qtiles<ZIG>(p, w, [&](int t, int h, const Seg& sq, int qt) {
        const int st = t % NS;
        const uint32_t n = static_cast<uint32_t>(t / NS);
        const uint32_t dst = sbase + L::kStage + st * 2 * L::kTile;
        const int tile = ((w.bat * p.H + h) * p.X + sq.chunk) * p.nt + qt;
        const uint32_t ext = sbase + L::kExt + st * 2 * kExtBytes;
        // dO(t) and its extension (-D), once dV(t - NS) has read the slot
        if (t >= NS && !bounded_wait(bar(kBarEmptyO + st), (n - 1) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          return false;
        }
        mbar_arrive_expect_tx(bar(kBarFullO + st), L::kTile + kExtBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_rows(&tdo, dst + L::kTile + c * L::kChunk, bar(kBarFullO + st), p.layout, c, h,
                   sq.chunk, qt * 128, w.bat);
        tma_load_2d(ext + kExtBytes, &text, bar(kBarFullO + st), 0, (p.tiles + tile) * 128);
#pragma unroll
        for (int x = 0; x < NS; ++x) nfo[x] += (x == st);
        // Q(t) and its extension (-LSE/scale), once dK(t - NS) has read the slot
        if (t >= NS && !bounded_wait(bar(kBarEmpty + st), (n - 1) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          return false;
        }
        mbar_arrive_expect_tx(bar(kBarFull + st), L::kTile + kExtBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_rows(&tq, dst + c * L::kChunk, bar(kBarFull + st), p.layout, c, h, sq.chunk,
                   qt * 128, w.bat);
        tma_load_2d(ext, &text, bar(kBarFull + st), 0, tile * 128);
#pragma unroll
        for (int x = 0; x < NS; ++x) nfq[x] += (x == st);
        return true;
      });
      if (!ok) {
        record_failure(p, abort_flag);
        bounded_wait(bar(kBarFix), 0, kDrainNs, nullptr);
#pragma unroll
        for (int x = 0; x < NS; ++x) {
          if (nfq[x]) bounded_wait(bar(kBarFull + x), (nfq[x] - 1) & 1, kDrainNs, nullptr);
          if (nfo[x]) bounded_wait(bar(kBarFullO + x), (nfo[x] - 1) & 1, kDrainNs, nullptr);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    const uint32_t tDK = tmem + kColDK, tDV = tmem + kColDV;
    const uint32_t tS = tmem + kColS, tDP = tmem + kColDP;
    const uint64_t dK = smem_desc_sw128(sbase + L::kFix, 16, 1024);
    const uint64_t dV = smem_desc_sw128(sbase + L::kFix + L::kTile, 16, 1024);
    // Q (which = 0) or dO (which = 1) of stage st, K-major or MN-major
    auto sdesc = [&](int st, int which, bool mn) -> uint64_t {
      return smem_desc_sw128(sbase + L::kStage + st * 2 * L::kTile + which * L::kTile,
                             mn ? L::kChunk : 16, 1024);
    };
    // S^T (which = 0) or dP^T (which = 1) of stage st, with its extension slice
    const uint64_t dA = smem_desc_sw32(sbase + L::kAext);
    constexpr uint32_t kIdesc = idesc_bf16_f32(128, 128, false);
    // score buffer of tile t
    auto sbuf = [&](int t) -> uint32_t { return (kTwoS && (t & 1)) ? kColS1 : kColS; };
    auto sfbar = [&](int t) -> int { return (kTwoS && (t & 1)) ? kBarSF1 : kBarSF; };
    auto products = [&](int st, int which, int t) {
      const uint32_t d_tmem = which == 0 ? tmem + sbuf(t) : tmem + kColDP;
      issue_ss<D>(d_tmem, which == 0 ? dK : dV, sdesc(st, which, false));
      mma_ss(d_tmem, dA, smem_desc_sw32(sbase + L::kExt + st * 2 * kExtBytes + which * kExtBytes),
             kIdesc, 1u);
    };
    bool ok = __all_sync(0xffffffffu, bounded_wait(bar(kBarFix), 0, p.timeout_ns, abort_flag) &&
                                      bounded_wait(bar(kBarFull), 0, p.timeout_ns, abort_flag));
    if (ok) {
      tc_fence_after_sync();
      if (elect_one()) {
        products(0, 0, 0);  // S^T(0) = K Q^T - LSE/scale
        mma_commit(bar(kBarSF));
      }
      __syncwarp();
      ok = __all_sync(0xffffffffu, bounded_wait(bar(kBarFullO), 0, p.timeout_ns, abort_flag));
    }
    if (ok) {
      tc_fence_after_sync();
      if (elect_one()) {
        products(0, 1, 0);  // dP^T(0) = V dO^T - D
        mma_commit(bar(kBarDPF));
      }
      __syncwarp();
    }
    // Order per tile t: dV(t) | S^T(t+1) | dK(t) | dP^T(t+1). With two score buffers
    // (d = 64) S^T(t+1) goes first: its buffer last held A^T(t-1), which dV(t-1) read
    // before it in the same order of MMAs, and the workers were done with it at W1(t-1).
    for (int t = 0; t < T && ok; ++t) {
      const int st = t % NS, st1 = (t + 1) % NS;
      const uint32_t ph1 = static_cast<uint32_t>((t + 1) / NS) & 1;
      const bool has_next = t + 1 < T;
      const uint32_t par = static_cast<uint32_t>(t) & 1;
      auto next_scores = [&]() -> bool {
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarFull + st1), ph1, p.timeout_ns, abort_flag)))
          return false;
        tc_fence_after_sync();
        if (elect_one()) {
          products(st1, 0, t + 1);
          mma_commit(bar(sfbar(t + 1)));
        }
        __syncwarp();
        return true;
      };
      if (kTwoS && has_next && !next_scores()) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarW1), par, p.timeout_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (elect_one()) {
        issue_ts<D>(tDV, tmem + sbuf(t), sdesc(st, 1, true), t > 0);   // dV += A^T dO
        mma_commit(bar(kBarEmptyO + st));
      }
      __syncwarp();
      if (!kTwoS && has_next && !next_scores()) {
        ok = false;
        break;
      }
      if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarW2), par, p.timeout_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (elect_one()) {
        issue_ts<D>(tDK, tDP, sdesc(st, 0, true), t > 0);          // dK += dS^T Q
        mma_commit(bar(kBarEmpty + st));
        if (!has_next) mma_commit(bar(kBarDone));
      }
      __syncwarp();
      if (has_next) {
        if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarFullO + st1), ph1, p.timeout_ns, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) {
          products(st1, 1, t + 1);
          mma_commit(bar(kBarDPF));
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
    __syncwarp();
  } else {
    // ------------------------------------------------------------- workers
    const int quarter = warp & 3;      // TMEM lanes = key rows [32 quarter, 32 quarter + 32)
    const int half = warp >> 2;        // query columns [64 half, 64 half + 64)
    const int j = w.kt * 128 + quarter * 32 + lane;
    const bool valid = j < w.sk.len;
    const int kpos = w.sk.base + j * w.sk.stride;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS0 = tmem + kColS + lane_off + half * 64;
    const uint32_t tS1 = tmem + kColS1 + lane_off + half * 64;
    const uint32_t tDP = tmem + kColDP + lane_off + half * 64;
    const float2 cc = make_float2(p.scale_log2, p.scale_log2);
    // First local query row of the current query segment that sees this key (kept per
    // segment, so the striped layout divides by its stride once per segment, not per tile).
    int seg_key = -1, first_q = 0;
    bool ok = true;
    walk_qtiles<ZIG>(p, w, [&](int t, int, const Seg& sq, int qt) {
      const uint32_t par = static_cast<uint32_t>(t) & 1;
      // phase 1: A^T = exp2((S^T - LSE/scale) * scale * log2e), masked; the
      // products already subtracted LSE/scale. Score buffer t % 2 at d = 64 (each
      // buffer completes once every two tiles), the one buffer otherwise.
      const bool b1 = kTwoS && (t & 1);
      const uint32_t tS = b1 ? tS1 : tS0;
      const uint32_t spar = kTwoS ? (static_cast<uint32_t>(t) >> 1) & 1 : par;
      if (!__all_sync(0xffffffffu,
                      bounded_wait(bar(b1 ? kBarSF1 : kBarSF), spar, p.timeout_ns, abort_flag))) {
        ok = false;
        return false;
      }
      tc_fence_after_sync();
      float a[64];
      {
        uint32_t r[64];
        tmem_ld_x64(tS, r);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 x = fmul2(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), cc);
          a[c] = ex2(x.x);
          a[c + 1] = ex2(x.y);
        }
      }
      // Causal mask: the key at kpos sees the queries at or after it, a suffix
      // of the tile's columns. (Columns past the chunk's end hold -1e30 there.)
      int cf = 0;
      if (p.causal) {
        if (sq.base != seg_key) {
          seg_key = sq.base;
          first_q = kpos <= sq.base ? 0 : (kpos - sq.base + sq.stride - 1) / sq.stride;
        }
        cf = min(max(first_q - qt * 128, 0), 128) - half * 64;
      }
      if (__any_sync(0xffffffffu, cf > 0)) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c < cf) a[c] = 0.f;
      }
      {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) pk[c] = pack_bf16x2(a[2 * c], a[2 * c + 1]);
        tmem_st_x32(tS, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarW1));
      // phase 2: dS^T = A^T * (dP^T - D)
      if (!__all_sync(0xffffffffu, bounded_wait(bar(kBarDPF), par, p.timeout_ns, abort_flag))) {
        ok = false;
        return false;
      }
      tc_fence_after_sync();
      {
        // dS^T = A^T * (dP^T - D); the products already subtracted D
        uint32_t r[64];
        tmem_ld_x64(tDP, r);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 e = fmul2(make_float2(a[c], a[c + 1]),
                                 make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])));
          pk[c >> 1] = pack_bf16x2(e.x, e.y);
        }
        tmem_st_x32(tDP, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarW2));
      return true;
    });
    if (ok) ok = __all_sync(0xffffffffu, bounded_wait(bar(kBarDone), 0, p.timeout_ns, abort_flag));
    if (!ok) {
      if (lane == 0) record_failure(p, abort_flag);
    } else {
      tc_fence_after_sync();
      // dK = scale * sum dS^T Q, dV = sum A^T dO: this warp writes columns
      // [half * D/2, half * D/2 + D/2) of its key rows.
      const size_t off = ((static_cast<size_t>(w.bat) * p.N + (valid ? kpos : 0)) * p.G + w.g) * D;
      const bool out_ok = valid && in_bounds(off, D, kv_elems(p), p.status);
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float mul = which == 0 ? p.scale : 1.f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(which == 0 ? p.dk : p.dv) + off;
        const uint32_t src = tmem + (which == 0 ? kColDK : kColDV) + lane_off;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const int col = half * (D / 2) + c * 32;
          uint32_t r[32];
          tmem_ld_x32(src + col, r);
          if (out_ok) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * mul, __uint_as_float(r[8 * q + 1]) * mul);
              v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * mul, __uint_as_float(r[8 * q + 3]) * mul);
              v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * mul, __uint_as_float(r[8 * q + 5]) * mul);
              v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * mul, __uint_as_float(r[8 * q + 7]) * mul);
              d4[q] = v;
            }
          }
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

// --------------------------------------------------------------------------- dQ
struct QUnit {
  int bat, h, u, qt;
  Seg sq;         // segment of shard u that holds the query rows
  int qpos_max;   // latest global position among the tile's rows
};

__device__ __forceinline__ QUnit decode_qunit(const BwdParams& p, int idx) {
  const int per_bh = p.X * p.nt;
  const int bh = idx / per_bh;
  const int r = idx - bh * per_bh;
  // Latest query positions first: under a causal mask they see the most keys.
  // Striped tiles go in blocks of 4 tile indices per shard (as in the forward).
  const int key = per_bh - 1 - r;
  int c, qt;
  if (p.layout == kStriped) {
    const int QB = (p.nt % 4 == 0) ? 4 : 1;
    const int blk = key / (QB * p.P), rem = key - blk * QB * p.P;
    c = rem / QB;
    qt = blk * QB + (rem - c * QB);
  } else {
    c = key / p.nt;
    qt = key - c * p.nt;
  }
  QUnit w;
  w.bat = bh / p.H;
  w.h = bh - w.bat * p.H;
  w.qt = qt;
  int seg = 0;
  if (p.layout == kZigzag) {
    w.u = c < p.P ? c : 2 * p.P - 1 - c;
    seg = c < p.P ? 0 : 1;
  } else {
    w.u = c;
  }
  w.sq = seg_of(p.layout, p.S, p.P, w.u, seg);
  const int last = min(qt * 128 + 127, w.sq.len - 1);
  w.qpos_max = w.sq.base + last * w.sq.stride;
  return w;
}

// Calls f(t, sk, kt) for every key tile the query tile sees, in the order every
// role walks: blocks b = (u + s) mod P (the reverse ring), then segments, then
// the visible prefix of tiles. Stops when f returns false.
template <bool ZIG, typename F>
__device__ __forceinline__ void walk_ktiles(const BwdParams& p, const QUnit& w, F&& f) {
  int t = 0;
  for (int s = 0; s < p.P; ++s) {
    const int b = ring_mod(w.u + s, p.P);
    for (int ks = 0; ks < (ZIG ? 2 : 1); ++ks) {
      const Seg sk = seg_of(p.layout, p.S, p.P, b, ks);
      const int nk = (seg_visible(sk, p.causal, 0, sk.len, w.qpos_max) + 127) >> 7;
      for (int kt = 0; kt < nk; ++kt, ++t)
        if (!f(t, sk, kt)) return;
    }
  }
}

template <int D, bool ZIG>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tq,
              const __grid_constant__ CUtensorMap tdo, const __grid_constant__ CUtensorMap tk,
              const __grid_constant__ CUtensorMap tv) {
  using L = DqSmem<D>;
  constexpr int NS = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = smem_u32(smem);
  // barriers: kBarFix, then NS full, NS empty, and the per-step ones after them
  constexpr int kFull = 1, kEmpty = 1 + NS, kSF = 1 + 2 * NS, kDPF = kSF + 1, kW1 = kSF + 2,
                kW2 = kSF + 3, kDone = kSF + 4, kDrain = kSF + 5, kSF1 = kSF + 6,
                kBars = kSF + 7;
  static_assert(8 * kBars + 8 <= 256, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kBar + 8 * kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kBar + 8 * kBars + 4);
  auto bar = [&](int i) -> uint32_t { return sbase + L::kBar + 8 * i; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const QUnit w = decode_qunit(p, blockIdx.x);

  int T = 0;
  walk_ktiles<ZIG>(p, w, [&](int, const Seg&, int) { ++T; return true; });

  if (T == 0) {
    if (threadIdx.x < 128) {
      const int i = w.qt * 128 + threadIdx.x;
      const int qpos = w.sq.base + i * w.sq.stride;
      const size_t off = ((static_cast<size_t>(w.bat) * p.N + qpos) * p.H + w.h) * D;
      if (i < w.sq.len && in_bounds(off, D, q_elems(p), p.status)) {
        uint4* a = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.dq) + off);
#pragma unroll
        for (int c = 0; c < D / 8; ++c) a[c] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < kBars; ++i) mbar_init(bar(i), 1);
    mbar_init(bar(kBarFix), kWorkers);   // the workers put Q and dO into TMEM
    mbar_init(bar(kW1), kWorkers);
    mbar_init(bar(kW2), kWorkers);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kTmaWarp && lane == 0) {
    prefetch_tensormap(&tk);
    prefetch_tensormap(&tv);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // TMEM: S, dP (fp32), dQ (fp32), and the stationary Q and dO tiles as bf16
  // pairs, the A operands of S = Q K^T and dP = dO V^T. At d = 64 a second score
  // buffer fits: tile t's scores go to buffer t % 2, so the next tile's scores need
  // not wait for the workers to have read this tile's.
  constexpr bool kTwoS = (D == 64);
  constexpr uint32_t kColS = 0, kColS1 = 128, kColDP = kTwoS ? 256 : 128,
                     kColDQ = kColDP + 128, kColQ = kColDQ + D, kColDO = kColQ + D / 2;
  static_assert(kColDO + D / 2 <= kTmemCols, "TMEM columns");

  if (warp == kTmaWarp) {
    // ------------------------------------------------------------------ TMA
    if (lane == 0) {
      uint32_t nf[NS] = {};   // loads issued per stage (for the drain on abort)
      bool ok = true;
      const int g = (w.h * p.G) / p.H;
      walk_ktiles<ZIG>(p, w, [&](int t, const Seg& sk, int kt) {
        const int st = t % NS;
        const uint32_t n = static_cast<uint32_t>(t / NS);
        if (t >= NS && !bounded_wait(bar(kEmpty + st), (n - 1) & 1, p.timeout_ns, abort_flag)) {
          ok = false;
          return false;
        }
        const uint32_t dst = sbase + L::kStage + st * 2 * L::kTile;
        mbar_arrive_expect_tx(bar(kFull + st), 2 * L::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_rows(&tk, dst + c * L::kChunk, bar(kFull + st), p.layout, c, g, sk.chunk,
                   kt * 128, w.bat);
          tma_rows(&tv, dst + L::kTile + c * L::kChunk, bar(kFull + st), p.layout, c, g,
                   sk.chunk, kt * 128, w.bat);
        }
#pragma unroll
        for (int x = 0; x < NS; ++x) nf[x] += (x == st);
        return true;
      });
      if (!ok) {
        record_failure(p, abort_flag);
#pragma unroll
        for (int x = 0; x < NS; ++x)
          if (nf[x]) bounded_wait(bar(kFull + x), (nf[x] - 1) & 1, kDrainNs, nullptr);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------------ MMA
    const uint32_t tS = tmem + kColS, tDP = tmem + kColDP, tDQ = tmem + kColDQ;
    const uint32_t tQ = tmem + kColQ, tDO = tmem + kColDO;
    // K (K-major for S, MN-major for dQ) and V (K-major) of stage st
    auto kdesc = [&](int st, bool mn) -> uint64_t {
      return smem_desc_sw128(sbase + L::kStage + st * 2 * L::kTile, mn ? L::kChunk : 16, 1024);
    };
    auto vdesc = [&](int st) -> uint64_t {
      return smem_desc_sw128(sbase + L::kStage + st * 2 * L::kTile + L::kTile, 16, 1024);
    };
    bool ok = __all_sync(0xffffffffu, bounded_wait(bar(kBarFix), 0, p.timeout_ns, abort_flag) &&
                                      bounded_wait(bar(kFull), 0, p.timeout_ns, abort_flag));
    if (ok) {
      tc_fence_after_sync();
      if (elect_one()) {
        issue_ts_kmajor<D>(tS, tQ, kdesc(0, false));    // S(0) = Q K^T, score buffer 0
        mma_commit(bar(kSF));
        issue_ts_kmajor<D>(tDP, tDO, vdesc(0));        // dP(0) = dO V^T
        mma_commit(bar(kDPF));
      }
      __syncwarp();
    }
    for (int t = 0; t < T && ok; ++t) {
      const int st = t % NS, st1 = (t + 1) % NS;
      const uint32_t ph1 = static_cast<uint32_t>((t + 1) / NS) & 1;
      const bool has_next = t + 1 < T;
      const uint32_t par = static_cast<uint32_t>(t) & 1;
      if (has_next) {
        // One score buffer: the workers have read S(t), so S(t+1) may overwrite it. Two
        // (d = 64): S(t+1) goes to the buffer of S(t-1), which the workers finished
        // reading before they wrote dS(t-1), and that was waited for (W2) before dQ(t-1).
        const bool ready = kTwoS ? bounded_wait(bar(kFull + st1), ph1, p.timeout_ns, abort_flag)
                                 : bounded_wait(bar(kW1), par, p.timeout_ns, abort_flag) &&
                                       bounded_wait(bar(kFull + st1), ph1, p.timeout_ns, abort_flag);
        if (!__all_sync(0xffffffffu, ready)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (elect_one()) {
          const bool b1 = kTwoS && ((t + 1) & 1);
          issue_ts_kmajor<D>(b1 ? tmem + kColS1 : tS, tQ, kdesc(st1, false));
          mma_commit(bar(b1 ? kSF1 : kSF));
        }
        __syncwarp();
      }
      if (!__all_sync(0xffffffffu, bounded_wait(bar(kW2), par, p.timeout_ns, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (elect_one()) {
        issue_ts<D>(tDQ, tDP, kdesc(st, true), t > 0);   // dQ += dS K
        mma_commit(bar(kEmpty + st));
        if (has_next) {
          issue_ts_kmajor<D>(tDP, tDO, vdesc(st1));
          mma_commit(bar(kDPF));
        } else {
          mma_commit(bar(kDone));
        }
      }
      __syncwarp();
    }
    if (!ok) {
      if (lane == 0) record_failure(p, abort_flag);
      if (elect_one()) mma_commit(bar(kDrain));
      __syncwarp();
      bounded_wait(bar(kDrain), 0, kDrainNs, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- workers
    const int quarter = warp & 3;      // TMEM lanes = query rows
    const int half = warp >> 2;        // key columns [64 half, 64 half + 64)
    const int i = w.qt * 128 + quarter * 32 + lane;
    const bool valid = i < w.sq.len;
    const int qpos = valid ? w.sq.base + i * w.sq.stride : -1;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t tS0 = tmem + kColS + lane_off + half * 64;
    const uint32_t tS1 = tmem + kColS1 + lane_off + half * 64;
    const uint32_t tDP = tmem + kColDP + lane_off + half * 64;
    const float* st_row = stats_tile(p, w.bat, w.h, w.sq.chunk, w.qt) + quarter * 32 + lane;
    const bool st_ok = in_bounds(static_cast<size_t>(st_row - p.ws), 129, stats_elems(p), p.status);
    const float l2 = st_ok ? st_row[0] : INFINITY;     // +inf past the chunk's end
    const float drow = st_ok ? st_row[128] : 0.f;
    // this row of q, dout and dq lies in its tensor
    const bool row_ok =
        valid && in_bounds(((static_cast<size_t>(w.bat) * p.N + qpos) * p.H + w.h) * D, D,
                           q_elems(p), p.status);
    const float2 cc = make_float2(p.scale_log2, p.scale_log2);
    const float2 ml = make_float2(-l2, -l2);
    const float2 dd = make_float2(drow, drow);
    {
      // Half 0 stores this row of Q, half 1 this row of dO, into TMEM as bf16
      // pairs (the memory order of the row); rows past the chunk's end are 0.
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const __nv_bfloat16*>(half == 0 ? p.q : p.dout) +
          ((static_cast<size_t>(w.bat) * p.N + (valid ? qpos : 0)) * p.H + w.h) * D);
      const uint32_t dst = tmem + (half == 0 ? kColQ : kColDO) + lane_off;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        uint32_t r[32];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 x = row_ok ? src[c * 8 + j] : make_uint4(0u, 0u, 0u, 0u);
          r[4 * j] = x.x;
          r[4 * j + 1] = x.y;
          r[4 * j + 2] = x.z;
          r[4 * j + 3] = x.w;
        }
        tmem_st_x32(dst + c * 32, r);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarFix));
    }
    // this row's visible keys of the current key segment, a prefix (kept per segment)
    int seg_key = -1, row_vis = 0;
    bool ok = true;
    walk_ktiles<ZIG>(p, w, [&](int t, const Seg& sk, int kt) {
      const uint32_t par = static_cast<uint32_t>(t) & 1;
      if (sk.base != seg_key || kt == 0) {
        seg_key = sk.base;
        row_vis = seg_visible(sk, p.causal, 0, sk.len, qpos);
      }
      // score buffer t % 2 at d = 64 (each completes once every two tiles)
      const bool b1 = kTwoS && (t & 1);
      const uint32_t spar = kTwoS ? (static_cast<uint32_t>(t) >> 1) & 1 : par;
      if (!__all_sync(0xffffffffu,
                      bounded_wait(bar(b1 ? kSF1 : kSF), spar, p.timeout_ns, abort_flag))) {
        ok = false;
        return false;
      }
      tc_fence_after_sync();
      float a[64];
      {
        uint32_t r[64];
        tmem_ld_x64(b1 ? tS1 : tS0, r);
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 x = ffma2(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])), cc, ml);
          a[c] = ex2(x.x);
          a[c + 1] = ex2(x.y);
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kW1));
      // causal / segment-tail mask: the visible keys of the tile are a prefix
      const int cnt = min(max(row_vis - kt * 128, 0), 128) - half * 64;
      if (__any_sync(0xffffffffu, cnt < 64)) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= cnt) a[c] = 0.f;
      }
      if (!__all_sync(0xffffffffu, bounded_wait(bar(kDPF), par, p.timeout_ns, abort_flag))) {
        ok = false;
        return false;
      }
      tc_fence_after_sync();
      {
        uint32_t r[64];
        tmem_ld_x64(tDP, r);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float2 e = fmul2(make_float2(a[c], a[c + 1]),
                                 fadd2(make_float2(__uint_as_float(r[c]), __uint_as_float(r[c + 1])),
                                       make_float2(-dd.x, -dd.y)));
          pk[c >> 1] = pack_bf16x2(e.x, e.y);
        }
        tmem_st_x32(tDP, pk);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kW2));
      return true;
    });
    if (ok) ok = __all_sync(0xffffffffu, bounded_wait(bar(kDone), 0, p.timeout_ns, abort_flag));
    if (!ok) {
      if (lane == 0) record_failure(p, abort_flag);
    } else {
      tc_fence_after_sync();
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.dq) +
                           ((static_cast<size_t>(w.bat) * p.N + (valid ? qpos : 0)) * p.H + w.h) * D;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = half * (D / 2) + c * 32;
        uint32_t r[32];
        tmem_ld_x32(tmem + kColDQ + lane_off + col, r);
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + col);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * p.scale, __uint_as_float(r[8 * q + 1]) * p.scale);
            v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * p.scale, __uint_as_float(r[8 * q + 3]) * p.scale);
            v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * p.scale, __uint_as_float(r[8 * q + 5]) * p.scale);
            v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * p.scale, __uint_as_float(r[8 * q + 7]) * p.scale);
            d4[q] = v;
          }
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

// Sets the dynamic shared-memory limit of a kernel once per device context.
template <typename K>
cudaError_t set_smem_once(K kernel, int bytes, OncePerContext& once) {
  return once.run(
      [&] { return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes); });
}

template <int D, bool ZIG>
cudaError_t launch_dkdv_d(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                          const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& text,
                          cudaStream_t st) {
  static OncePerContext done;
  const int smem = BwdSmem<D>::kAlloc;
  cudaError_t e = set_smem_once(bwd_dkdv_kernel<D, ZIG>, smem, done);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.B) * p.G * p.X * p.nt;
  if (grid <= 0) return cudaSuccess;
  bwd_dkdv_kernel<D, ZIG><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(p, tq, tdo, tk, tv,
                                                                                text);
  return cudaGetLastError();
}

template <int D, bool ZIG>
cudaError_t launch_dq_d(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                        const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  static OncePerContext done;
  const int smem = DqSmem<D>::kAlloc;
  cudaError_t e = set_smem_once(bwd_dq_kernel<D, ZIG>, smem, done);
  if (e != cudaSuccess) return e;
  const long long grid = static_cast<long long>(p.B) * p.H * p.X * p.nt;
  if (grid <= 0) return cudaSuccess;
  bwd_dq_kernel<D, ZIG><<<static_cast<unsigned>(grid), kThreads, smem, st>>>(p, tq, tdo, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_prep(const BwdParams& p, cudaStream_t st) {
  const long long rows = static_cast<long long>(p.B) * p.H * p.X * p.nt * 128;
  const int tpr = p.D / 8;
  long long blocks = (rows * tpr + 255) / 256;
  if (blocks > 152 * 64) blocks = 152 * 64;
  if (blocks < 1) blocks = 1;
  if (p.D == 64)
    bwd_prep_kernel<64><<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  else
    bwd_prep_kernel<128><<<static_cast<unsigned>(blocks), 256, 0, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd_dkdv(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                            const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& text,
                            cudaStream_t st) {
  const bool zig = p.layout == kZigzag;
  if (p.D == 64)
    return zig ? launch_dkdv_d<64, true>(p, tq, tdo, tk, tv, text, st)
               : launch_dkdv_d<64, false>(p, tq, tdo, tk, tv, text, st);
  return zig ? launch_dkdv_d<128, true>(p, tq, tdo, tk, tv, text, st)
             : launch_dkdv_d<128, false>(p, tq, tdo, tk, tv, text, st);
}

cudaError_t launch_bwd_dq(const BwdParams& p, const CUtensorMap& tq, const CUtensorMap& tdo,
                          const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
  const bool zig = p.layout == kZigzag;
  if (p.D == 64)
    return zig ? launch_dq_d<64, true>(p, tq, tdo, tk, tv, st)
               : launch_dq_d<64, false>(p, tq, tdo, tk, tv, st);
  return zig ? launch_dq_d<128, true>(p, tq, tdo, tk, tv, st)
             : launch_dq_d<128, false>(p, tq, tdo, tk, tv, st);
}

}  // namespace ra
