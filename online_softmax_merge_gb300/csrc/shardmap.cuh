// Shard ownership, global positions and causal visibility for the virtual ring.
// Shared by the host shard-map export and by every kernel, so that the maps the
// tests read back are the maps the kernels use.
//
// Layouts:
//  * contiguous — shard u holds tokens [u*S, (u+1)*S) ("Part 4: Ring Attention"
//    (Fofadiya) §4.3.1 "Initial State").
//  * striped — token t belongs to shard t mod P at local index t div P ("Ring
//    Attention" (aarnphm.xyz): Striped Attention alternates shard ownership).
//  * zigzag — 2P chunks of C = N / 2P tokens; shard u holds chunk u (local
//    0 .. C-1) then chunk 2P-1-u (local C .. 2C-1) ("Part 4" §4.8.3 "Zigzag
//    (Striped) Load Balancing").
// Causal visibility is on global positions: key position <= query position
// ("Ring Attention: what the near-infinite context paper actually says", "The
// causal masking complication").
//
// A shard is one or two *segments*: runs of local indices whose global positions
// grow by a fixed stride (contiguous: one run, stride 1; striped: one run, stride
// P; zigzag: two runs of C, stride 1). Within a segment the keys one query may
// see form a prefix, so a tile of queries x keys inside one segment each is
// empty, full or partial according to its corner positions ("Part 4" §4.8.1).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

enum : int { kContiguous = 0, kStriped = 1, kZigzag = 2 };
enum : int { kTileEmpty = 0, kTilePartial = 1, kTileFull = 2 };

// Global position (= original token index) of local index i of shard u.
RA_HD int32_t pos_of(int layout, int32_t S, int32_t P, int32_t u, int32_t i) {
  if (layout == kContiguous) return u * S + i;
  if (layout == kStriped) return i * P + u;
  const int32_t C = S / 2;
  return i < C ? u * C + i : (2 * P - 1 - u) * C + (i - C);
}
RA_HD int32_t owner_of(int layout, int32_t S, int32_t P, int32_t t) {
  if (layout == kContiguous) return t / S;
  if (layout == kStriped) return t % P;
  const int32_t c = t / (S / 2);
  return c < P ? c : 2 * P - 1 - c;
}
RA_HD int32_t local_of(int layout, int32_t S, int32_t P, int32_t t) {
  if (layout == kContiguous) return t % S;
  if (layout == kStriped) return t / P;
  const int32_t C = S / 2;
  return (t / C) < P ? t % C : C + t % C;
}

// A run of local indices [start, start + len) of a shard whose global positions
// are base + (i - start) * stride. chunk: the index along the tensor maps' shard
// (contiguous, striped) or chunk (zigzag) axis.
struct Seg {
  int32_t start, len, base, stride, chunk;
};

RA_HD int num_segs(int layout) { return layout == kZigzag ? 2 : 1; }

RA_HD Seg seg_of(int layout, int32_t S, int32_t P, int32_t u, int s) {
  Seg g;
  if (layout == kContiguous) {
    g.start = 0; g.len = S; g.base = u * S; g.stride = 1; g.chunk = u;
  } else if (layout == kStriped) {
    g.start = 0; g.len = S; g.base = u; g.stride = P; g.chunk = u;
  } else {
    const int32_t C = S / 2;
    const int32_t c = s == 0 ? u : 2 * P - 1 - u;
    g.start = s == 0 ? 0 : C; g.len = C; g.base = c * C; g.stride = 1; g.chunk = c;
  }
  return g;
}

// How many keys of segment g, counted from offset j0 inside it and at most
// `width` of them (never past its end), a query at global position qpos may
// see. Keys are visible iff base + j*stride <= qpos (always, if !causal); they
// form a prefix. qpos < 0 means "no query" and sees nothing under the mask.
RA_HD int32_t seg_visible(const Seg& g, int causal, int32_t j0, int32_t width, int32_t qpos) {
  int32_t lim = g.len - j0;
  if (lim > width) lim = width;
  if (lim < 0) lim = 0;
  if (!causal) return lim;
  const int32_t num = qpos - g.base - j0 * g.stride;
  int32_t cnt = num < 0 ? 0 : (g.stride == 1 ? num : num / g.stride) + 1;
  return cnt > lim ? lim : cnt;
}

// Whether local key j of shard b is visible to a query at global position qpos.
RA_HD bool key_visible(int layout, int32_t S, int32_t P, int causal, int32_t b, int32_t j,
                       int32_t qpos) {
  if (j < 0 || j >= S) return false;
  return !causal || pos_of(layout, S, P, b, j) <= qpos;
}

// Visible keys of shard b among local [j0, j0 + width), for a range that lies
// inside one segment (always true for contiguous and striped shards).
RA_HD int32_t visible_prefix(int layout, int32_t S, int32_t P, int causal, int32_t b,
                             int32_t j0, int32_t width, int32_t qpos) {
  const int s = (layout == kZigzag && j0 >= S / 2) ? 1 : 0;
  const Seg g = seg_of(layout, S, P, b, s);
  return seg_visible(g, causal, j0 - g.start, width, qpos);
}

// Class of the tile: rows [i0, i0+tm) of shard u x keys [j0, j0+tn) of shard b,
// counting only rows and keys < S. The tile is cut along segment boundaries;
// inside each piece positions grow with the local index, so two corner checks
// per piece decide it.
RA_HD int tile_class(int layout, int32_t S, int32_t P, int causal, int32_t u, int32_t b,
                     int32_t i0, int32_t tm, int32_t j0, int32_t tn) {
  int32_t i1 = i0 + tm;
  if (i1 > S) i1 = S;
  int32_t j1 = j0 + tn;
  if (j1 > S) j1 = S;
  if (i1 <= i0 || j1 <= j0) return kTileEmpty;
  bool any = false, all = true;
  for (int rs = 0; rs < num_segs(layout); ++rs) {
    const Seg gq = seg_of(layout, S, P, u, rs);
    const int32_t a0 = i0 > gq.start ? i0 : gq.start;
    const int32_t a1 = i1 < gq.start + gq.len ? i1 : gq.start + gq.len;
    if (a1 <= a0) continue;
    const int32_t q_first = gq.base + (a0 - gq.start) * gq.stride;
    const int32_t q_last = gq.base + (a1 - 1 - gq.start) * gq.stride;
    for (int ks = 0; ks < num_segs(layout); ++ks) {
      const Seg gk = seg_of(layout, S, P, b, ks);
      const int32_t c0 = j0 > gk.start ? j0 : gk.start;
      const int32_t c1 = j1 < gk.start + gk.len ? j1 : gk.start + gk.len;
      if (c1 <= c0) continue;
      const int32_t n = c1 - c0;
      if (seg_visible(gk, causal, c0 - gk.start, n, q_last) > 0) any = true;
      if (seg_visible(gk, causal, c0 - gk.start, n, q_first) < n) all = false;
    }
  }
  if (!any) return kTileEmpty;
  return all ? kTileFull : kTilePartial;
}

}  // namespace ra
