// Shard ownership, global positions and causal visibility for the virtual ring.
// Shared by the host shard-map export and by every kernel, so that the maps the
// tests read back are the maps the kernels use.
//
// Layouts:
//  * contiguous — shard u holds tokens [u*S, (u+1)*S) ("Part 4: Ring Attention"
//    (Fofadiya) §4.3.1 "Initial State").
//  * striped — token t belongs to shard t mod P at local index t div P ("Ring
//    Attention" (aarnphm.xyz): Striped Attention alternates shard ownership).
// Causal visibility is on global positions: key position <= query position
// ("Ring Attention: what the near-infinite context paper actually says", "The
// causal masking complication").  For both layouts the global position of local
// index i in a shard grows with i, so the keys of a shard that one query may see
// form a prefix of the shard, and a tile of queries x keys is empty, full or
// partial according to its two corner positions ("Part 4" §4.8.1).
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

namespace ra {

enum : int { kContiguous = 0, kStriped = 1 };
enum : int { kTileEmpty = 0, kTilePartial = 1, kTileFull = 2 };

// Global position (= original token index) of local index i of shard u.
RA_HD int32_t pos_of(int layout, int32_t S, int32_t P, int32_t u, int32_t i) {
  return layout == kContiguous ? u * S + i : i * P + u;
}
RA_HD int32_t owner_of(int layout, int32_t S, int32_t P, int32_t t) {
  return layout == kContiguous ? t / S : t % P;
}
RA_HD int32_t local_of(int layout, int32_t S, int32_t P, int32_t t) {
  return layout == kContiguous ? t % S : t / P;
}

// How many keys of shard b, counted from local index j0 and at most `width`
// of them (and never past the end of the shard), a query at global position
// qpos may see. Keys are visible iff pos(b, j) <= qpos (always, if !causal);
// the visible keys are a prefix, so the count is the prefix length.
// qpos < 0 means "no query" and sees nothing under the causal mask.
RA_HD int32_t visible_prefix(int layout, int32_t S, int32_t P, int causal, int32_t b,
                             int32_t j0, int32_t width, int32_t qpos) {
  int32_t lim = S - j0;
  if (lim > width) lim = width;
  if (lim < 0) lim = 0;
  if (!causal) return lim;
  int32_t cnt;
  if (layout == kContiguous) {
    cnt = qpos - (b * S + j0) + 1;          // b*S + j0 + c <= qpos
  } else {
    const int32_t num = qpos - b;            // (j0 + c)*P + b <= qpos
    cnt = num < 0 ? 0 : num / P - j0 + 1;
  }
  if (cnt < 0) cnt = 0;
  return cnt > lim ? lim : cnt;
}

// Class of the tile: rows [i0, i0+tm) of shard u x keys [j0, j0+tn) of shard b,
// counting only rows and keys < S.
RA_HD int tile_class(int layout, int32_t S, int32_t P, int causal, int32_t u, int32_t b,
                     int32_t i0, int32_t tm, int32_t j0, int32_t tn) {
  int32_t i_last = i0 + tm;
  if (i_last > S) i_last = S;
  i_last -= 1;
  int32_t n_keys = S - j0;
  if (n_keys > tn) n_keys = tn;
  if (i_last < i0 || n_keys <= 0) return kTileEmpty;
  const int32_t late = visible_prefix(layout, S, P, causal, b, j0, tn, pos_of(layout, S, P, u, i_last));
  if (late == 0) return kTileEmpty;
  const int32_t early = visible_prefix(layout, S, P, causal, b, j0, tn, pos_of(layout, S, P, u, i0));
  return early == n_keys ? kTileFull : kTilePartial;
}

}  // namespace ra
