// TMA coordinates of the tensor views every tiled kernel loads through.
//
// The host encodes each [B, N, heads, d] bf16 tensor as a 5-D tensor map whose
// box is 64 columns of one head over a run of local rows of one chunk: the
// contiguous and zigzag layouts as (d, heads, L, X, B) — X chunks of L tokens,
// the chunk index of a segment (a contiguous shard, or a zigzag half-shard) —
// and the striped layout as (d, heads, P, S, B), token i*P + u of shard u.
#pragma once
#include <stdint.h>

#include "ptx.cuh"
#include "shardmap.cuh"

namespace ra {

// Loads the box of rows [i0, i0 + box rows) of `chunk` (the segment's chunk
// index), columns [64 dchunk, 64 dchunk + 64) of `head`, batch `bat`, into dst;
// completion is counted on bar. Rows past the chunk's end arrive as zeros.
__device__ __forceinline__ void tma_rows(const CUtensorMap* map, uint32_t dst, uint32_t bar,
                                         int layout, int dchunk, int head, int chunk, int i0,
                                         int bat) {
  if (layout == kStriped)
    tma_load_5d(dst, map, bar, dchunk * 64, head, chunk, i0, bat);
  else
    tma_load_5d(dst, map, bar, dchunk * 64, head, i0, chunk, bat);
}

}  // namespace ra
