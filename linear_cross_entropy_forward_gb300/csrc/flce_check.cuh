// Bounds predicates of the in-kernel checks that the FLCE_DEBUG build compiles in,
// a stand-in for a memory sanitizer: before each TMA load and each epilogue store the
// kernel checks the access against the extents of its array; a failing check records
// FLCE_DEVERR_BOUNDS in the device error word, stops both CTAs of the pair, and the
// access is skipped, so the GPU never sees it.  The predicates are plain host/device
// functions so that they can be tested on the CPU.
#pragma once

#include <stdint.h>

#ifndef FLCE_DEBUG
#define FLCE_DEBUG 0
#endif

namespace flce {

// The widest tile extent along any dimension of the GEMMs (pair tiles are 256 rows
// by 256 columns; k-blocks are 64 deep).
constexpr int64_t kTileSpan = 256;

__host__ __device__ inline int64_t round_up_span(int64_t x) {
  return (x + kTileSpan - 1) / kTileSpan * kTileSpan;
}

// A TMA box starting at (x, y) of a tensor map over a [outer, inner] array.  Past the
// array's edge the engine reads zeros, and the ragged last tile of a dimension uses
// that, so a box may start past the edge -- but never beyond the tile-padded extent.
// x must also sit on a 16-byte boundary (8 bf16 elements).
__host__ __device__ inline bool tma_box_ok(int64_t x, int64_t y, int64_t inner, int64_t outer) {
  return x >= 0 && y >= 0 && x < round_up_span(inner) && y < round_up_span(outer) &&
         (x & 7) == 0;
}

// n consecutive elements from column `col` of a row `ld` elements long.
__host__ __device__ inline bool row_run_ok(int64_t col, int64_t n, int64_t ld) {
  return col >= 0 && n >= 0 && col + n <= ld;
}

// Index `i` of an array of `count` elements.
__host__ __device__ inline bool index_ok(int64_t i, int64_t count) { return i >= 0 && i < count; }

// Columns [col, col + n) of the 512-column TMEM allocation, read by warp `warp` from
// the lane quadrant `quadrant` (a warp may only reach the quadrant warp % 4).
__host__ __device__ inline bool tmem_ok(int64_t col, int64_t n, int quadrant, int warp) {
  return col >= 0 && n >= 0 && col + n <= 512 && quadrant == (warp & 3);
}

}  // namespace flce
