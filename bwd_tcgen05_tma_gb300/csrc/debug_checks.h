// Bounds predicates of the checking build (compiled with -DATTN_DEBUG): pure
// functions of plain integers.  The kernels evaluate them before a copy or a
// store and, when one fails, record ATTN_ERR_DEVICE_BOUNDS with the site and
// skip the access (no trap); the CPU tests compile the same header for the
// host and check the predicates themselves.
#pragma once
#include <stdint.h>

#if defined(__CUDACC__)
#define ATTN_HD __host__ __device__ __forceinline__
#else
#define ATTN_HD inline
#endif

namespace attn_dbg {

// A tiled TMA copy of the box {box_x, 1, box_z} at coordinates (x, y, z) of a
// tensor with extents {nx, ny, nz} and elem_bytes-byte elements:
//  - x starts on a 16-byte boundary (the copy engine's rule for the
//    innermost coordinate) and the box stays inside the row;
//  - y names an existing index of the middle dimension;
//  - a load may start before row 0 or run past the last row (the copy fills
//    zeros there) as long as one of its rows is inside the tensor;
//  - a store or a reduce starts at a row inside the tensor (never negative;
//    rows past the end are clipped by the copy engine).
ATTN_HD bool tma_box_ok(int64_t x, int64_t box_x, int64_t nx, int elem_bytes, int64_t y,
                        int64_t ny, int64_t z, int64_t box_z, int64_t nz, bool store) {
  if (x < 0 || (x * elem_bytes) % 16 != 0 || x + box_x > nx) return false;
  if (y < 0 || y >= ny) return false;
  if (store) return z >= 0 && z < nz;
  return z > -box_z && z < nz;
}

// The elements [first, first + count) lie inside an array of `size` elements.
ATTN_HD bool span_ok(int64_t first, int64_t count, int64_t size) {
  return first >= 0 && count >= 0 && first <= size - count;
}

// The elements [col, col + n) of row `row` of a row-strided tensor with
// `nrows` rows of `width` elements (the part of the row the tensor owns), at
// an address `addr` aligned to the `vec`-byte vector access that writes them.
ATTN_HD bool row_span_ok(int64_t row, int64_t nrows, int64_t col, int64_t n, int64_t width,
                         uint64_t addr, int vec) {
  return row >= 0 && row < nrows && col >= 0 && n >= 0 && col <= width - n &&
         addr % (uint64_t)vec == 0;
}

}  // namespace attn_dbg
