// Host-side construction of the TMA tensor maps the kernels use.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

namespace dsa {

// 3-D map over x [T, H, width] bf16 with a 64-column x `box_heads` x 1 box
// and 128-byte swizzle: one K-major chunk of a head group per load.
cudaError_t make_head_tile_map(CUtensorMap* map, const void* x, int T, int H, int width,
                               int box_heads);

// 2-D map over a row-major bf16 matrix [rows, cols] with a 64-column x
// `box_rows` box and 128-byte swizzle.
cudaError_t make_matrix_map(CUtensorMap* map, const void* x, long long rows, int cols,
                            int box_rows);

}  // namespace dsa
