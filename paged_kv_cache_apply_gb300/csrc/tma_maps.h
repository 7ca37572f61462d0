// TMA tensor maps over row-major bf16 matrices with 128-byte swizzled boxes.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace astr {

// A [rows, cols] bf16 matrix (row stride cols * 2 bytes) read in boxes of box_rows x box_cols
// (box_cols * 2 <= 128) into the 128-byte swizzled shared-memory layout; out-of-range rows
// read as zero. Returns false if the driver rejects the map.
bool encode_map_bf16_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                        uint32_t box_cols, uint32_t box_rows);

}  // namespace astr
