// Host helper: TMA tensor maps over bf16 [rows x 64] matrices.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mita {

// Fills `map` for a row-major bf16 matrix of `rows` rows of 64 elements at
// `base` (16-byte aligned), loaded as boxes of box_rows x 64 with the 128-byte
// swizzle. Returns false if the driver entry point is unavailable or an
// argument is rejected.
bool make_row_tmap(CUtensorMap* map, const void* base, uint64_t rows, uint32_t box_rows);

// 3-D map over per-head row matrices: element (c, r, h) is at
// base + (h * head_stride_rows + r * row_stride_rows) * 64 + c (bf16), for
// r < rows_per_head, h < heads; loaded as boxes of box_rows x 64 of one head
// in the 128-byte swizzle. A row stride > 1 reads a strided sample of rows;
// rows past rows_per_head read as zeros.
bool make_head_tmap(CUtensorMap* map, const void* base, uint64_t rows_per_head, uint64_t heads,
                    uint64_t row_stride_rows, uint64_t head_stride_rows, uint32_t box_rows);

}  // namespace mita
