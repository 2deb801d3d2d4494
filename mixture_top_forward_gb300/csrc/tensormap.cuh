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

}  // namespace mita
