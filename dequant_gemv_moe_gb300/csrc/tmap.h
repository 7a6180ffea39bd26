// tmap.h — host-side creation of 2-D TMA tensor maps over quantized weight
// matrices: rows of `row_bytes` bytes viewed as 16-bit elements, boxes of
// `box_bytes` x `box_rows`.  The driver entry point is fetched once through
// the runtime, so the library does not link libcuda directly.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace dqmoe {

// Returns false if the driver refuses the map (alignment, sizes).
bool make_weight_tmap(CUtensorMap* map, const void* base, uint64_t rows, uint64_t row_bytes,
                      uint32_t box_bytes, uint32_t box_rows);

// fp16 activations [rows][K] (K contiguous): boxes of 64 elements (128 B) x 32
// rows, written to shared memory in the 128-byte swizzled layout.
bool make_act_tmap_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t K);

}  // namespace dqmoe
