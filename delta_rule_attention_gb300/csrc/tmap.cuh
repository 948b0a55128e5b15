// Tensor maps (TMA descriptors) for bf16 activation tensors [mats][rows][cols],
// encoded on the host.  The library links only the CUDA runtime, so the
// driver's encoder is reached through the runtime's driver entry point.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace falcon {

// 3-D row-major bf16 tensor [mats][rows][cols] with a box of box_rows rows x
// box_cols columns (box_cols * 2 <= 128 bytes) and the 128-byte swizzle, so a
// box lands in (or leaves from) shared memory as a 128B-swizzled tile: the
// 16-byte chunk c of box row r at chunk position c ^ (r & 7).  Loads outside
// the tensor read zeros; stores outside it are dropped.  Returns false if the
// encoder is unavailable or rejects the arguments (base 16-byte aligned,
// cols * 2 a multiple of 16).
bool encode_rows_bf16(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                      uint64_t mats, uint32_t box_cols, uint32_t box_rows);

}  // namespace falcon
