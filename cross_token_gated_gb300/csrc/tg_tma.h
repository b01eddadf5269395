// Host-side creation of TMA tensor maps (driver entry point fetched through the
// runtime, so the library does not link libcuda directly).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace tg {

// Tiled bf16 tensor map over a row-major matrix [rows, cols] with row pitch
// `pitch_elems`, box [box_rows, box_cols], 128-byte swizzle when box_cols * 2 == 128
// (64 bytes / 32 bytes for narrower boxes), zero fill outside the matrix.
cudaError_t make_tmap_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch_elems,
                         uint32_t box_rows, uint32_t box_cols);

// Same over a [batch, rows, cols] tensor (row pitch cols, batch pitch rows*cols),
// box [1, box_rows, box_cols]; out-of-range rows of one batch read as zero
// instead of running into the next batch.
cudaError_t make_tmap_3d(CUtensorMap* map, const void* base, uint64_t batch, uint64_t rows, uint64_t cols,
                         uint32_t box_rows, uint32_t box_cols);

// Over a [batch, rows, heads, head_pitch] tensor of which the first head_cols columns of
// each head are read (row pitch heads * head_pitch), box [1, box_rows, 1, box_cols]:
// columns past a head's head_cols read as zero instead of running into the padding or
// the next head.  head_pitch * 2 must be a multiple of 16.
cudaError_t make_tmap_4d_heads(CUtensorMap* map, const void* base, uint64_t batch, uint64_t rows, uint64_t heads,
                               uint64_t head_cols, uint64_t head_pitch, uint32_t box_rows, uint32_t box_cols);

}  // namespace tg
