// qh_tmap.h -- host-side TMA tensor-map helpers and tensor-core launchers.
#pragma once

#include <cuda.h>

#include "qh_internal.cuh"

namespace qh {

// fp16 row-major matrix [rows, cols], box of 64 columns x box_rows rows,
// 128-byte swizzle (the tensor core's K-major SW128 layout).
bool tmap_rows_f16_sw128(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                         uint32_t box_rows);

// Packed uint32 head [rows, words_per_row], box of box_words x box_rows, no swizzle.
bool tmap_packed_rows(CUtensorMap* map, const uint32_t* wq, uint64_t words_per_row, uint64_t rows,
                      uint32_t box_words, uint32_t box_rows);

int tc_fwd_smem_bytes(int bits);
cudaError_t launch_tc_fwd(const CUtensorMap& tmap_h, const CUtensorMap& tmap_w,
                          const __half* scales, const __half* biases, int64_t V, int H, int bits,
                          float cap, const int* count, Partial* part, int* S_out, int* err,
                          int grid, cudaStream_t st);

}  // namespace qh
