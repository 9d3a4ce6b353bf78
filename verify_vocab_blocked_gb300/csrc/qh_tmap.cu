// qh_tmap.cu -- TMA tensor maps for the tensor-core kernels.  The encoder
// (cuTensorMapEncodeTiled) is looked up once through the runtime's driver
// entry-point query, so the library does not link libcuda directly.
#include <mutex>

#include "qh_tc.cuh"
#include "qh_tmap.h"

namespace qh {

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
               uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
               CUtensorMapSwizzle swz) {
    EncodeTiledFn fn = encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tmap_rows_f16_sw128(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows,
                         uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, cols, rows, cols * 2, 64,
                     box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_packed_rows(CUtensorMap* map, const uint32_t* wq, uint64_t words_per_row, uint64_t rows,
                      uint32_t box_words, uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, words_per_row, rows,
                     words_per_row * 4, box_words, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

bool tmap_packed_rows_sw128(CUtensorMap* map, const uint32_t* wq, uint64_t words_per_row,
                            uint64_t rows, uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, words_per_row, rows,
                     words_per_row * 4, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool tmap_packed_rows_swz(CUtensorMap* map, const uint32_t* wq, uint64_t words_per_row,
                          uint64_t rows, uint32_t box_words, uint32_t box_rows) {
    const CUtensorMapSwizzle swz = box_words * 4 == 32   ? CU_TENSOR_MAP_SWIZZLE_32B
                                   : box_words * 4 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                   : box_words * 4 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                                          : CU_TENSOR_MAP_SWIZZLE_NONE;
    if (swz == CU_TENSOR_MAP_SWIZZLE_NONE) return false;
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, wq, words_per_row, rows,
                     words_per_row * 4, box_words, box_rows, swz);
}

bool tmap_group_rows(CUtensorMap* map, const void* scales, uint64_t groups, uint64_t rows,
                     uint32_t box_groups, uint32_t box_rows) {
    return encode_2d(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, groups, rows, groups * 2,
                     box_groups, box_rows, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace qh
