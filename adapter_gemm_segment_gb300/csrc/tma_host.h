// Host-side creation of TMA tensor maps (driver entry point fetched through the runtime, so
// the library does not link libcuda directly).
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace lora {
namespace tc {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Row-major [rows, cols] 16-bit matrix, box {64 columns, box_rows rows}, 128-byte swizzle,
// out-of-bounds elements read as zero.
inline int make_map(CUtensorMap* m, const void* base, int bf16, uint64_t cols, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {64u, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return LORA_OK;
}

// Row-major [rows, cols] 16-bit matrix seen as [chunks][rows][64] (chunk = 64 columns, so the
// chunk stride is 128 bytes): one box {64, box_rows, box_chunks} lands as box_chunks
// consecutive [box_rows][64] tiles with 128-byte swizzle -- the layout of box_chunks
// consecutive 2-D boxes, fetched by a single TMA instruction.  cols must be a multiple of 64.
inline int make_map_chunked(CUtensorMap* m, const void* base, int bf16, uint64_t cols, uint64_t rows,
                            uint32_t box_rows, uint32_t box_chunks) {
    auto fn = encode_fn();
    if (!fn) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[3] = {64, rows, cols / 64};
    const cuuint64_t strides[2] = {cols * 2, 128};
    const cuuint32_t box[3] = {64u, box_rows, box_chunks};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled (chunked) failed (%d)", (int)r);
    return LORA_OK;
}

// Row-major [rows, cols] 16-bit matrix with row stride ld elements (0: ld = cols), box
// {box_cols, box_rows}, no swizzle (for stores of row-major shared-memory tiles).
inline int make_map_plain(CUtensorMap* m, const void* base, int bf16, uint64_t cols, uint64_t rows, uint32_t box_cols,
                          uint32_t box_rows, uint64_t ld = 0) {
    auto fn = encode_fn();
    if (!fn) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {(ld ? ld : cols) * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return LORA_OK;
}

// A pool's B slab [rows][r_max] (16-bit) seen as [rows][r_max / 8][8]: one box is one 8-column
// chunk of 128 consecutive rows, landing as [128][8] (16 bytes per row), no swizzle.
inline int make_map_bchunks(CUtensorMap* m, const void* base, int bf16, uint64_t r_max, uint64_t rows) {
    auto fn = encode_fn();
    if (!fn) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled is unavailable");
    const cuuint64_t dims[3] = {8, r_max / 8, rows};
    const cuuint64_t strides[2] = {16, r_max * 2};
    const cuuint32_t box[3] = {8u, 1u, 128u};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                          const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(LORA_ECUDA, "cuTensorMapEncodeTiled (B chunks) failed (%d)", (int)r);
    return LORA_OK;
}

}  // namespace tc
}  // namespace lora
