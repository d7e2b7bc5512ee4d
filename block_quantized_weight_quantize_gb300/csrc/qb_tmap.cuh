// qb_tmap.cuh -- tensor maps (the TMA engine's descriptors of a global
// tensor) for weight matrices as byte tensors, and the tiled copies that read
// boxes of them into shared memory.  One tiled copy moves a whole box (rows x
// bytes, or rows x blocks x bytes): one request to the copy engine where
// per-row bulk copies would issue one per row.
#pragma once

#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "qb_common.cuh"

namespace qb {

// cuTensorMapEncodeTiled from the driver, looked up once.
inline PFN_cuTensorMapEncodeTiled_v12000 tmap_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A matrix of `rows` records of `rec` bytes as a 2-D byte tensor [rows][rec],
// read in boxes of `bx` bytes x `by` rows (rows past the end read as zero).
inline bool tmap_rows(CUtensorMap *m, const void *W, int64_t rows, int64_t rec, int bx, int by) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)rec, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)rec};
    const cuuint32_t box[2] = {(cuuint32_t)bx, (cuuint32_t)by};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(W), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The blocks of a matrix as a 3-D byte tensor [rows][nb][bb] (block b of row r
// at r*rec + b*bb), read in boxes of bb bytes x `bn` blocks x `by` rows
// (blocks or rows past the end read as zero).
inline bool tmap_blocks(CUtensorMap *m, const void *W, int64_t rows, int64_t rec, int nb, int bb, int bn, int by) {
    auto enc = tmap_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)bb, (cuuint64_t)nb, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)bb, (cuuint64_t)rec};
    const cuuint32_t box[3] = {(cuuint32_t)bb, (cuuint32_t)bn, (cuuint32_t)by};
    const cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(W), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One box of a 2-D / 3-D tensor map into this CTA's shared memory, completing
// its bytes on `bar`.  x (the innermost coordinate, in bytes here) must be a
// multiple of 16.
__device__ __forceinline__ void tma_box_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
__device__ __forceinline__ void tma_box_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

}  // namespace qb
