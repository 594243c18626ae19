// tma.cuh -- 2-D tensor copies (TMA): the device-side copy instruction and
// the host-side encoding of a tensor map over a row-major byte matrix.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"

namespace qdg {

// 2-D tiled tensor copy global -> shared (TMA), completion counted on bar.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        cudaGetLastError();
    });
    return fn;
}

// Rank-2 map over a row-major matrix of `rows` rows of row_bytes bytes, read
// in boxes of box_bytes x box_rows (uint8 elements, or uint16 when u16).
// row_bytes, box_bytes and the base address must be multiples of 16.  Rows
// outside the matrix read as zero.
inline bool encode_rows(CUtensorMap* map, const void* base, int64_t row_bytes, int64_t rows, int box_bytes,
                        int box_rows, bool u16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const int esz = u16 ? 2 : 1;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(row_bytes / esz), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_bytes / esz), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1u, 1u};
    return enc(map, u16 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base),
               dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tiled tensor copy global -> shared (TMA), completion counted on bar.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

// Rank-3 map over a row-major byte matrix of `rows` rows of row_bytes bytes,
// seen as [column groups of seg_bytes][rows][bytes of a group] (dimension
// order inner to outer: byte within the group, row, group).  A box of
// (seg_bytes, box_rows, box_segs) lands in shared memory as box_segs
// consecutive slabs of box_rows x seg_bytes bytes.  seg_bytes, row_bytes and
// the base address must be multiples of 16; rows and groups outside the
// matrix read as zero.
inline bool encode_row_segments(CUtensorMap* map, const void* base, int64_t row_bytes, int64_t rows, int seg_bytes,
                                int box_rows, int box_segs) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(seg_bytes), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(row_bytes / seg_bytes)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(seg_bytes)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(seg_bytes), static_cast<cuuint32_t>(box_rows),
                               static_cast<cuuint32_t>(box_segs)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace qdg
