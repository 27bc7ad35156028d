// Host helpers shared by the kernels that load tiles with TMA: the driver's
// tensor-map encoder (resolved once through the runtime's entry-point query,
// so the library links no driver library itself), 2-D BF16 and FP32 maps,
// and the multiprocessor count of the current device.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

namespace kda {

inline PFN_cuTensorMapEncodeTiled_v12000 tma_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                            cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// BF16 (or, with `type`, another 16-bit type) [rows][cols] with a row pitch
// of `pitch_elems` elements, copied in boxes of box_cols x box_rows with the
// given shared-memory swizzle.  Rows past the end read as zero.
inline bool tma_map_bf16(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                         uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows,
                         CUtensorMapSwizzle swizzle,
                         CUtensorMapDataType type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
    auto fn = tma_encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {pitch_elems * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, type, 2, const_cast<void*>(base), gdim, gstride, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// BF16 [rows][cols] with a row pitch of `pitch_elems` elements, seen as
// groups of 8 consecutive columns: a box of `box_rows` rows x 128 columns
// lands in shared memory as [16 groups][box_rows][8], i.e. the MN-major
// core-matrix layout of an MMA operand whose N index is the column (K-adjacent
// core matrices 128 bytes apart, N-adjacent ones box_rows x 16 bytes).
inline bool tma_map_bf16_groups8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                                 uint64_t pitch_elems, uint32_t box_rows) {
    auto fn = tma_encode_fn();
    if (!fn || cols % 8 != 0) return false;
    cuuint64_t gdim[3] = {8, rows, cols / 8};
    cuuint64_t gstride[2] = {pitch_elems * 2, 16};
    cuuint32_t box[3] = {8, box_rows, 16};
    cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), gdim, gstride, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP32 [rows][cols] with a row pitch of `pitch_elems` elements, in boxes of
// box_cols x box_rows without swizzle (row-major in shared memory).
inline bool tma_map_f32(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows,
                        uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows) {
    auto fn = tma_encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {pitch_elems * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), gdim, gstride, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int sm_count() {
    static int counts[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (!counts[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        counts[dev] = n;
    }
    return counts[dev];
}

}  // namespace kda
