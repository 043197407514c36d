// Host helper of the tensor-core attention launches: tiled TMA descriptors
// for packed [T][H][D] bf16 tensors (boxes of 128 rows x 64 dims of one head,
// 128-byte swizzling: the operand layout of attn_tc.cuh).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace qa {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// dims {D, H, T} (innermost first), box {64, 1, box_rows} (128: a tile;
// 16: one page of a [pages * 16][H][D] pool).  Returns false when the driver
// rejects the descriptor (bad alignment or sizes).
// row_elems: elements between consecutive rows (0: packed, H * D).
inline bool make_rows_tmap(CUtensorMap *map, const void *base, int D, int H, long long T, int box_rows = 128,
                           long long row_elems = 0) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || T < 1 || T > 0x7fffffffLL) return false;
    if (row_elems == 0) row_elems = (long long)H * D;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)row_elems * 2};
    cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace qa
