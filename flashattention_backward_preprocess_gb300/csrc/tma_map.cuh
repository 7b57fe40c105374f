// tma_map.cuh -- host helper that builds the TMA tensor maps of the tcgen05 kernels:
// a 3-D view [heads][rows][cols] of a dense [B, heads, rows, cols] tensor, 128-byte
// swizzle, boxes of 128 bytes of columns by `box_rows` rows.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

typedef CUresult (*TmaEncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                     const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                     const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                     CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda needed).
inline TmaEncodeTiledFn tma_encode_fn() {
    static TmaEncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<TmaEncodeTiledFn>(ptr);
    }
    return fn;
}

// Columns past `cols` and rows past `rows` read as zeros (loads) and are skipped (stores,
// reduce-adds).  Returns false if the map cannot be encoded (alignment, sizes).
inline bool tma_map_3d(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize, int heads,
                       int rows, int cols, int box_rows) {
    TmaEncodeTiledFn enc = tma_encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)heads};
    const cuuint64_t strides[2] = {(cuuint64_t)cols * esize, (cuuint64_t)rows * cols * esize};
    const cuuint32_t box[3] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace fa
