// Tensor maps of the paged K/V pool for the TMA copies (cuTensorMapEncodeTiled, reached
// through the runtime's driver entry point so that the library links only the runtime).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "plan_layout.h"

namespace fa {
namespace tmap {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

// Pages [pool][Hkv][16][128] bf16 seen as a 4-D tensor (dims innermost first), read in boxes
// of 64 dims x 16 tokens of one head of one page, 128-byte swizzled in shared memory.
inline bool encode_pages(CUtensorMap *map, const void *pages, int64_t pool, int32_t hkv) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {cuuint64_t(fa::kHeadDim), cuuint64_t(fa::kPageSize), cuuint64_t(hkv),
                                cuuint64_t(pool)};
    const cuuint64_t strides[3] = {cuuint64_t(fa::kHeadDim * 2), cuuint64_t(fa::kPageSize * fa::kHeadDim * 2),
                                   cuuint64_t(hkv) * fa::kPageSize * fa::kHeadDim * 2};
    const cuuint32_t box[4] = {64, cuuint32_t(fa::kPageSize), 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(pages), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// V pages seen as a 5-D tensor (64 dims, 16 tokens, 2 dim-halves, Hkv, pool) so that one box
// of 64 x 16 x 2 lands a whole page-head (4 KiB) in shared memory as [half][token][64 dims],
// 128-byte swizzled: half the requests of two 64 x 16 boxes.
inline bool encode_pages_whole(CUtensorMap *map, const void *pages, int64_t pool, int32_t hkv) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[5] = {64, cuuint64_t(fa::kPageSize), 2, cuuint64_t(hkv), cuuint64_t(pool)};
    const cuuint64_t strides[4] = {cuuint64_t(fa::kHeadDim * 2), 128,
                                   cuuint64_t(fa::kPageSize * fa::kHeadDim * 2),
                                   cuuint64_t(hkv) * fa::kPageSize * fa::kHeadDim * 2};
    const cuuint32_t box[5] = {64, cuuint32_t(fa::kPageSize), 2, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(pages), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tmap
}  // namespace fa
