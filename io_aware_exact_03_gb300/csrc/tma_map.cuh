// Tensor-map encoding for the TMA loads of the tensor-core kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "attn_internal.h"

namespace attn {
namespace tma {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda); nullptr if the driver does not provide it.
inline EncodeTiledFn get_encode() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// [B, N, H, d] tensor seen as a 4-D map {d, H, N, B}; box = one swizzle chunk
// of d (chunk_elems) x 1 head x box_rows rows x 1 batch.  The swizzle is
// 128-byte when the chunk is 128 bytes wide, else 64-byte.
inline bool encode_map(CUtensorMap* m, const void* base, int dtype, int B, int N, int H, int d,
                       int chunk_elems, int box_rows) {
    EncodeTiledFn enc = get_encode();
    if (!enc) return false;
    const int E = dtype == kE4M3 ? 1 : 2;
    const CUtensorMapDataType dt = dtype == kBF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                   : dtype == kFP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)(N > 0 ? N : 1),
                                (cuuint64_t)B};
    const cuuint64_t strides[3] = {(cuuint64_t)d * E, (cuuint64_t)H * d * E,
                                   (cuuint64_t)(N > 0 ? N : 1) * H * d * E};
    const cuuint32_t box[4] = {(cuuint32_t)chunk_elems, 1, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapSwizzle sw =
        chunk_elems * E == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace tma
}  // namespace attn
