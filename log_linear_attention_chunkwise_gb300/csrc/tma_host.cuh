// Host side of TMA: tiled tensor maps, built through the driver entry point
// the CUDA runtime hands out (so liblla.so does not link libcuda directly).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lla {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A [n2][n1][n0] bf16 tensor (n0 innermost, contiguous) read in boxes of
// box0 x box1 x 1 with 128-byte swizzle; out-of-range elements read as 0.
// Requires n0 * 2 bytes to be a multiple of 16 and a 16-byte aligned base.
inline bool make_map_bf16_3d(CUtensorMap *map, const void *base, uint64_t n0, uint64_t n1,
                             uint64_t n2, uint32_t box0, uint32_t box1)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {n0, n1, n2};
    cuuint64_t strides[2] = {n0 * 2, n0 * n1 * 2};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The same for fp32 (box0 <= 32 so a box row is at most 128 bytes).
inline bool make_map_f32_3d(CUtensorMap *map, const void *base, uint64_t n0, uint64_t n1, uint64_t n2,
                            uint32_t box0, uint32_t box1)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {n0, n1, n2};
    cuuint64_t strides[2] = {n0 * 4, n0 * n1 * 4};
    cuuint32_t box[3] = {box0, box1, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims,
                     strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace lla
