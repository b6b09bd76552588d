// Shared device helpers of liblla.so (bit tricks, dtype loads).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lla.h"

namespace lla {

// bit_length(x): number of binary digits, 0 for x == 0.
__host__ __device__ __forceinline__ int bit_length_u32(uint32_t x)
{
#ifdef __CUDA_ARCH__
    return 32 - __clz(x);
#else
    int n = 0;
    while (x) { n++; x >>= 1; }
    return n;
#endif
}

__host__ __device__ __forceinline__ int bit_length_u64(uint64_t x)
{
#ifdef __CUDA_ARCH__
    return 64 - __clzll((long long)x);
#else
    int n = 0;
    while (x) { n++; x >>= 1; }
    return n;
#endif
}

// trailing zeros of x > 0
__host__ __device__ __forceinline__ int ctz_u32(uint32_t x)
{
#ifdef __CUDA_ARCH__
    return __ffs((int)x) - 1;
#else
    int n = 0;
    while ((x & 1u) == 0u) { n++; x >>= 1; }
    return n;
#endif
}

__host__ __device__ __forceinline__ int ctz_u64(uint64_t x)
{
#ifdef __CUDA_ARCH__
    return __ffsll((long long)x) - 1;
#else
    int n = 0;
    while ((x & 1u) == 0u) { n++; x >>= 1; }
    return n;
#endif
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x)
{
    return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x)
{
    return __float2bfloat16_rn(x);
}

__host__ __device__ __forceinline__ size_t align_up(size_t x, size_t a)
{
    return (x + a - 1) / a * a;
}

// lla_fwd's checks before the workspace (shape, dtypes, the empty case,
// pointers, alignment); *empty is set for a valid B*H*T == 0 call.
lla_status fwd_args_status(const void *q, const void *k, const void *v, const float *g,
                           const float *lambda, const void *out, int B, int H, int T, int dk,
                           int dv, int chunk, lla_dtype in_dt, lla_dtype out_dt, bool *empty);

}  // namespace lla
