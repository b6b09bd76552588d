// Sums of weighted outer products on CUDA cores,
//     acc += sum_t (sa_t a_t)(sb_t b_t)^T,  a_t in R^Da, b_t in R^Db,
// over runs of consecutive tokens.  Used where a state is a weighted K^T V
// style product: chunk states, prefill bucket states, the backward's
// block states.  A CTA of 256 threads tiles the Da x Db result (Da, Db <= 128,
// multiples of 8) as 16 x 16 thread tiles of 8 x 8; a step stages
// kOuterSub tokens of a and b as fp32 in shared memory and every thread
// reads its 8 a-values and 8 b-values as float4 pairs.
#pragma once

#include "lla_common.cuh"

namespace lla {

constexpr int kOuterThreads = 256;
constexpr int kOuterSub = 32;  // tokens staged per step

template <typename T> __device__ __forceinline__ void load8(const T *p, float *x, bool vec);

template <> __device__ __forceinline__ void load8<float>(const float *p, float *x, bool vec)
{
    if (vec) {
        const float4 u = reinterpret_cast<const float4 *>(p)[0], w = reinterpret_cast<const float4 *>(p)[1];
        x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
        x[4] = w.x; x[5] = w.y; x[6] = w.z; x[7] = w.w;
    } else {
#pragma unroll
        for (int q = 0; q < 8; q++) x[q] = p[q];
    }
}

template <> __device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *p, float *x, bool vec)
{
    if (vec) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&u);
#pragma unroll
        for (int q = 0; q < 8; q++) x[q] = __bfloat162float(b[q]);
    } else {
#pragma unroll
        for (int q = 0; q < 8; q++) x[q] = __bfloat162float(p[q]);
    }
}

// dst[tt][x] = scale[tt] * src[tt][x] for tt < n (scale == nullptr: 1), and 0
// for n <= tt < kOuterSub.  src holds n consecutive rows of width W.
template <typename T>
__device__ __forceinline__ void outer_stage(float *dst, const T *src, const float *scale, int n, int W)
{
    const int W8 = W / 8;
    const bool vec = (reinterpret_cast<uintptr_t>(src) & 15) == 0;
    for (int e = threadIdx.x; e < kOuterSub * W8; e += kOuterThreads) {
        const int tt = e / W8, x = (e - tt * W8) * 8;
        float v[8];
        if (tt < n) {
            load8<T>(src + (long long)tt * W + x, v, vec);
            const float s = scale ? scale[tt] : 1.f;
#pragma unroll
            for (int q = 0; q < 8; q++) v[q] *= s;
        } else {
#pragma unroll
            for (int q = 0; q < 8; q++) v[q] = 0.f;
        }
        float4 *d = reinterpret_cast<float4 *>(dst + tt * W + x);
        d[0] = make_float4(v[0], v[1], v[2], v[3]);
        d[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
}

__device__ __forceinline__ void outer_zero(float (&acc)[8][8])
{
#pragma unroll
    for (int a = 0; a < 8; a++)
#pragma unroll
        for (int b = 0; b < 8; b++) acc[a][b] = 0.f;
}

// acc (rows 8 ty.., columns 8 tx..) += sum over the n staged tokens.
__device__ __forceinline__ void outer_accumulate(float (&acc)[8][8], const float *as, const float *bs, int n,
                                                 int Da, int Db)
{
    const int r0 = 8 * ((threadIdx.x >> 4) & 15), c0 = 8 * (threadIdx.x & 15);
    if (r0 >= Da || c0 >= Db) return;
    for (int tt = 0; tt < n; tt++) {
        const float4 a0 = *reinterpret_cast<const float4 *>(as + tt * Da + r0);
        const float4 a1 = *reinterpret_cast<const float4 *>(as + tt * Da + r0 + 4);
        const float4 b0 = *reinterpret_cast<const float4 *>(bs + tt * Db + c0);
        const float4 b1 = *reinterpret_cast<const float4 *>(bs + tt * Db + c0 + 4);
        const float ra[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        const float rb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
        for (int a = 0; a < 8; a++)
#pragma unroll
            for (int b = 0; b < 8; b++) acc[a][b] = fmaf(ra[a], rb[b], acc[a][b]);
    }
}

// out[r][c] (row-major Da x Db) = acc, or += acc when add is set.
__device__ __forceinline__ void outer_store(float *out, const float (&acc)[8][8], int Da, int Db, bool add)
{
    const int r0 = 8 * ((threadIdx.x >> 4) & 15), c0 = 8 * (threadIdx.x & 15);
    if (r0 >= Da || c0 >= Db) return;
#pragma unroll
    for (int a = 0; a < 8; a++) {
        float4 *d = reinterpret_cast<float4 *>(out + (long long)(r0 + a) * Db + c0);
        float4 x0 = make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        float4 x1 = make_float4(acc[a][4], acc[a][5], acc[a][6], acc[a][7]);
        if (add) {
            const float4 y0 = d[0], y1 = d[1];
            x0.x += y0.x; x0.y += y0.y; x0.z += y0.z; x0.w += y0.w;
            x1.x += y1.x; x1.y += y1.y; x1.z += y1.z; x1.w += y1.w;
        }
        d[0] = x0;
        d[1] = x1;
    }
}

}  // namespace lla
