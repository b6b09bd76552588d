// Level weights from a two-layer MLP ("Adaptive memory decay for Log-Linear
// Attention", §Method "LambdaMLPSoftplus"):
//     h = d W1 (width 2L),   lambda = softplus(h W2 + b),
// one d vector of width Dd per (token, head), weights shared by the heads.
// A CTA of 128 threads handles 128 rows; the weights sit in shared memory and
// every thread reads the same weight at the same time (broadcast).
#include "lambda_mlp.cuh"

namespace lla {
namespace {

constexpr int kRows = 128;

__device__ __forceinline__ float softplus_f(float z)
{
    return fmaxf(z, 0.f) + log1pf(__expf(-fabsf(z)));
}

// LMAX bounds the register arrays; the layouts use the runtime L.
template <typename Tin, int LMAX>
__global__ void __launch_bounds__(kRows)
lambda_mlp_kernel(const Tin *__restrict__ d, const float *__restrict__ W1, const float *__restrict__ W2,
                  const float *__restrict__ bias, float *__restrict__ lam, long long N, int Dd, int L)
{
    const int Hd = 2 * L;
    extern __shared__ float sm[];
    float *w1 = sm;              // [Dd][Hd]
    float *w2 = w1 + Dd * Hd;    // [Hd][L]
    float *bs = w2 + Hd * L;     // [L]
    for (int e = threadIdx.x; e < Dd * Hd; e += kRows) w1[e] = W1[e];
    for (int e = threadIdx.x; e < Hd * L; e += kRows) w2[e] = W2[e];
    for (int e = threadIdx.x; e < L; e += kRows) bs[e] = bias[e];
    __syncthreads();
    const long long n = (long long)blockIdx.x * kRows + threadIdx.x;
    if (n >= N) return;
    const Tin *dr = d + n * Dd;
    float h[2 * LMAX];
#pragma unroll
    for (int j = 0; j < 2 * LMAX; j++) h[j] = 0.f;
    for (int k = 0; k < Dd; k++) {
        const float x = to_f32(dr[k]);
#pragma unroll
        for (int j = 0; j < 2 * LMAX; j++)
            if (j < Hd) h[j] = fmaf(x, w1[k * Hd + j], h[j]);
    }
    float *out = lam + n * L;
    for (int l = 0; l < L; l++) {
        float z = bs[l];
#pragma unroll
        for (int j = 0; j < 2 * LMAX; j++)
            if (j < Hd) z = fmaf(h[j], w2[j * L + l], z);
        out[l] = softplus_f(z);
    }
}

template <typename Tin, int LMAX>
cudaError_t launch_l(const LambdaMlpArgs &A)
{
    const long long N = (long long)A.B * A.H * A.T;
    const size_t smem = sizeof(float) * ((size_t)A.Dd * 2 * A.L + 2 * (size_t)A.L * A.L + A.L);
    auto kern = lambda_mlp_kernel<Tin, LMAX>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((N + kRows - 1) / kRows), kRows, smem, (cudaStream_t)A.stream>>>(
        (const Tin *)A.d, A.W1, A.W2, A.bias, A.lam, N, A.Dd, A.L);
    return cudaPeekAtLastError();
}

template <typename Tin>
cudaError_t launch_t(const LambdaMlpArgs &A)
{
    if (A.L <= 8) return launch_l<Tin, 8>(A);
    if (A.L <= 12) return launch_l<Tin, 12>(A);
    if (A.L <= 16) return launch_l<Tin, 16>(A);
    return launch_l<Tin, 32>(A);
}

}  // namespace

cudaError_t lambda_mlp(const LambdaMlpArgs &A)
{
    return A.in_dt == LLA_F32 ? launch_t<float>(A) : launch_t<__nv_bfloat16>(A);
}

}  // namespace lla
