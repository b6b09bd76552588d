// Level weights from a two-layer MLP ("Adaptive memory decay for Log-Linear
// Attention", §Method "LambdaMLPSoftplus"):
//     h = d W1 (width 2L),   lambda = softplus(h W2 + b),
// one d vector of width Dd per (token, head), weights shared by the heads.
// A CTA of 128 threads handles 128 consecutive rows.  The rows' d block and
// their lambda block are each one contiguous span of memory, so both move
// through shared memory with coalesced accesses; each thread then computes
// its row against weights held in shared memory (zero-padded to HP hidden
// columns so every weight row is read as float4 broadcasts).
#include "lambda_mlp.cuh"

namespace lla {
namespace {

constexpr int kRows = 128;

__device__ __forceinline__ float softplus_f(float z)
{
    return fmaxf(z, 0.f) + log1pf(__expf(-fabsf(z)));
}

template <typename Tin>
__device__ __forceinline__ void stage_rows(const Tin *__restrict__ src, float *sd, int rows, int Dd)
{
    const int ld = Dd + 1;
    const int total = rows * Dd;
    for (int e = threadIdx.x; e < total; e += kRows) sd[(e / Dd) * ld + e % Dd] = to_f32(src[e]);
}

// 8 bf16 per 16-byte load when the block starts 16-byte aligned.
template <>
__device__ __forceinline__ void stage_rows<__nv_bfloat16>(const __nv_bfloat16 *__restrict__ src,
                                                           float *sd, int rows, int Dd)
{
    const int ld = Dd + 1;
    const int total = rows * Dd;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const int nvec = total / 8;
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
        for (int i = threadIdx.x; i < nvec; i += kRows) {
            const uint4 u = s4[i];
            const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&u);
#pragma unroll
            for (int q = 0; q < 8; q++) {
                const int e = 8 * i + q;
                sd[(e / Dd) * ld + e % Dd] = __bfloat162float(b[q]);
            }
        }
        done = nvec * 8;
    }
    for (int e = done + threadIdx.x; e < total; e += kRows) sd[(e / Dd) * ld + e % Dd] = __bfloat162float(src[e]);
}

// HP: hidden width padded to a multiple of 4 (>= 2L).
template <typename Tin, int HP>
__global__ void __launch_bounds__(kRows)
lambda_mlp_kernel(const Tin *__restrict__ d, const float *__restrict__ W1, const float *__restrict__ W2,
                  const float *__restrict__ bias, float *__restrict__ lam, long long N, int Dd, int L)
{
    const int Hd = 2 * L;
    extern __shared__ __align__(16) float sm[];
    float *w1 = sm;                  // [Dd][HP]  W1, columns >= Hd zero
    float *w2t = w1 + Dd * HP;       // [L][HP]   W2 transposed, columns >= Hd zero
    float *bs = w2t + L * HP;        // [L]
    float *sd = bs + ((L + 3) & ~3); // [kRows][Dd+1]
    float *so = sd + kRows * (Dd + 1);  // [kRows][L+1]
    for (int e = threadIdx.x; e < Dd * HP; e += kRows) {
        const int k = e / HP, j = e % HP;
        w1[e] = j < Hd ? W1[k * Hd + j] : 0.f;
    }
    for (int e = threadIdx.x; e < L * HP; e += kRows) {
        const int l = e / HP, j = e % HP;
        w2t[e] = j < Hd ? W2[j * L + l] : 0.f;
    }
    for (int e = threadIdx.x; e < L; e += kRows) bs[e] = bias[e];
    const long long n0 = (long long)blockIdx.x * kRows;
    const int rows = (int)min((long long)kRows, N - n0);
    stage_rows<Tin>(d + n0 * Dd, sd, rows, Dd);
    __syncthreads();
    const int r = threadIdx.x;
    if (r < rows) {
        float h[HP];
#pragma unroll
        for (int j = 0; j < HP; j++) h[j] = 0.f;
        const float *dr = sd + r * (Dd + 1);
        for (int k = 0; k < Dd; k++) {
            const float x = dr[k];
            const float4 *w = reinterpret_cast<const float4 *>(w1 + k * HP);
#pragma unroll
            for (int j4 = 0; j4 < HP / 4; j4++) {
                const float4 c = w[j4];
                h[4 * j4 + 0] = fmaf(x, c.x, h[4 * j4 + 0]);
                h[4 * j4 + 1] = fmaf(x, c.y, h[4 * j4 + 1]);
                h[4 * j4 + 2] = fmaf(x, c.z, h[4 * j4 + 2]);
                h[4 * j4 + 3] = fmaf(x, c.w, h[4 * j4 + 3]);
            }
        }
        for (int l = 0; l < L; l++) {
            const float4 *w = reinterpret_cast<const float4 *>(w2t + l * HP);
            float z = bs[l];
#pragma unroll
            for (int j4 = 0; j4 < HP / 4; j4++) {
                const float4 c = w[j4];
                z = fmaf(h[4 * j4 + 0], c.x, z);
                z = fmaf(h[4 * j4 + 1], c.y, z);
                z = fmaf(h[4 * j4 + 2], c.z, z);
                z = fmaf(h[4 * j4 + 3], c.w, z);
            }
            so[r * (L + 1) + l] = softplus_f(z);
        }
    }
    __syncthreads();
    float *out = lam + n0 * L;
    for (int e = threadIdx.x; e < rows * L; e += kRows) out[e] = so[(e / L) * (L + 1) + e % L];
}

size_t smem_bytes(int Dd, int L, int HP)
{
    return sizeof(float) * ((size_t)Dd * HP + (size_t)L * HP + ((L + 3) & ~3) +
                            (size_t)kRows * (Dd + 1) + (size_t)kRows * (L + 1));
}

template <typename Tin, int HP>
cudaError_t launch_l(const LambdaMlpArgs &A)
{
    const long long N = (long long)A.B * A.H * A.T;
    const size_t smem = smem_bytes(A.Dd, A.L, HP);
    auto kern = lambda_mlp_kernel<Tin, HP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)((N + kRows - 1) / kRows), kRows, smem, (cudaStream_t)A.stream>>>(
        (const Tin *)A.d, A.W1, A.W2, A.bias, A.lam, N, A.Dd, A.L);
    return cudaPeekAtLastError();
}

template <typename Tin>
cudaError_t launch_t(const LambdaMlpArgs &A)
{
    if (A.L <= 8) return launch_l<Tin, 16>(A);
    if (A.L <= 12) return launch_l<Tin, 24>(A);
    if (A.L <= 16) return launch_l<Tin, 32>(A);
    if (A.L <= 24) return launch_l<Tin, 48>(A);
    return launch_l<Tin, 64>(A);
}

}  // namespace

cudaError_t lambda_mlp(const LambdaMlpArgs &A)
{
    return A.in_dt == LLA_F32 ? launch_t<float>(A) : launch_t<__nv_bfloat16>(A);
}

}  // namespace lla
