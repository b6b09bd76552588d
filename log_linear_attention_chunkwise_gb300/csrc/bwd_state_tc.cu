// Chunk states of the backward's rebuilt forward nodes on the tensor cores
// (bf16 k, v; dk = dv = 128; chunk 64):
//     H_i = K_i^T diag(exp(Gam_i - gamma)) V_i   ("Log-Linear Attention" §2.3),
// written to node slot i+1 for i < N-1, and Gam_i for every chunk (the
// chunk-gate prefix and the Fenwick scan that follow turn them into nodes).
// A CTA takes the chunk pair (2p, 2p+1) as one 128-token tile: TMA brings K,
// the MN-major A operand (M = dk); thread = token row scales its V row by
// exp(Gam - gamma) and splits it into a bf16 high part and a bf16 remainder
// (the MN-major B operand, N = dv), so each product keeps about 16 bits of
// the scaled values (K is exact); one thread issues, per chunk, four K = 16
// steps for each part into that chunk's tensor-memory accumulator.
#include "bwd_simt.cuh"
#include "sm100.cuh"
#include "tma_host.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kST = 128;  // tokens of a CTA: two chunks of 64
constexpr int kSD = 128;  // dk = dv
constexpr uint32_t kSB = kST * kSD * 2;  // bf16 128 x 128: 32 KB
constexpr uint32_t kSH = kSB / 2;
constexpr int kSThreads = 128;
constexpr uint32_t kSWait = 1u << 22;

struct __align__(1024) StateSmem {
    uint8_t k[kSB];
    uint8_t vhi[kSB], vlo[kSB];
    uint64_t bar_load, bar_mma;
    uint32_t tmem;
};

__global__ void __launch_bounds__(kSThreads, 2)
bwd_state_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __nv_bfloat16 *__restrict__ v,
                    const float *__restrict__ gamma, float *__restrict__ gam_tot, float *__restrict__ nodes, int T,
                    int N, int *__restrict__ err)
{
    extern __shared__ uint8_t smem_raw[];
    StateSmem &s = *reinterpret_cast<StateSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int p = threadIdx.x;
    const int c0 = 2 * blockIdx.x;
    const int bh = blockIdx.y;
    const long long t0 = (long long)c0 * 64;
    if (p == 0) {
        mbar_init(&s.bar_load, 1);
        mbar_init(&s.bar_mma, 1);
        fence_mbar_init();
        tma_prefetch_map(&map_k);
        mbar_arrive_expect_tx(&s.bar_load, kSB);
        tma_load_3d(s.k, &map_k, &s.bar_load, 0, (int)t0, bh);  // rows past T read as zero
        tma_load_3d(s.k + kSH, &map_k, &s.bar_load, 64, (int)t0, bh);
    }
    if (p < 32) {
        tmem_alloc(&s.tmem, 256);
        tmem_relinquish();
    }
    // token row p: exp(Gam_c - gamma_t) v_t, split
    const int c = c0 + (p >> 6);
    const bool ok = c < N;
    const long long t = t0 + p;
    float w = 0.f;
    if (ok) {
        const float Gam = gamma[(long long)bh * T + (long long)c * 64 + 63];
        w = __expf(Gam - gamma[(long long)bh * T + t]);
        if ((p & 63) == 0) gam_tot[(long long)bh * N + c] = Gam;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(v + ((long long)bh * T + (ok ? t : t0)) * kSD);
#pragma unroll 4
    for (int ch = 0; ch < 16; ch++) {
        const uint4 raw = ok ? src[ch] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t h4[4] = {raw.x, raw.y, raw.z, raw.w};
        uint4 hi, lo;
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&hi);
        __nv_bfloat162 *l2 = reinterpret_cast<__nv_bfloat162 *>(&lo);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const float x0 = __uint_as_float(h4[u] << 16) * w;  // bf16 -> fp32: the high half of the word
            const float x1 = __uint_as_float(h4[u] & 0xffff0000u) * w;
            const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
            const float2 hf = __bfloat1622float2(hv);
            h2[u] = hv;
            l2[u] = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
        }
        const uint32_t off = (ch >> 3) * kSH + sw128_offset(p, ch & 7);
        *reinterpret_cast<uint4 *>(s.vhi + off) = hi;
        *reinterpret_cast<uint4 *>(s.vlo + off) = lo;
    }
    fence_proxy_async_smem();
    if (!mbar_wait(&s.bar_load, 0, kSWait)) atomicCAS(err, 0, 1);
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;
    // chunk c0 + h has a state to write when c0 + h < N - 1
    const int nst = max(0, min(2, N - 1 - c0));
    if (p == 0) {
        const uint32_t idesc = idesc_bf16_f32(128, 128, true, true);
        for (int h = 0; h < nst; h++) {
#pragma unroll
            for (int kk = 4 * h; kk < 4 * h + 4; kk++) {
                const uint64_t a = desc_sw128(smem_u32(s.k) + kk * 2048, kSH, 1024);
                umma_bf16(tm + 128 * h, a, desc_sw128(smem_u32(s.vhi) + kk * 2048, kSH, 1024), idesc,
                          kk > 4 * h ? 1u : 0u);
                umma_bf16(tm + 128 * h, a, desc_sw128(smem_u32(s.vlo) + kk * 2048, kSH, 1024), idesc, 1u);
            }
        }
        umma_commit(&s.bar_mma);
    }
    if (!mbar_wait(&s.bar_mma, 0, kSWait)) atomicCAS(err, 0, 2);
    tc_fence_after_sync();
    // each state through shared memory (the operand stages are free now), then
    // to node slot c0 + h + 1 as whole rows: row p (tensor-memory lane p) is
    // staged by thread p at a 132-float stride, and the warps write 512-byte rows
    float *stg = reinterpret_cast<float *>(s.k);  // [128][132] fp32 = 66 KB of the 96 KB stages
    constexpr int kLds = kSD + 4;
    const uint32_t lane_off = (uint32_t)((p >> 5) * 32) << 16;
    for (int h = 0; h < nst; h++) {
#pragma unroll 1
        for (int cb = 0; cb < kSD; cb += 16) {
            float x[16];
            tmem_ld16(tm + 128 * h + lane_off + cb, x);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 4; u++)
                *reinterpret_cast<float4 *>(stg + p * kLds + cb + 4 * u) =
                    make_float4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
        }
        __syncthreads();
        float4 *dst = reinterpret_cast<float4 *>(nodes + ((long long)bh * N + c0 + h + 1) * kSD * kSD);
        for (int e = p; e < kSD * kSD / 4; e += kSThreads) {
            const int r = e >> 5, c4 = e & 31;
            dst[e] = *reinterpret_cast<const float4 *>(stg + r * kLds + 4 * c4);
        }
        __syncthreads();  // the staging is rewritten by the next state
    }
    tc_fence_before_sync();
    __syncthreads();
    if (p < 32) tmem_dealloc(tm, 256);
}

}  // namespace

bool bwd_state_tc_supported(const BwdArgs &A)
{
    return A.in_dt == LLA_BF16 && A.dk == kSD && A.dv == kSD && A.C == 64 && ((uintptr_t)A.k & 15) == 0 &&
           ((uintptr_t)A.v & 15) == 0;
}

cudaError_t bwd_state_tc(const BwdArgs &A, const float *gamma, float *gam_tot, float *nodes, int *err)
{
    const int BH = A.B * A.H, N = A.T / A.C;
    CUtensorMap mk;
    if (!make_map_bf16_3d(&mk, A.k, kSD, A.T, BH, 64, kST)) return cudaErrorInvalidValue;
    const size_t smem = sizeof(StateSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd_state_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_state_tc_kernel<<<dim3((N + 1) / 2, BH), kSThreads, smem, (cudaStream_t)A.stream>>>(
        mk, (const __nv_bfloat16 *)A.v, gamma, gam_tot, nodes, A.T, N, err);
    return cudaPeekAtLastError();
}

}  // namespace lla
