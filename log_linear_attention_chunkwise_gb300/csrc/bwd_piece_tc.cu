// Block-state pieces of the backward on the tensor cores (bf16 q; dk = dv =
// 128; chunk 64):  piece = sum_t w_t q_t dO_t^T over a run of tokens of one
// (level m, block b), w_t = lambda_t[c+1+m] exp(G_t - G_ref) (see the
// CUDA-core backward).  A CTA takes one piece (up to 16 chunks) in 128-token
// tiles: TMA brings the q tile; two threads per token row scale half the dO
// row each by w (0 for tokens outside the piece) and split it into bf16 high
// and remainder parts, stored side by side; one thread issues
// [piece_hi | piece_lo] += Q^T [(w dO)_hi | (w dO)_lo] (M = dk, N = 2 dv,
// K = 128 tokens: one MMA per K step) into two tensor-memory accumulators,
// added when the piece is written.  The dO rows of a tile are prefetched
// into L2 two tiles ahead.  The finished piece is
// written to its own slot; the reduction that follows sums a block's pieces
// in order.
#include "bwd_simt.cuh"
#include "sm100.cuh"
#include "split_stage.cuh"
#include "tma_host.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kPT = 128;
constexpr int kPDm = 128;
constexpr uint32_t kPB = kPT * kPDm * 2;  // 32 KB
constexpr uint32_t kPH = kPB / 2;
constexpr int kPThreads = 256;  // (token row, column half)
constexpr uint32_t kPWait = 1u << 22;

// S stages of (q tile, split dO tile).  With one stage (96 KB) two CTAs share
// an SM, so one CTA's dO split and drain overlap the other's loads and
// products; with two, one CTA overlaps its own next load.
template <int S>
struct __align__(1024) PieceSmem {
    uint8_t q[S][kPB];
    struct __align__(1024) {
        uint8_t hi[kPB], lo[kPB];  // the four 64-column blocks of one N = 256 operand
    } b[S];
    uint64_t bar_load[S], bar_mma[S], bar_done;
    uint32_t tmem;
};

template <int S>
__global__ void __launch_bounds__(kPThreads, 3 - S)
bwd_piece_tc_kernel(const __grid_constant__ CUtensorMap map_q, const float *__restrict__ dout,
                    const float *__restrict__ gamma, const float *__restrict__ lam, const double *__restrict__ P,
                    float *__restrict__ part, int T, int N, int L, int cbits, int nlev, int Pc,
                    int *__restrict__ err)
{
    extern __shared__ uint8_t smem_raw[];
    PieceSmem<S> &s = *reinterpret_cast<PieceSmem<S> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int p = tid & 127, half = tid >> 7;  // token row of a tile, half of its columns
    const int bh = blockIdx.y;
    // locate (m, b, piece) as the CUDA-core kernel does
    int idx = blockIdx.x, m = -1, b = 0, pc = 0;
    for (int mm = 0; mm < nlev; mm++) {
        const int nb = (N + (1 << mm) - 1) >> mm;
        const int pp = ((1 << mm) + Pc - 1) / Pc;
        const int cnt = (nb / 2) * pp;
        if (idx < cnt) {
            m = mm;
            b = 2 * (idx / pp) + 1;
            pc = idx % pp;
            break;
        }
        idx -= cnt;
    }
    if (m < 0) return;
    const int c0 = b << m;
    const int blk_end = min(N, (b + 1) << m);
    const int p0 = c0 + pc * Pc, p1 = min(blk_end, p0 + Pc);
    if (p0 >= p1) return;
    const int lev = cbits + 1 + m;
    const double *Pb = P + (long long)bh * (N + 1);
    const double Pref = Pb[c0];
    const long long t_lo = (long long)p0 << cbits, t_hi = (long long)p1 << cbits;
    const int ntiles = (int)((t_hi - t_lo + kPT - 1) / kPT);
    if (tid == 0) {
        for (int i = 0; i < S; i++) {
            mbar_init(&s.bar_load[i], 1);
            mbar_init(&s.bar_mma[i], 1);
        }
        mbar_init(&s.bar_done, 1);
        fence_mbar_init();
        tma_prefetch_map(&map_q);
    }
    if (tid < 32) {
        tmem_alloc(&s.tmem, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;
    auto load_q = [&](int n) {
        const int st = n % S;
        mbar_arrive_expect_tx(&s.bar_load[st], kPB);
        tma_load_3d(s.q[st], &map_q, &s.bar_load[st], 0, (int)(t_lo + (long long)n * kPT), bh);
        tma_load_3d(s.q[st] + kPH, &map_q, &s.bar_load[st], 64, (int)(t_lo + (long long)n * kPT), bh);
    };
    auto prefetch_dout = [&](int n) {  // the dO rows of tile n (rows past the piece are not needed)
        if (tid == 0 && n < ntiles) {
            const long long r0 = t_lo + (long long)n * kPT;
            const long long rows = min((long long)kPT, t_hi - r0);
            const float *src = dout + ((long long)bh * T + r0) * kPDm;
            for (long long r = 0; r < rows; r += 64)  // pieces of at most 32 KB
                bulk_prefetch_l2(src + r * kPDm, (uint32_t)(min(64LL, rows - r) * kPDm * 4));
        }
    };
    if (tid == 0)
        for (int n = 0; n < min(S, ntiles); n++) load_q(n);
    prefetch_dout(0);
    prefetch_dout(1);
    const uint32_t idesc = idesc_bf16_f32(128, 256, true, true);
    for (int n = 0; n < ntiles; n++) {
        const int st = n % S;
        prefetch_dout(n + 2);
        if (S == 2 && tid == 0 && n >= 1 && n + 1 < ntiles) {  // q stage of tile n-1 is free once its product is done
            if (!mbar_wait(&s.bar_mma[(n - 1) & 1], ((n - 1) >> 1) & 1, kPWait)) atomicCAS(err, 0, 2);
            load_q(n + 1);
        }
        // the stage is free once the product of tile n - S is done
        if (n >= S && !mbar_wait(&s.bar_mma[st], ((n - S) / S) & 1, kPWait)) atomicCAS(err, 0, 2);
        if (S == 1 && tid == 0 && n >= 1) load_q(n);
        // token row p of the tile: w dO, split
        const long long t = t_lo + (long long)n * kPT + p;
        float w = 0.f;
        if (t < t_hi) {
            const long long gi = (long long)bh * T + t;
            w = lam[gi * L + lev] * __expf((float)(Pb[t >> cbits] - Pref) + gamma[gi]);
        }
        const float4 *src = reinterpret_cast<const float4 *>(dout + ((long long)bh * T + (t < t_hi ? t : t_lo)) * kPDm);
        float4 av[8], cv[8];  // all of the half row's loads first
#pragma unroll
        for (int q8 = 0; q8 < 8; q8++) {
            const int ch = 8 * half + q8;
            av[q8] = cv[q8] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < t_hi) {
                av[q8] = src[2 * ch];
                cv[q8] = src[2 * ch + 1];
            }
        }
#pragma unroll
        for (int q8 = 0; q8 < 8; q8++) {
            const int ch = 8 * half + q8;
            const float4 a = av[q8], c = cv[q8];
            const float x[8] = {a.x * w, a.y * w, a.z * w, a.w * w, c.x * w, c.y * w, c.z * w, c.w * w};
            uint4 h, l;
            __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&h);
            __nv_bfloat162 *l2 = reinterpret_cast<__nv_bfloat162 *>(&l);
#pragma unroll
            for (int u = 0; u < 4; u++) {
                const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * u], x[2 * u + 1]);
                const float2 hf = __bfloat1622float2(hv);
                h2[u] = hv;
                l2[u] = __floats2bfloat162_rn(x[2 * u] - hf.x, x[2 * u + 1] - hf.y);
            }
            const uint32_t off = (ch >> 3) * kPH + sw128_offset(p, ch & 7);
            *reinterpret_cast<uint4 *>(s.b[st].hi + off) = h;
            *reinterpret_cast<uint4 *>(s.b[st].lo + off) = l;
        }
        fence_proxy_async_smem();
        if (!mbar_wait(&s.bar_load[st], (n / S) & 1, kPWait)) atomicCAS(err, 0, 1);
        __syncthreads();
        if (tid == 0) {
            tc_fence_after_sync();
#pragma unroll
            for (int kk = 0; kk < 8; kk++)
                umma_bf16(tm, desc_sw128(smem_u32(s.q[st]) + kk * 2048, kPH, 1024),
                          desc_sw128(smem_u32(s.b[st].hi) + kk * 2048, kPH, 1024), idesc, (n > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&s.bar_mma[st]);
        }
    }
    if (tid == 0) umma_commit(&s.bar_done);
    if (!mbar_wait(&s.bar_done, 0, kPWait)) atomicCAS(err, 0, 2);
    tc_fence_after_sync();
    // the piece through shared memory (64 KB from the first q stage on, free
    // once every product is done) and out as whole rows
    float *tile = reinterpret_cast<float *>(s.q[0]);
    const uint32_t lane_off = (uint32_t)((p >> 5) * 32) << 16;
#pragma unroll 1
    for (int cb = 64 * half; cb < 64 * half + 64; cb += 16) {
        float x[16], y[16];  // piece_hi + piece_lo
        tmem_ld16(tm + lane_off + cb, x);
        tmem_ld16(tm + lane_off + kPDm + cb, y);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 4; u++)
            *out_tile_piece(tile, p, cb / 4 + u) = make_float4(x[4 * u] + y[4 * u], x[4 * u + 1] + y[4 * u + 1],
                                                               x[4 * u + 2] + y[4 * u + 2], x[4 * u + 3] + y[4 * u + 3]);
    }
    __syncthreads();
    out_tile_store<kPThreads, false>(part + (((long long)bh * gridDim.x) + blockIdx.x) * kPDm * kPDm, tile, kPT);
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tm, 256);
}

}  // namespace

bool bwd_piece_tc_supported(const BwdArgs &A)
{
    return A.in_dt == LLA_BF16 && A.dk == kPDm && A.dv == kPDm && A.C == 64 && ((uintptr_t)A.q & 15) == 0 &&
           ((uintptr_t)A.dout & 15) == 0;
}

cudaError_t bwd_piece_tc(const BwdArgs &A, const float *gamma, const double *P, float *part, int nlev, int Pc,
                         int nitems, int *err)
{
    const int BH = A.B * A.H, N = A.T / A.C;
    CUtensorMap mq;
    if (!make_map_bf16_3d(&mq, A.q, kPDm, A.T, BH, 64, kPT)) return cudaErrorInvalidValue;
    constexpr int S = 1;
    const size_t smem = sizeof(PieceSmem<S>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd_piece_tc_kernel<S>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_piece_tc_kernel<S><<<dim3(nitems, BH), kPThreads, smem, (cudaStream_t)A.stream>>>(
        mq, A.dout, gamma, A.lam, P, part, A.T, N, A.L, ctz_u32((uint32_t)A.C), nlev, Pc, err);
    return cudaPeekAtLastError();
}

}  // namespace lla
