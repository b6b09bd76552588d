// Key side of the backward on the tensor cores (bf16 k, v; dk = dv = 128;
// chunk 64).
//
// For chunk i and level m with bit m of i clear, the later chunks of block
// b = (i >> m) + 1 contribute  dk_s += f_s R_{m,b} v_s,  dv_s += f_s R_{m,b}^T k_s
// with f_s = exp(G_ref - G_s), ref = the last token before the block (see the
// CUDA-core backward).  A CTA takes the pair of chunks (2p, 2p+1) as one
// 128-row tile.  For m >= 1 both chunks see the same block, and
// f_s = c_m rho_s with c_m = exp(P_{b 2^m} - P_{2p+2}) (block start to pair
// end) and rho_s = exp(P_{2p+2} - G_s) (token to pair end), both <= 1, so
// c_m R_m is staged per level and every level accumulates into one pair of
// tensor-memory accumulators:  dK = rho . sum_m V (c_m R_m)^T,
// dV = rho . sum_m K (c_m R_m).  Level 0 concerns chunk 2p alone (its block
// is chunk 2p+1) and goes to a second pair of accumulators, weighted by f_s
// for the first 64 rows and 0 for the others.  R is fp32: each staged
// c_m R_m is split into a bf16 high part and a bf16 remainder, and both are
// multiplied (k and v are exact in bf16), so the products keep about 16
// bits.  The staged R serves as the K-major B operand of the dk product and
// the MN-major B operand of the dv product.  Results are added to dk, dv.
#include "bwd_simt.cuh"
#include "sm100.cuh"
#include "split_stage.cuh"
#include "tma_host.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kKT = 128;                      // tile rows (two chunks of 64)
constexpr int kKD = 128;                      // dk = dv
constexpr uint32_t kKBuf = kKT * kKD * 2;     // bf16 128 x 128: 32 KB
constexpr uint32_t kKHalf = kKBuf / 2;
constexpr int kKThreads = 256;  // staging: twice the loads in flight; drain: a row's two column halves
constexpr int kKAllThreads = kKThreads + 32;  // plus one warp whose lane 0 issues the products
constexpr uint32_t kKWait = 1u << 22;

struct __align__(1024) KeySmem {
    uint8_t k[kKBuf];
    uint8_t v[kKBuf];
    uint8_t rhi[2][kKBuf];
    uint8_t rlo[2][kKBuf];
    uint64_t bar_load, bar_mma[2], bar_done, bar_staged[2];
    uint32_t tmem;
};

__device__ __forceinline__ void work_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

__device__ __forceinline__ void key_err(int *err, int code) { atomicCAS(err, 0, code); }

// 8 MMAs over K = 128, A K-major; B K-major (kmaj) or MN-major.
__device__ __forceinline__ void mma8(uint32_t d, const uint8_t *a, const uint8_t *b, uint32_t idesc, bool b_kmaj,
                                     bool acc)
{
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
        const uint32_t offa = (kk >> 2) * kKHalf + (kk & 3) * 32;
        const uint64_t bd = b_kmaj ? desc_sw128(smem_u32(b) + offa, 16, 1024)
                                   : desc_sw128(smem_u32(b) + kk * 2048, kKHalf, 1024);
        umma_bf16(d, desc_sw128(smem_u32(a) + offa, 16, 1024), bd, idesc, (acc || kk > 0) ? 1u : 0u);
    }
}

__global__ void __launch_bounds__(kKAllThreads, 1)
bwd_key_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  const float *__restrict__ gamma, const double *__restrict__ P, const float *__restrict__ R,
                  const float *__restrict__ part, float *__restrict__ dk, float *__restrict__ dv, int T, int N,
                  int nlev, int nblocks, int Pc, int nitems, int *__restrict__ err)
{
    extern __shared__ uint8_t smem_raw[];
    KeySmem &s = *reinterpret_cast<KeySmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int p = tid & 127, half = tid >> 7;  // tile row, column half of the drain
    const int pair = blockIdx.x;
    const int bh = blockIdx.y;
    const int c0 = 2 * pair;                 // first chunk of the pair
    const int pend = min(N, c0 + 2);         // chunk index after the pair
    const double *Pb = P + (long long)bh * (N + 1);
    // levels of the pair: m >= 1 shared, m = 0 only for chunk c0
    bool lev0 = (c0 + 1) < N;
    int levs[24];
    int nl = 0;
    for (int m = 1; m < nlev; m++)
        if (((c0 >> m) & 1) == 0 && (((long long)(c0 >> m) + 1) << m) < N) levs[nl++] = m;
    if (!lev0 && nl == 0) return;
    if (tid == 0) {
        mbar_init(&s.bar_load, 1);
        mbar_init(&s.bar_mma[0], 1);
        mbar_init(&s.bar_mma[1], 1);
        mbar_init(&s.bar_done, 1);
        mbar_init(&s.bar_staged[0], kKThreads);
        mbar_init(&s.bar_staged[1], kKThreads);
        fence_mbar_init();
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        mbar_arrive_expect_tx(&s.bar_load, 2 * kKBuf);
        for (int h = 0; h < 2; h++) {
            tma_load_3d(s.k + h * kKHalf, &map_k, &s.bar_load, h * 64, pair * kKT, bh);
            tma_load_3d(s.v + h * kKHalf, &map_v, &s.bar_load, h * 64, pair * kKT, bh);
        }
    }
    if (tid < 32) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;
    const uint32_t acc_k = tm, acc_v = tm + 128, acc_k0 = tm + 256, acc_v0 = tm + 384;
    const uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_kmn = idesc_bf16_f32(128, 128, false, true);
    const double Pend = Pb[pend];
    // stage c * R (fp32 [128][128]) as bf16 high and remainder parts, 128-byte swizzled
    auto stage = [&](int buf, const float *Rm, float c) {
        uint8_t *dst[2] = {s.rhi[buf], s.rlo[buf]};
        stage_split_tile<2, kKThreads, 8>(dst, Rm, kKD, nullptr, c, kKD);
    };
    // the level sequence: level 0 first (if any), then the shared levels
    const int total = (lev0 ? 1 : 0) + nl;
    auto level_of = [&](int n) { return (lev0 && n == 0) ? 0 : levs[n - (lev0 ? 1 : 0)]; };
    // the block states are read from DRAM: each is prefetched into L2 two
    // levels before it is staged
    auto prefetch_state = [&](int n) {
        if (tid == 0 && n < total) {
            const int m = level_of(n);
            const float *src = block_state(R, part, bh, m, (c0 >> m) + 1, N, Pc, nitems, nblocks, kKD * kKD);
            bulk_prefetch_l2(src, kKD * kKD * 2);
            bulk_prefetch_l2(src + kKD * kKD / 2, kKD * kKD * 2);
        }
    };
    prefetch_state(0);
    prefetch_state(1);
    // The 256 staging threads stage level n into buffer n & 1 and signal it;
    // one thread of the extra warp issues its products, so no staging thread
    // waits for the issue.
    if (tid >= kKThreads) {
        if (tid == kKThreads) {
            bool acc_started = false;
            if (!mbar_wait(&s.bar_load, 0, kKWait)) key_err(err, 1);
            for (int n = 0; n < total; n++) {
                const int buf = n & 1;
                const bool is0 = lev0 && n == 0;
                if (!mbar_wait(&s.bar_staged[buf], (n >> 1) & 1, kKWait)) key_err(err, 2);
                tc_fence_after_sync();
                const uint32_t dk_acc = is0 ? acc_k0 : acc_k, dv_acc = is0 ? acc_v0 : acc_v;
                const bool acc = is0 ? false : acc_started;
                mma8(dk_acc, s.v, s.rhi[buf], id_kk, true, acc);
                mma8(dk_acc, s.v, s.rlo[buf], id_kk, true, true);
                mma8(dv_acc, s.k, s.rhi[buf], id_kmn, false, acc);
                mma8(dv_acc, s.k, s.rlo[buf], id_kmn, false, true);
                umma_commit(&s.bar_mma[buf]);
                if (!is0) acc_started = true;
            }
            umma_commit(&s.bar_done);
        }
    } else {
    for (int n = 0; n < total; n++) {
        const int buf = n & 1;
        const bool is0 = lev0 && n == 0;
        const int m = level_of(n);
        const int b = (c0 >> m) + 1;
        prefetch_state(n + 2);
        const float *Rm = block_state(R, part, bh, m, b, N, Pc, nitems, nblocks, kKD * kKD);
        const float c = is0 ? 1.f : expf((float)(Pb[b << m] - Pend));
        if (n >= 2 && !mbar_wait(&s.bar_mma[buf], ((n - 2) >> 1) & 1, kKWait)) key_err(err, 2);
        stage(buf, Rm, c);
        fence_proxy_async_smem();
        mbar_arrive(&s.bar_staged[buf]);
    }
    if (!mbar_wait(&s.bar_done, 0, kKWait)) key_err(err, 2);
    tc_fence_after_sync();
    // drain: row p; weights rho (shared levels) and f0 (level 0, first chunk)
    const long long row = (long long)pair * kKT + p;
    const int chunk = c0 + (p >> 6);
    const float gam = (row < T) ? gamma[(long long)bh * T + row] : 0.f;
    const double Gs = Pb[min(chunk, N)] + (double)gam;
    const float rho = (row < T) ? expf((float)(Pend - Gs)) : 0.f;
    const float f0 = (lev0 && p < 64) ? expf((float)(Pb[c0 + 1] - Gs)) : 0.f;
    const uint32_t lane_off = (uint32_t)((p >> 5) * 32) << 16;
    const bool have_shared = nl > 0;
    // each result through shared memory (the k and v stages, free once every
    // product is done) and added to dk, dv as whole rows
    float *tile = reinterpret_cast<float *>(s.k);
    const int nrows = (int)min((long long)kKT, (long long)T - (long long)pair * kKT);
    for (int which = 0; which < 2; which++) {
        const uint32_t a_sh = which == 0 ? acc_k : acc_v, a_0 = which == 0 ? acc_k0 : acc_v0;
#pragma unroll 1
        for (int cb = half * 64; cb < half * 64 + 64; cb += 16) {
            float x[16], y[16];
            tmem_ld16(a_sh + lane_off + cb, x);
            tmem_ld16(a_0 + lane_off + cb, y);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 4; u++) {
                // an accumulator no level wrote holds no data: select, do not scale
                float a[4];
#pragma unroll
                for (int e = 0; e < 4; e++)
                    a[e] = (have_shared ? rho * x[4 * u + e] : 0.f) + (lev0 ? f0 * y[4 * u + e] : 0.f);
                *out_tile_piece(tile, p, cb / 4 + u) = make_float4(a[0], a[1], a[2], a[3]);
            }
        }
        work_sync();
        out_tile_store<kKThreads, true>((which == 0 ? dk : dv) + ((long long)bh * T + (long long)pair * kKT) * kKD,
                                        tile, nrows);
        work_sync();
    }
    }  // staging threads
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tm, 512);
}

}  // namespace

bool bwd_key_tc_supported(const BwdArgs &A)
{
    return A.in_dt == LLA_BF16 && A.dk == kKD && A.dv == kKD && A.C == 64 && ((uintptr_t)A.k & 15) == 0 &&
           ((uintptr_t)A.v & 15) == 0 && ((uintptr_t)A.dkey & 15) == 0 && ((uintptr_t)A.dval & 15) == 0;
}

cudaError_t bwd_key_tc(const BwdArgs &A, const float *gamma, const double *P, const float *R, const float *part,
                       int nlev, int nblocks, int Pc, int nitems, int *err)
{
    const int BH = A.B * A.H, N = A.T / A.C;
    CUtensorMap mk, mv;
    if (!make_map_bf16_3d(&mk, A.k, kKD, A.T, BH, 64, kKT) || !make_map_bf16_3d(&mv, A.v, kKD, A.T, BH, 64, kKT))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(KeySmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd_key_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_key_tc_kernel<<<dim3((N + 1) / 2, BH), kKAllThreads, smem, (cudaStream_t)A.stream>>>(
        mk, mv, gamma, P, R, part, A.dkey, A.dval, A.T, N, nlev, nblocks, Pc, nitems, err);
    return cudaPeekAtLastError();
}

}  // namespace lla
