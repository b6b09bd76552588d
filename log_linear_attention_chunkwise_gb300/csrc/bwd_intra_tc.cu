// Intra-chunk part of the backward on the tensor cores (bf16 q, k, v;
// dk = dv = 128; chunk 64).  A CTA takes the pair of chunks (2p, 2p+1) as one
// 128-row tile; the pairs inside a chunk form the two diagonal 64 x 64
// blocks of the tile's 128 x 128 score matrices:
//     S = Q K^T,  dP = dO V^T,  M[t][s] = lambda_t[l(t,s)] exp(gamma_t - gamma_s)
//     (s <= t, same chunk; 0 elsewhere),
//     W1 = M . dP,  W2 = M . S,  dlambda_t[l] = sum_{s in bucket l} exp(..) S dP,
//     dq = W1 K,  dk = W1^T Q,  dv = W2^T dO.
// S and dP come from the tensor cores (dO, fp32, split into bf16 high and
// remainder parts); thread = row reads its chunk's 64 columns of both, forms
// W1, W2 and the level gradients in fp32, and writes W1 (then W2) split into
// bf16 parts; the products dq, dk (and dv) follow on the tensor cores, are
// read back by rows into a shared tile and written out as whole rows.  dq, dk,
// dv and dlambda rows are fully written here (the node and block-state parts
// add to them afterwards).
#include "bwd_simt.cuh"
#include "sm100.cuh"
#include "split_stage.cuh"
#include "tma_host.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kIT = 128;
constexpr int kID = 128;
constexpr uint32_t kIB = kIT * kID * 2;  // 32 KB
constexpr uint32_t kIH = kIB / 2;
constexpr int kIThreads = 256;  // two threads per tile row: each takes half of the row's chunk columns
constexpr uint32_t kIWait = 1u << 22;

struct __align__(1024) IntraSmem {
    uint8_t q[kIB], k[kIB];
    uint8_t ohi[kIB], olo[kIB];  // dO split
    uint8_t v[kIB];              // V, then the high part of W1 / W2
    uint8_t wmid[kIB], wlo[kIB]; // the second and third parts of W1 / W2
    float gam[kIT];              // in-chunk gate sums of the tile's rows
    uint64_t bar_load, bar_mma;
    uint32_t tmem;
};

// c ? x : y as a predicated select (never a branch)
__device__ __forceinline__ float selp_f(bool c, float x, float y)
{
    float r;
    asm("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %3, 0;\n\tselp.f32 %0, %1, %2, p;\n\t}"
        : "=f"(r)
        : "f"(x), "f"(y), "r"((uint32_t)c));
    return r;
}

// 8 MMAs over K = 128 with the given operand majors (A K-major or MN-major,
// B K-major or MN-major; K-major rows are 128 B, MN-major K rows are 128 B).
__device__ __forceinline__ void mma8x(uint32_t d, const uint8_t *a, bool a_mn, const uint8_t *b, bool b_mn,
                                      uint32_t idesc, bool acc)
{
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
        const uint32_t offk = (kk >> 2) * kIH + (kk & 3) * 32;  // K-major step
        const uint32_t offm = kk * 2048;                        // MN-major step
        const uint64_t ad = a_mn ? desc_sw128(smem_u32(a) + offm, kIH, 1024) : desc_sw128(smem_u32(a) + offk, 16, 1024);
        const uint64_t bd = b_mn ? desc_sw128(smem_u32(b) + offm, kIH, 1024) : desc_sw128(smem_u32(b) + offk, 16, 1024);
        umma_bf16(d, ad, bd, idesc, (acc || kk > 0) ? 1u : 0u);
    }
}

// 8 NCH fp32 values of row `row` at columns [c0, c0 + 8 NCH) of a 128-wide
// tile (c0 a multiple of 8, inside one 64-column block) in three bf16 parts
// (high, middle, low: about 24 bits together), 128-byte swizzle.
template <int NCH>
__device__ __forceinline__ void put_split_x3(uint8_t *hi, uint8_t *mid, uint8_t *lo, int row, int c0, const float *x)
{
#pragma unroll
    for (int ch = 0; ch < NCH; ch++) {
        uint4 h, m, l;
        __nv_bfloat162 *h2 = reinterpret_cast<__nv_bfloat162 *>(&h);
        __nv_bfloat162 *m2 = reinterpret_cast<__nv_bfloat162 *>(&m);
        __nv_bfloat162 *l2 = reinterpret_cast<__nv_bfloat162 *>(&l);
#pragma unroll
        for (int u = 0; u < 4; u++) {
            float a = x[8 * ch + 2 * u], b = x[8 * ch + 2 * u + 1];
            const __nv_bfloat162 hv = __floats2bfloat162_rn(a, b);
            float2 f = __bfloat1622float2(hv);
            a -= f.x;
            b -= f.y;
            const __nv_bfloat162 mv = __floats2bfloat162_rn(a, b);
            f = __bfloat1622float2(mv);
            h2[u] = hv;
            m2[u] = mv;
            l2[u] = __floats2bfloat162_rn(a - f.x, b - f.y);
        }
        const uint32_t off = (c0 >> 6) * kIH + sw128_offset(row, ((c0 & 63) >> 3) + ch);
        *reinterpret_cast<uint4 *>(hi + off) = h;
        *reinterpret_cast<uint4 *>(mid + off) = m;
        *reinterpret_cast<uint4 *>(lo + off) = l;
    }
}

// Zeros at columns [c0, c0 + 8 NCH) of row `row` in two tiles.
template <int NCH>
__device__ __forceinline__ void put_zero_x(uint8_t *a, uint8_t *b, int row, int c0)
{
    const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int ch = 0; ch < NCH; ch++) {
        const uint32_t off = (c0 >> 6) * kIH + sw128_offset(row, ((c0 & 63) >> 3) + ch);
        *reinterpret_cast<uint4 *>(a + off) = z;
        *reinterpret_cast<uint4 *>(b + off) = z;
    }
}

__global__ void __launch_bounds__(kIThreads, 1)
bwd_intra_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                    const __grid_constant__ CUtensorMap map_v, const float *__restrict__ dout,
                    const float *__restrict__ gamma, const float *__restrict__ lam, float *__restrict__ dq,
                    float *__restrict__ dk, float *__restrict__ dv, float *__restrict__ dlam, int T, int L,
                    const __nv_bfloat16 *__restrict__ q16, const __nv_bfloat16 *__restrict__ k16,
                    const __nv_bfloat16 *__restrict__ v16, int nsm, int *__restrict__ err)
{
    extern __shared__ uint8_t smem_raw[];
    IntraSmem &s = *reinterpret_cast<IntraSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int t = tid & (kIT - 1), hh = tid >> 7;  // tile row, half of the row's chunk columns
    const int pair = blockIdx.x, bh = blockIdx.y;
    const long long trow = (long long)pair * kIT + t;
    const bool row_ok = trow < T;
    const long long tok = (long long)bh * T + trow;
    const int cb = t & 64;         // first column of this row's chunk in the tile
    const int ch0 = cb + 32 * hh;  // first of this thread's 32 columns of it
    if (tid == 0) {
        mbar_init(&s.bar_load, 1);
        mbar_init(&s.bar_mma, 1);
        fence_mbar_init();
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        mbar_arrive_expect_tx(&s.bar_load, 3 * kIB);
        for (int h = 0; h < 2; h++) {
            tma_load_3d(s.q + h * kIH, &map_q, &s.bar_load, h * 64, pair * kIT, bh);
            tma_load_3d(s.k + h * kIH, &map_k, &s.bar_load, h * 64, pair * kIT, bh);
            tma_load_3d(s.v + h * kIH, &map_v, &s.bar_load, h * 64, pair * kIT, bh);
        }
    }
    if (tid < 32) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    // dO tile, split
    {
        uint8_t *d[2] = {s.ohi, s.olo};
        stage_split_tile<2, kIThreads, 8>(d, dout + ((long long)bh * T + (long long)pair * kIT) * kID, kID, nullptr, 1.f,
                            (int)min((long long)kIT, (long long)T - (long long)pair * kIT));
    }
    const float gam_t = row_ok ? gamma[tok] : 0.f;
    if (hh == 0) s.gam[t] = gam_t;
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;
    const uint32_t tS = tm, tP = tm + 128, tQ = tm, tK = tm + 128, tV = tm + 256;
    const uint32_t lane_off = (uint32_t)((t >> 5) * 32) << 16;
    const uint32_t id_kk = idesc_bf16_f32(128, 128, false, false);
    const uint32_t id_kmn = idesc_bf16_f32(128, 128, false, true);
    const uint32_t id_mnmn = idesc_bf16_f32(128, 128, true, true);
    if (!mbar_wait(&s.bar_load, 0, kIWait)) atomicCAS(err, 0, 1);
    if (tid == 0) {
        tc_fence_after_sync();
        mma8x(tS, s.q, false, s.k, false, id_kk, false);    // S = Q K^T
        mma8x(tP, s.ohi, false, s.v, false, id_kk, false);  // dP = dO V^T
        mma8x(tP, s.olo, false, s.v, false, id_kk, true);
        umma_commit(&s.bar_mma);
    }
    if (!mbar_wait(&s.bar_mma, 0, kIWait)) atomicCAS(err, 0, 2);
    if (tid == 0) {
        // this tile's inputs are in: the CTA that will run next on this SM (one
        // CTA per SM, launched in order) gets its q, k, v and dO rows into L2
        // while this one computes, instead of all CTAs of a wave loading at once
        const long long nxt = (long long)blockIdx.y * gridDim.x + blockIdx.x + nsm;
        if (nxt < (long long)gridDim.x * gridDim.y) {
            const long long r0 = (nxt % gridDim.x) * kIT, b2 = nxt / gridDim.x;
            const long long rows = min((long long)kIT, (long long)T - r0);
            const long long e0 = (b2 * T + r0) * kID;
            prefetch_l2(dout + e0, rows * kID * 4);
            prefetch_l2(q16 + e0, rows * kID * 2);
            prefetch_l2(k16 + e0, rows * kID * 2);
            prefetch_l2(v16 + e0, rows * kID * 2);
        }
    }
    tc_fence_after_sync();
    // this thread's 32 columns of the row's chunk block: W1, W2 and the level
    // gradients (partial sums; the two halves meet before dlambda is written)
    float w1[32], w2[32];
    float dl[7];
#pragma unroll
    for (int l = 0; l < 7; l++) dl[l] = 0.f;
    {
        const int a = t & 63;
        const float *lam_t = lam + tok * L;
        float lamv[7];
#pragma unroll
        for (int l = 0; l < 7; l++) lamv[l] = (row_ok && l < L) ? lam_t[l] : 0.f;
#pragma unroll
        for (int c0 = 0; c0 < 32; c0 += 16) {
            float sv[16], pv[16];
            tmem_ld16(tS + lane_off + ch0 + c0, sv);
            tmem_ld16(tP + lane_off + ch0 + c0, pv);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; e++) {
                // branch-free: the level varies over the lanes, and a register
                // array indexed by it (or a branch per level) serialises the warp
                const int b = 32 * hh + c0 + e;  // key column inside the chunk
                const bool ok = b <= a && row_ok;
                const float dec = __expf(fminf(gam_t - s.gam[cb + b], 0.f));
                const uint32_t x = (uint32_t)(a ^ b);  // level = bit_length(x)
                float lm = lamv[0];
                lm = selp_f(x >= 1u, lamv[1], lm);
                lm = selp_f(x >= 2u, lamv[2], lm);
                lm = selp_f(x >= 4u, lamv[3], lm);
                lm = selp_f(x >= 8u, lamv[4], lm);
                lm = selp_f(x >= 16u, lamv[5], lm);
                lm = selp_f(x >= 32u, lamv[6], lm);
                const float m = selp_f(ok, lm * dec, 0.f);
                w1[c0 + e] = m * pv[e];
                w2[c0 + e] = m * sv[e];
                const float ds = selp_f(ok, dec * sv[e], 0.f);
                const int lev = 32 - __clz((int)x);
#pragma unroll
                for (int l = 0; l < 7; l++) dl[l] = fmaf(selp_f(lev == l, ds, 0.f), pv[e], dl[l]);
            }
        }
    }
    tc_fence_before_sync();
    // W1 (three parts) into the (now free) V stage and the two part stages
    put_split_x3<4>(s.v, s.wmid, s.wlo, t, ch0, w1);
    put_zero_x<4>(s.v, s.wmid, t, ch0 ^ 64);
    put_zero_x<4>(s.wlo, s.wlo, t, ch0 ^ 64);
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after_sync();
        mma8x(tQ, s.v, false, s.k, true, id_kmn, false);    // dq = W1 K   (B = K, MN-major)
        mma8x(tQ, s.wmid, false, s.k, true, id_kmn, true);
        mma8x(tQ, s.wlo, false, s.k, true, id_kmn, true);
        mma8x(tK, s.v, true, s.q, true, id_mnmn, false);    // dk = W1^T Q (A = W1 read MN-major)
        mma8x(tK, s.wmid, true, s.q, true, id_mnmn, true);
        mma8x(tK, s.wlo, true, s.q, true, id_mnmn, true);
        umma_commit(&s.bar_mma);
    }
    if (!mbar_wait(&s.bar_mma, 1, kIWait)) atomicCAS(err, 0, 2);
    tc_fence_after_sync();
    // W2 replaces W1
    put_split_x3<4>(s.v, s.wmid, s.wlo, t, ch0, w2);
    put_zero_x<4>(s.v, s.wmid, t, ch0 ^ 64);
    put_zero_x<4>(s.wlo, s.wlo, t, ch0 ^ 64);
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after_sync();
        mma8x(tV, s.v, true, s.ohi, true, id_mnmn, false);  // dv = W2^T dO
        mma8x(tV, s.v, true, s.olo, true, id_mnmn, true);
        mma8x(tV, s.wmid, true, s.ohi, true, id_mnmn, true);
        mma8x(tV, s.wlo, true, s.ohi, true, id_mnmn, true);
        umma_commit(&s.bar_mma);
    }
    // dq, dk while dv runs, then dv: each through shared memory (the q and k
    // stages, which no product reads any more) and out as whole rows.  The
    // tensor-memory loads are warp-collective: every lane issues them.
    float *tile = reinterpret_cast<float *>(s.q);
    const int nrows = (int)min((long long)kIT, (long long)T - (long long)pair * kIT);
    const long long row0 = (long long)bh * T + (long long)pair * kIT;
    auto put = [&](uint32_t src) {  // row t, columns [64 hh, 64 hh + 64)
#pragma unroll 1
        for (int c0 = 64 * hh; c0 < 64 * hh + 64; c0 += 16) {
            float x[16];
            tmem_ld16(src + lane_off + c0, x);
            tmem_ld_wait();
#pragma unroll
            for (int u = 0; u < 4; u++)
                *out_tile_piece(tile, t, c0 / 4 + u) = make_float4(x[4 * u], x[4 * u + 1], x[4 * u + 2], x[4 * u + 3]);
        }
    };
    for (int o = 0; o < 2; o++) {
        put(o == 0 ? tQ : tK);
        __syncthreads();
        out_tile_store<kIThreads, false>((o == 0 ? dq : dk) + row0 * kID, tile, nrows);
        __syncthreads();
    }
    // the level gradients: the second half's partial sums through the (free) tile
    if (hh == 1)
#pragma unroll
        for (int l = 0; l < 7; l++) tile[t * 8 + l] = dl[l];
    __syncthreads();
    if (hh == 0 && row_ok) {
        float *dlr = dlam + tok * L;
        for (int l = 0; l < L; l++) dlr[l] = l < 7 ? dl[l] + tile[t * 8 + l] : 0.f;
    }
    __syncthreads();  // the tile is staged again below
    if (!mbar_wait(&s.bar_mma, 0, kIWait)) atomicCAS(err, 0, 2);
    tc_fence_after_sync();
    put(tV);
    __syncthreads();
    out_tile_store<kIThreads, false>(dv + row0 * kID, tile, nrows);
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tm, 512);
}

}  // namespace

bool bwd_intra_tc_supported(const BwdArgs &A)
{
    return A.in_dt == LLA_BF16 && A.dk == kID && A.dv == kID && A.C == 64 && ((uintptr_t)A.q & 15) == 0 &&
           ((uintptr_t)A.k & 15) == 0 && ((uintptr_t)A.v & 15) == 0 && ((uintptr_t)A.dout & 15) == 0 &&
           ((uintptr_t)A.dq & 15) == 0 && ((uintptr_t)A.dkey & 15) == 0 && ((uintptr_t)A.dval & 15) == 0;
}

cudaError_t bwd_intra_tc(const BwdArgs &A, const float *gamma, int *err)
{
    const int BH = A.B * A.H;
    CUtensorMap mq, mk, mv;
    if (!make_map_bf16_3d(&mq, A.q, kID, A.T, BH, 64, kIT) || !make_map_bf16_3d(&mk, A.k, kID, A.T, BH, 64, kIT) ||
        !make_map_bf16_3d(&mv, A.v, kID, A.T, BH, 64, kIT))
        return cudaErrorInvalidValue;
    const size_t smem = sizeof(IntraSmem) + 1024;
    cudaError_t e = cudaFuncSetAttribute(bwd_intra_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    bwd_intra_tc_kernel<<<dim3((A.T + kIT - 1) / kIT, BH), kIThreads, smem, (cudaStream_t)A.stream>>>(
        mq, mk, mv, A.dout, gamma, A.lam, A.dq, A.dkey, A.dval, A.dlam, A.T, A.L, (const __nv_bfloat16 *)A.q,
        (const __nv_bfloat16 *)A.k, (const __nv_bfloat16 *)A.v, bwd_sm_count(), err);
    return cudaPeekAtLastError();
}

}  // namespace lla
