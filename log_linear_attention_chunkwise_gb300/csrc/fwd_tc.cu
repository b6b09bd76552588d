// Chunked forward on the 5th-generation tensor cores (tcgen05, TMEM, TMA),
// bf16 q/k/v with fp32 accumulation, dk = dv = 128.
//
// Page "Log-Linear Attention" (gist.science 2506.04761), technical summary
// §2.2 (Fenwick buckets of [0,t), one state per bucket, lambda-weighted
// read-out) and §2.3 (the hierarchical mask computed chunkwise with matmuls).
//
// One CTA handles one tile of 128 tokens of one (batch, head); tiles are
// taken from a global ticket counter in (batch*head, tile) order, so a tile
// only ever waits on tiles that started before it.  With Gam_i the gate sum
// of tile i and P_i = Gam_0 + ... + Gam_{i-1} (fp64, from the prefix kernel),
// the earlier tiles of tile i form the tile-level Fenwick buckets ending at
// j = i, i - lowbit(i), ...; bucket j (level m = ctz(j)) holds the tiles
// [j - 2^m, j) decayed to the end of tile j-1:
//     Node_j = sum over those tiles' keys s of exp(P_j - G_s) k_s v_s^T.
// A key s of bucket j has level 7 + 1 + m for every query of tile i.
// Per tile:
//   S  = Q K^T                              (tcgen05, TMEM)
//   H  = K^T diag(exp(Gam - gamma)) V        (tcgen05, TMEM) -> Node_{i+1}
//        Node_{i+1} = H + sum_{m < ctz(i+1)} exp(P_{i+1} - P_{j_m}) Node_{j_m},
//        j_m = i + 1 - 2^m, published to global memory (fp32 + bf16 copy)
//   P  = S . M,  M[a][b] = lambda_a[bit_length(a^b)] exp(gamma_a - gamma_b), b <= a
//   O  = P V + sum_{path j} diag(lambda_.[8+m] exp(gamma_. + P_i - P_j)) Q Node_j
// Every product above is a tcgen05 MMA of M = N = 128, bf16 operands in
// 128-byte-swizzled shared memory, fp32 accumulators in tensor memory.
#include "fwd_tc.cuh"
#include "sm100.cuh"
#include "tma_host.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kTile = 128;       // tokens per tile (MMA M)
constexpr int kD = 128;          // dk = dv
constexpr int kTileLevels = 7;   // levels inside a tile: bit_length(a ^ b) <= 7
constexpr int kThreads = 128;
constexpr uint32_t kBuf = kTile * kD * 2;  // one bf16 128x128 operand: 32 KB
constexpr uint32_t kHalf = kBuf / 2;       // one 64-column swizzled block
constexpr uint32_t kWaitIters = 1u << 22;  // bounded waits (~0.5 s with back-off)
constexpr int kLamLd = 9;                  // padded row of the in-tile lambdas

// Error codes written to the workspace error word.
constexpr int kErrLoadTimeout = 1;
constexpr int kErrMmaTimeout = 2;
constexpr int kErrNodeTimeout = 3;

struct __align__(1024) TcSmem {
    uint8_t q[kBuf];
    uint8_t k[kBuf];
    uint8_t v[kBuf];
    uint8_t vs[kBuf];
    uint8_t p[kBuf];
    float gam[kTile];
    float lam[kTile * kLamLd];
    float wsum[4];
    uint64_t bar_load, bar_mma, bar_node[2], bar_stage[2], bar_done;
    uint32_t tmem;
    int ticket;
};

struct TcParams {
    const float *g, *lam;
    void *out;
    const double *P;   // [BH][NT+1]
    int *flags;        // [BH][NT+1]
    int *ticket;
    int *err;
    float *node32;     // [BH][NT][128][128]
    __nv_bfloat16 *node16;
    int T, NT, BH, L;
};

__device__ __forceinline__ void set_err(int *err, int code) { atomicCAS(err, 0, code); }

// Acquire-load of a publication flag, bounded.
__device__ __forceinline__ bool wait_flag(const int *flag, uint32_t max_iter)
{
    for (uint32_t it = 0; it < max_iter; it++) {
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v != 0) return true;
        __nanosleep(it < 32 ? 32 : 256);
    }
    return false;
}

__device__ __forceinline__ void release_flag(int *flag)
{
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(flag), "r"(1) : "memory");
}

// Row `row` of a 128x128 bf16 operand stored as two 64-column 128B-swizzled
// blocks: scale every element by w and write to the same place in dst.
__device__ __forceinline__ void scale_row(const uint8_t *src, uint8_t *dst, int row, float w)
{
#pragma unroll
    for (int blk = 0; blk < 2; blk++) {
#pragma unroll
        for (int c = 0; c < 8; c++) {
            const uint32_t off = blk * kHalf + row * 128 + c * 16;
            uint4 raw = *reinterpret_cast<const uint4 *>(src + off);
            __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&raw);
#pragma unroll
            for (int u = 0; u < 4; u++) {
                float2 f = __bfloat1622float2(h[u]);
                h[u] = __floats2bfloat162_rn(f.x * w, f.y * w);
            }
            *reinterpret_cast<uint4 *>(dst + off) = raw;
        }
    }
}

// 8 MMAs over K = 128: A and B K-major (rows of 128 B, K split in two blocks).
__device__ __forceinline__ void mma_kk(uint32_t d, const uint8_t *a, const uint8_t *b, uint32_t idesc,
                                       bool accumulate)
{
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
        const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
        umma_bf16(d, desc_sw128(smem_u32(a) + off, 16, 1024), desc_sw128(smem_u32(b) + off, 16, 1024),
                  idesc, (accumulate || kk > 0) ? 1u : 0u);
    }
}

// 8 MMAs over K = 128 with A K-major and B MN-major (rows = K index).
__device__ __forceinline__ void mma_kmn(uint32_t d, const uint8_t *a, const uint8_t *b, uint32_t idesc,
                                        bool accumulate)
{
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
        const uint32_t offa = (kk >> 2) * kHalf + (kk & 3) * 32;
        const uint32_t offb = kk * 2048;
        umma_bf16(d, desc_sw128(smem_u32(a) + offa, 16, 1024),
                  desc_sw128(smem_u32(b) + offb, kHalf, 1024), idesc,
                  (accumulate || kk > 0) ? 1u : 0u);
    }
}

// 8 MMAs over K = 128 with A and B MN-major (rows = K index).
__device__ __forceinline__ void mma_mnmn(uint32_t d, const uint8_t *a, const uint8_t *b,
                                         uint32_t idesc)
{
#pragma unroll
    for (int kk = 0; kk < 8; kk++) {
        const uint32_t off = kk * 2048;
        umma_bf16(d, desc_sw128(smem_u32(a) + off, kHalf, 1024),
                  desc_sw128(smem_u32(b) + off, kHalf, 1024), idesc, kk > 0 ? 1u : 0u);
    }
}

template <typename OutT>
__device__ __forceinline__ void store_out16(OutT *dst, const float (&r)[16]);

template <>
__device__ __forceinline__ void store_out16<float>(float *dst, const float (&r)[16])
{
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int u = 0; u < 4; u++) d4[u] = make_float4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
}

template <>
__device__ __forceinline__ void store_out16<__nv_bfloat16>(__nv_bfloat16 *dst, const float (&r)[16])
{
    uint4 w[2];
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(w);
#pragma unroll
    for (int u = 0; u < 8; u++) h[u] = __floats2bfloat162_rn(r[2 * u], r[2 * u + 1]);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    d4[0] = w[0];
    d4[1] = w[1];
}

template <typename OutT>
__global__ void __launch_bounds__(kThreads, 1)
lla_fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                  const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_node,
                  const TcParams prm)
{
    extern __shared__ uint8_t smem_raw[];
    TcSmem &s = *reinterpret_cast<TcSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                            ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;

    if (tid == 0) {
        mbar_init(&s.bar_load, 1);
        mbar_init(&s.bar_mma, 1);
        mbar_init(&s.bar_node[0], 1);
        mbar_init(&s.bar_node[1], 1);
        mbar_init(&s.bar_stage[0], 1);
        mbar_init(&s.bar_stage[1], 1);
        mbar_init(&s.bar_done, 1);
        fence_mbar_init();
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        tma_prefetch_map(&map_node);
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    // The ticket is taken only once this CTA holds its tensor memory, so a
    // tile with a ticket never waits on a CTA that cannot make progress.
    if (tid == 0) s.ticket = atomicAdd(prm.ticket, 1);
    __syncthreads();
    const uint32_t tm = s.tmem;
    const uint32_t tm_S = tm, tm_H = tm + 128, tm_O = tm + 256;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

    const int NT = prm.NT;
    const int ticket = s.ticket;
    const int bh = ticket / NT;
    const int i = ticket - bh * NT;
    const int tile_rows = min(kTile, prm.T - i * kTile);
    const bool has_node = i < NT - 1;  // the last tile starts no node
    const long long tok = (long long)bh * prm.T + (long long)i * kTile + tid;
    const double *Pb = prm.P + (long long)bh * (NT + 1);
    int *flags = prm.flags + (long long)bh * (NT + 1);

    // ---- loads: Q, K, V by TMA; gates and in-tile lambdas by the threads
    if (tid == 0) {
        mbar_arrive_expect_tx(&s.bar_load, 3 * kBuf);
#pragma unroll
        for (int h = 0; h < 2; h++) {
            tma_load_3d(s.q + h * kHalf, &map_q, &s.bar_load, h * 64, i * kTile, bh);
            tma_load_3d(s.k + h * kHalf, &map_k, &s.bar_load, h * 64, i * kTile, bh);
            tma_load_3d(s.v + h * kHalf, &map_v, &s.bar_load, h * 64, i * kTile, bh);
        }
    }
    const bool row_ok = tid < tile_rows;
    const float gv = row_ok ? prm.g[tok] : 0.f;
    const float *lam_row = prm.lam + tok * prm.L;
#pragma unroll
    for (int l = 0; l <= kTileLevels; l++)
        s.lam[tid * kLamLd + l] = (row_ok && l < prm.L) ? lam_row[l] : 0.f;
    // inclusive running sum of the gates over the tile
    float incl = gv;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, off);
        if ((tid & 31) >= off) incl += y;
    }
    if ((tid & 31) == 31) s.wsum[warp] = incl;
    __syncthreads();
    float base = 0.f;
    for (int w = 0; w < warp; w++) base += s.wsum[w];
    const float gam_a = base + incl;
    s.gam[tid] = gam_a;
    const float Gam = s.wsum[0] + s.wsum[1] + s.wsum[2] + s.wsum[3];

    if (!mbar_wait(&s.bar_load, 0, kWaitIters)) set_err(prm.err, kErrLoadTimeout);
    // V scaled by exp(Gam - gamma_s), row s = this thread's token
    if (has_node) scale_row(s.v, s.vs, tid, __expf(Gam - gam_a));
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();

    // ---- S = Q K^T and H = K^T Vs
    if (tid == 0) {
        tc_fence_after_sync();
        mma_kk(tm_S, s.q, s.k, idesc_bf16_f32(128, 128, false, false), false);
        if (has_node) mma_mnmn(tm_H, s.k, s.vs, idesc_bf16_f32(128, 128, true, true));
        umma_commit(&s.bar_mma);
    }
    if (!mbar_wait(&s.bar_mma, 0, kWaitIters)) set_err(prm.err, kErrMmaTimeout);
    tc_fence_after_sync();

    // ---- Node_{i+1} = H + decayed lower-level path nodes; thread = dk row
    if (has_node) {
        const int z = __ffs(i + 1) - 1;  // ctz(i+1)
        const double Pn = Pb[i + 1];
        float fac[24];
#pragma unroll
        for (int m = 0; m < 24; m++) fac[m] = 0.f;
        for (int m = 0; m < z; m++) {
            const int j = i + 1 - (1 << m);
            if (tid == 0 && !wait_flag(flags + j, kWaitIters)) set_err(prm.err, kErrNodeTimeout);
        }
        __syncthreads();
#pragma unroll
        for (int m = 0; m < 24; m++)
            if (m < z) fac[m] = __expf((float)(Pn - Pb[i + 1 - (1 << m)]));
        const long long nbase = ((long long)bh * NT) * (kD * kD);
        float *dst32 = prm.node32 + nbase + (long long)(i + 1) * kD * kD + tid * kD;
        __nv_bfloat16 *dst16 = prm.node16 + nbase + (long long)(i + 1) * kD * kD + tid * kD;
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 16) {
            float r[16];
            tmem_ld16(tm_H + lane_off + c0, r);
            tmem_ld_wait();
            for (int m = 0; m < z; m++) {
                const float4 *src = reinterpret_cast<const float4 *>(
                    prm.node32 + nbase + (long long)(i + 1 - (1 << m)) * kD * kD + tid * kD + c0);
                const float f = fac[m];
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    float4 x = __ldcg(src + u);
                    r[4 * u] = fmaf(f, x.x, r[4 * u]);
                    r[4 * u + 1] = fmaf(f, x.y, r[4 * u + 1]);
                    r[4 * u + 2] = fmaf(f, x.z, r[4 * u + 2]);
                    r[4 * u + 3] = fmaf(f, x.w, r[4 * u + 3]);
                }
            }
            float4 *d4 = reinterpret_cast<float4 *>(dst32 + c0);
#pragma unroll
            for (int u = 0; u < 4; u++) __stcg(d4 + u, make_float4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]));
            uint4 w[2];
            __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(w);
#pragma unroll
            for (int u = 0; u < 8; u++) h[u] = __floats2bfloat162_rn(r[2 * u], r[2 * u + 1]);
            __stcg(reinterpret_cast<uint4 *>(dst16 + c0), w[0]);
            __stcg(reinterpret_cast<uint4 *>(dst16 + c0) + 1, w[1]);
        }
        fence_proxy_async_global();  // the bf16 copy is read by other CTAs' TMA
        __threadfence();
        __syncthreads();
        if (tid == 0) release_flag(flags + i + 1);
    }

    // ---- P = S . M  (thread = query row a), bf16 into the K-major buffer
    {
        const int a = tid;
        const float *lam_a = s.lam + a * kLamLd;
#pragma unroll 1
        for (int c0 = 0; c0 < kTile; c0 += 16) {
            float r[16];
            tmem_ld16(tm_S + lane_off + c0, r);
            tmem_ld_wait();
            uint4 w[2];
            __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(w);
#pragma unroll
            for (int u = 0; u < 8; u++) {
                float x[2];
#pragma unroll
                for (int e = 0; e < 2; e++) {
                    const int b = c0 + 2 * u + e;
                    x[e] = 0.f;
                    if (b <= a && row_ok) {
                        const int lev = 32 - __clz(a ^ b);
                        x[e] = r[2 * u + e] * lam_a[lev] * __expf(gam_a - s.gam[b]);
                    }
                }
                h[u] = __floats2bfloat162_rn(x[0], x[1]);
            }
            const int blk = c0 >> 6;
            const int ch = (c0 & 63) >> 3;
            *reinterpret_cast<uint4 *>(s.p + blk * kHalf + sw128_offset(a, ch)) = w[0];
            *reinterpret_cast<uint4 *>(s.p + blk * kHalf + sw128_offset(a, ch + 1)) = w[1];
        }
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after_sync();
        mma_kmn(tm_O, s.p, s.v, idesc_bf16_f32(128, 128, false, true), false);
        umma_commit(&s.bar_mma);
    }

    // ---- read-out: O += (w_m . Q) Node_j over the tile-level Fenwick path
    // stage 0 uses the K / Vs buffers (free once S and H are done), stage 1
    // the P / V buffers (free once P V is done).
    uint8_t *wq_buf[2] = {s.k, s.p};
    uint8_t *nd_buf[2] = {s.vs, s.v};
    int n = 0;
    for (int j = i; j > 0; j -= (j & -j), n++) {
        const int st = n & 1;
        const int m = __ffs(j) - 1;
        const int lev = kTileLevels + 1 + m;
        if (n == 1) {
            if (!mbar_wait(&s.bar_mma, 1, kWaitIters)) set_err(prm.err, kErrMmaTimeout);
        } else if (n >= 2) {
            if (!mbar_wait(&s.bar_stage[st], ((n - 2) >> 1) & 1, kWaitIters))
                set_err(prm.err, kErrMmaTimeout);
        }
        tc_fence_after_sync();
        if (tid == 0) {
            if (!wait_flag(flags + j, kWaitIters)) set_err(prm.err, kErrNodeTimeout);
            fence_proxy_async_global();
            mbar_arrive_expect_tx(&s.bar_node[st], kBuf);
            tma_load_3d(nd_buf[st], &map_node, &s.bar_node[st], 0, 0, bh * NT + j);
            tma_load_3d(nd_buf[st] + kHalf, &map_node, &s.bar_node[st], 64, 0, bh * NT + j);
        }
        const float wl = row_ok ? lam_row[lev] * __expf(gam_a + (float)(Pb[i] - Pb[j])) : 0.f;
        scale_row(s.q, wq_buf[st], tid, wl);
        fence_proxy_async_smem();
        tc_fence_before_sync();
        __syncthreads();
        if (tid == 0) {
            if (!mbar_wait(&s.bar_node[st], (n >> 1) & 1, kWaitIters)) set_err(prm.err, kErrLoadTimeout);
            tc_fence_after_sync();
            mma_kmn(tm_O, wq_buf[st], nd_buf[st], idesc_bf16_f32(128, 128, false, true), true);
            umma_commit(&s.bar_stage[st]);
        }
    }
    if (tid == 0) umma_commit(&s.bar_done);
    if (!mbar_wait(&s.bar_done, 0, kWaitIters)) set_err(prm.err, kErrMmaTimeout);
    tc_fence_after_sync();

    // ---- O epilogue: thread = output row
    if (row_ok) {
        OutT *dst = reinterpret_cast<OutT *>(prm.out) + tok * kD;
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 16) {
            float r[16];
            tmem_ld16(tm_O + lane_off + c0, r);
            tmem_ld_wait();
            store_out16<OutT>(dst + c0, r);
        }
    } else {
        // keep every warp's tcgen05.ld collective: rows past T load and drop
#pragma unroll 1
        for (int c0 = 0; c0 < kD; c0 += 16) {
            float r[16];
            tmem_ld16(tm_O + lane_off + c0, r);
            tmem_ld_wait();
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// Per (batch*head): Gam_i of every tile in fp64, P_i = prefix sums, and the
// publication flags and ticket reset for the main kernel.
__global__ void __launch_bounds__(256)
lla_tile_gate_prefix_kernel(const float *__restrict__ g, double *__restrict__ P, int *__restrict__ flags,
                            int *__restrict__ ticket, int *__restrict__ err, int T, int NT)
{
    __shared__ double part[256];
    const long long bh = blockIdx.x;
    const float *gb = g + bh * (long long)T;
    double *Pb = P + bh * (long long)(NT + 1);
    int *fb = flags + bh * (long long)(NT + 1);
    double carry = 0.0;
    for (int t0 = 0; t0 < NT; t0 += 256) {
        const int tile = t0 + threadIdx.x;
        double s = 0.0;
        if (tile < NT) {
            const int lo = tile * kTile, hi = min(T, lo + kTile);
            for (int t = lo; t < hi; t++) s += (double)gb[t];
        }
        part[threadIdx.x] = s;
        __syncthreads();
        if (threadIdx.x == 0) {
            double run = carry;
            for (int u = 0; u < 256; u++) {
                double x = part[u];
                part[u] = run;
                run += x;
            }
            carry = run;
        }
        __syncthreads();
        if (tile < NT) Pb[tile] = part[threadIdx.x];
        __syncthreads();
    }
    if (threadIdx.x == 0) Pb[NT] = carry;
    for (int j = threadIdx.x; j <= NT; j += 256) fb[j] = 0;
    if (bh == 0 && threadIdx.x == 0) {
        *ticket = 0;
        *err = 0;
    }
}

}  // namespace

// Workspace: [P fp64 BH*(NT+1)] [flags int BH*(NT+1)] [ticket, err] [node32] [node16]
static size_t off_flags(int BH, int NT) { return align_up((size_t)BH * (NT + 1) * 8, 256); }
static size_t off_ticket(int BH, int NT) { return off_flags(BH, NT) + align_up((size_t)BH * (NT + 1) * 4, 256); }
static size_t off_node32(int BH, int NT) { return off_ticket(BH, NT) + 256; }
static size_t off_node16(int BH, int NT)
{
    return off_node32(BH, NT) + align_up((size_t)BH * NT * kD * kD * 4, 1024);
}

size_t tc_workspace_bytes(int B, int H, int T)
{
    const int BH = B * H, NT = (T + kTile - 1) / kTile;
    return off_node16(BH, NT) + align_up((size_t)BH * NT * kD * kD * 2, 1024);
}

bool tc_supported(int dk, int dv, lla_dtype in_dt)
{
    return in_dt == LLA_BF16 && dk == kD && dv == kD;
}

size_t tc_smem_bytes() { return sizeof(TcSmem) + 1024; }

cudaError_t tc_fwd(const TcFwdArgs &A)
{
    const int BH = A.B * A.H, NT = (A.T + kTile - 1) / kTile;
    char *ws = (char *)A.workspace;
    TcParams prm;
    prm.g = A.g;
    prm.lam = A.lam;
    prm.out = A.out;
    prm.P = (const double *)ws;
    prm.flags = (int *)(ws + off_flags(BH, NT));
    prm.ticket = (int *)(ws + off_ticket(BH, NT));
    prm.err = prm.ticket + 1;
    prm.node32 = (float *)(ws + off_node32(BH, NT));
    prm.node16 = (__nv_bfloat16 *)(ws + off_node16(BH, NT));
    prm.T = A.T;
    prm.NT = NT;
    prm.BH = BH;
    prm.L = A.L;
    CUtensorMap mq, mk, mv, mn;
    if (!make_map_bf16_3d(&mq, A.q, kD, A.T, BH, 64, kTile) ||
        !make_map_bf16_3d(&mk, A.k, kD, A.T, BH, 64, kTile) ||
        !make_map_bf16_3d(&mv, A.v, kD, A.T, BH, 64, kTile) ||
        !make_map_bf16_3d(&mn, prm.node16, kD, kD, (uint64_t)BH * NT, 64, kTile))
        return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)A.stream;
    lla_tile_gate_prefix_kernel<<<BH, 256, 0, st>>>(A.g, (double *)prm.P, prm.flags, prm.ticket, prm.err,
                                                   A.T, NT);
    const size_t smem = tc_smem_bytes();
    cudaError_t e;
    if (A.out_dt == LLA_F32) {
        e = cudaFuncSetAttribute(lla_fwd_tc_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        lla_fwd_tc_kernel<float><<<BH * NT, kThreads, smem, st>>>(mq, mk, mv, mn, prm);
    } else {
        e = cudaFuncSetAttribute(lla_fwd_tc_kernel<__nv_bfloat16>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        lla_fwd_tc_kernel<__nv_bfloat16><<<BH * NT, kThreads, smem, st>>>(mq, mk, mv, mn, prm);
    }
    return cudaPeekAtLastError();
}

}  // namespace lla
