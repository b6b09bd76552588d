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
#include "sm100.cuh"
#include "tma_host.cuh"

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


// ------------------------------------------------ tensor-core path
// bf16 d with Dd a multiple of 64 (<= 256): the first layer h = d W1 runs on
// the tensor cores.  d is exact in bf16; W1 is split into three bf16 parts
// (hi + mid + lo reproduce each fp32 weight to about 24 bits), stacked along
// N, so one product of N = 3 NP per K step gives d W1_hi, d W1_mid and
// d W1_lo in three fp32 accumulators, which the epilogue adds as
// hi + (mid + lo): h carries the error of an fp32 dot product, and a tile
// takes Dd / 16 MMAs instead of three times as many.  Per 128-row tile: TMA
// brings the d rows through a ring of up to four stages, one thread issues
// the products into one of two accumulator sets, and eight epilogue warps
// (two threads per row, each half of the row's float4 groups of L)
// read h, apply the second layer and softplus in fp32 and store their
// weights.  CTAs are persistent over the tiles.
constexpr int kTcRows = 128;
constexpr int kTcEpi = 256;             // epilogue threads (two per row)
constexpr int kTcParts = kTcEpi / kTcRows;
constexpr int kTcIssueWarp = kTcEpi / 32;
constexpr int kTcThreads = kTcEpi + 32;  // plus one issuing warp
constexpr uint32_t kTcWait = 1u << 22;

using namespace sm100;

// Sticky record of a bounded wait that gave up (1: load, 2: product) for
// calls that pass no device_error word; the kernel carries on, so the
// results of that call are not to be trusted.
__device__ int lla_lambda_tc_wait_err;

// tensor-memory columns of the two accumulator sets (3 NP columns each)
__host__ __device__ constexpr int tc_tmem_cols(int NP) { return 6 * NP <= 128 ? 128 : 6 * NP <= 256 ? 256 : 512; }

constexpr int kTcMaxStages = 4;
constexpr uint32_t kTcSmemMax = 227 * 1024 - 1024;

struct TcLayout {  // byte offsets in dynamic shared memory (1024-aligned base)
    uint32_t w1, w2, d0, dtile, bars, total;
    int stages;
};

__host__ __device__ inline TcLayout tc_layout(int Dd, int NP, int L)
{
    TcLayout t;
    const uint32_t w1bytes = 3u * (uint32_t)NP * 128 * (uint32_t)(Dd / 64);  // [Dd/64][3 NP rows][128 B]
    t.dtile = (uint32_t)kTcRows * 128 * (uint32_t)(Dd / 64);
    const int Lp = (L + 3) & ~3;
    const uint32_t tail = (((uint32_t)(NP * Lp + Lp) * 4 + 15) & ~15u) + (2 * kTcMaxStages + 4) * 8 + 16;
    t.w1 = 0;
    t.d0 = (w1bytes + 1023) & ~1023u;
    t.stages = kTcMaxStages;
    while (t.stages > 2 && t.d0 + t.stages * t.dtile + tail > kTcSmemMax) t.stages--;
    t.w2 = t.d0 + t.stages * t.dtile;
    t.bars = (t.w2 + (uint32_t)(NP * Lp + Lp) * 4 + 15) & ~15u;
    t.total = t.bars + (2 * kTcMaxStages + 4) * 8 + 16;
    return t;
}

template <int NP>
__global__ void __launch_bounds__(kTcThreads, 1)
lambda_tc_kernel(const __grid_constant__ CUtensorMap map_d, const float *__restrict__ W1,
                 const float *__restrict__ W2, const float *__restrict__ bias, float *__restrict__ lam,
                 long long N, int Dd, int L, int *err)
{
    if (err == nullptr) err = &lla_lambda_tc_wait_err;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const TcLayout lay = tc_layout(Dd, NP, L);
    const int Hd = 2 * L;
    const int nb = Dd / 64;
    const int NS = lay.stages;
    const uint32_t wblk = 3u * NP * 128;  // one 64-wide K block of the stacked W1^T parts
    const uint32_t dblk = (uint32_t)kTcRows * 128;
    const int Lp = (L + 3) & ~3;
    float *w2 = reinterpret_cast<float *>(sm + lay.w2);  // [NP][Lp] zero-padded, then bias [Lp]
    float *bs = w2 + NP * Lp;
    uint64_t *bar_load = reinterpret_cast<uint64_t *>(sm + lay.bars);  // [NS]
    uint64_t *bar_mma = bar_load + kTcMaxStages;                       // [2]
    uint64_t *bar_free = bar_mma + 2;                                  // [2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bar_free + 2);
    const int tid = threadIdx.x, warp = tid >> 5;
    // W1^T split into three bf16 parts, stacked along N (rows part NP + n) in
    // the K-major 128-byte-swizzled layout
    for (int e = tid; e < NP * Dd; e += kTcThreads) {
        const int n = e / Dd, k = e % Dd;
        float w = n < Hd ? W1[k * Hd + n] : 0.f;
#pragma unroll
        for (int part = 0; part < 3; part++) {
            const uint32_t off = (uint32_t)(k / 64) * wblk + sw128_offset(part * NP + n, (k % 64) / 8) + (k % 8) * 2;
            const __nv_bfloat16 b = __float2bfloat16_rn(w);
            *reinterpret_cast<__nv_bfloat16 *>(sm + lay.w1 + off) = b;
            w -= __bfloat162float(b);
        }
    }
    for (int e = tid; e < NP * Lp; e += kTcThreads) {
        const int j = e / Lp, l = e % Lp;
        w2[e] = (j < Hd && l < L) ? W2[j * L + l] : 0.f;
    }
    for (int e = tid; e < Lp; e += kTcThreads) bs[e] = e < L ? bias[e] : 0.f;
    if (tid == kTcEpi) {
        for (int b = 0; b < NS; b++) mbar_init(&bar_load[b], 1);
        for (int b = 0; b < 2; b++) {
            mbar_init(&bar_mma[b], 1);
            mbar_init(&bar_free[b], kTcEpi);
        }
        fence_mbar_init();
        tma_prefetch_map(&map_d);
    }
    if (warp == kTcIssueWarp) {
        tmem_alloc(tmem_slot, tc_tmem_cols(NP));
        tmem_relinquish();
    }
    fence_proxy_async_smem();  // W1 parts written by threads, read by the tensor cores
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = *tmem_slot;
    const long long ntiles = (N + kTcRows - 1) / kTcRows;
    const int my = (int)((ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x);  // tiles of this CTA
    if (warp == kTcIssueWarp) {
        if (tid == kTcEpi) {
            // tile i: load stage i % NS, accumulator set i % 2
            auto load = [&](int i) {
                const int ls = i % NS;
                const long long tile = blockIdx.x + (long long)i * gridDim.x;
                uint8_t *dst = sm + lay.d0 + ls * lay.dtile;
                mbar_arrive_expect_tx(&bar_load[ls], dblk * nb);
                for (int b = 0; b < nb; b++)
                    tma_load_3d(dst + b * dblk, &map_d, &bar_load[ls], 64 * b, (int)(tile * kTcRows), 0);
            };
            for (int i = 0; i < min(NS, my); i++) load(i);
            const uint32_t idesc = idesc_bf16_f32(128, 3 * NP, false, false);
            for (int i = 0; i < my; i++) {
                const int ls = i % NS, st = i & 1;
                if (!mbar_wait(&bar_load[ls], (i / NS) & 1, kTcWait)) atomicCAS(err, 0, 1);
                if (i >= 2 && !mbar_wait(&bar_free[st], ((i - 2) >> 1) & 1, kTcWait)) atomicCAS(err, 0, 2);
                tc_fence_after_sync();
                const uint32_t acc = tm + (uint32_t)(st * 3 * NP);
                const uint8_t *dt = sm + lay.d0 + ls * lay.dtile;
                for (int kk = 0; kk < 4 * nb; kk++) {
                    const uint32_t offa = (kk >> 2) * dblk + (kk & 3) * 32;
                    const uint32_t offb = (kk >> 2) * wblk + (kk & 3) * 32;
                    umma_bf16(acc, desc_sw128(smem_u32(dt) + offa, 16, 1024),
                              desc_sw128(smem_u32(sm + lay.w1) + offb, 16, 1024), idesc, kk > 0 ? 1u : 0u);
                }
                umma_commit(&bar_mma[st]);
                if (i + NS < my) {  // the stage is free once this tile's products are done
                    if (!mbar_wait(&bar_mma[st], (i >> 1) & 1, kTcWait)) atomicCAS(err, 0, 2);
                    load(i + NS);
                }
            }
        }
    } else {
        // epilogue: kTcParts threads per row of the tile (= tensor-memory lane);
        // part p takes the float4 groups g of lambda with g % kTcParts == p.
        // Tiles are taken in pairs (i, i + 1: accumulator sets 0 and 1), so that
        // every W2 load from shared memory serves two rows: those loads (about
        // four wavefronts each, although all lanes read one address) bound the
        // kernel.
        const int row_t = tid & (kTcRows - 1), part = tid >> 7;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const bool vec = (L & 3) == 0 && ((uintptr_t)lam & 15) == 0;  // every row 16-byte aligned
        // h = hi + (mid + lo) from the three accumulators of set st
        auto drain = [&](int i, float (&h)[NP]) {
            const int st = i & 1;
            if (!mbar_wait(&bar_mma[st], (i >> 1) & 1, kTcWait)) atomicCAS(err, 0, 2);
            tc_fence_after_sync();
            const uint32_t acc = tm + (uint32_t)(st * 3 * NP) + lane_off;
#pragma unroll
            for (int c = 0; c < NP; c += 16) {
                float m[16], l[16];
                tmem_ld16(acc + c, *reinterpret_cast<float(*)[16]>(h + c));
                tmem_ld16(acc + NP + c, m);
                tmem_ld16(acc + 2 * NP + c, l);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 16; u++) h[c + u] += m[u] + l[u];
            }
            tc_fence_before_sync();
            mbar_arrive(&bar_free[st]);
        };
        auto store = [&](long long row, const float4 &y, int l0) {
            float *out = lam + row * L;
            if (vec) {
                *reinterpret_cast<float4 *>(out + l0) = y;
            } else {
                const float yy[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
                for (int q = 0; q < 4; q++)
                    if (l0 + q < L) out[l0 + q] = yy[q];
            }
        };
        for (int i = 0; i < my; i += 2) {
            const bool two = i + 1 < my;
            const long long row0 = (blockIdx.x + (long long)i * gridDim.x) * kTcRows + row_t;
            const long long row1 = row0 + (long long)gridDim.x * kTcRows;
            float h0[NP], h1[NP];
            drain(i, h0);
            if (two) {
                drain(i + 1, h1);
            } else {
#pragma unroll
                for (int j = 0; j < NP; j++) h1[j] = 0.f;
            }
            for (int l0 = 4 * part; l0 < L; l0 += 4 * kTcParts) {
                float4 z0 = *reinterpret_cast<const float4 *>(bs + l0), z1 = z0;
#pragma unroll
                for (int j = 0; j < NP; j++) {
                    const float4 w = *reinterpret_cast<const float4 *>(w2 + j * Lp + l0);
                    z0.x = fmaf(h0[j], w.x, z0.x);
                    z0.y = fmaf(h0[j], w.y, z0.y);
                    z0.z = fmaf(h0[j], w.z, z0.z);
                    z0.w = fmaf(h0[j], w.w, z0.w);
                    z1.x = fmaf(h1[j], w.x, z1.x);
                    z1.y = fmaf(h1[j], w.y, z1.y);
                    z1.z = fmaf(h1[j], w.z, z1.z);
                    z1.w = fmaf(h1[j], w.w, z1.w);
                }
                if (row0 < N)
                    store(row0, make_float4(softplus_f(z0.x), softplus_f(z0.y), softplus_f(z0.z), softplus_f(z0.w)),
                          l0);
                if (two && row1 < N)
                    store(row1, make_float4(softplus_f(z1.x), softplus_f(z1.y), softplus_f(z1.z), softplus_f(z1.w)),
                          l0);
            }
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == kTcIssueWarp) tmem_dealloc(tm, tc_tmem_cols(NP));
}

template <int NP>
cudaError_t launch_tc_np(const LambdaMlpArgs &A)
{
    const long long N = (long long)A.B * A.H * A.T;
    CUtensorMap md;
    if (!make_map_bf16_3d(&md, A.d, (uint64_t)A.Dd, (uint64_t)N, 1, 64, kTcRows)) return cudaErrorInvalidValue;
    const size_t smem = tc_layout(A.Dd, NP, A.L).total + 1024;
    auto kern = lambda_tc_kernel<NP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const long long ntiles = (N + kTcRows - 1) / kTcRows;
    const int grid = (int)(ntiles < nsm ? ntiles : nsm);
    kern<<<grid, kTcThreads, smem, (cudaStream_t)A.stream>>>(md, A.W1, A.W2, A.bias, A.lam, N, A.Dd, A.L,
                                                          (int *)A.device_error);
    return cudaPeekAtLastError();
}

}  // namespace

bool lambda_tc_supported(const LambdaMlpArgs &A)
{
    return A.in_dt == LLA_BF16 && A.Dd % 64 == 0 && A.Dd <= 256 && 2 * A.L <= 64 &&
           ((uintptr_t)A.d & 15) == 0 && tc_layout(A.Dd, 64, A.L).total + 1024 <= 227 * 1024;
}

cudaError_t lambda_mlp(const LambdaMlpArgs &A)
{
    if (lambda_tc_supported(A)) {
        const int np = 2 * A.L <= 16 ? 16 : 2 * A.L <= 32 ? 32 : 2 * A.L <= 48 ? 48 : 64;
        switch (np) {
        case 16: return launch_tc_np<16>(A);
        case 32: return launch_tc_np<32>(A);
        case 48: return launch_tc_np<48>(A);
        default: return launch_tc_np<64>(A);
        }
    }
    return A.in_dt == LLA_F32 ? launch_t<float>(A) : launch_t<__nv_bfloat16>(A);
}

}  // namespace lla
