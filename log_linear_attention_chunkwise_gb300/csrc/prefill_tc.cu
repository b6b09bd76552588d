// Prefill bucket states on the tensor cores (bf16 k, v; dk = dv = 128).
//
// The decode state after a prefix [0, T) holds one state per Fenwick bucket
// of [0, T) ("Log-Linear Attention" §2.2): S_l = sum_{s in bucket l}
// exp(tail_s) k_s v_s^T with tail_s = g_{s+1} + ... + g_{T-1}.  Each bucket is
// a product K^T diag(w) V over its tokens, so a CTA takes a run of
// 128-token tiles of one bucket: TMA brings K and V tiles through a
// kPreStages ring, two threads per token scale their halves of the V row by w
// (0 outside the bucket) and split them into a bf16 high part and a bf16
// remainder stored right after it, and one thread issues
// [S_hi | S_lo] += K^T [V_hi | V_lo] (M = dk, N = 2 dv, K = 128 tokens: one
// MMA per K step) into two tensor-memory accumulators, added at the end: k
// is exact in bf16, so the two products keep about 16 bits of each scaled
// value instead of bf16's 8.  The partial state is added to the zeroed
// output state with float4 atomics.  Waits are bounded; a wait that
// gives up records a code in the workspace error word.
#include "decode.cuh"
#include "sm100.cuh"
#include "tma_host.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kPTile = 128;
constexpr int kPD = 128;
constexpr uint32_t kPBuf = kPTile * kPD * 2;  // one bf16 128 x 128 tile: 32 KB
constexpr uint32_t kPHalf = kPBuf / 2;        // one 64-column swizzled block
constexpr int kPreStages = 2;
constexpr int kPreThreads = 256;  // two per token: one 64-column block of its V row each
constexpr uint32_t kPreWait = 1u << 22;

struct __align__(1024) PreStage {
    uint8_t k[kPBuf];
    uint8_t v[kPBuf];    // scaled in place to the high part
    uint8_t vlo[kPBuf];  // the remainder: with v, the four 64-column blocks of one N = 256 operand
};

struct __align__(1024) PreSmem {
    PreStage st[kPreStages];
    uint64_t bar_load[kPreStages], bar_mma[kPreStages], bar_done;
    uint32_t tmem;
};

struct PreTable {
    long long start[40], len[40];
    int item_begin[41];
    int slot[40];
    int n;
};

__device__ __forceinline__ void pre_err(int *err, int code) { atomicCAS(err, 0, code); }

__global__ void __launch_bounds__(kPreThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                  const float *__restrict__ tail, float *__restrict__ S, PreTable tab, int T, int Ls,
                  int tpc, int *__restrict__ err)
{
    extern __shared__ uint8_t smem_raw[];
    PreSmem &s = *reinterpret_cast<PreSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int p = tid & (kPTile - 1), hb = tid >> 7;  // token row, 64-column block of V
    const long long bh = blockIdx.y;
    const int item = blockIdx.x;
    int li = 0;
    while (li + 1 < tab.n && tab.item_begin[li + 1] <= item) li++;
    const long long blo = tab.start[li], bhi = tab.start[li] + tab.len[li];
    const long long row0 = blo + (long long)(item - tab.item_begin[li]) * tpc * kPTile;
    const int ntiles = (int)min((long long)tpc, (bhi - row0 + kPTile - 1) / kPTile);
    if (tid == 0) {
        for (int b = 0; b < kPreStages; b++) {
            mbar_init(&s.bar_load[b], 1);
            mbar_init(&s.bar_mma[b], 1);
        }
        mbar_init(&s.bar_done, 1);
        fence_mbar_init();
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
    }
    if (tid < 32) {
        tmem_alloc(&s.tmem, 256);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;
    const float *tb = tail + bh * (long long)T;
    auto issue_load = [&](int n) {
        const int ls = n % kPreStages;
        const int y = (int)(row0 + (long long)n * kPTile);
        mbar_arrive_expect_tx(&s.bar_load[ls], 2 * kPBuf);
        tma_load_3d(s.st[ls].k, &map_k, &s.bar_load[ls], 0, y, (int)bh);
        tma_load_3d(s.st[ls].k + kPHalf, &map_k, &s.bar_load[ls], 64, y, (int)bh);
        tma_load_3d(s.st[ls].v, &map_v, &s.bar_load[ls], 0, y, (int)bh);
        tma_load_3d(s.st[ls].v + kPHalf, &map_v, &s.bar_load[ls], 64, y, (int)bh);
    };
    auto weight = [&](int n) {  // exp(tail) of this thread's token of tile n, 0 outside the bucket
        const long long r = row0 + (long long)n * kPTile + p;
        return (n < ntiles && r < bhi) ? __expf(tb[r]) : 0.f;
    };
    if (tid == 0)
        for (int n = 0; n < min(kPreStages, ntiles); n++) issue_load(n);
    float w = weight(0);
    const uint32_t idesc = idesc_bf16_f32(128, 256, true, true);
    for (int n = 0; n < ntiles; n++) {
        const int ls = n % kPreStages;
        if (tid == 0 && n >= 1 && n - 1 + kPreStages < ntiles) {
            // the stage of tile n-1 is free once its product is done
            const int pn = n - 1;
            if (!mbar_wait(&s.bar_mma[pn % kPreStages], (pn / kPreStages) & 1, kPreWait)) pre_err(err, 2);
            issue_load(pn + kPreStages);
        }
        const float wn = weight(n + 1);
        if (!mbar_wait(&s.bar_load[ls], (n / kPreStages) & 1, kPreWait)) pre_err(err, 1);
        // block hb of V row p scaled in place
        {
            const int h = hb;
#pragma unroll
            for (int c = 0; c < 8; c++) {
                const uint32_t off = h * kPHalf + sw128_offset(p, c);
                uint4 *q4 = reinterpret_cast<uint4 *>(s.st[ls].v + off);
                uint4 raw = *q4, rlo;
                __nv_bfloat162 *hv = reinterpret_cast<__nv_bfloat162 *>(&raw);
                __nv_bfloat162 *lv = reinterpret_cast<__nv_bfloat162 *>(&rlo);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    const float2 f = __bfloat1622float2(hv[u]);
                    const float a = f.x * w, b = f.y * w;
                    const __nv_bfloat162 hi = __floats2bfloat162_rn(a, b);
                    const float2 hf = __bfloat1622float2(hi);
                    hv[u] = hi;
                    lv[u] = __floats2bfloat162_rn(a - hf.x, b - hf.y);
                }
                *q4 = raw;
                *reinterpret_cast<uint4 *>(s.st[ls].vlo + off) = rlo;
            }
        }
        w = wn;
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after_sync();
            // [S_hi | S_lo] += K^T [V_hi | V_lo]: A = K^T (M = dk, MN-major), B = the
            // four 64-column blocks of v and vlo (N = 2 dv, MN-major, 16 KB apart)
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                const uint32_t off = kk * 2048;
                umma_bf16(tm, desc_sw128(smem_u32(s.st[ls].k) + off, kPHalf, 1024),
                          desc_sw128(smem_u32(s.st[ls].v) + off, kPHalf, 1024), idesc, (n > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&s.bar_mma[ls]);
        }
    }
    if (tid == 0) umma_commit(&s.bar_done);
    if (!mbar_wait(&s.bar_done, 0, kPreWait)) pre_err(err, 2);
    tc_fence_after_sync();
    // thread (p, hb) = columns [64 hb, 64 hb + 64) of dk row p of the partial
    // state, S_hi + S_lo; add it to the slot
    float4 *dst = reinterpret_cast<float4 *>(S + ((bh * Ls + tab.slot[li]) * kPD + p) * kPD);
    const uint32_t lane_off = (uint32_t)(((tid >> 5) & 3) * 32) << 16;
#pragma unroll
    for (int c0 = 64 * hb; c0 < 64 * hb + 64; c0 += 16) {
        float x[16], y[16];
        tmem_ld16(tm + lane_off + c0, x);
        tmem_ld16(tm + lane_off + kPD + c0, y);
        tmem_ld_wait();
        if (ntiles > 0) {
#pragma unroll
            for (int u = 0; u < 4; u++)
                atomicAdd(dst + c0 / 4 + u, make_float4(x[4 * u] + y[4 * u], x[4 * u + 1] + y[4 * u + 1],
                                                        x[4 * u + 2] + y[4 * u + 2], x[4 * u + 3] + y[4 * u + 3]));
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tm, 256);
}

}  // namespace

bool prefill_tc_supported(const PrefillArgs &A)
{
    return A.in_dt == LLA_BF16 && A.dk == kPD && A.dv == kPD &&
           ((uintptr_t)A.k & 15) == 0 && ((uintptr_t)A.v & 15) == 0 && ((uintptr_t)A.S & 15) == 0;
}

size_t prefill_tc_smem_bytes() { return sizeof(PreSmem) + 1024; }

// tail, the zeroed state and the error word are ready on the stream.
cudaError_t prefill_tc(const PrefillArgs &A, const float *tail, int *err)
{
    const long long BH = (long long)A.B * A.H;
    // tiles per CTA: about four CTAs per SM over the whole grid (one resident
    // at a time), so a CTA's set-up and hand-off overlap other CTAs' streaming
    long long tiles = 0;
    for (int l = 1; l <= A.Ls && l <= 40; l++)
        if (((long long)A.T >> (l - 1)) & 1) tiles += ((1LL << (l - 1)) + kPTile - 1) / kPTile;
    int dev = 0, nsm = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const long long want = (tiles * BH + 4LL * nsm - 1) / (4LL * (nsm > 0 ? nsm : 1));
    const int tpc = (int)(want < 1 ? 1 : (want > 64 ? 64 : want));
    PreTable tab{};
    int nitems = 0;
    for (int l = 1; l <= A.Ls && l <= 40; l++) {
        if (!(((long long)A.T >> (l - 1)) & 1)) continue;
        const long long start = ((long long)A.T >> l) << l;
        const long long len = 1LL << (l - 1);
        tab.start[tab.n] = start;
        tab.len[tab.n] = len;
        tab.slot[tab.n] = l - 1;
        tab.item_begin[tab.n] = nitems;
        nitems += (int)((len + (long long)tpc * kPTile - 1) / ((long long)tpc * kPTile));
        tab.n++;
    }
    tab.item_begin[tab.n] = nitems;
    if (nitems == 0) return cudaSuccess;
    CUtensorMap mk, mv;
    if (!make_map_bf16_3d(&mk, A.k, kPD, A.T, BH, 64, kPTile) ||
        !make_map_bf16_3d(&mv, A.v, kPD, A.T, BH, 64, kPTile))
        return cudaErrorInvalidValue;
    const size_t smem = prefill_tc_smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    prefill_tc_kernel<<<dim3(nitems, (unsigned)BH), kPreThreads, smem, (cudaStream_t)A.stream>>>(
        mk, mv, tail, A.S, tab, A.T, A.Ls, tpc, err);
    return cudaPeekAtLastError();
}

}  // namespace lla
