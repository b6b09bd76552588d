// Query side of the backward on the tensor cores (bf16 q, k; dk = dv = 128;
// chunk 64): the read-out of the forward's chunk-level Fenwick nodes.
//
// For a row t of chunk i and each node j on the Fenwick path of i (level
// l = c + 1 + ctz(j)), with U_t = Node_j dO_t and w_t = exp(G_t - P_j) <= 1:
//     dq_t += lambda_t[l] w_t U_t,   dlambda_t[l] += w_t q_t . U_t.
// A CTA takes the pair of chunks (2p, 2p+1) as one 128-row tile: the path
// of 2p+1 is node 2p+1 followed by the path of 2p, so every node of the pair
// is one product over all 128 rows, with weight 0 on the rows it does not
// concern.  U = dO Node^T runs on the tensor cores with dO and the node (both
// fp32) split into bf16 high and remainder parts (three products: hi.hi,
// hi.lo, lo.hi: dO_hi times [Node_hi | Node_lo] as one N = 256 product into
// two accumulators, then dO_lo times Node_hi into the first, and the drain
// adds the two); a two-deep ring of node stages and of accumulator pairs lets the
// staging of node n+1 and the product of node n overlap the drain of node
// n-1.  Eight warps drain: thread = (row, half of the 128 columns); the two
// halves' q.U partial sums meet in shared memory.  Results are added to dq
// and dlambda.
#include "bwd_simt.cuh"
#include "sm100.cuh"
#include "split_stage.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kQT = 128;
constexpr int kQD = 128;
constexpr uint32_t kQBuf = kQT * kQD * 2;  // bf16 128 x 128: 32 KB
constexpr uint32_t kQHalf = kQBuf / 2;
constexpr int kQThreads = 256;
constexpr uint32_t kQWait = 1u << 22;
constexpr int kQMaxPath = 20;

struct __align__(1024) QuerySmem {
    uint8_t ohi[kQBuf], olo[kQBuf];     // dO tile, high and remainder parts
    uint8_t nd[2][2 * kQBuf];           // node stages: per 64-column K block, the high part's
                                        // 128 rows then the remainder's (one N = 256 operand)
    float part[2][kQT];                 // q.U partial sums of the second half
    float wt[kQMaxPath][kQT];           // per path node and row: exp(G_t - P_j) (0 where it does not apply)
    float lwt[kQMaxPath][kQT];          // the same times lambda_t at the node's level
    uint64_t bar_mma[2];
    uint32_t tmem;
};

__device__ __forceinline__ void q_err(int *err, int code) { atomicCAS(err, 0, code); }

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

template <typename Tin>
__global__ void __launch_bounds__(kQThreads, 1)
bwd_query_tc_kernel(const Tin *__restrict__ q, const float *__restrict__ dout, const float *__restrict__ gamma,
                    const float *__restrict__ lam, const double *__restrict__ P, const float *__restrict__ nodes,
                    float *__restrict__ dq, float *__restrict__ dlam, int T, int N, int L, int cbits,
                    int *__restrict__ err)
{
    extern __shared__ uint8_t smem_raw[];
    QuerySmem &s = *reinterpret_cast<QuerySmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int row = tid & (kQT - 1), half = tid >> 7;
    const int pair = blockIdx.x, bh = blockIdx.y;
    const int c0 = 2 * pair;
    // the pair's nodes: 2p+1 (second chunk only, if it exists), then the path of 2p
    int js[kQMaxPath];
    int np = 0;
    if (c0 + 1 < N) js[np++] = c0 + 1;
    for (int j = c0; j > 0; j -= (j & -j)) js[np++] = j;
    if (np == 0) return;
    const double *Pb = P + (long long)bh * (N + 1);
    const long long trow = (long long)pair * kQT + row;
    const bool row_ok = trow < T;
    const int chunk = c0 + (row >> 6);
    const long long tok = (long long)bh * T + trow;
    if (tid == 0) {
        mbar_init(&s.bar_mma[0], 1);
        mbar_init(&s.bar_mma[1], 1);
        fence_mbar_init();
    }
    if (tid < 32) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    // read-out weights of every path node for this row (the halves split the
    // nodes): w = exp(G_t - P_j) from one fp64 difference, lw = lambda_t[l] w
    {
        const double Gt = Pb[min(chunk, N)] + (double)(row_ok ? gamma[tok] : 0.f);
        const float *lam_row = lam + tok * L;
        for (int n = half; n < np; n += 2) {
            const int j = js[n];
            const bool mine = row_ok && (j <= chunk);  // node 2p+1 concerns the second chunk only
            const float w = mine ? expf((float)(Gt - Pb[j])) : 0.f;
            s.wt[n][row] = w;
            s.lwt[n][row] = mine ? lam_row[cbits + 1 + (__ffs(j) - 1)] * w : 0.f;
        }
    }
    // dO tile and the first node
    const int nrows = (int)min((long long)kQT, (long long)T - (long long)pair * kQT);
    {
        uint8_t *d0[2] = {s.ohi, s.olo};
        stage_split_tile<2, kQThreads, 8>(d0, dout + ((long long)bh * T + (long long)pair * kQT) * kQD, kQD,
                                          nullptr, 1.f, nrows);
    }
    const float *node_base = nodes + (long long)bh * N * kQD * kQD;
    // the fp32 nodes come from DRAM: each is prefetched into L2 two nodes
    // before it is staged
    auto prefetch_node = [&](int n) {
        if (tid == 0 && n < np) {
            const float *src = node_base + (long long)js[n] * kQD * kQD;
            bulk_prefetch_l2(src, kQD * kQD * 2);
            bulk_prefetch_l2(src + kQD * kQD / 2, kQD * kQD * 2);
        }
    };
    prefetch_node(1);
    prefetch_node(2);
    {
        uint8_t *d1[2] = {s.nd[0], s.nd[0] + kQHalf};
        stage_split_tile<2, kQThreads, 8, 2 * kQHalf>(d1, node_base + (long long)js[0] * kQD * kQD, kQD, nullptr, 1.f,
                                                      kQD);
    }
    fence_proxy_async_smem();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;
    const uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
    const uint32_t idesc2 = idesc_bf16_f32(128, 256, false, false);
    // this thread's q half row (16-byte loads), and G_t
    float qv[64];
    {
        const uint4 *qr = reinterpret_cast<const uint4 *>(q + tok * kQD + half * 64);
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const uint4 w4 = row_ok ? qr[u] : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t h4[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int e = 0; e < 4; e++) {
                qv[8 * u + 2 * e] = __uint_as_float(h4[e] << 16);  // bf16 -> fp32: the high half of the word
                qv[8 * u + 2 * e + 1] = __uint_as_float(h4[e] & 0xffff0000u);
            }
        }
    }
    float dqa[64];
#pragma unroll
    for (int c = 0; c < 64; c++) dqa[c] = 0.f;
    const uint32_t lane_off = (uint32_t)((tid >> 5) & 3) * 32 << 16;
    auto issue = [&](int n) {
        const int b = n & 1;
        tc_fence_after_sync();
        const uint32_t acc = tm + b * 256;  // [dO_hi Node_hi^T + dO_lo Node_hi^T | dO_hi Node_lo^T]
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
            const uint32_t offa = (kk >> 2) * kQHalf + (kk & 3) * 32, offb = (kk >> 2) * (2 * kQHalf) + (kk & 3) * 32;
            umma_bf16(acc, desc_sw128(smem_u32(s.ohi) + offa, 16, 1024), desc_sw128(smem_u32(s.nd[b]) + offb, 16, 1024),
                      idesc2, kk > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int kk = 0; kk < 8; kk++) {
            const uint32_t offa = (kk >> 2) * kQHalf + (kk & 3) * 32, offb = (kk >> 2) * (2 * kQHalf) + (kk & 3) * 32;
            umma_bf16(acc, desc_sw128(smem_u32(s.olo) + offa, 16, 1024), desc_sw128(smem_u32(s.nd[b]) + offb, 16, 1024),
                      idesc, 1u);
        }
        umma_commit(&s.bar_mma[b]);
    };
    auto drain = [&](int n) {
        const int b = n & 1;
        const int j = js[n];
        const int lev = cbits + 1 + (__ffs(j) - 1);
        const bool mine = row_ok && (j <= chunk);
        const float w = s.wt[n][row], lw = s.lwt[n][row];
        if (!mbar_wait(&s.bar_mma[b], (n >> 1) & 1, kQWait)) q_err(err, 2);
        tc_fence_after_sync();
        float dot = 0.f;
#pragma unroll
        for (int c0c = 0; c0c < 64; c0c += 16) {
            float u[16], u2[16];
            tmem_ld16(tm + b * 256 + lane_off + half * 64 + c0c, u);
            tmem_ld16(tm + b * 256 + 128 + lane_off + half * 64 + c0c, u2);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; e++) u[e] += u2[e];
#pragma unroll
            for (int e = 0; e < 16; e++) {
                dqa[c0c + e] = fmaf(lw, u[e], dqa[c0c + e]);
                dot = fmaf(qv[c0c + e], u[e], dot);
            }
        }
        tc_fence_before_sync();
        if (half == 1) s.part[b][row] = dot;
        named_sync(1, kQThreads);
        if (half == 0 && mine) dlam[tok * L + lev] += w * (dot + s.part[b][row]);
    };
    if (tid == 0) issue(0);
    for (int n = 0; n < np; n++) {
        if (n + 1 < np) {
            // stage node n+1 into the other buffer once node n-1's product is done
            const int b1 = (n + 1) & 1;
            if (n >= 1 && !mbar_wait(&s.bar_mma[b1], ((n - 1) >> 1) & 1, kQWait)) q_err(err, 2);
            prefetch_node(n + 3);
            uint8_t *d1[2] = {s.nd[b1], s.nd[b1] + kQHalf};
            stage_split_tile<2, kQThreads, 8, 2 * kQHalf>(d1, node_base + (long long)js[n + 1] * kQD * kQD, kQD,
                                                          nullptr, 1.f, kQD);
            fence_proxy_async_smem();
        }
        drain(n);  // contains a barrier of all threads: node n+1 is staged and U_{n-1} drained
        if (n + 1 < np && tid == 0) issue(n + 1);
    }
    // dq through shared memory (the dO stages, free once every product is
    // done) and added as whole rows
    float *tile = reinterpret_cast<float *>(s.ohi);
#pragma unroll
    for (int u = 0; u < 16; u++)
        *out_tile_piece(tile, row, half * 16 + u) = make_float4(dqa[4 * u], dqa[4 * u + 1], dqa[4 * u + 2], dqa[4 * u + 3]);
    __syncthreads();
    out_tile_store<kQThreads, true>(dq + ((long long)bh * T + (long long)pair * kQT) * kQD, tile, nrows);
    tc_fence_before_sync();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tm, 512);
}

}  // namespace

bool bwd_query_tc_supported(const BwdArgs &A)
{
    return A.in_dt == LLA_BF16 && A.dk == kQD && A.dv == kQD && A.C == 64 && ((uintptr_t)A.dout & 15) == 0 &&
           ((uintptr_t)A.dq & 15) == 0;
}

cudaError_t bwd_query_tc(const BwdArgs &A, const float *gamma, const double *P, const float *nodes, int *err)
{
    const int BH = A.B * A.H, N = A.T / A.C;
    const int cbits = ctz_u32((uint32_t)A.C);  // 6: the supported chunk is 64
    const size_t smem = sizeof(QuerySmem) + 1024;
    auto kern = bwd_query_tc_kernel<__nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3((N + 1) / 2, BH), kQThreads, smem, (cudaStream_t)A.stream>>>(
        (const __nv_bfloat16 *)A.q, A.dout, gamma, A.lam, P, nodes, A.dq, A.dlam, A.T, N, A.L, cbits, err);
    return cudaPeekAtLastError();
}

}  // namespace lla
