// Internal interface of the backward (CUDA cores, fp32 arithmetic).
#pragma once

#include <stddef.h>

#include "lla_common.cuh"

namespace lla {

struct BwdArgs {
    const void *q, *k, *v;
    const float *g, *lam, *dout;
    float *dq, *dkey, *dval, *dg, *dlam;
    int B, H, T, dk, dv, C, L;
    lla_dtype in_dt;
    void *workspace;
    int32_t *device_error;  // caller's word, or nullptr (the workspace word is used)
    void *stream;
};

// The state R_{m,b} of block b at level m ([Dk][Dv] fp32, E = Dk Dv): a block
// of several pieces has the sum of its pieces in its R slot (block slots flat
// by level); a block that is a single piece is read from that piece's slot
// directly (the reduction skips it).  Piece slots are flat by level, (b / 2)
// times pieces-per-block within a level.
__device__ __forceinline__ const float *block_state(const float *R, const float *part, long long bh, int m, int b,
                                                    int N, int Pc, int nitems, int nblocks, int E)
{
    int off = 0, first = 0;
    for (int mm = 0; mm < m; mm++) {
        const int nb = (N + (1 << mm) - 1) >> mm;
        off += nb;
        first += (nb / 2) * (((1 << mm) + Pc - 1) / Pc);
    }
    const int pp = ((1 << m) + Pc - 1) / Pc;
    const int blk_end = min(N, (b + 1) << m);
    if (blk_end - (b << m) <= Pc)
        return part + ((bh * nitems) + first + (long long)(b / 2) * pp) * (long long)E;
    return R + ((bh * nblocks) + off + b) * (long long)E;
}

size_t bwd_workspace_bytes(const BwdArgs &A);
size_t bwd_smem_bytes(const BwdArgs &A);
cudaError_t bwd(const BwdArgs &A);
// Key side on the tensor cores (bf16, dk = dv = 128, chunk 64): adds to dk, dv.
bool bwd_key_tc_supported(const BwdArgs &A);
cudaError_t bwd_key_tc(const BwdArgs &A, const float *gamma, const double *P, const float *R, const float *part,
                       int nlev, int nblocks, int Pc, int nitems, int *err);
// Query side (node read-out) on the tensor cores, same conditions: adds to dq, dlambda.
bool bwd_query_tc_supported(const BwdArgs &A);
cudaError_t bwd_query_tc(const BwdArgs &A, const float *gamma, const double *P, const float *nodes, int *err);
// Intra-chunk part on the tensor cores, same conditions: writes dq, dk, dv, dlambda.
bool bwd_intra_tc_supported(const BwdArgs &A);
cudaError_t bwd_intra_tc(const BwdArgs &A, const float *gamma, int *err);
// Chunk states of the rebuilt forward nodes on the tensor cores, same conditions:
// the chunk gate totals (every chunk) and H_i in node slot i+1 (i < N-1).
bool bwd_state_tc_supported(const BwdArgs &A);
cudaError_t bwd_state_tc(const BwdArgs &A, const float *gamma, float *gam_tot, float *nodes, int *err);
// Block-state pieces on the tensor cores, same conditions: writes every piece slot it owns.
bool bwd_piece_tc_supported(const BwdArgs &A);
cudaError_t bwd_piece_tc(const BwdArgs &A, const float *gamma, const double *P, float *part, int nlev, int Pc,
                         int nitems, int *err);


// Number of SMs of the current device (the tensor-core backward kernels run
// one CTA per SM, so the CTA that follows CTA x on an SM is about x + this).
inline int bwd_sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        n <= 0)
        n = 148;
    return n;
}

// Prefetch [p, p + bytes) into L2 (bytes a multiple of 16, p 16-byte aligned),
// in pieces of at most 32 KB.
__device__ __forceinline__ void prefetch_l2(const void *p, long long bytes)
{
    const char *c = static_cast<const char *>(p);
    for (long long o = 0; o < bytes; o += 32768) {
        const long long n = bytes - o < 32768 ? bytes - o : 32768;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c + o), "r"((uint32_t)n) : "memory");
    }
}

}  // namespace lla
