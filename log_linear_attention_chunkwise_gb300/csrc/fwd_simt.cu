// Chunked forward on CUDA cores (fp32 arithmetic): every supported shape and
// the fp32-input path.  Four launches per call:
//   1. chunk states  H_i = K_i^T diag(exp(Gam_i - gamma)) V_i, gate totals Gam_i
//   2. chunk-gate prefix P_j = Gam_0 + ... + Gam_{j-1} (fp64)
//   3. chunk-level Fenwick scan of the states into tree nodes
//   4. per chunk: masked intra-chunk product + lambda-weighted node read-out
// Page "Log-Linear Attention" (gist.science 2506.04761), technical summary:
// §2.2 (Fenwick buckets, per-level states, output equation) and §2.3 (the
// chunked, matmul-rich parallel form).
//
// Notation: chunk i holds tokens [iC, iC+C), C = 2^c.  gamma_a is the
// inclusive gate sum inside the chunk, Gam_i its value at the chunk's last
// token, P_i = G_{iC-1} the gate sum of all earlier chunks.  A key s in chunk
// j < i has level c + bit_length(i XOR j) for every query of chunk i, so the
// earlier chunks split into the chunk-level Fenwick buckets of [0, i): for
// each set bit m of i, the bucket [i' - 2^m, i') with i' = i with bits below
// m cleared.  Node_j (j >= 1) holds the chunks [j - lowbit(j), j) decayed to
// the last token of chunk j-1:
//   Node_j = H_{j-1} + sum_{k < ctz(j)} exp(P_j - P_{j-2^k}) Node_{j-2^k}.
// Query row a of chunk i adds, for the bucket ending at j (m = ctz(j)),
//   lambda_a[c+1+m] * exp(gamma_a + P_i - P_j) * q_a^T Node_j.
#include "fwd_simt.cuh"
#include "outer_simt.cuh"

namespace lla {
namespace {

constexpr int kThreads = 256;
constexpr int kSub = 32;  // tokens staged per step of the state kernel

// Inclusive running sum of C <= 128 gates, by warp 0; src may be global.
__device__ __forceinline__ void chunk_cumsum_warp0(const float *src, float *dst, int C)
{
    if (threadIdx.x >= 32) return;
    const int lane = threadIdx.x;
    const int per = (C + 31) / 32;
    float loc[4];
    float run = 0.f;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        int idx = lane * per + u;
        float x = (u < per && idx < C) ? src[idx] : 0.f;
        run += x;
        loc[u] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    float excl = incl - run;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        int idx = lane * per + u;
        if (u < per && idx < C) dst[idx] = excl + loc[u];
    }
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
simt_chunk_state_kernel(const Tin *__restrict__ k, const Tin *__restrict__ v,
                        const float *__restrict__ g, float *__restrict__ gam,
                        float *__restrict__ nodes, int T, int dk, int dv, int C, int N)
{
    static_assert(kThreads == kOuterThreads && kSub == kOuterSub, "outer-product tiling");
    extern __shared__ __align__(16) float sm[];
    float *gl = sm;                // [128] gamma
    float *sc = gl + 128;          // [kSub] row scales exp(Gam - gamma)
    float *ks = sc + kSub;         // [kSub][dk]
    float *vs = ks + kSub * dk;    // [kSub][dv], rows scaled
    const int i = blockIdx.x;
    const long long bh = blockIdx.y;
    const long long tok0 = bh * (long long)T + (long long)i * C;

    chunk_cumsum_warp0(g + tok0, gl, C);
    __syncthreads();
    const float Gam = gl[C - 1];
    if (threadIdx.x == 0) gam[bh * N + i] = Gam;
    if (i == N - 1) return;  // the last chunk's state starts no node

    float acc[8][8];
    outer_zero(acc);
    for (int s0 = 0; s0 < C; s0 += kSub) {
        const int ns = min(kSub, C - s0);
        if (threadIdx.x < kSub) sc[threadIdx.x] = threadIdx.x < ns ? expf(Gam - gl[s0 + threadIdx.x]) : 0.f;
        __syncthreads();
        outer_stage<Tin>(ks, k + (tok0 + s0) * dk, nullptr, ns, dk);
        outer_stage<Tin>(vs, v + (tok0 + s0) * dv, sc, ns, dv);
        __syncthreads();
        outer_accumulate(acc, ks, vs, ns, dk, dv);
    }
    outer_store(nodes + (bh * N + (i + 1)) * (long long)dk * dv, acc, dk, dv, false);
}

// P[bh][j] = sum_{i<j} gam[bh][i] in fp64, j = 0..N.
__global__ void __launch_bounds__(kThreads)
simt_gate_prefix_kernel(const float *__restrict__ gam, double *__restrict__ P, int N)
{
    __shared__ double wsum[kThreads / 32];
    const long long bh = blockIdx.x;
    const int per = (N + kThreads - 1) / kThreads;
    const int lo = min(N, (int)threadIdx.x * per), hi = min(N, lo + per);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    double s = 0.0;
    for (int j = lo; j < hi; j++) s += (double)gam[bh * N + j];
    // exclusive prefix of the per-thread sums: within the warp, then over warps
    double incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
        const double xw = lane < kThreads / 32 ? wsum[lane] : 0.0;
        double wi = xw;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, wi, off);
            if (lane >= off) wi += y;
        }
        if (lane < kThreads / 32) wsum[lane] = wi - xw;  // sum over earlier warps
    }
    __syncthreads();
    double run = (incl - s) + wsum[w];
    double *Pb = P + bh * (long long)(N + 1);
    for (int j = lo; j < hi; j++) {
        Pb[j] = run;
        run += (double)gam[bh * N + j];
    }
    if (threadIdx.x == kThreads - 1) Pb[N] = run;
}

// In-place Fenwick scan, level by level: slot j (1..N-1) holds H_{j-1} and becomes
//     Node_j = H_{j-1} + sum_{m < ctz(j)} exp(P_j - P_{j-2^m}) Node_{j-2^m}.
// Every node of level z reads only nodes of lower levels, so the nodes of one
// level are independent.  The CTA forms the weights of a batch of up to
// kScanBatch nodes of one level in shared memory (one fp64 difference each,
// shared by every element), then each thread updates four adjacent elements
// (float4) of four nodes at a time, all loads of the four before their stores.
constexpr int kScanBatch = 256;
constexpr int kScanMaxZ = 20;  // levels of a chunk index below 2^20

__global__ void __launch_bounds__(kThreads)
simt_fenwick_scan_kernel(const double *__restrict__ P, float *__restrict__ nodes, int N, int E)
{
    __shared__ float wt[kScanBatch * kScanMaxZ];
    const long long bh = blockIdx.y;
    const int e4 = blockIdx.x * kThreads + threadIdx.x;  // float4 index within a node
    const bool act = 4 * e4 < E;
    const double *Pb = P + bh * (long long)(N + 1);
    float4 *base = reinterpret_cast<float4 *>(nodes + bh * (long long)N * E) + e4;
    const long long E4 = E / 4;
    for (int z = 1; (1 << z) < N; z++) {
        const int step = 2 << z;
        const int nz = (N - (1 << z) + step - 1) / step;  // nodes of level z: j = 2^z + n step
        for (int n0 = 0; n0 < nz; n0 += kScanBatch) {
            const int nb = min(kScanBatch, nz - n0);
            __syncthreads();  // the previous batch's weights are no longer read
            for (int x = threadIdx.x; x < nb * z; x += kThreads) {
                const int n = x / z, m = x % z;
                const int j = (1 << z) + (n0 + n) * step;
                wt[n * kScanMaxZ + m] = expf((float)(Pb[j] - Pb[j - (1 << m)]));
            }
            __syncthreads();
            if (!act) continue;
            for (int n = 0; n < nb; n += 4) {
                float4 val[4];
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    if (n + u >= nb) break;
                    const int j = (1 << z) + (n0 + n + u) * step;
                    val[u] = base[(long long)j * E4];
                    const float *w = wt + (n + u) * kScanMaxZ;
                    for (int m = 0; m < z; m++) {
                        const float4 lo = base[(long long)(j - (1 << m)) * E4];
                        val[u].x = fmaf(w[m], lo.x, val[u].x);
                        val[u].y = fmaf(w[m], lo.y, val[u].y);
                        val[u].z = fmaf(w[m], lo.z, val[u].z);
                        val[u].w = fmaf(w[m], lo.w, val[u].w);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    if (n + u >= nb) break;
                    base[(long long)((1 << z) + (n0 + n + u) * step) * E4] = val[u];
                }
            }
        }
    }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads)
simt_chunk_output_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k,
                         const Tin *__restrict__ v, const float *__restrict__ g,
                         const float *__restrict__ lam, const double *__restrict__ P,
                         const float *__restrict__ nodes, Tout *__restrict__ out,
                         int T, int dk, int dv, int C, int cbits, int N, int L)
{
    extern __shared__ float sm[];
    const int ldkv = (dk > dv ? dk : dv) + 1;
    float *gl = sm;                    // [128]
    float *Qs = gl + 128;              // [C][dk]
    float *KVs = Qs + C * dk;          // [C][ldkv]: K rows, then V rows
    float *Ps = KVs + C * ldkv;        // [C][C] masked scores
    float *Nt = Ps + C * C;            // [16][dv] node rows
    float *Ls = Nt + 16 * dv;          // [C][L] lambda rows
    const int i = blockIdx.x;
    const long long bh = blockIdx.y;
    const long long tok0 = bh * (long long)T + (long long)i * C;

    chunk_cumsum_warp0(g + tok0, gl, C);
    for (int e = threadIdx.x; e < C * dk; e += kThreads) {
        Qs[e] = to_f32(q[tok0 * dk + e]);
        int s = e / dk, r = e % dk;
        KVs[s * ldkv + r] = to_f32(k[tok0 * dk + e]);
    }
    for (int e = threadIdx.x; e < C * L; e += kThreads) Ls[e] = lam[tok0 * L + e];
    __syncthreads();

    // masked scores: M[a][b] = lambda_a[bit_length(a^b)] exp(gamma_a - gamma_b), b <= a
    for (int e = threadIdx.x; e < C * C; e += kThreads) {
        int a = e / C, b = e % C;
        float s = 0.f;
        if (b <= a) {
            float d = 0.f;
            for (int r = 0; r < dk; r++) d = fmaf(Qs[a * dk + r], KVs[b * ldkv + r], d);
            s = d * Ls[a * L + bit_length_u32((uint32_t)(a ^ b))] * expf(gl[a] - gl[b]);
        }
        Ps[e] = s;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < C * dv; e += kThreads) {
        int s = e / dv, cc = e % dv;
        KVs[s * ldkv + cc] = to_f32(v[tok0 * dv + e]);
    }
    __syncthreads();

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int RB = C / 16, CB = dv / 16;
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; a++)
#pragma unroll
        for (int b = 0; b < 8; b++) acc[a][b] = 0.f;
    for (int b = 0; b < C; b++) {
        float vc[8];
#pragma unroll
        for (int jj = 0; jj < 8; jj++) vc[jj] = (jj < CB) ? KVs[b * ldkv + tx + 16 * jj] : 0.f;
#pragma unroll
        for (int a = 0; a < 8; a++) {
            float p = (a < RB) ? Ps[(ty + 16 * a) * C + b] : 0.f;
#pragma unroll
            for (int jj = 0; jj < 8; jj++) acc[a][jj] = fmaf(p, vc[jj], acc[a][jj]);
        }
    }

    // read-out over the chunk-level Fenwick path of [0, i)
    const double *Pb = P + bh * (long long)(N + 1);
    for (int j = i; j > 0; j -= (j & -j)) {
        const int m = ctz_u32((uint32_t)j);
        const int lev = cbits + 1 + m;
        const float dP = (float)(Pb[i] - Pb[j]);
        const float *Nd = nodes + (bh * N + j) * (long long)dk * dv;
        float u[8][8];
#pragma unroll
        for (int a = 0; a < 8; a++)
#pragma unroll
            for (int b = 0; b < 8; b++) u[a][b] = 0.f;
        for (int r0 = 0; r0 < dk; r0 += 16) {
            __syncthreads();
            for (int e = threadIdx.x; e < 16 * dv; e += kThreads) Nt[e] = Nd[r0 * dv + e];
            __syncthreads();
            for (int rr = 0; rr < 16; rr++) {
                float nc[8];
#pragma unroll
                for (int jj = 0; jj < 8; jj++) nc[jj] = (jj < CB) ? Nt[rr * dv + tx + 16 * jj] : 0.f;
#pragma unroll
                for (int a = 0; a < 8; a++) {
                    float qv = (a < RB) ? Qs[(ty + 16 * a) * dk + r0 + rr] : 0.f;
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) u[a][jj] = fmaf(qv, nc[jj], u[a][jj]);
                }
            }
        }
#pragma unroll
        for (int a = 0; a < 8; a++) {
            if (a < RB) {
                int row = ty + 16 * a;
                float w = Ls[row * L + lev] * expf(gl[row] + dP);
#pragma unroll
                for (int jj = 0; jj < 8; jj++) acc[a][jj] = fmaf(w, u[a][jj], acc[a][jj]);
            }
        }
    }
#pragma unroll
    for (int a = 0; a < 8; a++)
#pragma unroll
        for (int jj = 0; jj < 8; jj++)
            if (a < RB && jj < CB)
                out[(tok0 + ty + 16 * a) * dv + tx + 16 * jj] = from_f32<Tout>(acc[a][jj]);
}

// Steps 1-3 only (chunk states, fp64 prefix, Fenwick scan) into the workspace.
template <typename Tin>
cudaError_t launch_nodes(const SimtFwdArgs &A, bool states = true)
{
    const int BH = A.B * A.H;
    const int N = A.T / A.C;
    cudaStream_t st = (cudaStream_t)A.stream;
    char *ws = (char *)A.workspace;
    float *gam = (float *)ws;
    double *P = (double *)(ws + simt_ws_offset_P(A));
    float *nodes = (float *)(ws + simt_ws_offset_nodes(A));
    if (states) {
        size_t sm1 = sizeof(float) * (128 + kSub + kSub * A.dk + kSub * A.dv);
        simt_chunk_state_kernel<Tin><<<dim3(N, BH), kThreads, sm1, st>>>(
            (const Tin *)A.k, (const Tin *)A.v, A.g, gam, nodes, A.T, A.dk, A.dv, A.C, N);
    }
    simt_gate_prefix_kernel<<<BH, kThreads, 0, st>>>(gam, P, N);
    const int E = A.dk * A.dv;  // a multiple of 256: every node row splits into float4s
    if (N > 1)
        simt_fenwick_scan_kernel<<<dim3((E / 4 + kThreads - 1) / kThreads, BH), kThreads, 0, st>>>(
            P, nodes, N, E);
    return cudaPeekAtLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_all(const SimtFwdArgs &A)
{
    const int BH = A.B * A.H;
    const int N = A.T / A.C;
    cudaStream_t st = (cudaStream_t)A.stream;
    char *ws = (char *)A.workspace;
    double *P = (double *)(ws + simt_ws_offset_P(A));
    float *nodes = (float *)(ws + simt_ws_offset_nodes(A));
    cudaError_t err = launch_nodes<Tin>(A);
    if (err != cudaSuccess) return err;
    const int ldkv = (A.dk > A.dv ? A.dk : A.dv) + 1;
    size_t sm4 = sizeof(float) * (128 + A.C * A.dk + A.C * ldkv + A.C * A.C + 16 * A.dv + A.C * A.L);
    auto kern = simt_chunk_output_kernel<Tin, Tout>;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm4);
    if (err != cudaSuccess) return err;
    int cbits = ctz_u32((uint32_t)A.C);
    kern<<<dim3(N, BH), kThreads, sm4, st>>>(
        (const Tin *)A.q, (const Tin *)A.k, (const Tin *)A.v, A.g, A.lam, P, nodes,
        (Tout *)A.out, A.T, A.dk, A.dv, A.C, cbits, N, A.L);
    return cudaPeekAtLastError();
}

}  // namespace

size_t simt_ws_offset_P(const SimtFwdArgs &A)
{
    const size_t BH = (size_t)A.B * A.H, N = (size_t)(A.T / A.C);
    return align_up(BH * N * sizeof(float), 256);
}

size_t simt_ws_offset_nodes(const SimtFwdArgs &A)
{
    const size_t BH = (size_t)A.B * A.H, N = (size_t)(A.T / A.C);
    return simt_ws_offset_P(A) + align_up(BH * (N + 1) * sizeof(double), 256);
}

size_t simt_workspace_bytes(const SimtFwdArgs &A)
{
    const size_t BH = (size_t)A.B * A.H, N = (size_t)(A.T / A.C);
    return simt_ws_offset_nodes(A) + align_up(BH * N * (size_t)A.dk * A.dv * sizeof(float), 256);
}

size_t simt_max_smem_bytes(const SimtFwdArgs &A)
{
    const int ldkv = (A.dk > A.dv ? A.dk : A.dv) + 1;
    return sizeof(float) * (128 + (size_t)A.C * A.dk + (size_t)A.C * ldkv + (size_t)A.C * A.C +
                            16 * (size_t)A.dv + (size_t)A.C * A.L);
}

cudaError_t simt_build_nodes(const SimtFwdArgs &A)
{
    return A.in_dt == LLA_F32 ? launch_nodes<float>(A) : launch_nodes<__nv_bfloat16>(A);
}

cudaError_t simt_nodes_from_states(const SimtFwdArgs &A)
{
    return launch_nodes<float>(A, false);  // the input type is not read
}

cudaError_t simt_fwd(const SimtFwdArgs &A)
{
    if (A.in_dt == LLA_F32 && A.out_dt == LLA_F32) return launch_all<float, float>(A);
    if (A.in_dt == LLA_BF16 && A.out_dt == LLA_F32) return launch_all<__nv_bfloat16, float>(A);
    return launch_all<__nv_bfloat16, __nv_bfloat16>(A);
}

}  // namespace lla
