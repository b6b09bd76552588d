// Backward of the chunked forward on CUDA cores (fp32 arithmetic).
//
// The pages give no gradients; these follow from the definition of
// "Log-Linear Attention" §2.2 (with the Mamba-2 gate of §3).  With
// A_ts = lambda_t[l(t,s)] exp(G_t - G_s) for s <= t and dO the incoming
// gradient of o:
//   dq_t      = sum_s A_ts (dO_t . v_s) k_s
//   dk_s      = sum_t A_ts (dO_t . v_s) q_t,   dv_s = sum_t A_ts (q_t . k_s) dO_t
//   dlam_t[l] = sum_{s: l(t,s) = l} exp(G_t - G_s) (q_t . k_s)(dO_t . v_s)
//   dG_u      = sum_l lam_u[l] dlam_u[l] - k_u . dk_u,   dg_r = sum_{u >= r} dG_u.
// Chunk i holds tokens [iC, iC+C).  The query side (dq, dlam) reads out the
// forward's chunk-level Fenwick nodes along the path of i: for the node j
// (level m = ctz(j)),  dq_t += lambda_t[c+1+m] w_t Node_j dO_t and
// dlam_t[c+1+m] += w_t q_t . (Node_j dO_t), w_t = exp(gamma_t + P_i - P_j).
// The key side (dk, dv) looks right: the chunks j > i with
// bit_length(i XOR j) = m+1 form the aligned block b = (i >> m) + 1 of 2^m
// chunks (bit m of i clear), every pair at level c+1+m, so one state per
// (level, block) serves them:
//   R_{m,b} = sum_{t in block} lambda_t[c+1+m] exp(G_t - G_ref) q_t dO_t^T,
//   ref = last token before the block;  dk_s += f_s R v_s,  dv_s += f_s R^T k_s,
//   f_s = exp(G_ref - G_s).  Pairs inside a chunk use the masked C x C scores.
// Every sum runs in a fixed order (no atomics), so the result is bitwise
// reproducible from call to call.
#include "bwd_simt.cuh"
#include "fwd_simt.cuh"
#include "outer_simt.cuh"

namespace lla {
namespace {

constexpr int kThreads = 256;

// gamma [BH][T]: inclusive gate sum inside each chunk (C <= 128), by one warp.
__global__ void __launch_bounds__(32)
bwd_gamma_kernel(const float *__restrict__ g, float *__restrict__ gamma, int T, int C)
{
    const long long tok0 = (long long)blockIdx.y * T + (long long)blockIdx.x * C;
    const int lane = threadIdx.x;
    const int per = (C + 31) / 32;
    float loc[4];
    float run = 0.f;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int idx = lane * per + u;
        run += (u < per && idx < C) ? g[tok0 + idx] : 0.f;
        loc[u] = run;
    }
    float incl = run;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
    }
    const float excl = incl - run;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        const int idx = lane * per + u;
        if (u < per && idx < C) gamma[tok0 + idx] = excl + loc[u];
    }
}

constexpr int kCk = 64;  // dv columns of a node staged at a time

size_t query_smem_floats(int C, int Dk, int Dv, int L)
{
    const size_t lk = Dk + 1, lv = Dv + 1;
    const size_t intra = 3 * (size_t)C * C;
    const size_t node = (size_t)kCk * Dk;
    const size_t scratch = intra > node ? intra : node;
    return 128 + 2 * (size_t)C * lk + 2 * (size_t)C * lv + scratch + 2 * (size_t)C * L;
}

// Per chunk: intra-chunk parts of dq, dk, dv, dlam, then the query side of
// the earlier chunks (dq, dlam) through the forward's Fenwick path nodes.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
bwd_query_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                 const float *__restrict__ dout, const float *__restrict__ gamma,
                 const float *__restrict__ lam, const double *__restrict__ P,
                 const float *__restrict__ nodes, float *__restrict__ dq, float *__restrict__ dk,
                 float *__restrict__ dv, float *__restrict__ dlam, int T, int Dk, int Dv, int C,
                 int cbits, int N, int L, int do_path)
{
    extern __shared__ float sm[];
    const int lk = Dk + 1, lv = Dv + 1;
    float *gl = sm;                 // [C]
    float *Qs = gl + 128;           // [C][lk]
    float *Ks = Qs + C * lk;        // [C][lk]
    float *Vs = Ks + C * lk;        // [C][lv]
    float *Ds = Vs + C * lv;        // [C][lv]  dO
    float *Ls = Ds + C * lv;        // [C][L]   lambda rows
    float *dL = Ls + C * L;         // [C][L]   dlam accumulators
    float *W1 = dL + C * L;         // [C][C]   M . (dO.v)      (intra phase)
    float *W2 = W1 + C * C;         // [C][C]   M . (q.k)
    float *X = W2 + C * C;          // [C][C]   decay . (q.k)(dO.v)
    float *Nt = W1;                 // [kCk][Dk] node columns, transposed (path phase)
    const int i = blockIdx.x;
    const long long bh = blockIdx.y;
    const long long tok0 = bh * (long long)T + (long long)i * C;
    for (int e = threadIdx.x; e < C; e += kThreads) gl[e] = gamma[tok0 + e];
    for (int e = threadIdx.x; e < C * Dk; e += kThreads) {
        const int t = e / Dk, r = e % Dk;
        Qs[t * lk + r] = to_f32(q[tok0 * Dk + e]);
        Ks[t * lk + r] = to_f32(k[tok0 * Dk + e]);
    }
    for (int e = threadIdx.x; e < C * Dv; e += kThreads) {
        const int t = e / Dv, c = e % Dv;
        Vs[t * lv + c] = to_f32(v[tok0 * Dv + e]);
        Ds[t * lv + c] = dout[tok0 * Dv + e];
    }
    for (int e = threadIdx.x; e < C * L; e += kThreads) Ls[e] = lam[tok0 * L + e];
    __syncthreads();
    // Masked pair weights.  Thread (ty, tx) computes the 4 x 4 block of
    // pairs t = 4 ty + i, s = 4 tx + j of S = Q K^T and dP = dO V^T.
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    {
        const int t0 = 4 * ty, s0 = 4 * tx;
        if (t0 < C && s0 < C && s0 <= t0 + 3) {
            float qk[4][4], ov[4][4];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) qk[i][j] = ov[i][j] = 0.f;
            for (int r = 0; r < Dk; r++) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; i++) a[i] = Qs[(t0 + i) * lk + r];
#pragma unroll
                for (int j = 0; j < 4; j++) b[j] = Ks[(s0 + j) * lk + r];
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int j = 0; j < 4; j++) qk[i][j] = fmaf(a[i], b[j], qk[i][j]);
            }
            for (int c = 0; c < Dv; c++) {
                float a[4], b[4];
#pragma unroll
                for (int i = 0; i < 4; i++) a[i] = Ds[(t0 + i) * lv + c];
#pragma unroll
                for (int j = 0; j < 4; j++) b[j] = Vs[(s0 + j) * lv + c];
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int j = 0; j < 4; j++) ov[i][j] = fmaf(a[i], b[j], ov[i][j]);
            }
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    const int t = t0 + i, s2 = s0 + j;
                    float w1 = 0.f, w2 = 0.f, x = 0.f;
                    if (s2 <= t) {
                        const float dec = expf(gl[t] - gl[s2]);
                        const float m = Ls[t * L + bit_length_u32((uint32_t)(t ^ s2))] * dec;
                        w1 = m * ov[i][j];
                        w2 = m * qk[i][j];
                        x = dec * qk[i][j] * ov[i][j];
                    }
                    W1[t * C + s2] = w1;
                    W2[t * C + s2] = w2;
                    X[t * C + s2] = x;
                }
        } else if (t0 < C && s0 < C) {  // blocks above the diagonal
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    W1[(t0 + i) * C + s0 + j] = 0.f;
                    W2[(t0 + i) * C + s0 + j] = 0.f;
                    X[(t0 + i) * C + s0 + j] = 0.f;
                }
        }
    }
    __syncthreads();
    // intra-chunk level gradients: level 0 is s = t, level l >= 1 the keys
    // s < t with bit l-1 the highest bit where s and t differ
    for (int e = threadIdx.x; e < C * L; e += kThreads) {
        const int t = e / L, l = e % L;
        float a = 0.f;
        if (l == 0) {
            a = X[t * C + t];
        } else if (l <= cbits && ((t >> (l - 1)) & 1)) {
            const int lo = (t >> l) << l, hi = lo + (1 << (l - 1));
            for (int s2 = lo; s2 < hi; s2++) a += X[t * C + s2];
        }
        dL[e] = a;
    }
    // Intra parts: dq_t = sum_s W1[t][s] k_s and, with t as a key,
    // dk_t = sum_u W1[u][t] q_u; dv_t = sum_u W2[u][t] dO_u.  Thread (ty, tx)
    // owns rows 4 ty .. 4 ty + 3 and columns tx, tx + 16, ... (conflict-free
    // row reads of K, Q, dO).
    {
        const int t0 = 4 * ty;
        const int RK = Dk / 16, RV = Dv / 16;
        if (t0 < C) {
            float aq[4][8], ak[4][8];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int c = 0; c < 8; c++) aq[i][c] = ak[i][c] = 0.f;
            for (int u = 0; u < C; u++) {
                float wq[4], wk[4], kv[8], qv[8];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    wq[i] = W1[(t0 + i) * C + u];  // t0+i as query, u as key
                    wk[i] = W1[u * C + t0 + i];    // u as query, t0+i as key
                }
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    kv[c] = c < RK ? Ks[u * lk + tx + 16 * c] : 0.f;
                    qv[c] = c < RK ? Qs[u * lk + tx + 16 * c] : 0.f;
                }
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int c = 0; c < 8; c++) {
                        aq[i][c] = fmaf(wq[i], kv[c], aq[i][c]);
                        ak[i][c] = fmaf(wk[i], qv[c], ak[i][c]);
                    }
            }
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int c = 0; c < 8; c++)
                    if (c < RK) {
                        dq[(tok0 + t0 + i) * Dk + tx + 16 * c] = aq[i][c];
                        dk[(tok0 + t0 + i) * Dk + tx + 16 * c] = ak[i][c];
                    }
            float av[4][8];
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int c = 0; c < 8; c++) av[i][c] = 0.f;
            for (int u = 0; u < C; u++) {
                float wv[4], dvv[8];
#pragma unroll
                for (int i = 0; i < 4; i++) wv[i] = W2[u * C + t0 + i];
#pragma unroll
                for (int c = 0; c < 8; c++) dvv[c] = c < RV ? Ds[u * lv + tx + 16 * c] : 0.f;
#pragma unroll
                for (int i = 0; i < 4; i++)
#pragma unroll
                    for (int c = 0; c < 8; c++) av[i][c] = fmaf(wv[i], dvv[c], av[i][c]);
            }
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int c = 0; c < 8; c++)
                    if (c < RV) dv[(tok0 + t0 + i) * Dv + tx + 16 * c] = av[i][c];
        }
    }
    __syncthreads();
    // Earlier chunks through the forward's path nodes.  Thread (ty, tx) owns
    // rows t0..t0+3 (t0 = 4 ty) and columns r0..r0+7 (r0 = 8 tx) of
    // U = dO Node_j^T; dq accumulates in registers over the path.
    const double *Pb = P + bh * (long long)(N + 1);
    const int t0 = 4 * ty, r0 = 8 * tx;
    const bool own = t0 < C && r0 < Dk;
    float dqa[4][8];
#pragma unroll
    for (int a = 0; a < 4; a++)
#pragma unroll
        for (int c = 0; c < 8; c++) dqa[a][c] = 0.f;
    for (int j = do_path ? i : 0; j > 0; j -= (j & -j)) {
        const int lev = cbits + 1 + ctz_u32((uint32_t)j);
        const float dP = (float)(Pb[i] - Pb[j]);
        const float *Nd = nodes + (bh * N + j) * (long long)Dk * Dv;
        float u[4][8];
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int c = 0; c < 8; c++) u[a][c] = 0.f;
        for (int c0 = 0; c0 < Dv; c0 += kCk) {
            const int nc = min(kCk, Dv - c0);
            __syncthreads();
            for (int e = threadIdx.x; e < Dk * (nc / 4); e += kThreads) {
                const int r = e % Dk, c4 = e / Dk;
                const float4 x = *reinterpret_cast<const float4 *>(Nd + (long long)r * Dv + c0 + 4 * c4);
                Nt[(4 * c4 + 0) * Dk + r] = x.x;
                Nt[(4 * c4 + 1) * Dk + r] = x.y;
                Nt[(4 * c4 + 2) * Dk + r] = x.z;
                Nt[(4 * c4 + 3) * Dk + r] = x.w;
            }
            __syncthreads();
            if (own) {
                for (int cc = 0; cc < nc; cc++) {
                    float dv4[4];
#pragma unroll
                    for (int a = 0; a < 4; a++) dv4[a] = Ds[(t0 + a) * lv + c0 + cc];
                    const float4 n0 = *reinterpret_cast<const float4 *>(Nt + cc * Dk + r0);
                    const float4 n1 = *reinterpret_cast<const float4 *>(Nt + cc * Dk + r0 + 4);
                    const float nn[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
#pragma unroll
                    for (int a = 0; a < 4; a++)
#pragma unroll
                        for (int c = 0; c < 8; c++) u[a][c] = fmaf(dv4[a], nn[c], u[a][c]);
                }
            }
        }
        // dq_t += lambda_t[lev] w_t U_t ;  dlam_t[lev] += w_t q_t . U_t
        float part[4];
#pragma unroll
        for (int a = 0; a < 4; a++) {
            const int t = min(t0 + a, C - 1);
            const float w = expf(gl[t] + dP);
            const float lw = Ls[t * L + lev] * w;
            float pr = 0.f;
#pragma unroll
            for (int c = 0; c < 8; c++) {
                dqa[a][c] = fmaf(lw, u[a][c], dqa[a][c]);
                pr = fmaf(own ? Qs[t * lk + r0 + c] : 0.f, u[a][c], pr);
            }
            part[a] = w * pr;
        }
#pragma unroll
        for (int a = 0; a < 4; a++)
#pragma unroll
            for (int off = 8; off > 0; off >>= 1) part[a] += __shfl_xor_sync(0xffffffffu, part[a], off, 16);
        if (tx == 0 && t0 < C) {
#pragma unroll
            for (int a = 0; a < 4; a++) dL[(t0 + a) * L + lev] += part[a];
        }
    }
    __syncthreads();
    if (own && i > 0 && do_path) {
#pragma unroll
        for (int a = 0; a < 4; a++) {
            float *dst = dq + (tok0 + t0 + a) * Dk + r0;
            float4 x0 = *reinterpret_cast<float4 *>(dst), x1 = *reinterpret_cast<float4 *>(dst + 4);
            x0.x += dqa[a][0]; x0.y += dqa[a][1]; x0.z += dqa[a][2]; x0.w += dqa[a][3];
            x1.x += dqa[a][4]; x1.y += dqa[a][5]; x1.z += dqa[a][6]; x1.w += dqa[a][7];
            *reinterpret_cast<float4 *>(dst) = x0;
            *reinterpret_cast<float4 *>(dst + 4) = x1;
        }
    }
    for (int e = threadIdx.x; e < C * L; e += kThreads) dlam[tok0 * L + e] = dL[e];
}

// Work items of the block states: level m, odd block b (chunks
// [b 2^m, min(N, (b+1) 2^m))) and a piece of at most Pc of those chunks.
// Level m has nb/2 odd blocks (nb = ceil(N / 2^m)), each cut into
// ceil(2^m / Pc) pieces (empty pieces of a short last block do nothing).
struct Item {
    int m, b, p, pp;
};

__device__ __forceinline__ bool decode_item(int idx, int N, int nlev, int Pc, Item *it)
{
    for (int m = 0; m < nlev; m++) {
        const int nb = (N + (1 << m) - 1) >> m;
        const int pp = ((1 << m) + Pc - 1) / Pc;
        const int cnt = (nb / 2) * pp;
        if (idx < cnt) {
            it->m = m;
            it->b = 2 * (idx / pp) + 1;
            it->p = idx % pp;
            it->pp = pp;
            return true;
        }
        idx -= cnt;
    }
    return false;
}

// One piece of R_{m,b} = sum_t lambda_t[c+1+m] exp(G_t - G_ref) q_t dO_t^T.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
bwd_block_piece_kernel(const Tin *__restrict__ q, const float *__restrict__ dout,
                       const float *__restrict__ gamma, const float *__restrict__ lam,
                       const double *__restrict__ P, float *__restrict__ part, int T, int Dk, int Dv,
                       int C, int cbits, int N, int L, int nlev, int Pc)
{
    __shared__ __align__(16) float qs[kOuterSub * 128];
    __shared__ __align__(16) float ds[kOuterSub * 128];
    __shared__ float sc[kOuterSub];
    const long long bh = blockIdx.y;
    Item it;
    if (!decode_item(blockIdx.x, N, nlev, Pc, &it)) return;
    const int c0 = it.b << it.m;
    const int blk_end = min(N, (it.b + 1) << it.m);
    const int p0 = c0 + it.p * Pc, p1 = min(blk_end, p0 + Pc);
    if (p0 >= p1) return;
    const int lev = cbits + 1 + it.m;
    const double *Pb = P + bh * (long long)(N + 1);
    const double Pref = Pb[c0];
    float acc[8][8];
    outer_zero(acc);
    const long long t_lo = (long long)p0 * C, t_hi = (long long)p1 * C;
    for (long long t0 = t_lo; t0 < t_hi; t0 += kOuterSub) {
        const int nt = (int)min((long long)kOuterSub, t_hi - t0);
        if (threadIdx.x < kOuterSub) {
            float w = 0.f;
            if ((int)threadIdx.x < nt) {
                const long long t = t0 + threadIdx.x;
                const long long gi = bh * T + t;
                w = lam[gi * L + lev] * expf((float)(Pb[t / C] - Pref) + gamma[gi]);
            }
            sc[threadIdx.x] = w;
        }
        __syncthreads();
        outer_stage<Tin>(qs, q + (bh * T + t0) * Dk, sc, nt, Dk);
        outer_stage<float>(ds, dout + (bh * T + t0) * Dv, nullptr, nt, Dv);
        __syncthreads();
        outer_accumulate(acc, qs, ds, nt, Dk, Dv);
    }
    outer_store(part + ((bh * gridDim.x) + blockIdx.x) * (long long)Dk * Dv, acc, Dk, Dv, false);
}

// R_{m,b} = sum of its pieces in piece order (bitwise reproducible).  One
// CTA per (odd block, slice of its elements) of the levels whose blocks span
// several pieces (2^m > Pc); a ragged last block of one piece exits
// (block_state reads the piece itself, as for every block of the lower
// levels).
__global__ void __launch_bounds__(kThreads)
bwd_block_reduce_kernel(const float *__restrict__ part, float *__restrict__ R, int Dk, int Dv, int N,
                        int nlev, int Pc, int nitems, int nblocks)
{
    const long long bh = blockIdx.y;
    int idx = blockIdx.x, m = 0, off = 0, first = 0;
    for (; m < nlev; m++) {
        const int nb = (N + (1 << m) - 1) >> m;
        const int pp = ((1 << m) + Pc - 1) / Pc;
        if (pp > 1) {
            if (idx < nb / 2) break;
            idx -= nb / 2;
        }
        off += nb;
        first += (nb / 2) * pp;
    }
    if (m >= nlev) return;
    const int b = 2 * idx + 1;
    const int pp = ((1 << m) + Pc - 1) / Pc;
    const int blk_end = min(N, (b + 1) << m);
    const int npieces = (blk_end - (b << m) + Pc - 1) / Pc;  // non-empty pieces
    if (npieces <= 1) return;
    const float4 *src = reinterpret_cast<const float4 *>(part) +
                        ((bh * nitems) + first + (b / 2) * pp) * (long long)(Dk * Dv / 4);
    float4 *dst = reinterpret_cast<float4 *>(R) + ((bh * nblocks) + off + b) * (long long)(Dk * Dv / 4);
    const int E4 = Dk * Dv / 4;
    // slice blockIdx.z of the block's elements; the pieces are added in piece
    // order, four loads issued before their additions
    const int per = (E4 + gridDim.z - 1) / gridDim.z;
    const int e_lo = blockIdx.z * per, e_hi = min(E4, e_lo + per);
    for (int e = e_lo + threadIdx.x; e < e_hi; e += kThreads) {
        float4 acc = src[e];
        int p = 1;
        for (; p + 3 < npieces; p += 4) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; u++) x[u] = src[(long long)(p + u) * E4 + e];
#pragma unroll
            for (int u = 0; u < 4; u++) {
                acc.x += x[u].x; acc.y += x[u].y; acc.z += x[u].z; acc.w += x[u].w;
            }
        }
        for (; p < npieces; p++) {
            const float4 x = src[(long long)p * E4 + e];
            acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
        }
        dst[e] = acc;
    }
}

constexpr int kRowsPer = 4;  // rows of a thread tile
constexpr int kColsPer = 8;  // columns of a thread tile

// Per chunk: the key side of the later chunks, over every level m whose
// right-hand block exists:  dk_s += f_s R v_s,  dv_s += f_s R^T k_s.
// Thread (ty, tx) owns rows s0..s0+3 and columns 8 tx..8 tx+7 of dk and of
// dv, accumulated in registers over the levels.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
bwd_key_kernel(const Tin *__restrict__ k, const Tin *__restrict__ v, const float *__restrict__ gamma,
               const double *__restrict__ P, const float *__restrict__ R, const float *__restrict__ part,
               float *__restrict__ dk, float *__restrict__ dv, int T, int Dk, int Dv, int C, int N, int nlev,
               int nblocks, int Pc, int nitems)
{
    extern __shared__ __align__(16) float sm[];
    const int lk = Dk + 1, lv = Dv + 1;
    float *Rb = sm;               // [Dk*Dv] R or R^T
    float *Ks = Rb + Dk * Dv;     // [C][lk]
    float *Vs = Ks + C * lk;      // [C][lv]
    float *gl = Vs + C * lv;      // [C]
    const int i = blockIdx.x;
    const long long bh = blockIdx.y;
    const long long tok0 = bh * (long long)T + (long long)i * C;
    for (int e = threadIdx.x; e < C * Dk; e += kThreads) Ks[(e / Dk) * lk + e % Dk] = to_f32(k[tok0 * Dk + e]);
    for (int e = threadIdx.x; e < C * Dv; e += kThreads) Vs[(e / Dv) * lv + e % Dv] = to_f32(v[tok0 * Dv + e]);
    for (int e = threadIdx.x; e < C; e += kThreads) gl[e] = gamma[tok0 + e];
    __syncthreads();
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int s0 = kRowsPer * ty, x0 = kColsPer * tx;
    const bool rows_ok = s0 < C;
    const bool own_k = rows_ok && x0 < Dk, own_v = rows_ok && x0 < Dv;
    float dka[kRowsPer][kColsPer], dva[kRowsPer][kColsPer];
#pragma unroll
    for (int a = 0; a < kRowsPer; a++)
#pragma unroll
        for (int c = 0; c < kColsPer; c++) dka[a][c] = dva[a][c] = 0.f;
    const double *Pb = P + bh * (long long)(N + 1);
    bool any = false;
    for (int m = 0; m < nlev; m++) {
        const int b = (i >> m) + 1;
        if (((i >> m) & 1) == 0 && ((long long)b << m) < N) {
            any = true;
            const float *Rm = block_state(R, part, bh, m, b, N, Pc, nitems, nblocks, Dk * Dv);
            const float dP = (float)(Pb[b << m] - Pb[i]);
            float f[kRowsPer];
#pragma unroll
            for (int a = 0; a < kRowsPer; a++) f[a] = expf(dP - gl[min(s0 + a, C - 1)]);
            // dk: reduce over c with R^T staged ([c][r])
            __syncthreads();
            for (int e = threadIdx.x; e < Dk * (Dv / 4); e += kThreads) {
                const int r = e % Dk, c4 = e / Dk;
                const float4 x = *reinterpret_cast<const float4 *>(Rm + (long long)r * Dv + 4 * c4);
                Rb[(4 * c4 + 0) * Dk + r] = x.x;
                Rb[(4 * c4 + 1) * Dk + r] = x.y;
                Rb[(4 * c4 + 2) * Dk + r] = x.z;
                Rb[(4 * c4 + 3) * Dk + r] = x.w;
            }
            __syncthreads();
            if (own_k) {
                float t[kRowsPer][kColsPer];
#pragma unroll
                for (int a = 0; a < kRowsPer; a++)
#pragma unroll
                    for (int c = 0; c < kColsPer; c++) t[a][c] = 0.f;
                for (int c = 0; c < Dv; c++) {
                    float va[kRowsPer];
#pragma unroll
                    for (int a = 0; a < kRowsPer; a++) va[a] = Vs[(s0 + a) * lv + c];
                    const float4 r0 = *reinterpret_cast<const float4 *>(Rb + c * Dk + x0);
                    const float4 r1 = *reinterpret_cast<const float4 *>(Rb + c * Dk + x0 + 4);
                    const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                    for (int a = 0; a < kRowsPer; a++)
#pragma unroll
                        for (int cc = 0; cc < kColsPer; cc++) t[a][cc] = fmaf(va[a], rr[cc], t[a][cc]);
                }
#pragma unroll
                for (int a = 0; a < kRowsPer; a++)
#pragma unroll
                    for (int cc = 0; cc < kColsPer; cc++) dka[a][cc] = fmaf(f[a], t[a][cc], dka[a][cc]);
            }
            // dv: reduce over r with R staged as is ([r][c])
            __syncthreads();
            for (int e = threadIdx.x; e < Dk * Dv / 4; e += kThreads)
                reinterpret_cast<float4 *>(Rb)[e] = reinterpret_cast<const float4 *>(Rm)[e];
            __syncthreads();
            if (own_v) {
                float t[kRowsPer][kColsPer];
#pragma unroll
                for (int a = 0; a < kRowsPer; a++)
#pragma unroll
                    for (int c = 0; c < kColsPer; c++) t[a][c] = 0.f;
                for (int r = 0; r < Dk; r++) {
                    float ka[kRowsPer];
#pragma unroll
                    for (int a = 0; a < kRowsPer; a++) ka[a] = Ks[(s0 + a) * lk + r];
                    const float4 r0 = *reinterpret_cast<const float4 *>(Rb + r * Dv + x0);
                    const float4 r1 = *reinterpret_cast<const float4 *>(Rb + r * Dv + x0 + 4);
                    const float rr[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                    for (int a = 0; a < kRowsPer; a++)
#pragma unroll
                        for (int cc = 0; cc < kColsPer; cc++) t[a][cc] = fmaf(ka[a], rr[cc], t[a][cc]);
                }
#pragma unroll
                for (int a = 0; a < kRowsPer; a++)
#pragma unroll
                    for (int cc = 0; cc < kColsPer; cc++) dva[a][cc] = fmaf(f[a], t[a][cc], dva[a][cc]);
            }
        }
    }
    if (!any) return;
    auto add8 = [](float *dst, const float *x) {
        float4 a = *reinterpret_cast<float4 *>(dst), b = *reinterpret_cast<float4 *>(dst + 4);
        a.x += x[0]; a.y += x[1]; a.z += x[2]; a.w += x[3];
        b.x += x[4]; b.y += x[5]; b.z += x[6]; b.w += x[7];
        *reinterpret_cast<float4 *>(dst) = a;
        *reinterpret_cast<float4 *>(dst + 4) = b;
    };
#pragma unroll
    for (int a = 0; a < kRowsPer; a++) {
        if (own_k) add8(dk + (tok0 + s0 + a) * Dk + x0, dka[a]);
        if (own_v) add8(dv + (tok0 + s0 + a) * Dv + x0, dva[a]);
    }
}

// dG_u = sum_l lam_u[l] dlam_u[l] - k_u . dk_u, a warp per pair of tokens (fp32
// sums; the long running sum over tokens below is fp64).  With 16-byte aligned
// k and dk (VEC) each lane reads four consecutive elements of a row per load;
// both tokens' loads are issued before their sums.
template <typename Tin> struct Vec4;
template <> struct Vec4<float> {
    using type = float4;
    __device__ static void to_f32(const float4 &x, float (&f)[4]) { f[0] = x.x; f[1] = x.y; f[2] = x.z; f[3] = x.w; }
};
template <> struct Vec4<__nv_bfloat16> {
    using type = uint2;
    __device__ static void to_f32(const uint2 &x, float (&f)[4])
    {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&x);
        const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    }
};

template <typename Tin, bool VEC>
__global__ void __launch_bounds__(kThreads)
bwd_gate_grad_kernel(const Tin *__restrict__ k, const float *__restrict__ lam,
                     const float *__restrict__ dlam, const float *__restrict__ dk,
                     double *__restrict__ dG, int T, int Dk, int L)
{
    const int lane = threadIdx.x & 31;
    const int u0 = 2 * (blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5));
    if (u0 >= T) return;
    float a[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int u = u0 + e;
        if (u < T) {
            const long long gi = (long long)blockIdx.y * T + u;
            for (int l = lane; l < L; l += 32) a[e] = fmaf(lam[gi * L + l], dlam[gi * L + l], a[e]);
            if (VEC) {
                using V = typename Vec4<Tin>::type;
                for (int r = 4 * lane; r < Dk; r += 128) {
                    const V kv = *reinterpret_cast<const V *>(k + gi * Dk + r);
                    const float4 dv = *reinterpret_cast<const float4 *>(dk + gi * Dk + r);
                    float kf[4];
                    Vec4<Tin>::to_f32(kv, kf);
                    a[e] = fmaf(-kf[0], dv.x, a[e]);
                    a[e] = fmaf(-kf[1], dv.y, a[e]);
                    a[e] = fmaf(-kf[2], dv.z, a[e]);
                    a[e] = fmaf(-kf[3], dv.w, a[e]);
                }
            } else {
                for (int r = lane; r < Dk; r += 32) a[e] = fmaf(-to_f32(k[gi * Dk + r]), dk[gi * Dk + r], a[e]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < 2; e++) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a[e] += __shfl_xor_sync(0xffffffffu, a[e], off);
    }
    if (lane < 2 && u0 + lane < T) dG[(long long)blockIdx.y * T + u0 + lane] = (double)(lane ? a[1] : a[0]);
}

// dg_r = sum_{u >= r} dG_u per (batch, head), fp64.  One CTA of 1024 threads
// per block of kGateBlk tokens: first the sum of every token after the block
// (coalesced loads, four in flight per thread; the later blocks are read
// once per earlier block, from L2), then the suffix sums inside the block,
// four consecutive tokens per thread.  Every sum runs in a fixed order.
constexpr int kGateBlk = 4096;

__device__ __forceinline__ double warp_sum_f64(double x)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__global__ void __launch_bounds__(1024)
bwd_gate_scan_kernel(const double *__restrict__ dG, float *__restrict__ dg, int T)
{
    __shared__ double wsum[32];
    __shared__ double after_sh;
    const long long bh = blockIdx.y;
    const double *src = dG + bh * T;
    const int b0 = blockIdx.x * kGateBlk, b1 = min(T, b0 + kGateBlk);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    // the tokens after the block
    double a0 = 0.0, a1 = 0.0, a2 = 0.0, a3 = 0.0;
    int u = b1 + tid;
    for (; u + 3 * 1024 < T; u += 4 * 1024) {
        a0 += src[u];
        a1 += src[u + 1024];
        a2 += src[u + 2048];
        a3 += src[u + 3072];
    }
    for (; u < T; u += 1024) a0 += src[u];
    const double a = warp_sum_f64((a0 + a1) + (a2 + a3));
    if (lane == 0) wsum[w] = a;
    __syncthreads();
    if (w == 0) {
        const double x = warp_sum_f64(wsum[lane]);
        if (lane == 0) after_sh = x;
    }
    __syncthreads();
    const double after = after_sh;
    // the block
    const int t0 = b0 + 4 * tid;
    double x[4];
#pragma unroll
    for (int e = 0; e < 4; e++) x[e] = t0 + e < b1 ? src[t0 + e] : 0.0;
    const double sum4 = (x[0] + x[1]) + (x[2] + x[3]);
    double incl = sum4;  // inclusive suffix within the warp (lanes >= this one)
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32) incl += y;
    }
    if (lane == 0) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
        const double xw = wsum[lane];
        double wi = xw;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double y = __shfl_down_sync(0xffffffffu, wi, off);
            if (lane + off < 32) wi += y;
        }
        wsum[lane] = wi - xw;  // sum over later warps
    }
    __syncthreads();
    double run = after + (incl - sum4) + wsum[w];  // every token after this thread's four
#pragma unroll
    for (int e = 3; e >= 0; e--) {
        run += x[e];
        if (t0 + e < b1) dg[bh * T + t0 + e] = (float)run;
    }
}

int block_levels(int N) { return N > 1 ? bit_length_u32((uint32_t)(N - 1)) : 0; }

// R slots: every block of every level (odd ones used), flat by level.
int total_blocks(int N)
{
    int tot = 0;
    for (int m = 0; m < block_levels(N); m++) tot += (N + (1 << m) - 1) >> m;
    return tot;
}

int piece_chunks(int C) { return 1024 / C > 1 ? 1024 / C : 1; }

// Odd blocks of the levels whose blocks span several pieces (the reduction's CTAs).
int multi_piece_blocks(int N, int Pc)
{
    int tot = 0;
    for (int m = 0; m < block_levels(N); m++)
        if (((1 << m) + Pc - 1) / Pc > 1) tot += ((N + (1 << m) - 1) >> m) / 2;
    return tot;
}

int total_items(int N, int Pc)
{
    int tot = 0;
    for (int m = 0; m < block_levels(N); m++)
        tot += (((N + (1 << m) - 1) >> m) / 2) * (((1 << m) + Pc - 1) / Pc);
    return tot;
}

size_t key_smem_floats(int C, int Dk, int Dv)
{
    return (size_t)Dk * Dv + (size_t)C * (Dk + 1) + (size_t)C * (Dv + 1) + C;
}

SimtFwdArgs node_args(const BwdArgs &A)
{
    SimtFwdArgs F;
    F.q = A.q; F.k = A.k; F.v = A.v; F.g = A.g; F.lam = A.lam; F.out = nullptr;
    F.B = A.B; F.H = A.H; F.T = A.T; F.dk = A.dk; F.dv = A.dv; F.C = A.C; F.L = A.L;
    F.in_dt = A.in_dt; F.out_dt = LLA_F32; F.workspace = A.workspace; F.stream = A.stream;
    return F;
}

// Workspace: the CUDA-core forward's (chunk gate sums, P, nodes), then
// gamma [BH][T] fp32, R [BH][total_blocks][Dk][Dv] fp32,
// pieces [BH][total_items][Dk][Dv] fp32, dG [BH][T] fp64.
struct BwdLayout {
    size_t gamma, R, parts, dG, err, end;
};

BwdLayout layout(const BwdArgs &A)
{
    SimtFwdArgs F = node_args(A);
    const size_t BH = (size_t)A.B * A.H, st = (size_t)A.dk * A.dv * 4;
    const int N = A.T / A.C;
    BwdLayout l;
    l.gamma = simt_workspace_bytes(F);
    l.R = l.gamma + align_up(BH * A.T * 4, 256);
    l.parts = l.R + align_up(BH * (size_t)total_blocks(N) * st, 256);
    l.dG = l.parts + align_up(BH * (size_t)total_items(N, piece_chunks(A.C)) * st, 256);
    l.err = l.dG + align_up(BH * A.T * 8, 256);
    l.end = l.err + 256;
    return l;
}

template <typename Tin>
cudaError_t launch_bwd(const BwdArgs &A)
{
    const int BH = A.B * A.H, N = A.T / A.C;
    const int cbits = ctz_u32((uint32_t)A.C);
    cudaStream_t st = (cudaStream_t)A.stream;
    SimtFwdArgs F = node_args(A);
    char *ws = (char *)A.workspace;
    const BwdLayout lay = layout(A);
    const double *P = (const double *)(ws + simt_ws_offset_P(F));
    float *nodes = (float *)(ws + simt_ws_offset_nodes(F));
    float *gamma = (float *)(ws + lay.gamma);
    float *R = (float *)(ws + lay.R);
    float *parts = (float *)(ws + lay.parts);
    double *dG = (double *)(ws + lay.dG);
    // bounded waits of the tensor-core parts report into the caller's word,
    // else into a workspace word cleared before each part
    int *const err = A.device_error ? (int *)A.device_error : (int *)(ws + lay.err);
    auto clear_err = [&]() { return A.device_error ? cudaSuccess : cudaMemsetAsync(err, 0, sizeof(int), st); };
    bwd_gamma_kernel<<<dim3(N, BH), 32, 0, st>>>(A.g, gamma, A.T, A.C);
    cudaError_t e;
    if (bwd_state_tc_supported(A)) {
        // the forward's chunk states on the tensor cores, then its prefix and scan
        e = clear_err();
        if (e != cudaSuccess) return e;
        e = bwd_state_tc(A, gamma, (float *)ws, nodes, err);
        if (e != cudaSuccess) return e;
        e = simt_nodes_from_states(F);
    } else {
        e = simt_build_nodes(F);
    }
    if (e != cudaSuccess) return e;
    if (bwd_intra_tc_supported(A)) {
        e = clear_err();
        if (e != cudaSuccess) return e;
        e = bwd_intra_tc(A, gamma, err);
        if (e != cudaSuccess) return e;
    } else {
        const size_t smq = sizeof(float) * query_smem_floats(A.C, A.dk, A.dv, A.L);
        e = cudaFuncSetAttribute(bwd_query_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
        if (e != cudaSuccess) return e;
        bwd_query_kernel<Tin><<<dim3(N, BH), kThreads, smq, st>>>(
            (const Tin *)A.q, (const Tin *)A.k, (const Tin *)A.v, A.dout, gamma, A.lam, P, nodes, A.dq,
            A.dkey, A.dval, A.dlam, A.T, A.dk, A.dv, A.C, cbits, N, A.L, bwd_query_tc_supported(A) ? 0 : 1);
    }
    if (bwd_query_tc_supported(A) && N > 1) {
        e = clear_err();
        if (e != cudaSuccess) return e;
        e = bwd_query_tc(A, gamma, P, nodes, err);
        if (e != cudaSuccess) return e;
    }
    const int nlev = block_levels(N), nblocks = total_blocks(N);
    const int Pc = piece_chunks(A.C), nitems = total_items(N, Pc);
    if (nitems > 0) {
        if (bwd_piece_tc_supported(A)) {
            e = bwd_piece_tc(A, gamma, P, parts, nlev, Pc, nitems, err);
            if (e != cudaSuccess) return e;
        } else {
            bwd_block_piece_kernel<Tin><<<dim3(nitems, BH), kThreads, 0, st>>>(
                (const Tin *)A.q, A.dout, gamma, A.lam, P, parts, A.T, A.dk, A.dv, A.C, cbits, N, A.L, nlev,
                Pc);
        }
        const int nred = multi_piece_blocks(N, Pc);
        if (nred > 0)
            bwd_block_reduce_kernel<<<dim3(nred, BH, 8), kThreads, 0, st>>>(parts, R, A.dk, A.dv, N, nlev, Pc, nitems,
                                                                         nblocks);
        if (bwd_key_tc_supported(A)) {
            e = clear_err();
            if (e != cudaSuccess) return e;
            e = bwd_key_tc(A, gamma, P, R, parts, nlev, nblocks, Pc, nitems, err);
            if (e != cudaSuccess) return e;
        } else {
            const size_t smk = sizeof(float) * key_smem_floats(A.C, A.dk, A.dv);
            e = cudaFuncSetAttribute(bwd_key_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
            if (e != cudaSuccess) return e;
            bwd_key_kernel<Tin><<<dim3(N, BH), kThreads, smk, st>>>(
                (const Tin *)A.k, (const Tin *)A.v, gamma, P, R, parts, A.dkey, A.dval, A.T, A.dk, A.dv, A.C, N,
                nlev, nblocks, Pc, nitems);
        }
    }
    {
        const dim3 grid((A.T + kThreads / 16 - 1) / (kThreads / 16), BH);  // two tokens per warp
        if ((((uintptr_t)A.k | (uintptr_t)A.dkey) & 15u) == 0)
            bwd_gate_grad_kernel<Tin, true><<<grid, kThreads, 0, st>>>((const Tin *)A.k, A.lam, A.dlam, A.dkey, dG,
                                                                       A.T, A.dk, A.L);
        else
            bwd_gate_grad_kernel<Tin, false><<<grid, kThreads, 0, st>>>((const Tin *)A.k, A.lam, A.dlam, A.dkey, dG,
                                                                        A.T, A.dk, A.L);
    }
    bwd_gate_scan_kernel<<<dim3((A.T + kGateBlk - 1) / kGateBlk, BH), 1024, 0, st>>>(dG, A.dg, A.T);
    return cudaPeekAtLastError();
}

}  // namespace

size_t bwd_workspace_bytes(const BwdArgs &A) { return layout(A).end; }

size_t bwd_smem_bytes(const BwdArgs &A)
{
    const size_t q = query_smem_floats(A.C, A.dk, A.dv, A.L), k = key_smem_floats(A.C, A.dk, A.dv);
    return sizeof(float) * (q > k ? q : k);
}

cudaError_t bwd(const BwdArgs &A)
{
    return A.in_dt == LLA_F32 ? launch_bwd<float>(A) : launch_bwd<__nv_bfloat16>(A);
}

}  // namespace lla
