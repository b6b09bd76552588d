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

namespace lla {
namespace {

constexpr int kThreads = 256;
constexpr int kSub = 32;

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

size_t query_smem_floats(int C, int Dk, int Dv, int L)
{
    const size_t lk = Dk + 1, lv = Dv + 1;
    const size_t scratch = 3 * (size_t)C * C > (size_t)C * lk ? 3 * (size_t)C * C : (size_t)C * lk;
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
                 int cbits, int N, int L)
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
    float *U = W1;                  // [C][lk]  q_t[r] (Node dO_t)[r]  (path phase)
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
    // masked pair weights
    for (int e = threadIdx.x; e < C * C; e += kThreads) {
        const int t = e / C, s = e % C;
        float w1 = 0.f, w2 = 0.f, x = 0.f;
        if (s <= t) {
            float qk = 0.f, ov = 0.f;
            for (int r = 0; r < Dk; r++) qk = fmaf(Qs[t * lk + r], Ks[s * lk + r], qk);
            for (int c = 0; c < Dv; c++) ov = fmaf(Ds[t * lv + c], Vs[s * lv + c], ov);
            const float dec = expf(gl[t] - gl[s]);
            const float m = Ls[t * L + bit_length_u32((uint32_t)(t ^ s))] * dec;
            w1 = m * ov;
            w2 = m * qk;
            x = dec * qk * ov;
        }
        W1[e] = w1;
        W2[e] = w2;
        X[e] = x;
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
            for (int s = lo; s < hi; s++) a += X[t * C + s];
        }
        dL[e] = a;
    }
    // intra parts: dq_t = sum_s W1[t][s] k_s ; dk_s = sum_t W1[t][s] q_t ; dv_s = sum_t W2[t][s] dO_t
    for (int e = threadIdx.x; e < C * Dk; e += kThreads) {
        const int t = e / Dk, r = e % Dk;
        float a = 0.f, b = 0.f;
        for (int s = 0; s < C; s++) {
            a = fmaf(W1[t * C + s], Ks[s * lk + r], a);   // t as query
            b = fmaf(W1[s * C + t], Qs[s * lk + r], b);   // t as key
        }
        dq[(tok0 + t) * Dk + r] = a;
        dk[(tok0 + t) * Dk + r] = b;
    }
    for (int e = threadIdx.x; e < C * Dv; e += kThreads) {
        const int s = e / Dv, c = e % Dv;
        float a = 0.f;
        for (int t = 0; t < C; t++) a = fmaf(W2[t * C + s], Ds[t * lv + c], a);
        dv[(tok0 + s) * Dv + c] = a;
    }
    __syncthreads();
    // earlier chunks through the forward's path nodes
    const double *Pb = P + bh * (long long)(N + 1);
    for (int j = i; j > 0; j -= (j & -j)) {
        const int lev = cbits + 1 + ctz_u32((uint32_t)j);
        const float dP = (float)(Pb[i] - Pb[j]);
        const float *Nd = nodes + (bh * N + j) * (long long)Dk * Dv;
        for (int e = threadIdx.x; e < C * Dk; e += kThreads) {
            const int r = e / C, t = e % C;  // consecutive threads share a node row
            float u = 0.f;
            for (int c = 0; c < Dv; c++) u = fmaf(Nd[r * Dv + c], Ds[t * lv + c], u);
            const float w = expf(gl[t] + dP);
            dq[(tok0 + t) * Dk + r] += Ls[t * L + lev] * w * u;
            U[t * lk + r] = w * Qs[t * lk + r] * u;
        }
        __syncthreads();
        for (int t = threadIdx.x; t < C; t += kThreads) {
            float a = 0.f;
            for (int r = 0; r < Dk; r++) a += U[t * lk + r];
            dL[t * L + lev] += a;
        }
        __syncthreads();
    }
    for (int e = threadIdx.x; e < C * L; e += kThreads) dlam[tok0 * L + e] = dL[e];
}

// R_{m,b} for every level m and block b (odd b below N; other CTAs exit).
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
bwd_block_state_kernel(const Tin *__restrict__ q, const float *__restrict__ dout,
                       const float *__restrict__ gamma, const float *__restrict__ lam,
                       const double *__restrict__ P, float *__restrict__ R, int T, int Dk, int Dv,
                       int C, int cbits, int N, int L, int nlev)
{
    __shared__ float qs[kSub * 128];
    __shared__ float ds[kSub * 128];
    const long long bh = blockIdx.y;
    // locate (m, b) from the flat index: level m has ceil(N / 2^m) blocks
    int idx = blockIdx.x, m = 0, nb = N;
    while (m < nlev && idx >= nb) {
        idx -= nb;
        m++;
        nb = (N + (1 << m) - 1) >> m;
    }
    if (m >= nlev) return;
    const int b = idx;
    if ((b & 1) == 0 || ((long long)b << m) >= N) return;
    const int c0 = b << m, c1 = min(N, (b + 1) << m);  // chunks of the block
    const int lev = cbits + 1 + m;
    const double *Pb = P + bh * (long long)(N + 1);
    const double Pref = Pb[c0];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    const int RB = Dk / 16, CB = Dv / 16;
    float acc[8][8];
#pragma unroll
    for (int a = 0; a < 8; a++)
#pragma unroll
        for (int cc = 0; cc < 8; cc++) acc[a][cc] = 0.f;
    const long long t_lo = (long long)c0 * C, t_hi = (long long)c1 * C;
    for (long long t0 = t_lo; t0 < t_hi; t0 += kSub) {
        const int nt = (int)min((long long)kSub, t_hi - t0);
        __syncthreads();
        for (int e = threadIdx.x; e < kSub * Dk; e += kThreads) {
            const int tt = e / Dk, r = e % Dk;
            float x = 0.f;
            if (tt < nt) {
                const long long t = t0 + tt;
                const int j = (int)(t / C);
                const long long gi = bh * T + t;
                const float w = lam[gi * L + lev] * expf((float)(Pb[j] - Pref) + gamma[gi]);
                x = w * to_f32(q[gi * Dk + r]);
            }
            qs[e] = x;
        }
        for (int e = threadIdx.x; e < kSub * Dv; e += kThreads) {
            const int tt = e / Dv, c = e % Dv;
            ds[e] = (tt < nt) ? dout[(bh * T + t0 + tt) * Dv + c] : 0.f;
        }
        __syncthreads();
        for (int tt = 0; tt < nt; tt++) {
            float qr[8], dc[8];
#pragma unroll
            for (int a = 0; a < 8; a++) qr[a] = (a < RB) ? qs[tt * Dk + ty + 16 * a] : 0.f;
#pragma unroll
            for (int cc = 0; cc < 8; cc++) dc[cc] = (cc < CB) ? ds[tt * Dv + tx + 16 * cc] : 0.f;
#pragma unroll
            for (int a = 0; a < 8; a++)
#pragma unroll
                for (int cc = 0; cc < 8; cc++) acc[a][cc] = fmaf(qr[a], dc[cc], acc[a][cc]);
        }
    }
    float *out = R + ((bh * gridDim.x) + blockIdx.x) * (long long)Dk * Dv;
#pragma unroll
    for (int a = 0; a < 8; a++)
#pragma unroll
        for (int cc = 0; cc < 8; cc++)
            if (a < RB && cc < CB) out[(ty + 16 * a) * Dv + tx + 16 * cc] = acc[a][cc];
}

// Per chunk: the key side of the later chunks, dk_s += f_s R v_s, dv_s += f_s R^T k_s.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
bwd_key_kernel(const Tin *__restrict__ k, const Tin *__restrict__ v, const float *__restrict__ gamma,
               const double *__restrict__ P, const float *__restrict__ R, float *__restrict__ dk,
               float *__restrict__ dv, int T, int Dk, int Dv, int C, int N, int nlev, int nblocks)
{
    extern __shared__ float sm[];
    const int lk = Dk + 1, lv = Dv + 1;
    float *Ks = sm;               // [C][lk]
    float *Vs = Ks + C * lk;      // [C][lv]
    float *gl = Vs + C * lv;      // [C]
    const int i = blockIdx.x;
    const long long bh = blockIdx.y;
    const long long tok0 = bh * (long long)T + (long long)i * C;
    for (int e = threadIdx.x; e < C * Dk; e += kThreads) Ks[(e / Dk) * lk + e % Dk] = to_f32(k[tok0 * Dk + e]);
    for (int e = threadIdx.x; e < C * Dv; e += kThreads) Vs[(e / Dv) * lv + e % Dv] = to_f32(v[tok0 * Dv + e]);
    for (int e = threadIdx.x; e < C; e += kThreads) gl[e] = gamma[tok0 + e];
    __syncthreads();
    const double *Pb = P + bh * (long long)(N + 1);
    int off = 0;
    for (int m = 0; m < nlev; m++) {
        const int nb = (N + (1 << m) - 1) >> m;
        const int b = (i >> m) + 1;
        if (((i >> m) & 1) == 0 && ((long long)b << m) < N) {
            const float *Rm = R + ((bh * nblocks) + off + b) * (long long)Dk * Dv;
            const float dP = (float)(Pb[b << m] - Pb[i]);
            for (int e = threadIdx.x; e < C * Dk; e += kThreads) {
                const int r = e / C, s = e % C;
                float a = 0.f;
                for (int c = 0; c < Dv; c++) a = fmaf(Rm[r * Dv + c], Vs[s * lv + c], a);
                dk[(tok0 + s) * Dk + r] += expf(dP - gl[s]) * a;
            }
            for (int e = threadIdx.x; e < C * Dv; e += kThreads) {
                const int c = e / C, s = e % C;
                float a = 0.f;
                for (int r = 0; r < Dk; r++) a = fmaf(Rm[r * Dv + c], Ks[s * lk + r], a);
                dv[(tok0 + s) * Dv + c] += expf(dP - gl[s]) * a;
            }
        }
        off += nb;
    }
}

// dG_u = sum_l lam_u[l] dlam_u[l] - k_u . dk_u, then dg = reverse running sum (fp64).
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
bwd_gate_kernel(const Tin *__restrict__ k, const float *__restrict__ lam, const float *__restrict__ dlam,
                const float *__restrict__ dk, float *__restrict__ dg, int T, int Dk, int L)
{
    __shared__ double part[kThreads];
    const long long bh = blockIdx.x;
    const int per = (T + kThreads - 1) / kThreads;
    const int lo = min(T, (int)threadIdx.x * per), hi = min(T, lo + per);
    auto dG = [&](int u) -> double {
        const long long gi = bh * T + u;
        double a = 0.0;
        for (int l = 0; l < L; l++) a += (double)lam[gi * L + l] * (double)dlam[gi * L + l];
        for (int r = 0; r < Dk; r++) a -= (double)to_f32(k[gi * Dk + r]) * (double)dk[gi * Dk + r];
        return a;
    };
    double s = 0.0;
    for (int u = lo; u < hi; u++) s += dG(u);
    part[threadIdx.x] = s;
    __syncthreads();
    if (threadIdx.x == 0) {  // exclusive suffix sums of the partials
        double run = 0.0;
        for (int w = kThreads - 1; w >= 0; w--) {
            const double x = part[w];
            part[w] = run;
            run += x;
        }
    }
    __syncthreads();
    double run = part[threadIdx.x];
    for (int u = hi - 1; u >= lo; u--) {
        run += dG(u);
        dg[bh * T + u] = (float)run;
    }
}

int block_levels(int N) { return N > 1 ? bit_length_u32((uint32_t)(N - 1)) : 0; }

int total_blocks(int N)
{
    int tot = 0;
    for (int m = 0; m < block_levels(N); m++) tot += (N + (1 << m) - 1) >> m;
    return tot;
}

SimtFwdArgs node_args(const BwdArgs &A)
{
    SimtFwdArgs F;
    F.q = A.q; F.k = A.k; F.v = A.v; F.g = A.g; F.lam = A.lam; F.out = nullptr;
    F.B = A.B; F.H = A.H; F.T = A.T; F.dk = A.dk; F.dv = A.dv; F.C = A.C; F.L = A.L;
    F.in_dt = A.in_dt; F.out_dt = LLA_F32; F.workspace = A.workspace; F.stream = A.stream;
    return F;
}

template <typename Tin>
cudaError_t launch_bwd(const BwdArgs &A)
{
    const int BH = A.B * A.H, N = A.T / A.C;
    const int cbits = ctz_u32((uint32_t)A.C);
    cudaStream_t st = (cudaStream_t)A.stream;
    SimtFwdArgs F = node_args(A);
    cudaError_t e = simt_build_nodes(F);
    if (e != cudaSuccess) return e;
    char *ws = (char *)A.workspace;
    const double *P = (const double *)(ws + simt_ws_offset_P(F));
    const float *nodes = (const float *)(ws + simt_ws_offset_nodes(F));
    float *gamma = (float *)(ws + simt_workspace_bytes(F));
    float *R = (float *)(ws + simt_workspace_bytes(F) + align_up((size_t)BH * A.T * 4, 256));
    bwd_gamma_kernel<<<dim3(N, BH), 32, 0, st>>>(A.g, gamma, A.T, A.C);
    const size_t smq = sizeof(float) * query_smem_floats(A.C, A.dk, A.dv, A.L);
    e = cudaFuncSetAttribute(bwd_query_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smq);
    if (e != cudaSuccess) return e;
    bwd_query_kernel<Tin><<<dim3(N, BH), kThreads, smq, st>>>(
        (const Tin *)A.q, (const Tin *)A.k, (const Tin *)A.v, A.dout, gamma, A.lam, P, nodes, A.dq,
        A.dkey, A.dval, A.dlam, A.T, A.dk, A.dv, A.C, cbits, N, A.L);
    const int nlev = block_levels(N), nblocks = total_blocks(N);
    if (nblocks > 0) {
        bwd_block_state_kernel<Tin><<<dim3(nblocks, BH), kThreads, 0, st>>>(
            (const Tin *)A.q, A.dout, gamma, A.lam, P, R, A.T, A.dk, A.dv, A.C, cbits, N, A.L, nlev);
        const size_t smk = sizeof(float) * ((size_t)A.C * (A.dk + 1) + (size_t)A.C * (A.dv + 1) + A.C);
        e = cudaFuncSetAttribute(bwd_key_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smk);
        if (e != cudaSuccess) return e;
        bwd_key_kernel<Tin><<<dim3(N, BH), kThreads, smk, st>>>(
            (const Tin *)A.k, (const Tin *)A.v, gamma, P, R, A.dkey, A.dval, A.T, A.dk, A.dv, A.C, N, nlev,
            nblocks);
    }
    bwd_gate_kernel<Tin><<<BH, kThreads, 0, st>>>((const Tin *)A.k, A.lam, A.dlam, A.dkey, A.dg, A.T,
                                                   A.dk, A.L);
    return cudaPeekAtLastError();
}

}  // namespace

size_t bwd_workspace_bytes(const BwdArgs &A)
{
    SimtFwdArgs F = node_args(A);
    const size_t BH = (size_t)A.B * A.H;
    const int N = A.T / A.C;
    return simt_workspace_bytes(F) + align_up(BH * A.T * 4, 256) +
           align_up(BH * (size_t)total_blocks(N) * A.dk * A.dv * 4, 256);
}

size_t bwd_smem_bytes(const BwdArgs &A) { return sizeof(float) * query_smem_floats(A.C, A.dk, A.dv, A.L); }

cudaError_t bwd(const BwdArgs &A)
{
    return A.in_dt == LLA_F32 ? launch_bwd<float>(A) : launch_bwd<__nv_bfloat16>(A);
}

}  // namespace lla
