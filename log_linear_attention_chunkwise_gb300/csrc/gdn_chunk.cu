// Log-Linear Gated DeltaNet forward, chunkwise form.
//
// The per-token model is the one of the decode step (each Fenwick bucket
// keeps its own state S_l, dk x dv; every state takes each token's
// transition A_t = alpha_t (I - beta_t k_t k_t^T), alpha_t = exp(g_t); the
// read-out is sum_l lambda_t[l] S_l^T q_t; see "Log-Linear Attention" §3 for
// the hierarchical-mask construction and §2.3 for the chunked evaluation).
// Over a chunk of C = 64 tokens the product of the undecayed factors has the
// compact (UT / WY) form
//     (I - beta_{C-1} k k^T) ... (I - beta_0 k k^T) = I - K^T T K,
//     T = (I + strict_lower(diag(beta) K K^T))^{-1} diag(beta),
// and the decay is a scalar, so with gam_a = g_0 + ... + g_a (inclusive):
//   * state read-out at local row a: exp(gam_a) S^T qt_a,
//     qt_a = q_a - sum_{b <= a} (q_a . k_b) w_b,  W = T K;
//   * chunk transition: S <- exp(gam_{C-1}) (S - K^T (W S));
//   * the chunk's own contribution at its end: H = K^T T diag(exp(gam_{C-1} - gam)) V;
//   * intra-chunk output: o_a = sum_{s <= a} lambda_a[l(a,s)] exp(gam_a - gam_s) Cm[a,s] v_s,
//     Cm = inclusive_lower(Q K^T) T  (Cm[a,a] = beta_a q_a.k_a: level 0).
// Two launches.  gdn_chunk_prep_kernel does everything that is local to a
// chunk, for all chunks at once (one CTA per chunk; the 16 x 16 diagonal
// blocks of the inverse by forward substitution and the blocks below them by
// block substitution), writing the intra-chunk output, the rows of q~ and W,
// H and exp(gam_{C-1}).  gdn_chunk_scan_kernel walks the chunks of one
// (batch, head) in order for 8 value columns (a state column only mixes with
// itself), keeping the chunk-level Fenwick states in shared memory: read-out
// added to the output, transition, and the fold of H into the new level; the
// next chunk's operands are prefetched with cp.async while one is worked.
// Both run their products as warp-level TF32 tensor-core tiles with every
// fp32 operand split into a high part and a remainder.
#include "gdn.cuh"

namespace lla {
namespace {

constexpr int kGC = 64;        // chunk length
constexpr int kGCBits = 6;     // log2(kGC)
constexpr int kGT = 256;       // threads of both kernels
constexpr int kLdm = kGC + 4;  // row stride of the 64 x 64 matrices in shared memory (fragment rows: distinct banks)
constexpr int kGW = 8;         // value columns of a scan CTA
constexpr size_t kMaxSmem = 227 * 1024;  // dynamic shared memory of one CTA

// acc[i][j] += sum_{k < K} A(ty + 16 i, k) B(k, tx + 16 j), A(r, k) = A[r ar + k ak],
// B(k, c) = B[k bk + c bc]: fp32 CUDA cores, for the few products of any K
// (the buckets of a ragged end).
template <int RI, int CJ>
__device__ __forceinline__ void mm16(float (&acc)[RI][CJ], const float *A, int ar, int ak, const float *B, int bk,
                                     int bc, int K, int ty, int tx)
{
    const float *pa = A + ty * ar;
    const float *pb = B + tx * bc;
#pragma unroll 4
    for (int k = 0; k < K; k++) {
        float a[RI], b[CJ];
#pragma unroll
        for (int i = 0; i < RI; i++) a[i] = pa[16 * i * ar + k * ak];
#pragma unroll
        for (int j = 0; j < CJ; j++) b[j] = pb[k * bk + 16 * j * bc];
#pragma unroll
        for (int i = 0; i < RI; i++)
#pragma unroll
            for (int j = 0; j < CJ; j++) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
}

// Dynamic shared memory of this launch, in bytes: a kernel whose layout does
// not fit returns before touching shared memory.
__device__ __forceinline__ uint32_t dynamic_smem_bytes()
{
    uint32_t x;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(x));
    return x;
}

// One 16-byte piece of the input (8 bf16 or 4 fp32) as fp32, or zeros.
template <typename Tin>
__device__ __forceinline__ void load16_f32(const Tin *p, bool ok, float (&x)[16 / sizeof(Tin)])
{
    constexpr int n = 16 / (int)sizeof(Tin);
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (ok) w = *reinterpret_cast<const uint4 *>(p);
    if constexpr (sizeof(Tin) == 4) {
        x[0] = __uint_as_float(w.x);
        x[1] = __uint_as_float(w.y);
        x[2] = __uint_as_float(w.z);
        x[3] = __uint_as_float(w.w);
    } else {
        const uint32_t h[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < n / 2; u++) {
            x[2 * u] = __uint_as_float(h[u] << 16);            // bf16 -> fp32: the high half of the word
            x[2 * u + 1] = __uint_as_float(h[u] & 0xffff0000u);
        }
    }
}

template <int RI, int CJ>
__device__ __forceinline__ void zero(float (&acc)[RI][CJ])
{
#pragma unroll
    for (int i = 0; i < RI; i++)
#pragma unroll
        for (int j = 0; j < CJ; j++) acc[i][j] = 0.f;
}

__device__ __forceinline__ uint32_t to_tf32(float x)
{
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void split_tf32(float x, uint32_t &hi, uint32_t &lo)
{
    hi = to_tf32(x);
    lo = to_tf32(x - __uint_as_float(hi));
}

// d += a b, m16n8k8, A row-major 16 x 8, B column-major 8 x 8, TF32 in, fp32 accumulate.
__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
                 "{%8, %9}, {%0, %1, %2, %3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}


// Warp-level tensor-core product on m16n8k8 TF32 tiles: acc[i] is the tile
// tt = warp + 8 i of an (16 MT) x (8 NT) result (row block tt % MT, column
// block tt / MT; tiles past MT x NT are skipped), lane 4 g + t holding rows
// g, g + 8 and columns 2 t, 2 t + 1:
//   acc += sum_k A(r, k) B(k, c),  A(r, k) = A[r ar + k ak], B(k, c) = B[k bk + c bc].
// SA / SB split that operand into TF32 high and remainder parts (an operand
// exact in TF32, such as a bf16 input, is used whole); the partial products
// hi.hi, hi.lo, lo.hi keep about 21 bits.  Triangular operands skip k-steps:
// ALOW (A(r, k) = 0 for k > r), BLOW (B(k, c) = 0 for c > k); OUTLOW skips
// tiles wholly above the diagonal (the caller keeps the lower part only).
template <int NTW, int MT, int NT, bool SA, bool SB, bool ALOW, bool BLOW, bool OUTLOW>
__device__ __forceinline__ void warp_mma(float (&acc)[NTW][4], const float *A, int ar, int ak, const float *B, int bk,
                                         int bc, int K, int warp, int g, int t)
{
#pragma unroll
    for (int i = 0; i < NTW; i++) {
        acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
        const int tt = warp + 8 * i;
        if (tt >= MT * NT) continue;
        const int mt = tt % MT, nt = tt / MT;
        const float *a0 = A + (16 * mt + g) * ar + t * ak;
        const float *b0 = B + t * bk + (8 * nt + g) * bc;
        const int k_lo = BLOW ? 8 * nt : 0;
        int k_hi = ALOW ? min(K, 16 * mt + 16) : K;
        if (OUTLOW && 8 * nt > 16 * mt + 15) k_hi = k_lo;
#pragma unroll 2
        for (int k0 = k_lo; k0 < k_hi; k0 += 8) {
            const float ax[4] = {a0[k0 * ak], a0[8 * ar + k0 * ak], a0[(k0 + 4) * ak], a0[8 * ar + (k0 + 4) * ak]};
            const float bx[2] = {b0[k0 * bk], b0[(k0 + 4) * bk]};
            uint32_t ah[4], al[4], bh[2], bl[2];
#pragma unroll
            for (int e = 0; e < 4; e++) {
                if (SA) split_tf32(ax[e], ah[e], al[e]);
                else ah[e] = __float_as_uint(ax[e]);
            }
#pragma unroll
            for (int e = 0; e < 2; e++) {
                if (SB) split_tf32(bx[e], bh[e], bl[e]);
                else bh[e] = __float_as_uint(bx[e]);
            }
            mma_tf32(acc[i], ah, bh[0], bh[1]);
            if (SB) mma_tf32(acc[i], ah, bl[0], bl[1]);
            if (SA) mma_tf32(acc[i], al, bh[0], bh[1]);
        }
    }
}

// Calls f(row, col, value) for every element of the warp's tiles of warp_mma.
template <int NTW, int MT, int NT, typename F>
__device__ __forceinline__ void warp_tiles(const float (&acc)[NTW][4], int warp, int g, int t, F &&f)
{
#pragma unroll
    for (int i = 0; i < NTW; i++) {
        const int tt = warp + 8 * i;
        if (tt >= MT * NT) continue;
        const int r = 16 * (tt % MT) + g, c = 8 * (tt / MT) + 2 * t;
        f(r, c, acc[i][0], acc[i][1]);
        f(r + 8, c, acc[i][2], acc[i][3]);
    }
}

// Shared memory of the prep kernel, in floats after the 64 running gate sums.
struct PrepLayout {
    int ldk, ldq, ldv;
    size_t k, q, v, m1, m2, x, y, lam, beta, floats;
};

__host__ __device__ inline PrepLayout prep_layout(int dk, int dv, int L)
{
    PrepLayout P;
    // strides = 4 (mod 32) words: a fragment's rows g and columns t land in
    // 4 g + t, 32 distinct banks; V (read as k-rows t, columns g) uses 8 (mod 32)
    P.ldk = dk + 4;
    P.ldq = (dk > dv ? dk : dv) + 4;       // Q, later U = T' V
    P.ldv = dv + 8;
    P.k = kGC;                             // after gam[64]
    P.q = P.k + (size_t)kGC * P.ldk;
    P.v = P.q + (size_t)kGC * P.ldq;
    P.m1 = P.v + (size_t)kGC * P.ldv;
    P.m2 = P.m1 + (size_t)kGC * kLdm;
    P.x = P.m2 + (size_t)kGC * kLdm;
    P.y = P.x + (size_t)kGC * kLdm;        // [3][16][17] block products of the inverse
    P.lam = P.y + 3 * 16 * 17;
    P.beta = P.lam + (size_t)kGC * L;
    P.floats = P.beta + kGC;
    return P;
}

// Workspace: [BH][N][128][dk] (rows of q~, then of W), [BH][N][dk][dv] (H), [BH][N] exp(gam_{C-1}).
struct WsLayout {
    size_t qw, h, gend, bytes;
};

inline WsLayout ws_layout(long long BH, int N, int dk, int dv)
{
    WsLayout W;
    W.qw = 0;
    W.h = W.qw + align_up((size_t)BH * N * 2 * dk * kGC * sizeof(float), 256);
    W.gend = W.h + align_up((size_t)BH * N * dk * dv * sizeof(float), 256);
    W.bytes = W.gend + align_up((size_t)BH * N * sizeof(float), 256);
    return W;
}

// Steps 7 to 9 of the prep kernel for dv = 16 CJ: the intra-chunk output,
// the chunk state H, and the low-bit states of a ragged last chunk.  SIN:
// the inputs (K, V) need splitting for TF32 (fp32 inputs; bf16 are exact).
template <int DK, int CJ, bool SIN>
__device__ __forceinline__ void prep_tail(float *M1, const float *M2, const float *Xs, const float *Ks, float *Qs,
                                          const float *Vs, const float *gam, float *__restrict__ out,
                                          float *__restrict__ ws_h, float *__restrict__ ws_gend,
                                          float *__restrict__ state_out, long long tok0, long long bh, int ci, int N,
                                          int nv, int dv, int ldq, int ldv, int Ls_out)
{
    constexpr int DV = 16 * CJ;
    const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
    const int warp = tid >> 5, g = (tid & 31) >> 2, t = tid & 3;
    // 7. intra-chunk output M V
    {
        float acc[CJ][4];
        warp_mma<CJ, 4, DV / 8, true, SIN, true, false, false>(acc, M2, kLdm, 1, Vs, ldv, 1, kGC, warp, g, t);
        warp_tiles<CJ, 4, DV / 8>(acc, warp, g, t, [&](int r, int c, float x, float y) {
            if (r < nv) *reinterpret_cast<float2 *>(out + (tok0 + r) * dv + c) = make_float2(x, y);
        });
    }
    __syncthreads();  // M1 (Cm) and Qs are free

    // 8. T' = T diag(exp(gam_{C-1} - gam)) into M1, U = T' V into Qs, H = K^T U
    const float Gam = gam[kGC - 1];
    for (int e = tid; e < kGC * kGC; e += kGT) {
        const int r = e >> kGCBits, b = e & (kGC - 1);
        M1[r * kLdm + b] = Xs[r * kLdm + b] * expf(Gam - gam[b]);
    }
    __syncthreads();
    constexpr int HT = (DK / 16) * (DV / 8);  // m16n8 tiles of H
    auto kt_u = [&](int lo, int hi, float *dst) {
        // U = T'[:, lo:hi] V[lo:hi, :] into Qs, then dst = K^T U (dk x dv)
        if (lo == 0 && hi == kGC) {
            float acc[CJ][4];
            warp_mma<CJ, 4, DV / 8, true, SIN, true, false, false>(acc, M1, kLdm, 1, Vs, ldv, 1, kGC, warp, g, t);
            warp_tiles<CJ, 4, DV / 8>(acc, warp, g, t, [&](int r, int c, float x, float y) {
                *reinterpret_cast<float2 *>(Qs + r * ldq + c) = make_float2(x, y);
            });
        } else {
            float acc[4][CJ];
            zero(acc);
            mm16<4, CJ>(acc, M1 + lo, kLdm, 1, Vs + lo * ldv, ldv, 1, hi - lo, ty, tx);
#pragma unroll
            for (int i = 0; i < 4; i++)
#pragma unroll
                for (int j = 0; j < CJ; j++) Qs[(ty + 16 * i) * ldq + tx + 16 * j] = acc[i][j];
        }
        __syncthreads();
        float acc[(HT + 7) / 8][4];
        // A(r, a) = K[a][r], B(a, c) = U[a][c]
        warp_mma<(HT + 7) / 8, DK / 16, DV / 8, SIN, true, false, false, false>(acc, Ks, 1, DK + 4, Qs, ldq, 1, kGC,
                                                                                warp, g, t);
        warp_tiles<(HT + 7) / 8, DK / 16, DV / 8>(acc, warp, g, t, [&](int r, int c, float x, float y) {
            *reinterpret_cast<float2 *>(dst + r * dv + c) = make_float2(x, y);
        });
    };
    kt_u(0, kGC, ws_h + (bh * N + ci) * (long long)DK * dv);
    if (tid == 0) ws_gend[bh * N + ci] = expf(Gam);

    // 9. after a ragged last chunk the sequence's low bits are buckets inside
    //    it: slot j (bit j of T) holds K^T T'[:, B_j] V[B_j, :] over its tokens
    if (state_out && ci == N - 1 && nv < kGC) {
        for (int j = 0; j < kGCBits; j++) {
            if (!((nv >> j) & 1)) continue;
            const int hi = nv - (nv & ((1 << j) - 1)), lo = hi - (1 << j);
            __syncthreads();  // Qs is reused
            kt_u(lo, hi, state_out + ((bh * Ls_out + j) * DK) * (long long)dv);
        }
    }
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kGT, DK <= 64 ? 2 : 1)
gdn_chunk_prep_kernel(const Tin *__restrict__ q, const Tin *__restrict__ k, const Tin *__restrict__ v,
                      const float *__restrict__ g, const float *__restrict__ beta, const float *__restrict__ lam,
                      float *__restrict__ out, float *__restrict__ ws_qw, float *__restrict__ ws_h,
                      float *__restrict__ ws_gend, float *__restrict__ state_out, int T, int N, int H, int dv,
                      int L, int Ls_out)
{
    extern __shared__ __align__(16) float sm[];
    const PrepLayout P = prep_layout(DK, dv, L);
    if (P.floats * sizeof(float) > dynamic_smem_bytes()) return;
    const int ldk = P.ldk, ldq = P.ldq, ldv = P.ldv;
    constexpr bool SIN = sizeof(Tin) == 4;  // fp32 inputs are split for TF32; bf16 are exact
    float *gam = sm;
    float *Ks = sm + P.k, *Qs = sm + P.q, *Vs = sm + P.v;
    float *M1 = sm + P.m1, *M2 = sm + P.m2, *Xs = sm + P.x, *Ys = sm + P.y;
    float *ls = sm + P.lam, *bs = sm + P.beta;
    const int tid = threadIdx.x;
    const int warp = tid >> 5, fg = (tid & 31) >> 2, ft = tid & 3;  // fragment lane: row group, column
    const int ci = blockIdx.x;
    const long long bh = (long long)blockIdx.z * H + blockIdx.y;
    const long long tok0 = bh * T + (long long)ci * kGC;
    const int nv = min(kGC, T - ci * kGC);
    const int cj = dv / 16;

    // 1. the chunk's inputs, zero past T (a padded token has k = v = 0, beta = 0,
    //    g = 0: its factor is the identity and it adds nothing)
    //    (16-byte vector loads: every row starts on a 16-byte boundary)
    constexpr int EPV = 16 / (int)sizeof(Tin);  // elements per 16-byte piece
    for (int e = tid; e < kGC * DK / EPV; e += kGT) {
        const int a = e / (DK / EPV), r = (e % (DK / EPV)) * EPV;
        float xk[EPV], xq[EPV];
        load16_f32<Tin>(k + tok0 * DK + (long long)e * EPV, a < nv, xk);
        load16_f32<Tin>(q + tok0 * DK + (long long)e * EPV, a < nv, xq);
#pragma unroll
        for (int u = 0; u < EPV; u++) {
            Ks[a * ldk + r + u] = xk[u];
            Qs[a * ldq + r + u] = xq[u];
        }
    }
    for (int e = tid; e < kGC * dv / EPV; e += kGT) {
        float xv[EPV];
        const int a = e * EPV / dv, c = e * EPV % dv;
        load16_f32<Tin>(v + tok0 * dv + (long long)e * EPV, a < nv, xv);
#pragma unroll
        for (int u = 0; u < EPV; u++) Vs[a * ldv + c + u] = xv[u];
    }
    for (int e = tid; e < kGC * L; e += kGT) ls[e] = e / L < nv ? lam[tok0 * L + e] : 0.f;
    for (int e = tid; e < kGC * kLdm; e += kGT) Xs[e] = 0.f;
    if (tid < kGC) bs[tid] = tid < nv ? beta[tok0 + tid] : 0.f;
    if (tid < 32) {  // inclusive running sum of the gates (fp64, stored fp32), two tokens per lane
        const int a0 = 2 * tid;
        const double g0 = a0 < nv ? (double)g[tok0 + a0] : 0.0;
        const double g1 = a0 + 1 < nv ? (double)g[tok0 + a0 + 1] : 0.0;
        double s = g0 + g1;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double y = __shfl_up_sync(0xffffffffu, s, off);
            if (tid >= off) s += y;
        }
        gam[a0 + 1] = (float)s;
        gam[a0] = (float)(s - g1);
    }
    __syncthreads();

    // 2. M1 = strict_lower(diag(beta) K K^T), M2 = inclusive_lower(Q K^T)
    {
        float ak[4][4], aq[4][4];
        // A(a, r) = K[a][r] (or Q), B(r, b) = K[b][r]
        warp_mma<4, 4, 8, SIN, SIN, false, false, true>(ak, Ks, ldk, 1, Ks, 1, ldk, DK, warp, fg, ft);
        warp_mma<4, 4, 8, SIN, SIN, false, false, true>(aq, Qs, ldq, 1, Ks, 1, ldk, DK, warp, fg, ft);
        warp_tiles<4, 4, 8>(ak, warp, fg, ft, [&](int r, int c, float x, float y) {
            M1[r * kLdm + c] = c < r ? bs[r] * x : 0.f;
            M1[r * kLdm + c + 1] = c + 1 < r ? bs[r] * y : 0.f;
        });
        warp_tiles<4, 4, 8>(aq, warp, fg, ft, [&](int r, int c, float x, float y) {
            M2[r * kLdm + c] = c <= r ? x : 0.f;
            M2[r * kLdm + c + 1] = c + 1 <= r ? y : 0.f;
        });
    }
    __syncthreads();

    // 3. X = (I + M1)^{-1}: the four 16 x 16 diagonal blocks by forward
    //    substitution (a lane per column, the column in registers), then the
    //    blocks below the diagonal, one block diagonal at a time:
    //    X_ij = -X_ii sum_{j <= m < i} M1_im X_mj
    if (tid < 128 && (tid & 31) < 16) {
        const int w = tid >> 5, l = tid & 31;
        const float *Lw = M1 + 16 * w * kLdm + 16 * w;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; r++) {
            float s = r == l ? 1.f : 0.f;
#pragma unroll
            for (int j = 0; j < r; j++) s = fmaf(-Lw[r * kLdm + j], x[j], s);
            x[r] = s;
        }
#pragma unroll
        for (int r = 0; r < 16; r++) Xs[(16 * w + r) * kLdm + 16 * w + l] = x[r];
    }
    __syncthreads();
    {
        const int r = tid >> 4, c = tid & 15;
        for (int d = 1; d < 4; d++) {
            for (int blk = 0; blk + d < 4; blk++) {
                const int bi = blk + d, bj = blk;
                float y = 0.f;
                for (int m = bj; m < bi; m++)
#pragma unroll
                    for (int e = 0; e < 16; e++)
                        y = fmaf(M1[(16 * bi + r) * kLdm + 16 * m + e], Xs[(16 * m + e) * kLdm + 16 * bj + c], y);
                Ys[(blk * 16 + r) * 17 + c] = y;
            }
            __syncthreads();
            for (int blk = 0; blk + d < 4; blk++) {
                const int bi = blk + d, bj = blk;
                float x = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e++)
                    x = fmaf(Xs[(16 * bi + r) * kLdm + 16 * bi + e], Ys[(blk * 16 + e) * 17 + c], x);
                Xs[(16 * bi + r) * kLdm + 16 * bj + c] = -x;
            }
            __syncthreads();
        }
    }
    // 4. T = X diag(beta), in place
    for (int e = tid; e < kGC * kGC; e += kGT) {
        const int a = e >> kGCBits, b = e & (kGC - 1);
        Xs[a * kLdm + b] *= bs[b];
    }
    __syncthreads();

    // 5. Cm = M2 T (lower triangular) into M1; the intra-chunk weights
    //    lambda_a[l(a,s)] exp(gam_a - gam_s) Cm[a,s] into M2
    {
        float acc[4][4];
        warp_mma<4, 4, 8, true, true, true, true, false>(acc, M2, kLdm, 1, Xs, kLdm, 1, kGC, warp, fg, ft);
        __syncthreads();  // every read of M1 (done) and M2 precedes the writes
        warp_tiles<4, 4, 8>(acc, warp, fg, ft, [&](int r, int c, float x, float y) {
            const float v2[2] = {x, y};
#pragma unroll
            for (int u = 0; u < 2; u++) {
                const int s2 = c + u;
                M1[r * kLdm + s2] = v2[u];
                float m = 0.f;
                if (s2 <= r && r < nv) {
                    const int lev = 32 - __clz(r ^ s2);
                    m = ls[r * L + lev] * expf(gam[r] - gam[s2]) * v2[u];
                }
                M2[r * kLdm + s2] = m;
            }
        });
    }
    __syncthreads();

    // 6. q~ = diag(exp(gam)) (Q - Cm K) and W = T K, rows [a][r]: q~ in rows 0..63, W in 64..127
    {
        float *qw_ws = ws_qw + (bh * N + ci) * (2LL * DK * kGC);
        constexpr int NTW = DK / 16;
        float aw[NTW][4], ac[NTW][4];
        // A(a, b) = T[a][b] (or Cm), B(b, r) = K[b][r]
        warp_mma<NTW, 4, DK / 8, true, SIN, true, false, false>(aw, Xs, kLdm, 1, Ks, ldk, 1, kGC, warp, fg, ft);
        warp_mma<NTW, 4, DK / 8, true, SIN, true, false, false>(ac, M1, kLdm, 1, Ks, ldk, 1, kGC, warp, fg, ft);
        warp_tiles<NTW, 4, DK / 8>(aw, warp, fg, ft, [&](int r, int c, float x, float y) {
            *reinterpret_cast<float2 *>(qw_ws + (kGC + r) * DK + c) = make_float2(x, y);
        });
        warp_tiles<NTW, 4, DK / 8>(ac, warp, fg, ft, [&](int r, int c, float x, float y) {
            const float ea = expf(gam[r]);
            *reinterpret_cast<float2 *>(qw_ws + r * DK + c) =
                make_float2(ea * (Qs[r * ldq + c] - x), ea * (Qs[r * ldq + c + 1] - y));
        });
    }
    switch (cj) {
    case 1: prep_tail<DK, 1, SIN>(M1, M2, Xs, Ks, Qs, Vs, gam, out, ws_h, ws_gend, state_out, tok0, bh, ci, N, nv, dv, ldq, ldv, Ls_out); break;
    case 2: prep_tail<DK, 2, SIN>(M1, M2, Xs, Ks, Qs, Vs, gam, out, ws_h, ws_gend, state_out, tok0, bh, ci, N, nv, dv, ldq, ldv, Ls_out); break;
    case 4: prep_tail<DK, 4, SIN>(M1, M2, Xs, Ks, Qs, Vs, gam, out, ws_h, ws_gend, state_out, tok0, bh, ci, N, nv, dv, ldq, ldv, Ls_out); break;
    default: prep_tail<DK, 8, SIN>(M1, M2, Xs, Ks, Qs, Vs, gam, out, ws_h, ws_gend, state_out, tok0, bh, ci, N, nv, dv, ldq, ldv, Ls_out); break;
    }
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async4(void *dst, const void *src, int src_bytes)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Shared memory of the scan kernel: states, W S rows, then one or two stages.
// The scan's products have 8 columns (one CTA's value slice), so they run as
// warp-level m16n8k8 TF32 tensor-core products; every fp32 operand is split
// into a TF32 high part and a TF32 remainder and the three significant
// partial products (hi.hi, hi.lo, lo.hi) are accumulated in fp32, which keeps
// about 21 bits (bf16 keys are exact in TF32 and need no split).  The staged
// q~ / W and key rows are stored with their 16-byte pieces XOR-permuted by
// row, so the fragment loads (lane 4 g + t reads row g, column t, or row t,
// columns g) fall in distinct banks without padding.
struct ScanLayout {
    size_t S, WS, stage, qw, kr, h, lam, gend, stage_bytes, bytes;
};

__host__ __device__ inline ScanLayout scan_layout(int dk, int N, int nlv, int nst, int tin_bytes)
{
    ScanLayout Y;
    const int NS = bit_length_u32((uint32_t)N);                     // slots (the last fold included)
    const int nl = bit_length_u32((uint32_t)(N - 1));               // slots live at some chunk < N
    const int nws = nl > 1 ? nl : 1;
    Y.S = 0;                                                        // [NS][dk][kGW] fp32
    Y.WS = Y.S + (size_t)NS * dk * kGW * 4;                         // [nws][64][kGW] fp32
    Y.stage = align_up(Y.WS + (size_t)nws * kGC * kGW * 4, 16);
    Y.qw = 0;                                                       // [128][dk] fp32, permuted
    Y.kr = Y.qw + (size_t)2 * kGC * dk * 4;                         // [64][dk] input type, permuted
    Y.h = Y.kr + (size_t)kGC * dk * tin_bytes;                      // H slice [dk][kGW]
    Y.lam = Y.h + (size_t)dk * kGW * 4;                             // chunk-level lambda [64][nlv]
    Y.gend = Y.lam + (size_t)kGC * nlv * 4;
    Y.stage_bytes = align_up(Y.gend + 16, 16);
    Y.bytes = Y.stage + (size_t)nst * Y.stage_bytes;
    return Y;
}

// Element offset of (row, c) in a staged q~ / W tile: piece c/4 of the row
// is stored at piece (c/4) ^ (row & 7) (fewer pieces per row: fewer bits).
template <int DK>
__device__ __forceinline__ int qw_off(int row, int c)
{
    constexpr int msk = (DK / 4 < 8 ? DK / 4 : 8) - 1;
    return row * DK + ((((c >> 2) ^ (row & msk)) << 2) | (c & 3));
}

// Element offset of (a, r) in a staged key tile: the 16-byte piece holding r
// is moved by a & 3 pieces (bf16) or 2 (a & 3) pieces (fp32, whose 8
// consecutive columns span two pieces).
template <int DK, typename Tin>
__device__ __forceinline__ int k_piece_xor(int a)
{
    constexpr int cpr = DK * (int)sizeof(Tin) / 16;
    return (sizeof(Tin) == 2 ? (a & 3) : ((a & 3) << 1)) & (cpr - 1);
}

template <int DK, typename Tin>
__device__ __forceinline__ int k_off(int a, int r)
{
    constexpr int epc = 16 / (int)sizeof(Tin);
    return a * DK + ((((r / epc) ^ k_piece_xor<DK, Tin>(a)) * epc) + (r % epc));
}

// The next (up to) four slots of rem, lowest first; returns how many.
__device__ __forceinline__ int take_slots(uint32_t &rem, int (&mm)[4])
{
    int nu = 0;
#pragma unroll
    for (int u = 0; u < 4; u++) {
        mm[u] = rem ? __ffs((int)rem) - 1 : mm[0];
        if (rem) {
            nu = u + 1;
            rem &= rem - 1;
        }
    }
    return nu;
}

// Read-out and W S of a warp's 16 rows of [q~; W] (rows r0..r0+15 of the
// 128) against live slots mm[0..NU): d[u] is the m16n8 result tile.
template <int NU, int DK>
__device__ __forceinline__ void scan_rows(const float *__restrict__ QWs, const float *__restrict__ S,
                                          const int (&mm)[4], int r0, int g, int t, float (&d)[4][4])
{
#pragma unroll
    for (int u = 0; u < NU; u++) d[u][0] = d[u][1] = d[u][2] = d[u][3] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < DK / 8; kk++) {
        uint32_t ah[4], al[4];
        split_tf32(QWs[qw_off<DK>(r0 + g, 8 * kk + t)], ah[0], al[0]);
        split_tf32(QWs[qw_off<DK>(r0 + g + 8, 8 * kk + t)], ah[1], al[1]);
        split_tf32(QWs[qw_off<DK>(r0 + g, 8 * kk + t + 4)], ah[2], al[2]);
        split_tf32(QWs[qw_off<DK>(r0 + g + 8, 8 * kk + t + 4)], ah[3], al[3]);
#pragma unroll
        for (int u = 0; u < NU; u++) {
            const float *Sm = S + (mm[u] * DK + 8 * kk + t) * kGW + g;
            uint32_t bh0, bl0, bh1, bl1;
            split_tf32(Sm[0], bh0, bl0);
            split_tf32(Sm[4 * kGW], bh1, bl1);
            mma_tf32(d[u], ah, bh0, bh1);
            mma_tf32(d[u], ah, bl0, bl1);
            mma_tf32(d[u], al, bh0, bh1);
        }
    }
}

// The transition of live slots mm[0..NU) on a warp's 16 state rows r0..r0+15:
// S[r, :] <- ge (S[r, :] - sum_a K[a][r] (W S)[a, :]).
template <int NU, int DK, typename Tin>
__device__ __forceinline__ void scan_transition(const Tin *__restrict__ Kr, const float *__restrict__ WS, float *S,
                                                const int (&mm)[4], int r0, int g, int t, float ge)
{
    float d[4][4];
#pragma unroll
    for (int u = 0; u < NU; u++) d[u][0] = d[u][1] = d[u][2] = d[u][3] = 0.f;
#pragma unroll 2
    for (int kk = 0; kk < kGC / 8; kk++) {  // A(row r, col a) = K[a][r]
        const int a0 = 8 * kk + t, a1 = a0 + 4;
        const float x[4] = {to_f32(Kr[k_off<DK, Tin>(a0, r0 + g)]), to_f32(Kr[k_off<DK, Tin>(a0, r0 + g + 8)]),
                            to_f32(Kr[k_off<DK, Tin>(a1, r0 + g)]), to_f32(Kr[k_off<DK, Tin>(a1, r0 + g + 8)])};
        uint32_t ah[4], al[4];
#pragma unroll
        for (int e = 0; e < 4; e++) {
            if (sizeof(Tin) == 2) {
                ah[e] = __float_as_uint(x[e]);  // a bf16 value is exact in TF32
                al[e] = 0u;
            } else {
                split_tf32(x[e], ah[e], al[e]);
            }
        }
#pragma unroll
        for (int u = 0; u < NU; u++) {
            const float *W0 = WS + (mm[u] * kGC + 8 * kk + t) * kGW + g;
            uint32_t bh0, bl0, bh1, bl1;
            split_tf32(W0[0], bh0, bl0);
            split_tf32(W0[4 * kGW], bh1, bl1);
            mma_tf32(d[u], ah, bh0, bh1);
            mma_tf32(d[u], ah, bl0, bl1);
            if (sizeof(Tin) == 4) mma_tf32(d[u], al, bh0, bh1);
        }
    }
#pragma unroll
    for (int u = 0; u < NU; u++) {
#pragma unroll
        for (int h = 0; h < 2; h++) {
            float2 *sp = reinterpret_cast<float2 *>(S + (mm[u] * DK + r0 + g + 8 * h) * kGW + 2 * t);
            float2 x = *sp;
            x.x = ge * (x.x - d[u][2 * h]);
            x.y = ge * (x.y - d[u][2 * h + 1]);
            *sp = x;
        }
    }
}

template <typename Tin, int DK>
__global__ void __launch_bounds__(kGT, 2)
gdn_chunk_scan_kernel(const Tin *__restrict__ k, const float *__restrict__ lam, float *__restrict__ out,
                      const float *__restrict__ ws_qw, const float *__restrict__ ws_h,
                      const float *__restrict__ ws_gend, float *__restrict__ state_out, int T, int N, int H, int dv,
                      int L, int Ls_out, int nst)
{
    extern __shared__ __align__(16) uint8_t smb[];
    const int NS = bit_length_u32((uint32_t)N);  // chunk-level slots: slot m = level kGCBits + 1 + m
    const int nlv = max(L - (kGCBits + 1), 0);
    const ScanLayout Y = scan_layout(DK, N, nlv, nst, (int)sizeof(Tin));
    if (Y.bytes > dynamic_smem_bytes()) return;
    float *S = reinterpret_cast<float *>(smb + Y.S);
    float *WS = reinterpret_cast<float *>(smb + Y.WS);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, t = lane & 3;
    const int col0 = blockIdx.x * kGW;
    const long long bh = (long long)blockIdx.z * H + blockIdx.y;
    const bool ragged = (T % kGC) != 0;

    auto stage_ptr = [&](int st) { return smb + Y.stage + (size_t)st * Y.stage_bytes; };
    auto load = [&](int st, int ci) {
        uint8_t *b = stage_ptr(st);
        const int nvc = min(kGC, T - ci * kGC);
        const long long row0 = bh * T + (long long)ci * kGC;
        const float *qw = ws_qw + (bh * N + ci) * (2LL * DK * kGC);
        constexpr int qpr = DK / 4;  // 16-byte pieces per q~ / W row
        for (int e = tid; e < 2 * kGC * qpr; e += kGT) {
            const int r = e / qpr, p = e % qpr;
            cp_async16(b + Y.qw + (size_t)qw_off<DK>(r, 4 * p) * 4, qw + r * DK + 4 * p, 16);
        }
        constexpr int cpr = DK * (int)sizeof(Tin) / 16;  // 16-byte pieces per key row
        for (int e = tid; e < kGC * cpr; e += kGT) {
            const int a = e / cpr, p = e % cpr;
            const Tin *src = k + (row0 + min(a, nvc - 1)) * DK + p * (16 / (int)sizeof(Tin));
            cp_async16(b + Y.kr + ((size_t)a * cpr + (p ^ k_piece_xor<DK, Tin>(a))) * 16, src, a < nvc ? 16 : 0);
        }
        const float *h = ws_h + (bh * N + ci) * (long long)DK * dv + col0;
        for (int e = tid; e < DK * kGW / 4; e += kGT) {
            const int r = e / (kGW / 4), p = e % (kGW / 4);
            cp_async16(b + Y.h + 16 * e, h + (long long)r * dv + 4 * p, 16);
        }
        for (int e = tid; e < kGC * nlv; e += kGT) {
            const int a = e / nlv, m = e % nlv;
            cp_async4(b + Y.lam + 4 * e, lam + (row0 + min(a, nvc - 1)) * L + kGCBits + 1 + m, a < nvc ? 4 : 0);
        }
        if (tid == 0) cp_async4(b + Y.gend, ws_gend + bh * N + ci, 4);
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    constexpr int MT = DK / 16;       // 16-row tiles of a state
    constexpr int NSP = 8 / MT;       // warps sharing one state tile (they split the slots)
    const int mt = warp % MT, sp = warp / MT;

    if (nst == 2) load(0, 0);
    for (int ci = 0; ci < N; ci++) {
        const int st = nst == 2 ? (ci & 1) : 0;
        if (nst == 1) load(0, ci);
        cp_async_wait_all();
        __syncthreads();  // stage ci is visible; chunk ci-1 is finished with the other stage
        if (nst == 2 && ci + 1 < N) load((ci + 1) & 1, ci + 1);
        const uint8_t *b = stage_ptr(st);
        const float *QWs = reinterpret_cast<const float *>(b + Y.qw);
        const Tin *Kr = reinterpret_cast<const Tin *>(b + Y.kr);
        const float *Hs = reinterpret_cast<const float *>(b + Y.h);
        const float *lamc = reinterpret_cast<const float *>(b + Y.lam);
        const float ge = *reinterpret_cast<const float *>(b + Y.gend);
        const uint32_t live = (uint32_t)ci;  // slot m is live at chunk ci iff bit m of ci is set

        if (live) {
            // A. warp w takes rows 16w..16w+15 of [q~; W]: warps 0-3 read out into
            //    the output, warps 4-7 leave W S of each live slot for the transition
            const int r0 = 16 * warp;
            const bool readout = warp < 4;
            const int nvc = T - ci * kGC;
            float o[4] = {0.f, 0.f, 0.f, 0.f};
            float *orow[2];
            if (readout) {  // the intra-chunk output this adds to, loaded while the products run
#pragma unroll
                for (int h = 0; h < 2; h++) {
                    const int a = r0 + g + 8 * h;
                    orow[h] = out + (bh * T + (long long)ci * kGC + a) * dv + col0 + 2 * t;
                    if (a < nvc) {
                        const float2 x = *reinterpret_cast<const float2 *>(orow[h]);
                        o[2 * h] = x.x;
                        o[2 * h + 1] = x.y;
                    }
                }
            }
            uint32_t rem = live;
            while (rem) {
                int mm[4];
                const int nu = take_slots(rem, mm);
                float d[4][4];
                switch (nu) {
                case 1: scan_rows<1, DK>(QWs, S, mm, r0, g, t, d); break;
                case 2: scan_rows<2, DK>(QWs, S, mm, r0, g, t, d); break;
                case 3: scan_rows<3, DK>(QWs, S, mm, r0, g, t, d); break;
                default: scan_rows<4, DK>(QWs, S, mm, r0, g, t, d); break;
                }
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    if (u >= nu) break;
                    if (readout) {
                        const float l0 = lamc[(r0 + g) * nlv + mm[u]], l1 = lamc[(r0 + g + 8) * nlv + mm[u]];
                        o[0] = fmaf(l0, d[u][0], o[0]);
                        o[1] = fmaf(l0, d[u][1], o[1]);
                        o[2] = fmaf(l1, d[u][2], o[2]);
                        o[3] = fmaf(l1, d[u][3], o[3]);
                    } else {
                        float *w = WS + (mm[u] * kGC + r0 - kGC + g) * kGW + 2 * t;
                        *reinterpret_cast<float2 *>(w) = make_float2(d[u][0], d[u][1]);
                        *reinterpret_cast<float2 *>(w + 8 * kGW) = make_float2(d[u][2], d[u][3]);
                    }
                }
            }
            if (readout) {
#pragma unroll
                for (int h = 0; h < 2; h++)
                    if (r0 + g + 8 * h < nvc)
                        *reinterpret_cast<float2 *>(orow[h]) = make_float2(o[2 * h], o[2 * h + 1]);
            }
            __syncthreads();

            // B. transition: warp (tile mt, part sp) takes every NSP-th live slot
            uint32_t mine = 0;
            {
                uint32_t rem = live;
                for (int n = 0; rem; n++) {
                    const uint32_t low = rem & (0u - rem);
                    if (n % NSP == sp) mine |= low;
                    rem ^= low;
                }
            }
            while (mine) {
                int mm[4];
                const int nu = take_slots(mine, mm);
                switch (nu) {
                case 1: scan_transition<1, DK>(Kr, WS, S, mm, 16 * mt, g, t, ge); break;
                case 2: scan_transition<2, DK>(Kr, WS, S, mm, 16 * mt, g, t, ge); break;
                case 3: scan_transition<3, DK>(Kr, WS, S, mm, 16 * mt, g, t, ge); break;
                default: scan_transition<4, DK>(Kr, WS, S, mm, 16 * mt, g, t, ge); break;
                }
            }
            __syncthreads();
        }

        // C. the fold into slot ctz(ci+1) of the chunk's state and the slots below it
        if (ci + 1 < N || !ragged) {  // a ragged last chunk stays out of the chunk levels
            const int m0 = ctz_u32((uint32_t)ci + 1u);
            for (int e = tid; e < DK * kGW; e += kGT) {
                float sv = Hs[e];
                for (int m = 0; m < m0; m++) sv += S[m * DK * kGW + e];
                S[m0 * DK * kGW + e] = sv;
            }
        }
        if (nst == 1) __syncthreads();  // the single stage is reloaded next
    }

    // the state after the sequence in the decode layout (slot j = level j + 1,
    // live iff bit j of T); the slots below kGCBits that are live come from the
    // prep kernel's last chunk
    if (state_out) {
        __syncthreads();
        const long long nfull = T >> kGCBits;
        for (int j = 0; j < Ls_out; j++) {
            if (j < kGCBits && ((T >> j) & 1)) continue;
            const int m = j - kGCBits;
            const bool on = m >= 0 && m < NS && ((nfull >> m) & 1);
            for (int e = tid; e < DK * kGW; e += kGT) {
                const int r = e / kGW, c = e % kGW;
                state_out[((bh * Ls_out + j) * DK + r) * (long long)dv + col0 + c] =
                    on ? S[(m * DK + r) * kGW + c] : 0.f;
            }
        }
    }
}

int scan_stages(int dk, int N, int nlv, int tin_bytes)
{
    return scan_layout(dk, N, nlv, 2, tin_bytes).bytes <= kMaxSmem ? 2 : 1;
}

template <typename Tin, int DK>
cudaError_t launch_chunk_dk(const GdnFwdArgs &A)
{
    const int N = (A.T + kGC - 1) / kGC;
    const long long BH = (long long)A.B * A.H;
    const WsLayout W = ws_layout(BH, N, DK, A.dv);
    uint8_t *ws = (uint8_t *)A.workspace;
    float *ws_qw = (float *)(ws + W.qw), *ws_h = (float *)(ws + W.h), *ws_gend = (float *)(ws + W.gend);
    cudaStream_t s = (cudaStream_t)A.stream;

    const size_t psmem = prep_layout(DK, A.dv, A.L).floats * sizeof(float);
    auto prep = gdn_chunk_prep_kernel<Tin, DK>;
    cudaError_t e = cudaFuncSetAttribute(prep, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)psmem);
    if (e != cudaSuccess) return e;
    prep<<<dim3(N, A.H, A.B), kGT, psmem, s>>>((const Tin *)A.q, (const Tin *)A.k, (const Tin *)A.v, A.g, A.beta,
                                                A.lam, A.out, ws_qw, ws_h, ws_gend, A.state_out, A.T, N, A.H, A.dv,
                                                A.L, A.Ls_out);
    e = cudaPeekAtLastError();
    if (e != cudaSuccess) return e;

    const int nlv = A.L - (kGCBits + 1) > 0 ? A.L - (kGCBits + 1) : 0;
    const int nst = scan_stages(DK, N, nlv, (int)sizeof(Tin));
    const size_t ssmem = scan_layout(DK, N, nlv, nst, (int)sizeof(Tin)).bytes;
    auto scan = gdn_chunk_scan_kernel<Tin, DK>;
    e = cudaFuncSetAttribute(scan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)ssmem);
    if (e != cudaSuccess) return e;
    scan<<<dim3(A.dv / kGW, A.H, A.B), kGT, ssmem, s>>>((const Tin *)A.k, A.lam, A.out, ws_qw, ws_h, ws_gend,
                                                         A.state_out, A.T, N, A.H, A.dv, A.L, A.Ls_out, nst);
    return cudaPeekAtLastError();
}

template <typename Tin>
cudaError_t launch_chunk(const GdnFwdArgs &A)
{
    switch (A.dk) {
    case 16: return launch_chunk_dk<Tin, 16>(A);
    case 32: return launch_chunk_dk<Tin, 32>(A);
    case 64: return launch_chunk_dk<Tin, 64>(A);
    default: return launch_chunk_dk<Tin, 128>(A);
    }
}

}  // namespace

size_t gdn_fwd_workspace_bytes(int B, int H, int T, int dk, int dv)
{
    if ((long long)B * H * T <= 0) return 0;
    return ws_layout((long long)B * H, (T + kGC - 1) / kGC, dk, dv).bytes;
}

bool gdn_fwd_fits(int T, int dk, int dv, int L, int tin_bytes)
{
    const int N = (T + kGC - 1) / kGC;
    const int nlv = L - (kGCBits + 1) > 0 ? L - (kGCBits + 1) : 0;
    return prep_layout(dk, dv, L).floats * sizeof(float) <= kMaxSmem &&
           scan_layout(dk, N, nlv, 1, tin_bytes).bytes <= kMaxSmem;
}

cudaError_t gdn_fwd(const GdnFwdArgs &A)
{
    return A.in_dt == LLA_F32 ? launch_chunk<float>(A) : launch_chunk<__nv_bfloat16>(A);
}

}  // namespace lla
