// Log-Linear Gated DeltaNet, one decode step (the recurrent form).
//
// "Log-Linear Attention" §3 builds Log-Linear Gated DeltaNet by keeping the
// Gated DeltaNet state update and adding the hierarchical (Fenwick) mask; the
// pages give no formula.  Here every Fenwick bucket of the prefix keeps its
// own state S_l (dk x dv, the sum-of-k-v^T orientation) and all of them take
// each token's transition A_t = alpha_t (I - beta_t k_t k_t^T),
// alpha_t = exp(g_t).  Per token t (§2.3's recurrent form, slot i = level
// i+1, live iff bit i of t is set):
//   1. S_l <- A_t S_l for every live slot;
//   2. o_t = lam_t[0] beta_t (q_t.k_t) v_t + sum_live lam_t[l] S_l^T q_t;
//   3. slot m = ctz(t+1) receives beta_t k_t v_t^T + sum of slots below it.
// Column c of every state only ever mixes with itself: with
// P = q.S[:,c] and U = k.S[:,c] of the old state, the new column is
// alpha (S[:,c] - beta U k) and its read-out alpha (P - beta U (q.k)).
// The forward over whole sequences is the chunkwise form (gdn_chunk.cu).
#include "gdn.cuh"

namespace lla {
namespace {

// One decode step on the level state in global memory [B,H,Ls,dk,dv].
// A warp owns 32/SPLIT value columns of one (batch, head); SPLIT lanes share
// a column, each holding R = DK/SPLIT of its rows in registers, so the dot
// products over dk need only a SPLIT-lane shuffle and the state is read in
// full 32-byte sectors.  The slots below m = ctz(t+1) are only summed into
// the new slot, and because the transition is linear their transitioned sum
// is alpha (sum_i S_i - beta k sum_i (k.S_i)): one register column
// accumulates them as they stream in.  The other live slots are loaded into
// the same registers, transitioned and stored back.
template <typename Tin, int DK, int DV, int SPLIT>
__global__ void __launch_bounds__(32)
gdn_decode_kernel(float *__restrict__ S, const Tin *__restrict__ q, const Tin *__restrict__ k,
                  const Tin *__restrict__ v, const float *__restrict__ g, const float *__restrict__ beta,
                  const float *__restrict__ lam, float *__restrict__ out, const int64_t *__restrict__ pos,
                  int H, int Ls, int32_t *__restrict__ err)
{
    constexpr int dv = DV;
    constexpr int CW = 32 / SPLIT;  // columns per warp
    constexpr int R = DK / SPLIT;   // rows per lane
    __shared__ float qs[DK], ks[DK];
    const int lane = threadIdx.x;
    const int part = lane / CW;
    const int col = blockIdx.x * CW + lane % CW;
    const int b = blockIdx.z;
    const long long bh = (long long)b * H + blockIdx.y;
    const long long t64 = pos[b];
    if (t64 < 0 || bit_length_u64((uint64_t)(t64 + 1)) > Ls) {  // no room in the state
        if (err && lane == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicCAS(err, 0, 1 + b);
        return;
    }
    const uint64_t t = (uint64_t)t64;
    float qk = 0.f;
    for (int r = lane; r < DK; r += 32) {
        const float a = to_f32(q[bh * DK + r]), c = to_f32(k[bh * DK + r]);
        qs[r] = a;
        ks[r] = c;
        qk = fmaf(a, c, qk);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) qk += __shfl_xor_sync(0xffffffffu, qk, off);
    __syncwarp();
    const bool active = col < dv;  // inactive lanes still join the shuffles
    const float al = expf(g[bh]), be = beta[bh];
    const float vc = active ? to_f32(v[bh * dv + col]) : 0.f;
    const float *lt = lam + bh * (Ls + 1);
    float *Sb = S + bh * (long long)Ls * DK * dv + (long long)(part * R) * dv + (active ? col : 0);
    const float *qp = qs + part * R, *kp = ks + part * R;
    const int m = ctz_u64(t + 1u);
    float o = lt[0] * be * qk * vc;
    auto allsum = [](float x) {
#pragma unroll
        for (int off = CW; off < 32; off <<= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        return x;
    };
    float x[R];
    // slots 0..m-1: live, folded into slot m
#pragma unroll
    for (int r = 0; r < R; r++) x[r] = 0.f;
    float U = 0.f;
    for (int i = 0; i < m; i++) {
        const float *Si = Sb + (long long)i * DK * dv;
        float p = 0.f, u = 0.f;
#pragma unroll
        for (int r = 0; r < R; r++) {
            const float sv = active ? __ldcs(Si + (long long)r * dv) : 0.f;
            p = fmaf(qp[r], sv, p);
            u = fmaf(kp[r], sv, u);
            x[r] += sv;
        }
        p = allsum(p);
        u = allsum(u);
        U += u;
        o = fmaf(lt[i + 1], al * (p - be * u * qk), o);
    }
    if (active) {
        float *Sm = Sb + (long long)m * DK * dv;
        const float bu = be * U;
#pragma unroll
        for (int r = 0; r < R; r++) Sm[(long long)r * dv] = fmaf(be * kp[r], vc, al * (x[r] - bu * kp[r]));
    }
    // live slots above m: transitioned in place
    for (int i = m + 1; i < Ls; i++) {
        if (!((t >> i) & 1u)) continue;
        float *Si = Sb + (long long)i * DK * dv;
        float p = 0.f, u = 0.f;
#pragma unroll
        for (int r = 0; r < R; r++) {
            x[r] = active ? Si[(long long)r * dv] : 0.f;
            p = fmaf(qp[r], x[r], p);
            u = fmaf(kp[r], x[r], u);
        }
        p = allsum(p);
        u = allsum(u);
        const float bu = be * u;
        if (active) {
#pragma unroll
            for (int r = 0; r < R; r++) Si[(long long)r * dv] = al * (x[r] - bu * kp[r]);
        }
        o = fmaf(lt[i + 1], al * (p - bu * qk), o);
    }
    if (active && part == 0) out[bh * dv + col] = o;
}

template <typename Tin, int DK, int DV>
void launch_decode_dkv(const GdnDecodeArgs &A)
{
    constexpr int SPLIT = DK / 32 > 1 ? DK / 32 : 1;
    constexpr int CW = 32 / SPLIT;
    gdn_decode_kernel<Tin, DK, DV, SPLIT><<<dim3((DV + CW - 1) / CW, A.H, A.B), 32, 0, (cudaStream_t)A.stream>>>(
        A.S, (const Tin *)A.q, (const Tin *)A.k, (const Tin *)A.v, A.g, A.beta, A.lam, A.out, A.pos, A.H,
        A.Ls, A.err);
}

template <typename Tin, int DK>
void launch_decode_dk(const GdnDecodeArgs &A)
{
    switch (A.dv) {
    case 16: launch_decode_dkv<Tin, DK, 16>(A); break;
    case 32: launch_decode_dkv<Tin, DK, 32>(A); break;
    case 64: launch_decode_dkv<Tin, DK, 64>(A); break;
    default: launch_decode_dkv<Tin, DK, 128>(A); break;
    }
}

template <typename Tin>
cudaError_t launch_decode(const GdnDecodeArgs &A)
{
    switch (A.dk) {
    case 16: launch_decode_dk<Tin, 16>(A); break;
    case 32: launch_decode_dk<Tin, 32>(A); break;
    case 64: launch_decode_dk<Tin, 64>(A); break;
    default: launch_decode_dk<Tin, 128>(A); break;
    }
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t gdn_decode_step(const GdnDecodeArgs &A)
{
    return A.in_dt == LLA_F32 ? launch_decode<float>(A) : launch_decode<__nv_bfloat16>(A);
}

}  // namespace lla
