// Recurrent decode step and prefill -> decode state hand-off.
// Page "Log-Linear Attention" (gist.science 2506.04761), technical summary
// §2.3: decoding is recurrent, each step touching O(log T) level states;
// §2.2: one state per Fenwick bucket of the prefix [0, t).
//
// State of one (batch, head): S[Ls][dk][dv] fp32 (slot i = level i+1) and a
// log-decay D[Ls]; the true level state is exp(D_i) * S_i.  Slot i is live at
// token index t iff bit i of t is set.  Keeping the decay as a scalar per slot
// means a step reads the popcount(t) live slots once and writes one slot,
// instead of rescaling every live slot in memory.
#include <cooperative_groups.h>

#include "decode.cuh"
#include "outer_simt.cuh"
#include "sm100.cuh"

namespace lla {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxLs = 40;

// One cluster of kParts CTAs per (head, sequence); CTA `part` owns rows
// [part*dk/kParts, (part+1)*dk/kParts) of every slot, all dv columns: one
// contiguous chunk of each slot (16 KB at dk = dv = 128).  The live slots'
// chunks stream into shared memory by bulk copies through a ring of
// kRing buffers, issued as soon as the position is known (before the small
// vector loads), so each SM keeps about three CTAs x kRing chunks in
// flight.  Thread layout inside a CTA: cg = column group of 4 (float4),
// rg = row group; a thread owns rows rg, rg+R, ... of its 4 columns.  The
// partial read-outs are summed through distributed shared memory by CTA 0,
// which also writes the slot log-decays once every CTA of the cluster has
// read them.
constexpr int kParts = 4;
constexpr int kRing = 4;
constexpr uint32_t kCopyWait = 1u << 22;  // bounded waits on the slot copies

template <typename Tin, int DV>
__global__ void __cluster_dims__(kParts, 1, 1) __launch_bounds__(kThreads, 3)
decode_step_kernel(float *__restrict__ S, float *__restrict__ D, const Tin *__restrict__ q,
                   const Tin *__restrict__ k, const Tin *__restrict__ v,
                   const float *__restrict__ g, const float *__restrict__ lam,
                   float *__restrict__ out, const int64_t *__restrict__ pos, int H, int dk,
                   int Ls, int32_t *__restrict__ err)
{
    namespace cg = cooperative_groups;
    using namespace sm100;
    constexpr int dv = DV;
    constexpr int NC4 = DV / 4;                 // column groups
    constexpr int R = kThreads / NC4;           // row groups
    constexpr int RPT = (128 / kParts + R - 1) / R;  // rows per thread (dk <= 128)
    extern __shared__ __align__(128) uint8_t ring[];  // kRing chunks of rows x DV fp32
    __shared__ float qs[128], kss[128], vs[DV];
    __shared__ float wl[kMaxLs], el[kMaxLs], dnew[kMaxLs];
    __shared__ float red[R][DV];
    __shared__ float part_out[DV];
    __shared__ float qk_sh;
    __shared__ uint64_t bar[kRing];

    cg::cluster_group cluster = cg::this_cluster();
    const int part = (int)cluster.block_rank();
    const int h = blockIdx.x / kParts, b = blockIdx.y;
    const long long bh = (long long)b * H + h;
    const int64_t t = pos[b];
    // every CTA of the cluster takes the same branch (same sequence)
    if (t < 0 || bit_length_u64((uint64_t)t + 1) > Ls) {
        if (part == 0 && threadIdx.x == 0 && err != nullptr) *err = 1 + b;
        return;
    }
    const int tid = threadIdx.x;
    const int rows = dk / kParts, row0 = part * rows;
    const uint32_t chunk = (uint32_t)rows * DV * 4;  // bytes of this CTA's part of a slot
    const uint64_t live_all = (uint64_t)t & ((Ls >= 64) ? ~0ull : ((1ull << Ls) - 1));
    const int nlive = __popcll(live_all);
    // the k-th live slot's chunk into ring buffer k % kRing
    auto issue = [&](int kk, uint64_t rest) {
        const int l = ctz_u64(rest);
        uint64_t *bb = &bar[kk % kRing];
        mbar_arrive_expect_tx(bb, chunk);
        bulk_load(ring + (kk % kRing) * chunk, S + ((bh * Ls + l) * (long long)dk + row0) * dv, chunk, bb);
    };
    if (tid == 0) {
        for (int i = 0; i < kRing; i++) mbar_init(&bar[i], 1);
        fence_mbar_init();
        uint64_t rest = live_all;
        for (int kk = 0; kk < kRing && rest; kk++) {
            issue(kk, rest);
            rest &= rest - 1;
        }
    }
    for (int r = tid; r < dk; r += kThreads) {
        qs[r] = to_f32(q[bh * dk + r]);
        kss[r] = to_f32(k[bh * dk + r]);
    }
    for (int c = tid; c < dv; c += kThreads) vs[c] = to_f32(v[bh * dv + c]);
    const float gg = g[bh];
    if (tid < Ls) {
        const bool live = (t >> tid) & 1;
        const float dn = D[bh * Ls + tid] + (live ? gg : 0.f);
        dnew[tid] = dn;
        const float e = live ? expf(dn) : 0.f;
        el[tid] = e;
        wl[tid] = live ? lam[bh * (Ls + 1) + tid + 1] * e : 0.f;
    }
    __syncthreads();
    if (part == 0 && tid < 32) {
        float p = 0.f;
        for (int r = tid; r < dk; r += 32) p = fmaf(qs[r], kss[r], p);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) p += __shfl_xor_sync(0xffffffffu, p, off);
        if (tid == 0) qk_sh = p;
    }

    const int m = ctz_u64((uint64_t)t + 1);
    const int cg4 = tid % NC4, rg = tid / NC4;
    const int col = cg4 * 4;
    constexpr int ncol4 = DV / 4;
    float4 mrg[RPT];
#pragma unroll
    for (int i = 0; i < RPT; i++) mrg[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);

    // live slots in order, each from its ring buffer once its copy has landed;
    // a buffer is refilled with the slot kRing later once every thread is done
    uint64_t live = live_all, ahead = live_all;
    for (int i = 0; i < kRing && ahead; i++) ahead &= ahead - 1;  // the slots not yet issued
    for (int kk = 0; kk < nlive; kk++) {
        const int l0 = ctz_u64(live);
        live &= live - 1;
        if (!mbar_wait(&bar[kk % kRing], (kk / kRing) & 1, kCopyWait) && err != nullptr) atomicCAS(err, 0, -1);
        const float4 *S0 = reinterpret_cast<const float4 *>(ring + (kk % kRing) * chunk);
        float4 sv0[RPT];
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + R * i;
            sv0[i] = (r < rows) ? S0[r * NC4 + cg4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float w0 = wl[l0], e0 = (l0 < m) ? el[l0] : 0.f;
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + R * i;
            const float qr = (r < rows) ? qs[row0 + r] : 0.f;
            const float a0 = qr * w0;
            acc.x = fmaf(a0, sv0[i].x, acc.x);
            acc.y = fmaf(a0, sv0[i].y, acc.y);
            acc.z = fmaf(a0, sv0[i].z, acc.z);
            acc.w = fmaf(a0, sv0[i].w, acc.w);
            // slots below m are carried into the new slot (e = 0 for the others)
            mrg[i].x = fmaf(e0, sv0[i].x, mrg[i].x);
            mrg[i].y = fmaf(e0, sv0[i].y, mrg[i].y);
            mrg[i].z = fmaf(e0, sv0[i].z, mrg[i].z);
            mrg[i].w = fmaf(e0, sv0[i].w, mrg[i].w);
        }
        if (kk + kRing < nlive) {
            __syncthreads();  // every thread has read buffer kk % kRing
            if (tid == 0) issue(kk + kRing, ahead);
            ahead &= ahead - 1;
        }
    }
    red[rg][col + 0] = acc.x;
    red[rg][col + 1] = acc.y;
    red[rg][col + 2] = acc.z;
    red[rg][col + 3] = acc.w;
    // the new slot m (level m+1) is dead at t, so no CTA of this step reads it
    {
        float4 *Sm = reinterpret_cast<float4 *>(S + ((bh * Ls + m) * (long long)dk) * dv);
        const float4 vv = make_float4(vs[col], vs[col + 1], vs[col + 2], vs[col + 3]);
#pragma unroll
        for (int i = 0; i < RPT; i++) {
            const int r = rg + R * i;
            if (r < rows) {
                const float kr = kss[row0 + r];
                float4 o;
                o.x = fmaf(kr, vv.x, mrg[i].x);
                o.y = fmaf(kr, vv.y, mrg[i].y);
                o.z = fmaf(kr, vv.z, mrg[i].z);
                o.w = fmaf(kr, vv.w, mrg[i].w);
                __stcs(Sm + (long long)(row0 + r) * ncol4 + cg4, o);
            }
        }
    }
    __syncthreads();
    for (int c = tid; c < DV; c += kThreads) {
        float o = 0.f;
#pragma unroll 4
        for (int r = 0; r < R; r++) o += red[r][c];
        part_out[c] = o;
    }
    cluster.sync();  // partials ready; every CTA has read the old log-decays
    if (part == 0) {
        for (int c = tid; c < DV; c += kThreads) {
            float o = lam[bh * (Ls + 1)] * qk_sh * vs[c];
#pragma unroll
            for (int p2 = 0; p2 < kParts; p2++) o += cluster.map_shared_rank(part_out, p2)[c];
            out[bh * dv + c] = o;
        }
        if (tid < Ls) D[bh * Ls + tid] = (tid == m) ? 0.f : dnew[tid];
    }
    cluster.sync();  // keep every CTA's partials alive until CTA 0 has read them
}

// tail[bh][s] = sum_{r=s+1}^{T-1} g[bh][r], accumulated in fp64 and stored
// fp32, in two launches over chunks of kTailChunk tokens: chunk sums, then
// each chunk's suffix scan plus its carry (the sum of the later chunks' sums,
// formed by one warp of the chunk's CTA).
constexpr int kTailChunk = 1024;

__global__ void __launch_bounds__(256)
prefill_chunk_sum_kernel(const float *__restrict__ g, double *__restrict__ csum, int T, int nchunk)
{
    __shared__ double wsum[8];
    const long long bh = blockIdx.y;
    const int c = blockIdx.x;
    double a = 0.0;
    for (int i = threadIdx.x; i < kTailChunk; i += 256) {
        const long long r = (long long)c * kTailChunk + i;
        if (r < T) a += (double)g[bh * T + r];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = a;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < 8; w++) t += wsum[w];
        csum[bh * nchunk + c] = t;
    }
}

__global__ void __launch_bounds__(kTailChunk)
prefill_tail_kernel(const float *__restrict__ g, const double *__restrict__ csum, float *__restrict__ tail,
                    int T, int nchunk)
{
    __shared__ double wsum[kTailChunk / 32];
    __shared__ double carry_sh;
    const long long bh = blockIdx.y;
    const int c = blockIdx.x;
    const int i = threadIdx.x, lane = i & 31, w = i >> 5;
    if (w == 0) {  // the carry: the sums of the chunks after c, in a fixed order
        double a = 0.0;
        for (int c2 = c + 1 + lane; c2 < nchunk; c2 += 32) a += csum[bh * nchunk + c2];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a += __shfl_xor_sync(0xffffffffu, a, off);
        if (lane == 0) carry_sh = a;
    }
    const long long r = (long long)c * kTailChunk + i;
    const double x = r < T ? (double)g[bh * T + r] : 0.0;
    double incl = x;  // sum over this lane and the later lanes of the warp
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_down_sync(0xffffffffu, incl, off);
        if (lane + off < 32) incl += y;
    }
    if (lane == 0) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
        const double own = wsum[lane];
        double s = own;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double y = __shfl_down_sync(0xffffffffu, s, off);
            if (lane + off < 32) s += y;
        }
        wsum[lane] = s - own;  // later warps of the chunk
    }
    __syncthreads();
    if (r < T) tail[bh * T + r] = (float)(carry_sh + wsum[w] + (incl - x));
}

constexpr int kSeg = 1024;  // tokens per CTA of the bucket kernel

struct BucketTable {
    long long start[kMaxLs];
    long long len[kMaxLs];
    int seg_begin[kMaxLs + 1];
    int slot[kMaxLs];
    int n;
};

template <typename Tin>
__global__ void __launch_bounds__(kThreads)
prefill_bucket_kernel(const Tin *__restrict__ k, const Tin *__restrict__ v,
                      const float *__restrict__ tail, float *__restrict__ S, BucketTable tab,
                      int T, int dk, int dv, int Ls)
{
    __shared__ __align__(16) float ks[kOuterSub * 128];
    __shared__ __align__(16) float vs[kOuterSub * 128];
    __shared__ float sc[kOuterSub];
    const long long bh = blockIdx.y;
    const int sid = blockIdx.x;
    int li = 0;
    while (li + 1 < tab.n && tab.seg_begin[li + 1] <= sid) li++;
    const long long s_lo = tab.start[li] + (long long)(sid - tab.seg_begin[li]) * kSeg;
    const long long s_hi = min(s_lo + kSeg, tab.start[li] + tab.len[li]);
    float acc[8][8];
    outer_zero(acc);
    const Tin *kb = k + bh * (long long)T * dk;
    const Tin *vb = v + bh * (long long)T * dv;
    const float *tb = tail + bh * (long long)T;
    for (long long s0 = s_lo; s0 < s_hi; s0 += kOuterSub) {
        const int ns = (int)min((long long)kOuterSub, s_hi - s0);
        if (threadIdx.x < kOuterSub) sc[threadIdx.x] = (int)threadIdx.x < ns ? expf(tb[s0 + threadIdx.x]) : 0.f;
        __syncthreads();
        outer_stage<Tin>(ks, kb + s0 * dk, nullptr, ns, dk);
        outer_stage<Tin>(vs, vb + s0 * dv, sc, ns, dv);
        __syncthreads();
        outer_accumulate(acc, ks, vs, ns, dk, dv);
    }
    const int r0 = 8 * (threadIdx.x >> 4), c0 = 8 * (threadIdx.x & 15);
    if (r0 >= dk || c0 >= dv) return;
    float *Sl = S + (bh * Ls + tab.slot[li]) * (long long)dk * dv;
#pragma unroll
    for (int a = 0; a < 8; a++)
#pragma unroll
        for (int b = 0; b < 8; b++) atomicAdd(Sl + (r0 + a) * dv + c0 + b, acc[a][b]);
}

template <typename Tin, int DV>
void launch_decode_dv(const DecodeArgs &A)
{
    const size_t smem = (size_t)kRing * (A.dk / kParts) * DV * 4;
    if (smem > 48 * 1024)
        cudaFuncSetAttribute(decode_step_kernel<Tin, DV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    decode_step_kernel<Tin, DV><<<dim3(A.H * kParts, A.B), kThreads, smem, (cudaStream_t)A.stream>>>(
        A.S, A.D, (const Tin *)A.q, (const Tin *)A.k, (const Tin *)A.v, A.g, A.lam, A.out, A.pos,
        A.H, A.dk, A.Ls, A.err);
}

template <typename Tin>
cudaError_t launch_decode(const DecodeArgs &A)
{
    switch (A.dv) {
    case 16: launch_decode_dv<Tin, 16>(A); break;
    case 32: launch_decode_dv<Tin, 32>(A); break;
    case 64: launch_decode_dv<Tin, 64>(A); break;
    default: launch_decode_dv<Tin, 128>(A); break;
    }
    return cudaPeekAtLastError();
}

template <typename Tin>
cudaError_t launch_prefill(const PrefillArgs &A)
{
    cudaStream_t st = (cudaStream_t)A.stream;
    const long long BH = (long long)A.B * A.H;
    cudaError_t err = cudaMemsetAsync(A.S, 0, sizeof(float) * BH * A.Ls * A.dk * A.dv, st);
    if (err != cudaSuccess) return err;
    err = cudaMemsetAsync(A.D, 0, sizeof(float) * BH * A.Ls, st);
    if (err != cudaSuccess) return err;
    if (A.T == 0) return cudaSuccess;
    BucketTable tab{};
    int nseg = 0;
    for (int l = 1; l <= A.Ls && l <= 40; l++) {
        if (!(((long long)A.T >> (l - 1)) & 1)) continue;
        const long long start = ((long long)A.T >> l) << l;
        const long long len = 1LL << (l - 1);
        tab.start[tab.n] = start;
        tab.len[tab.n] = len;
        tab.slot[tab.n] = l - 1;
        tab.seg_begin[tab.n] = nseg;
        nseg += (int)((len + kSeg - 1) / kSeg);
        tab.n++;
    }
    tab.seg_begin[tab.n] = nseg;
    float *tail = (float *)A.workspace;
    const int nchunk = (A.T + kTailChunk - 1) / kTailChunk;
    const size_t tail_bytes = align_up((size_t)BH * A.T * sizeof(float), 256);
    double *csum = (double *)((char *)A.workspace + tail_bytes);
    prefill_chunk_sum_kernel<<<dim3(nchunk, (unsigned)BH), 256, 0, st>>>(A.g, csum, A.T, nchunk);
    prefill_tail_kernel<<<dim3(nchunk, (unsigned)BH), kTailChunk, 0, st>>>(A.g, csum, tail, A.T, nchunk);
    if (prefill_tc_supported(A)) {
        int *dev_err = A.device_error ? (int *)A.device_error
                                      : (int *)((char *)(csum + align_up((size_t)BH * nchunk, 32)));
        if (!A.device_error) {
            err = cudaMemsetAsync(dev_err, 0, sizeof(int), st);
            if (err != cudaSuccess) return err;
        }
        return prefill_tc(A, tail, dev_err);
    }
    prefill_bucket_kernel<Tin><<<dim3(nseg, (unsigned)BH), kThreads, 0, st>>>(
        (const Tin *)A.k, (const Tin *)A.v, tail, A.S, tab, A.T, A.dk, A.dv, A.Ls);
    return cudaPeekAtLastError();
}

}  // namespace

cudaError_t decode_step(const DecodeArgs &A)
{
    if (A.in_dt == LLA_F32) return launch_decode<float>(A);
    return launch_decode<__nv_bfloat16>(A);
}

size_t prefill_workspace_bytes(int B, int H, int T)
{
    // per-token tails, chunk sums (fp64), the tensor-core path's error word
    const size_t BH = (size_t)B * H;
    const size_t nchunk = (size_t)((T > 0 ? T : 1) + kTailChunk - 1) / kTailChunk;
    return align_up(BH * (size_t)(T > 0 ? T : 1) * sizeof(float), 256) +
           align_up(BH * nchunk, 32) * sizeof(double) + 256;
}

cudaError_t prefill_state(const PrefillArgs &A)
{
    if (A.in_dt == LLA_F32) return launch_prefill<float>(A);
    return launch_prefill<__nv_bfloat16>(A);
}

}  // namespace lla
