// Chunked forward on the 5th-generation tensor cores (tcgen05, TMEM, TMA),
// bf16 q/k/v with fp32 accumulation, dk = dv = D for D = 64 or 128.
//
// Page "Log-Linear Attention" (gist.science 2506.04761), technical summary
// §2.2 (Fenwick buckets of [0,t), one state per bucket, lambda-weighted
// read-out) and §2.3 (the hierarchical mask computed chunkwise with matmuls).
//
// Five launches.  Two small kernels form the fp64 tile-gate prefix sums.  Node
// walkers (one CTA per head and segment of tiles, the whole dv width, walking in order
// with the Fenwick stack in tensor memory) compute each tile's state and
// publish the tile-level Fenwick nodes; a fix-up kernel chains the nodes that
// span segments.  The read-out consumer (persistent: one CTA per SM taking
// tiles from a queue, the next tile's inputs loading while the current one
// computes) forms the masked intra-tile product and the lambda-weighted
// read-out of the nodes.  With Gam_i the gate sum of tile i and
// P_i = Gam_0 + ... + Gam_{i-1} (fp64, from the prefix kernels), the earlier
// tiles of tile i form the tile-level Fenwick buckets ending at
// j = i, i - lowbit(i), ...; bucket j (level m = ctz(j)) holds the tiles
// [j - 2^m, j) decayed to the end of tile j-1:
//     Node_j = sum over those tiles' keys s of exp(P_j - G_s) k_s v_s^T.
// A key s of bucket j has level 7 + 1 + m for every query of tile i.
// Per tile:
//   S  = Q K^T                              (tcgen05, TMEM)
//   H  = K^T diag(exp(Gam - gamma)) V        (tcgen05, TMEM) -> Node_{i+1}
//        Node_{i+1} = H + sum_{m < ctz(i+1)} exp(P_{i+1} - P_{j_m}) Node_{j_m},
//        j_m = i + 1 - 2^m, published to global memory in bf16
//   P  = S . M,  M[a][b] = lambda_a[bit_length(a^b)] exp(gamma_a - gamma_b), b <= a
//   O  = P V + sum_{path j} diag(lambda_.[8+m] exp(gamma_. + P_i - P_j)) (Q Node_j)
// Every product above is a tcgen05 MMA of M = 128 (tokens, or dk padded to
// 128 rows for D = 64), bf16 operands in 128-byte-swizzled shared memory,
// fp32 accumulators in tensor memory.  The read-out forms U_j = Q Node_j per
// path node in tensor memory and applies the per-row weights in fp32 while
// draining it.
#include <atomic>

#include "fwd_tc.cuh"
#include "sm100.cuh"
#include "tma_host.cuh"

namespace lla {
namespace {

using namespace sm100;

constexpr int kTile = 128;       // tokens per tile (MMA M)
constexpr int kTileLevels = 7;   // levels inside a tile: bit_length(a ^ b) <= 7
constexpr uint32_t kBlk = kTile * 128;  // one 64-column swizzled block of a 128-row bf16 tile: 16 KB
constexpr uint32_t kWaitIters = 1u << 22;  // bounded waits (~0.5 s with back-off)
constexpr uint32_t kWithheldWaitIters = 4096;  // the waits while the test hook withholds a product
constexpr int kMaxPath = 17;               // levels of a tile index (T <= 2^24, so NT <= 2^17)
constexpr int kLamMax = 25;                // lambda entries per token: L <= 1 + bit_length(2^24 - 1)
constexpr int kMlpHidden = 32;             // hidden width of the in-kernel lambda MLP (2L <= 32)

// Error codes (lla_device_error) written to the error word.
constexpr int kErrLoadTimeout = LLA_DEVERR_COPY_TIMEOUT;
constexpr int kErrMmaTimeout = LLA_DEVERR_SYNC_TIMEOUT;

struct TcParams {
    const float *g, *lam;
    void *out;
    const double *P;        // [BH][NT+1] tile-gate prefix sums
    float *gamma;           // [BH][NT][128] inclusive gate sum inside each tile (fp32)
    int *err;               // first bounded wait that gave up (0: none): the caller's word or the workspace's
    int *queue;             // next work item of the read-out consumer (reset to 0 by the gate-sum kernel)
    float *segtot;          // [BH][nseg_full][D][D] decayed segment totals
    __nv_bfloat16 *node16;  // [BH][NT][D][D] Fenwick nodes (index 0 unused)
    int T, NT, BH, L, nseg_full;
    // lambda from the two-layer MLP on the key tile ("Adaptive memory decay for
    // Log-Linear Attention", LambdaMLPSoftplus) instead of a lambda input
    const float *W1, *W2, *bmlp;  // [D][2L], [2L][L], [L] fp32
    int mlp;
    uint32_t wait_iters;    // polls before a wait gives up
    uint32_t s_wait_iters;  // the same for the waits on S = Q K^T (short while it is withheld)
    int withhold;           // test hook: the consumer issues no S = Q K^T and no signal for it
};

__device__ __forceinline__ void set_err(int *err, int code) { atomicCAS(err, 0, code); }

// MMAs over K = D with A and B K-major (rows of 128 B, K split in 64-column blocks).
template <int D>
__device__ __forceinline__ void mma_kk(uint32_t d, const uint8_t *a, const uint8_t *b, uint32_t idesc)
{
#pragma unroll
    for (int kk = 0; kk < D / 16; kk++) {
        const uint32_t off = (kk >> 2) * kBlk + (kk & 3) * 32;
        umma_bf16(d, desc_sw128(smem_u32(a) + off, 16, 1024), desc_sw128(smem_u32(b) + off, 16, 1024),
                  idesc, kk > 0 ? 1u : 0u);
    }
}

// MMAs over K = D with A K-major and B MN-major (rows = K index, N in
// 64-column blocks of D rows each).
template <int D>
__device__ __forceinline__ void mma_kmn(uint32_t d, const uint8_t *a, const uint8_t *b, uint32_t idesc)
{
#pragma unroll
    for (int kk = 0; kk < D / 16; kk++) {
        const uint32_t offa = (kk >> 2) * kBlk + (kk & 3) * 32;
        const uint32_t offb = kk * 2048;
        umma_bf16(d, desc_sw128(smem_u32(a) + offa, 16, 1024),
                  desc_sw128(smem_u32(b) + offb, (uint32_t)D * 128, 1024), idesc, kk > 0 ? 1u : 0u);
    }
}

// ======================================================= node walkers
// The tile-level Fenwick nodes Node_j (j = 1 .. NT-1) are built by walkers:
// one CTA per (batch*head, segment of 8 tiles) goes through its segment in
// order.  For tile i it forms the whole state H_i (D x D) on the tensor
// cores and closes Node_{i+1}:
//     Node_{i+1} = H_i + sum_{m < ctz(i+1)} exp(P_{i+1} - P_{i+1-2^m}) Node_{i+1-2^m},
// keeping the latest node of each level (the Fenwick stack, three levels) in
// fp32 in tensor memory, so nothing crosses CTAs and nothing waits.  Only
// the node that closes a full segment reaches back before the segment; the
// walker writes that segment's decayed total instead, and the fix-up kernel
// forms the nodes at segment granularity from the totals.  Nodes are
// published in bf16, the read-out's MMA operand.  Each K and V tile is read
// once; a ring of three tiles keeps the loads in flight.  For D = 64 the
// product's M (= dk) is padded to 128: the second 64-row block of the K^T
// operand reads whatever shared memory follows the tile, and those rows of
// H are never read.

// fp32 tile of 128 rows staged as 32-column boxes of 128 rows x 128 B:
// byte offset of the 4-float chunk holding columns [4c, 4c+4) of row r.
__device__ __forceinline__ uint32_t f32_stage_off(int r, int c)
{
    return (uint32_t)(c >> 3) * (kTile * 128) + sw128_offset(r, c & 7);
}

constexpr int kSegLog = 3;
constexpr int kSeg = 1 << kSegLog;       // tiles per segment
constexpr int kWalkStages = 2;           // K/V tiles in flight per walker
constexpr int kWalkEpi = 512;            // warps 0-15: node epilogue, four threads per dk row
constexpr int kWalkPrep = 128;           // warps 8-11: tile preparation, thread = token row
constexpr int kWalkThreads = kWalkEpi + kWalkPrep + 64;  // warp 16: loader, warp 17: MMA issuer

template <int D>
struct __align__(1024) WalkSmem {
    uint8_t k[kWalkStages][kTile * D * 2];  // K tiles
    uint8_t v[kWalkStages][kTile * D * 2];  // V tiles, scaled in place by exp(Gam - gamma)
    uint8_t nst[2][D * D * 2];              // closed nodes in bf16, staged for their TMA stores (two in turn)
    float gm[kWalkStages][kTile];           // the tile's inclusive gate sums gamma
    double P[kSeg + 1];                     // P_{i0} .. P_{i0+kSeg}
    uint64_t bar_load[kWalkStages], bar_scaled[kWalkStages], bar_h, bar_hfree;
    uint32_t tmem;
};

// the epilogue threads of a walker: four per dk row
template <int D>
__device__ __forceinline__ void wepi_sync()
{
    asm volatile("bar.sync 2, %0;" ::"n"((kWalkEpi / 128) * D) : "memory");
}

// tensor-memory columns of a walker: the stack's kSegLog levels and H, D each
template <int D>
constexpr uint32_t walk_tmem_cols()
{
    return (kSegLog + 1) * D <= 256 ? 256u : 512u;
}


// Warp-specialised, every hand-off through an mbarrier: a loader warp keeps
// the ring of K/V tiles full (tile n+3 as soon as tile n's product is done),
// the preparation warps scale V by exp(Gam - gamma), an MMA warp issues the
// state product of each scaled tile, and the epilogue warps fold tile n-1's
// state into the Fenwick stack and publish the node.
template <int D>
__global__ void __launch_bounds__(kWalkThreads, 1)
lla_node_walker_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                       const __grid_constant__ CUtensorMap map_node, const TcParams prm)
{
    constexpr uint32_t kT = kTile * D * 2;
    extern __shared__ uint8_t smem_raw[];
    WalkSmem<D> &s = *reinterpret_cast<WalkSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                      ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int seg = blockIdx.x, bh = blockIdx.y;
    const int NT = prm.NT;
    const int i0 = seg * kSeg, i1 = min(i0 + kSeg, NT - 1);  // tiles i0..i1-1 close Node_{i+1}
    const int ntiles = i1 - i0;
    const double *Pb = prm.P + (long long)bh * (NT + 1);

    if (tid == 0) {
        for (int b = 0; b < kWalkStages; b++) {
            mbar_init(&s.bar_load[b], 1);
            mbar_init(&s.bar_scaled[b], kWalkPrep);
        }
        mbar_init(&s.bar_h, 1);
        mbar_init(&s.bar_hfree, (kWalkEpi / 128) * D);
        fence_mbar_init();
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        tma_prefetch_map(&map_node);
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, walk_tmem_cols<D>());
        tmem_relinquish();
    }
    // a tile's K and V (inputs), then its 128 gamma values (from the gate
    // launches: one aligned 512-byte run), on one barrier
    auto issue_kv = [&](int n) {
        const int ls = n % kWalkStages, i = i0 + n;
        mbar_arrive_expect_tx(&s.bar_load[ls], 2 * kT + kTile * 4);
#pragma unroll
        for (int h = 0; h < D / 64; h++) {
            tma_load_3d(s.k[ls] + h * kBlk, &map_k, &s.bar_load[ls], h * 64, i * kTile, bh);
            tma_load_3d(s.v[ls] + h * kBlk, &map_v, &s.bar_load[ls], h * 64, i * kTile, bh);
        }
    };
    auto issue_gamma = [&](int n) {
        const int ls = n % kWalkStages, i = i0 + n;
        bulk_load(s.gm[ls], prm.gamma + ((long long)bh * NT + i) * kTile, kTile * 4, &s.bar_load[ls]);
    };
    auto issue_load = [&](int n) {
        issue_kv(n);
        issue_gamma(n);
    };
    constexpr int kLoader = kWalkEpi + kWalkPrep;  // the loader lane
    __syncthreads();  // the barriers are initialised
    // the first tiles' K and V load while the gate launches finish; gamma and
    // P only after them
    if (tid == kLoader)
        for (int n = 0; n < kWalkStages && n < ntiles; n++) issue_kv(n);
    grid_dependency_wait();
    grid_launch_dependents();  // the fix-up and read-out may start in this grid's tail (after the gates)
    if (tid == kLoader)
        for (int n = 0; n < kWalkStages && n < ntiles; n++) issue_gamma(n);
    for (int j = tid; j <= kSeg; j += kWalkThreads) s.P[j] = (i0 + j <= NT) ? Pb[i0 + j] : 0.0;
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;
    // columns: stack level m at [D m, D m + D) for m < kSegLog; H after it
    const uint32_t tm_h = tm + kSegLog * D;

    if (tid >= kWalkEpi + kWalkPrep + 32) {
        // ---------------- MMA issuer (one lane): tile n's product once its V is
        // scaled and tile n-1's state has been drained from the accumulator
        if ((tid & 31) == 0) {
            const uint32_t idesc = idesc_bf16_f32(128, D, true, true);
            for (int n = 0; n < ntiles; n++) {
                const int ls = n % kWalkStages;
                if (!mbar_wait(&s.bar_scaled[ls], (n / kWalkStages) & 1, prm.wait_iters))
                    set_err(prm.err, kErrMmaTimeout);
                if (n >= 1 && !mbar_wait(&s.bar_hfree, (n - 1) & 1, prm.wait_iters))
                    set_err(prm.err, kErrMmaTimeout);
                tc_fence_after_sync();
                // H = K^T Vs: A = K^T (M = 128 >= dk, MN-major), B = Vs (N = D, MN-major)
                const uint64_t da = desc_sw128(smem_u32(s.k[ls]), kBlk, 1024);
                const uint64_t db = desc_sw128(smem_u32(s.v[ls]), kBlk, 1024);
#pragma unroll
                for (int kk = 0; kk < 8; kk++)  // K step of 16 rows = 2048 bytes = 128 in the address field
                    umma_bf16(tm_h, da + kk * 128, db + kk * 128, idesc, kk > 0 ? 1u : 0u);
                umma_commit(&s.bar_h);
            }
        }
    } else if (tid >= kWalkEpi + kWalkPrep) {
        // ---------------- loader (one lane): a stage is refilled once the
        // product of the tile it held is done
        if ((tid & 31) == 0)
            for (int n = kWalkStages; n < ntiles; n++) {  // the first stages were issued above
                if (!mbar_wait(&s.bar_h, (n - kWalkStages) & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                issue_load(n);
            }
    } else if (tid >= kWalkEpi) {
        // ---------------- preparation warps: thread = token row
        const int prow = tid - kWalkEpi;
        for (int n = 0; n < ntiles; n++) {
            const int ls = n % kWalkStages;
            if (!mbar_wait(&s.bar_load[ls], (n / kWalkStages) & 1, prm.wait_iters)) set_err(prm.err, kErrLoadTimeout);
            const float w = __expf(s.gm[ls][kTile - 1] - s.gm[ls][prow]);
            // V row prow scaled in place by exp(Gam - gamma), eight 16-byte chunks at a
            // time: all loads first, then the products, then the stores
            uint8_t *const vrow = s.v[ls] + prow * 128;
            const uint32_t sw = (uint32_t)(prow & 7);
#pragma unroll
            for (int c0 = 0; c0 < D / 8; c0 += 8) {
                uint4 raw[8];
#pragma unroll
                for (int c = 0; c < 8; c++)
                    raw[c] = *reinterpret_cast<const uint4 *>(vrow + ((c0 + c) >> 3) * kBlk + ((c ^ sw) << 4));
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&raw[c]);
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const float2 f = __bfloat1622float2(h[u]);
                        h[u] = __floats2bfloat162_rn(f.x * w, f.y * w);
                    }
                }
#pragma unroll
                for (int c = 0; c < 8; c++)
                    *reinterpret_cast<uint4 *>(vrow + ((c0 + c) >> 3) * kBlk + ((c ^ sw) << 4)) = raw[c];
            }
            fence_proxy_async_smem();
            mbar_arrive(&s.bar_scaled[ls]);
        }
    } else if ((tid & 127) < D) {
        // ---------------- epilogue warps: thread = (dk row, quarter of the columns)
        constexpr int kC = D / (kWalkEpi / 128);  // columns per thread
        const int r = tid & 127, q = tid >> 7;
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t c0 = q * kC;
        int nstage = 0;  // nodes published so far: the staging buffer alternates
        for (int n = 0; n < ntiles; n++) {
            const int J = i0 + n + 1;
            const int z = __ffs(J) - 1;
            const bool cross = (J == i0 + kSeg);  // closes a full segment
            // the tile before a segment-closing one (whose epilogue folds nothing)
            // combines the stack, decayed to the segment's end, into level 0, so
            // the closing tile folds that one level instead of kSegLog
            const bool pre = (J == i0 + kSeg - 1) && (ntiles == kSeg);
            const int mlim = cross ? 1 : z;
            if (!mbar_wait(&s.bar_h, n & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
            tc_fence_after_sync();
            float acc[kC];
#pragma unroll
            for (int c = 0; c < kC; c += 16) tmem_ld16(tm_h + lane_off + c0 + c, *reinterpret_cast<float(*)[16]>(acc + c));
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(&s.bar_hfree);  // the next tile's product may overwrite H
            const double PJ = s.P[J - i0];
            for (int m = 0; m < mlim; m++) {
                const float f = cross ? 1.f : __expf((float)(PJ - s.P[J - (1 << m) - i0]));
#pragma unroll
                for (int c = 0; c < kC; c += 16) {
                    float x[16];
                    tmem_ld16(tm + m * D + lane_off + c0 + c, x);
                    tmem_ld_wait();
#pragma unroll
                    for (int u = 0; u < 16; u++) acc[c + u] = fmaf(f, x[u], acc[c + u]);
                }
            }
            if (!cross) {
                if (z < kSegLog && !pre) {
#pragma unroll
                    for (int c = 0; c < kC; c += 16)
                        tmem_st16(tm + z * D + lane_off + c0 + c, *reinterpret_cast<float(*)[16]>(acc + c));
                    tmem_st_wait();
                }
                // the node in bf16 through shared memory (the layout of its TMA box:
                // 64-column blocks of D rows, 128-byte swizzle) and one TMA store;
                // a staging buffer is reused once the store two nodes back has read it
                uint8_t *const nst = s.nst[nstage & 1];
                if (tid == 0) tma_store_wait_read_all_but_one();
                wepi_sync<D>();
#pragma unroll
                for (int c = 0; c < kC / 8; c++) {
                    const int cg = (c0 >> 3) + c;  // 8-column chunk of the row
                    uint4 w;
                    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w);
#pragma unroll
                    for (int u = 0; u < 4; u++) h[u] = __floats2bfloat162_rn(acc[8 * c + 2 * u], acc[8 * c + 2 * u + 1]);
                    *reinterpret_cast<uint4 *>(nst + (cg >> 3) * (D * 128) + sw128_offset(r, cg & 7)) = w;
                }
                fence_proxy_async_smem();
                wepi_sync<D>();
                if (tid == 0) {
#pragma unroll
                    for (int h = 0; h < D / 64; h++)
                        tma_store_3d(&map_node, nst + h * (D * 128), h * 64, 0, bh * NT + J);
                    tma_store_commit();
                }
                nstage++;
                if (pre) {
                    // this node and the stack levels above it, each decayed to the
                    // segment's end P_{i0 + kSeg}: the segment total less the next
                    // tile's state
                    const double PE = s.P[kSeg];
                    const float f0 = __expf((float)(PE - PJ));
#pragma unroll
                    for (int u = 0; u < kC; u++) acc[u] *= f0;
                    for (int m = 1; m < kSegLog; m++) {
                        const float f = __expf((float)(PE - s.P[kSeg - (1 << m)]));
#pragma unroll
                        for (int c = 0; c < kC; c += 16) {
                            float x[16];
                            tmem_ld16(tm + m * D + lane_off + c0 + c, x);
                            tmem_ld_wait();
#pragma unroll
                            for (int u = 0; u < 16; u++) acc[c + u] = fmaf(f, x[u], acc[c + u]);
                        }
                    }
#pragma unroll
                    for (int c = 0; c < kC; c += 16)
                        tmem_st16(tm + lane_off + c0 + c, *reinterpret_cast<float(*)[16]>(acc + c));
                    tmem_st_wait();
                }
            } else {
                float4 *dst = reinterpret_cast<float4 *>(
                    prm.segtot + (((long long)bh * prm.nseg_full + seg) * D + r) * D + c0);
#pragma unroll
                for (int u = 0; u < kC / 4; u++)
                    dst[u] = make_float4(acc[4 * u], acc[4 * u + 1], acc[4 * u + 2], acc[4 * u + 3]);
            }
        }
        if (tid == 0) tma_store_wait_all();  // the staging is read before the CTA ends
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, walk_tmem_cols<D>());
}

// Nodes that close full segments, each on its own from the segment totals:
// node u SEG covers segments [u - lowbit(u), u), so
//   Node_{u SEG} = sum_{sigma in [u - lowbit(u), u)} exp(P_{u SEG} - P_{(sigma+1) SEG}) Tot_sigma.
// One CTA per (2048 state elements, u, batch*head): a thread owns 8 elements
// (two float4 at a 1024-element stride, so the CTA's loads are coalesced) and
// the totals are summed two segments at a time with all loads in flight.
constexpr int kFixThreads = 256;
constexpr int kFixElems = kFixThreads * 8;
template <int D>
__global__ void __launch_bounds__(kFixThreads)
lla_node_fixup_kernel(const TcParams prm)
{
    grid_launch_dependents();
    grid_dependency_wait();  // the walkers' segment totals
    const long long bh = blockIdx.z;
    const int u = blockIdx.y + 1;
    const int NT = prm.NT, nseg = prm.nseg_full;
    const int e0 = blockIdx.x * kFixElems + threadIdx.x * 4;  // elements [e0, e0+4) and [e0+1024, e0+1028)
    const double *Pb = prm.P + bh * (NT + 1);
    const double Pu = Pb[u * kSeg];
    const int first = u - (u & -u);
    float4 va = make_float4(0.f, 0.f, 0.f, 0.f), vb = va;
    for (int sg = first; sg < u; sg += 2) {
        const bool two = sg + 1 < u;
        const float *t0 = prm.segtot + ((bh * nseg) + sg) * (D * D);
        const float4 a0 = *reinterpret_cast<const float4 *>(t0 + e0);
        const float4 b0 = *reinterpret_cast<const float4 *>(t0 + e0 + 1024);
        float4 a1 = make_float4(0.f, 0.f, 0.f, 0.f), b1 = a1;
        if (two) {
            a1 = *reinterpret_cast<const float4 *>(t0 + D * D + e0);
            b1 = *reinterpret_cast<const float4 *>(t0 + D * D + e0 + 1024);
        }
        const float f0 = __expf((float)(Pu - Pb[(sg + 1) * kSeg]));
        const float f1 = two ? __expf((float)(Pu - Pb[(sg + 2) * kSeg])) : 0.f;
        va.x = fmaf(f0, a0.x, fmaf(f1, a1.x, va.x));
        va.y = fmaf(f0, a0.y, fmaf(f1, a1.y, va.y));
        va.z = fmaf(f0, a0.z, fmaf(f1, a1.z, va.z));
        va.w = fmaf(f0, a0.w, fmaf(f1, a1.w, va.w));
        vb.x = fmaf(f0, b0.x, fmaf(f1, b1.x, vb.x));
        vb.y = fmaf(f0, b0.y, fmaf(f1, b1.y, vb.y));
        vb.z = fmaf(f0, b0.z, fmaf(f1, b1.z, vb.z));
        vb.w = fmaf(f0, b0.w, fmaf(f1, b1.w, vb.w));
    }
    __nv_bfloat16 *dst = prm.node16 + (bh * NT + (long long)u * kSeg) * (D * D);
    *reinterpret_cast<__nv_bfloat162 *>(dst + e0) = __floats2bfloat162_rn(va.x, va.y);
    *reinterpret_cast<__nv_bfloat162 *>(dst + e0 + 2) = __floats2bfloat162_rn(va.z, va.w);
    *reinterpret_cast<__nv_bfloat162 *>(dst + e0 + 1024) = __floats2bfloat162_rn(vb.x, vb.y);
    *reinterpret_cast<__nv_bfloat162 *>(dst + e0 + 1026) = __floats2bfloat162_rn(vb.z, vb.w);
}

// ======================================================= read-out consumer
// Persistent: one CTA per SM takes tiles from a queue (a counter in the
// workspace) in order, last tiles first and tile-major across heads, so
// co-running tiles share their deep nodes and the nodes written last are
// still in L2.  Eighteen warps:
//   warps 0-15 epilogue (thread = (row, quarter of the columns)): the mask
//              P, the drains of P V and of every U = Q Node_j with its fp32
//              per-row weight, the output staged in shared memory; four
//              threads per row keep enough warps in flight to hide the
//              tensor-memory and barrier latencies;
//   warp 16    producer: writes out (TMA store) the output staged in a stage,
//              then takes the next tile and brings its q, k, v, gamma,
//              lambda and path P values into that stage (two stages), and
//              its path nodes into L2;
//   warp 17    MMA issuer (one lane): S, P V, the node loads and the U's.
// Tile n uses stage n & 1 and tensor-memory region n & 1, so the MMAs and
// loads of tile n+1 proceed while the epilogue drains tile n.  The roles
// hand off through mbarriers only; the barriers used a variable number of
// times per tile are waited with running completion counts.

constexpr int kEpiThreads = 512;   // 16 epilogue warps: 4 threads per row
constexpr int kConsThreads = kEpiThreads + 64;  // plus a producer warp and an MMA warp
constexpr int kProdWarp = kEpiThreads / 32, kMmaWarp = kProdWarp + 1;
constexpr int kParts = kEpiThreads / kTile;  // threads per row

template <int D>
struct __align__(1024) ConsStage {
    uint8_t q[kTile * D * 2];
    uint8_t k[kTile * D * 2];  // K, then path node 0, 2, ...; with q the fp32 output staging
    uint8_t v[kTile * D * 2];  // V, then path node 1, 3, ...
};

// Shared memory after the stages: either the lambda rows of each stage
// ([128][L] fp32, loaded with the tile), or, with the in-kernel lambda MLP,
// the first layer's weights as bf16 high and low parts in the K-major
// swizzled layout of one N = 64 MMA operand (per 64-wide K block, the 32
// hidden rows of the high part, then those of the low part), the second
// layer and bias (fp32) and one [128][L] staging of the tile's lambdas.
template <int D>
struct MlpLayout {
    static constexpr uint32_t kW1Part = kMlpHidden * D * 2;
    static constexpr uint32_t kW2 = 2 * kW1Part;                        // [2L][L] fp32
    static constexpr uint32_t kBias = kW2 + kMlpHidden * 16 * 4;        // L <= 16
    static constexpr uint32_t kLam = kBias + 16 * 4;                    // [128][L] fp32
    static constexpr uint32_t kEnd = kLam + kTile * 16 * 4;
};
constexpr uint32_t kLamStage = kTile * kLamMax * 4;
template <int D>
constexpr uint32_t aux_bytes()
{
    return MlpLayout<D>::kEnd > 2 * kLamStage ? MlpLayout<D>::kEnd : 2 * kLamStage;
}

template <int D>
struct __align__(1024) ConsSmem {
    ConsStage<D> st[2];
    uint8_t aux[aux_bytes<D>()];    // lambda stages, or the MLP's weights and lambda staging
    float gam[2][kTile];
    float kf[kTile];                // exp(gamma_e - gamma_b), e = last key of b's 16-key chunk
    double pj[2][kMaxPath + 1];     // P at the path nodes of the stage's tile, then P_i
    int item[2];                    // the stage's work item, -1 when the queue is empty
    uint64_t bar_load[2], bar_staged[2], bar_tfree[2];
    uint64_t bar_s, bar_pready, bar_pv, bar_pvfree, bar_h;
    uint64_t bar_node[2], bar_u[2], bar_ufree[2];
    uint32_t tmem;
};

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 512;" ::: "memory"); }

// Work item w -> tile (i, bh): tile-major, last tiles first.
__device__ __forceinline__ void item_tile(int w, int NT, int BH, int *i, int *bh)
{
    const int rev = NT * BH - 1 - w;
    *i = rev / BH;
    *bh = rev - *i * BH;
}

template <int D, typename OutT>
__global__ void __launch_bounds__(kConsThreads, 1)
lla_readout_consumer_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                            const __grid_constant__ CUtensorMap map_v,
                            const __grid_constant__ CUtensorMap map_node,
                            const __grid_constant__ CUtensorMap map_out, const TcParams prm)
{
    constexpr uint32_t kT = kTile * D * 2;  // bytes of one bf16 tile
    constexpr uint32_t kRegion = 128 + D;   // tensor-memory columns per tile: S / P / U even, then P V / U odd
    extern __shared__ uint8_t smem_raw[];
    ConsSmem<D> &s = *reinterpret_cast<ConsSmem<D> *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                      ~uintptr_t(1023));
    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int NT = prm.NT, BH = prm.BH, L = prm.L;
    const int total = NT * BH;

    if (tid == kEpiThreads) {
        for (int b = 0; b < 2; b++) {
            mbar_init(&s.bar_load[b], 1);
            mbar_init(&s.bar_staged[b], 1);
            mbar_init(&s.bar_tfree[b], kEpiThreads);
            mbar_init(&s.bar_node[b], 1);
            mbar_init(&s.bar_u[b], 1);
            mbar_init(&s.bar_ufree[b], kEpiThreads);
        }
        mbar_init(&s.bar_s, 1);
        mbar_init(&s.bar_pready, kEpiThreads);
        mbar_init(&s.bar_pv, 1);
        mbar_init(&s.bar_pvfree, kEpiThreads);
        mbar_init(&s.bar_h, 1);
        fence_mbar_init();
        tma_prefetch_map(&map_q);
        tma_prefetch_map(&map_k);
        tma_prefetch_map(&map_v);
        tma_prefetch_map(&map_node);
        tma_prefetch_map(&map_out);
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem, 512);
        tmem_relinquish();
    }
    using ML = MlpLayout<D>;
    if (prm.mlp) {
        // W1 split into bf16 high and low parts (together about 16 bits of every
        // weight; the keys are exact in bf16), transposed into the K-major
        // operand layout, hidden columns past 2L zero; W2 and the bias in fp32
        const int Hd = 2 * L;
        for (int e = tid; e < kMlpHidden * D; e += kConsThreads) {
            const int n = e / D, kx = e % D;
            const float w = n < Hd ? prm.W1[kx * Hd + n] : 0.f;
            const __nv_bfloat16 hi = __float2bfloat16_rn(w);
            const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
            // per 64-wide K block: rows [0, 32) the high part, [32, 64) the low part
            const uint32_t blk = (uint32_t)(kx >> 6) * (2 * kMlpHidden * 128), in = (kx & 7) * 2;
            *reinterpret_cast<__nv_bfloat16 *>(s.aux + blk + sw128_offset(n, (kx & 63) >> 3) + in) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(s.aux + blk + sw128_offset(kMlpHidden + n, (kx & 63) >> 3) + in) = lo;
        }
        float *w2 = reinterpret_cast<float *>(s.aux + ML::kW2);  // [32][L], rows past 2L zero
        for (int e = tid; e < kMlpHidden * L; e += kConsThreads) w2[e] = e < Hd * L ? prm.W2[e] : 0.f;
        for (int e = tid; e < L; e += kConsThreads) reinterpret_cast<float *>(s.aux + ML::kBias)[e] = prm.bmlp[e];
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tm = s.tmem;

    if (warp == kProdWarp) {
        // ---------------- producer
        // The output of the tile that last used a stage, staged there by the
        // epilogue, is written out by TMA from here before the stage is
        // refilled, so the epilogue never waits for the store.
        auto issue_store = [&](int sgx, int nx) {  // lane 0: tile nx of stage sgx
            if (!mbar_wait(&s.bar_staged[sgx], (nx >> 1) & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
            int io, bho;
            item_tile(s.item[sgx], NT, BH, &io, &bho);
            const ConsStage<D> &t = s.st[sgx];
            if (sizeof(OutT) == 4) {
#pragma unroll
                for (int b = 0; b < D / 32; b++) tma_store_3d(&map_out, t.q + b * (kTile * 128), b * 32, io * kTile, bho);
            } else {
#pragma unroll
                for (int h = 0; h < D / 64; h++) tma_store_3d(&map_out, t.q + h * kBlk, h * 64, io * kTile, bho);
            }
            tma_store_commit();
        };
        bool dep_done = false;
        for (int n = 0;; n++) {
            const int sg = n & 1;
            // the next work item and the P values at its path nodes, fetched while
            // the tile that last used this stage may still be reading out
            int w = 0;
            if (lane == 0) w = atomicAdd(prm.queue, 1);
            w = __shfl_sync(0xffffffffu, w, 0);
            const bool have = w < total;
            int i = 0, bh = 0, j = 0;
            double pv = 0.0;
            if (have) {
                item_tile(w, NT, BH, &i, &bh);
                const double *Pb = prm.P + (long long)bh * (NT + 1);
                // lane c clears the c lowest set bits of i; lane 31 takes P_i
                j = i;
                for (int c = 0; c < lane && j > 0; c++) j -= (j & -j);
                if (lane < kMaxPath && j > 0) pv = Pb[j];
                if (lane == 31) pv = Pb[i];
            }
            if (n >= 2 && lane == 0) issue_store(sg, n - 2);
            __syncwarp();
            if (!have) {
                if (lane == 0) {
                    s.item[sg] = -1;
                    mbar_arrive(&s.bar_load[sg]);
                    if (n >= 1) issue_store(sg ^ 1, n - 1);  // the last tile taken
                    tma_store_wait_read();  // the stores read shared memory before the CTA ends
                }
                break;
            }
            if (lane < kMaxPath && j > 0) s.pj[sg][lane] = pv;
            if (lane == 31) s.pj[sg][kMaxPath] = pv;
            if (lane == 0) s.item[sg] = w;
            __syncwarp();
            if (lane == 0) {
                const int rows = min(kTile, prm.T - i * kTile);
                const uint32_t lam_bytes = prm.mlp ? 0u : (uint32_t)rows * L * 4;
                uint64_t *bar = &s.bar_load[sg];
                mbar_arrive_expect_tx(bar, 3 * kT + lam_bytes + kTile * 4);
                ConsStage<D> &t = s.st[sg];
                // V, lambda and gamma first; q and k once the store has read the
                // output staged in their buffers
#pragma unroll
                for (int h = 0; h < D / 64; h++) tma_load_3d(t.v + h * kBlk, &map_v, bar, h * 64, i * kTile, bh);
                const long long tok0 = (long long)bh * prm.T + (long long)i * kTile;
                if (!prm.mlp)
                    bulk_load(s.aux + sg * kLamStage, prm.lam + tok0 * L, lam_bytes, bar);
                bulk_load(s.gam[sg], prm.gamma + ((long long)bh * NT + i) * kTile, kTile * 4, bar);
                if (n >= 2) tma_store_wait_read();
#pragma unroll
                for (int h = 0; h < D / 64; h++) {
                    tma_load_3d(t.q + h * kBlk, &map_q, bar, h * 64, i * kTile, bh);
                    tma_load_3d(t.k + h * kBlk, &map_k, bar, h * 64, i * kTile, bh);
                }
            }
            // the tile's path nodes into L2 ahead of their loads (lane c: node c);
            // they come from the previous launches, so wait for those once
            if (i > 0) {
                if (!dep_done) {
                    grid_dependency_wait();
                    dep_done = true;
                }
                if (lane < kMaxPath && j > 0)
                    bulk_prefetch_l2(prm.node16 + ((long long)bh * NT + j) * (D * D), (uint32_t)D * D * 2);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMA issuer (one lane)
        if (lane == 0) {
            const uint32_t id_s = idesc_bf16_f32(128, 128, false, false);
            const uint32_t id_kmn = idesc_bf16_f32(128, D, false, true);
            const uint32_t id_h = idesc_bf16_f32(128, 2 * kMlpHidden, false, false);
            // [K W1_hi | K W1_lo] (one N = 64 product per K step) into slot 1 of the tile's region
            auto issue_h = [&](uint32_t slot1, const uint8_t *kt) {
#pragma unroll
                for (int kk = 0; kk < D / 16; kk++) {
                    const uint32_t offa = (kk >> 2) * kBlk + (kk & 3) * 32;
                    const uint32_t offb = (kk >> 2) * (2 * kMlpHidden * 128) + (kk & 3) * 32;
                    umma_bf16(slot1, desc_sw128(smem_u32(kt) + offa, 16, 1024),
                              desc_sw128(smem_u32(s.aux) + offb, 16, 1024), id_h, kk ? 1u : 0u);
                }
                umma_commit(&s.bar_h);
            };
            // parities of the completions so far of bar_node[b] and bar_u[b] (bit b):
            // only parities are ever waited on
            uint32_t par_node = 0, par_u = 0;
            bool dep_done = false;
            bool s_early = false;  // this tile's S was issued while the previous tile read out
            for (int n = 0;; n++) {
                const int sg = n & 1;
                if (!mbar_wait(&s.bar_load[sg], (n >> 1) & 1, prm.wait_iters)) set_err(prm.err, kErrLoadTimeout);
                const int w = s.item[sg];
                if (w < 0) break;
                int i, bh;
                item_tile(w, NT, BH, &i, &bh);
                const int npath = __popc(i);
                if (!s_early && n >= 2 && !mbar_wait(&s.bar_tfree[sg], ((n - 2) >> 1) & 1, prm.wait_iters))
                    set_err(prm.err, kErrMmaTimeout);
                tc_fence_after_sync();
                // slot b at slot0 + 128 b; node buffer b is k (b = 0) or v (b = 1)
                const uint32_t slot0 = tm + sg * kRegion;
                ConsStage<D> &t = s.st[sg];
                auto nd = [&](int b) { return t.k + b * kT; };
                auto load_node = [&](int b, int jn) {  // a D x D bf16 node, D/64 boxes of 64 columns
                    mbar_arrive_expect_tx(&s.bar_node[b], (uint32_t)D * D * 2);
#pragma unroll
                    for (int h = 0; h < D / 64; h++)
                        tma_load_3d(nd(b) + h * (D * 128), &map_node, &s.bar_node[b], h * 64, 0, bh * NT + jn);
                };
                auto wait_node = [&](int b) {
                    if (!mbar_wait(&s.bar_node[b], (par_node >> b) & 1, prm.wait_iters))
                        set_err(prm.err, kErrLoadTimeout);
                    par_node ^= 1u << b;
                };
                auto issue_u = [&](int b) {
                    tc_fence_after_sync();
                    mma_kmn<D>(slot0 + 128 * b, t.q, nd(b), id_kmn);
                    umma_commit(&s.bar_u[b]);
                    par_u ^= 1u << b;
                };
                // parity of the completion of the latest U issued into slot b
                auto last_u_par = [&](int b) { return ((par_u >> b) & 1) ^ 1; };
                if (!s_early) {
                    if (!prm.withhold) {  // withheld: nothing is left in flight, the waits on bar_s run out
                        mma_kk<D>(slot0, t.q, t.k, id_s);
                        umma_commit(&s.bar_s);
                    }
                    if (prm.mlp) issue_h(slot0 + 128, t.k);
                }
                s_early = false;
                int jnext = i;
                if (npath > 0) {
                    if (!mbar_wait(&s.bar_s, n & 1, prm.s_wait_iters)) set_err(prm.err, kErrMmaTimeout);
                    // with the lambda MLP, h = K W1 was issued after S and reads K too
                    if (prm.mlp && !mbar_wait(&s.bar_h, n & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                    if (!dep_done) {
                        // the nodes come from the previous launches; everything before this
                        // point reads only inputs and the gate sums
                        grid_dependency_wait();
                        dep_done = true;
                    }
                    load_node(0, jnext);  // the K buffer is free once S (and h) are done
                    jnext -= (jnext & -jnext);
                }
                // O = P V: P from tensor memory once the epilogue has stored it
                if (!mbar_wait(&s.bar_pready, n & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                tc_fence_after_sync();
                // P of keys [32p, 32p+32) sits packed in columns [32p, 32p+16)
#pragma unroll
                for (int kk = 0; kk < 8; kk++)
                    umma_bf16_tmem_a(slot0 + 128, slot0 + (kk >> 1) * 32 + (kk & 1) * 8,
                                     desc_sw128(smem_u32(t.v) + kk * 2048, kBlk, 1024), id_kmn, kk > 0 ? 1u : 0u);
                umma_commit(&s.bar_pv);
                if (npath > 0) {
                    if (!mbar_wait(&s.bar_pv, n & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                    if (npath > 1) {
                        load_node(1, jnext);  // the V buffer is free once P V is done
                        jnext -= (jnext & -jnext);
                    }
                    // path node 0 into slot 0 (P has been consumed)
                    wait_node(0);
                    issue_u(0);
                }
                {   // the next tile's S, if its inputs have landed and its region is free,
                    // so that the epilogue finds it done when it gets there
                    const int n1 = n + 1, sg1 = n1 & 1;
                    if (mbar_test(&s.bar_load[sg1], (n1 >> 1) & 1) && s.item[sg1] >= 0 &&
                        (n1 < 2 || mbar_test(&s.bar_tfree[sg1], ((n1 - 2) >> 1) & 1))) {
                        tc_fence_after_sync();
                        if (!prm.withhold) {
                            mma_kk<D>(tm + sg1 * kRegion, s.st[sg1].q, s.st[sg1].k, id_s);
                            umma_commit(&s.bar_s);
                        }
                        if (prm.mlp) issue_h(tm + sg1 * kRegion + 128, s.st[sg1].k);
                        s_early = true;
                    }
                }
                // Node k+2 goes into buffer b as soon as U_k has read it, before U_{k+1}
                // waits for its own node
                for (int k = 0; k < npath; k++) {
                    const int b = k & 1, b1 = b ^ 1;
                    if (k + 2 < npath) {
                        // node buffer b is free once U_k's product is done
                        if (!mbar_wait(&s.bar_u[b], last_u_par(b), prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                        load_node(b, jnext);
                        jnext -= (jnext & -jnext);
                    }
                    if (k + 1 < npath) {
                        // slot b1 is free once U_{k-1} (or, for k = 0, P V) is drained
                        if (k == 0) {
                            if (!mbar_wait(&s.bar_pvfree, n & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                        } else {
                            // the drain of U_{k-1}, the latest U in slot b1
                            if (!mbar_wait(&s.bar_ufree[b1], last_u_par(b1), prm.wait_iters))
                                set_err(prm.err, kErrMmaTimeout);
                        }
                        wait_node(b1);
                        issue_u(b1);
                    }
                }
            }
        }
        __syncwarp();
    } else {
        // ---------------- epilogue warps
        const int row = tid & (kTile - 1);
        const int part = tid >> 7;                      // keys [32 part, +32), columns [kCols part, +kCols)
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        constexpr int kCols = D / kParts;               // output columns per thread
        uint32_t par_u = 0;  // parity of the completions of bar_u[b] consumed so far (bit b)
        for (int n = 0;; n++) {
            const int sg = n & 1;
            if (!mbar_wait(&s.bar_load[sg], (n >> 1) & 1, prm.wait_iters)) set_err(prm.err, kErrLoadTimeout);
            const int w = s.item[sg];
            if (w < 0) break;
            int i, bh;
            item_tile(w, NT, BH, &i, &bh);
            const int npath = __popc(i);
            const bool row_ok = row < prm.T - i * kTile;
            const float *gam = s.gam[sg];
            const float gam_a = gam[row];
            const uint32_t slot0 = tm + sg * kRegion, slot1 = slot0 + 128;
            const float *lam_a;
            if (prm.mlp) {
                // lambda_l = softplus(b_l + sum_j h_j W2[j][l]) for l = part, part + 4, ...;
                // h (the row's 2L hidden values) from tensor memory
                if (!mbar_wait(&s.bar_h, n & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                tc_fence_after_sync();
                // h = K W1_hi + K W1_lo
                float h[kMlpHidden];
                {
                    float hl[16];
#pragma unroll
                    for (int c = 0; c < kMlpHidden; c += 16) {
                        tmem_ld16(slot1 + lane_off + c, *reinterpret_cast<float(*)[16]>(h + c));
                        tmem_ld16(slot1 + lane_off + kMlpHidden + c, hl);
                        tmem_ld_wait();
#pragma unroll
                        for (int u = 0; u < 16; u++) h[c + u] += hl[u];
                    }
                }
                const float *w2 = reinterpret_cast<const float *>(s.aux + ML::kW2);
                const float *bs = reinterpret_cast<const float *>(s.aux + ML::kBias);
                float *lst = reinterpret_cast<float *>(s.aux + ML::kLam);
                for (int l = part; l < L; l += kParts) {
                    float z = bs[l];
#pragma unroll
                    for (int jh = 0; jh < kMlpHidden; jh++) z = fmaf(h[jh], w2[jh * L + l], z);
                    lst[row * L + l] = fmaxf(z, 0.f) + log1pf(__expf(-fabsf(z)));
                }
                lam_a = lst + row * L;
            } else {
                lam_a = reinterpret_cast<const float *>(s.aux + sg * kLamStage) + row * L;
            }
            if (part == 0) s.kf[row] = __expf(gam[row | 15] - gam_a);
            epi_sync();
            // P = S . M  (thread = query row a, keys [32 part, 32 part + 32)), written
            // back packed (keys 2c, 2c+1 in one column) into columns
            // [32 part, 32 part + 16): columns this thread has already read, so no
            // other thread's S is overwritten.  A warp's 32 rows form one 32-row
            // block, so the case is uniform over the warp: keys all above its rows
            // (part > a/32), all below them (two 16-key chunks of one level each),
            // or the diagonal block, where each lane has the 16-key chunk holding
            // its own row (the lower chunk for rows 0-15 of the block, the upper one
            // for rows 16-31) and one chunk wholly below (or above) the row.
            // Below the row, with e the last key of the chunk,
            //   exp(gamma_a - gamma_b) = exp(gamma_a - gamma_e) exp(gamma_e - gamma_b),
            // both factors <= 1; inside the row's own chunk one exp per key.
            // The per-lane factors are formed before S is waited for.
            {
                const int a = row, rb = a >> 5, kb = part * 32;
                const bool hi = (a & 16) != 0;
                float cf0 = 0.f, cf1 = 0.f;  // lambda_a[level] exp(gamma_a - gamma_e) of each chunk
                if (part < rb) {
                    cf0 = lam_a[32 - __clz(a ^ kb)] * __expf(gam_a - gam[kb + 15]);
                    cf1 = lam_a[32 - __clz(a ^ (kb + 16))] * __expf(gam_a - gam[kb + 31]);
                } else if (part == rb && hi) {
                    // rows 16-31 of the block: keys [kb, kb + 16) lie below, at level 5
                    cf0 = lam_a[5] * __expf(gam_a - gam[kb + 15]);
                }
                if (!mbar_wait(&s.bar_s, n & 1, prm.s_wait_iters)) set_err(prm.err, kErrMmaTimeout);
                tc_fence_after_sync();
                uint32_t pk[16];
                auto pack = [](float x0, float x1) {
                    __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
                    return *reinterpret_cast<uint32_t *>(&h);
                };
                if (part > rb) {
#pragma unroll
                    for (int u = 0; u < 16; u++) pk[u] = 0u;
                } else {
                    // the loads are warp-collective: every lane of the warp issues them
                    float r0[16], r1[16];
                    tmem_ld16(slot0 + lane_off + kb, r0);
                    tmem_ld16(slot0 + lane_off + kb + 16, r1);
                    tmem_ld_wait();
                    const float4 *kf4 = reinterpret_cast<const float4 *>(s.kf + kb);
                    if (part < rb) {
#pragma unroll
                        for (int u = 0; u < 4; u++) {
                            const float4 f0 = kf4[u], f1 = kf4[4 + u];
                            pk[2 * u] = pack(r0[4 * u] * cf0 * f0.x, r0[4 * u + 1] * cf0 * f0.y);
                            pk[2 * u + 1] = pack(r0[4 * u + 2] * cf0 * f0.z, r0[4 * u + 3] * cf0 * f0.w);
                            pk[8 + 2 * u] = pack(r1[4 * u] * cf1 * f1.x, r1[4 * u + 1] * cf1 * f1.y);
                            pk[8 + 2 * u + 1] = pack(r1[4 * u + 2] * cf1 * f1.z, r1[4 * u + 3] * cf1 * f1.w);
                        }
                    } else {
                        const int cd = kb + (hi ? 16 : 0);  // the row's own chunk
#pragma unroll
                        for (int u = 0; u < 8; u++) {
                            float xd[2], xo[2];
#pragma unroll
                            for (int e = 0; e < 2; e++) {
                                const int j = 2 * u + e, b = cd + j;
                                // the level (0..4) varies over the lanes: a shared-memory
                                // lookup (a select chain over registers compiles to branches)
                                const float lj = lam_a[32 - __clz(a ^ b)];
                                const float ex = __expf(fminf(gam_a - gam[b], 0.f));
                                xd[e] = b <= a ? (hi ? r1[j] : r0[j]) * lj * ex : 0.f;
                                // the other chunk: below the row for rows 16-31 (cf0), above it
                                // for rows 0-15 (cf0 = 0)
                                xo[e] = (hi ? r0[j] : r1[j]) * cf0 * s.kf[kb + j];
                            }
                            const uint32_t pd = pack(xd[0], xd[1]), po = pack(xo[0], xo[1]);
                            pk[u] = hi ? po : pd;
                            pk[8 + u] = hi ? pd : po;
                        }
                    }
                }
                if (!row_ok) {  // a row past T
#pragma unroll
                    for (int u = 0; u < 16; u++) pk[u] = 0u;
                }
                tmem_st16(slot0 + lane_off + kb, *reinterpret_cast<const float(*)[16]>(pk));
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(&s.bar_pready);

            if (!mbar_wait(&s.bar_pv, n & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
            tc_fence_after_sync();
            float o[kCols];
#pragma unroll
            for (int c0 = 0; c0 < kCols; c0 += 16)
                tmem_ld16(slot1 + lane_off + part * kCols + c0, *reinterpret_cast<float(*)[16]>(o + c0));
            tmem_ld_wait();
            tc_fence_before_sync();
            mbar_arrive(&s.bar_pvfree);

            // read-out: U_k = Q Node_{j_k} in slot k & 1, drained with the fp32 weight
            //   lambda_a[8 + m_k] exp(gamma_a + P_i - P_{j_k}),  m_k = ctz(j_k)
            {
                const double Pi = s.pj[sg][kMaxPath];
                int j = i;
                for (int k = 0; k < npath; k++) {
                    const int b = k & 1;
                    const int m = __ffs(j) - 1;
                    j -= (j & -j);
                    const float wk = row_ok ? lam_a[kTileLevels + 1 + m] * __expf(gam_a + (float)(Pi - s.pj[sg][k]))
                                            : 0.f;
                    if (!mbar_wait(&s.bar_u[b], (par_u >> b) & 1, prm.wait_iters)) set_err(prm.err, kErrMmaTimeout);
                    par_u ^= 1u << b;
                    tc_fence_after_sync();
                    const uint32_t sl = slot0 + 128 * b;
                    float r[kCols];
#pragma unroll
                    for (int c0 = 0; c0 < kCols; c0 += 16)
                        tmem_ld16(sl + lane_off + part * kCols + c0, *reinterpret_cast<float(*)[16]>(r + c0));
                    tmem_ld_wait();
                    tc_fence_before_sync();
                    mbar_arrive(&s.bar_ufree[b]);
#pragma unroll
                    for (int u = 0; u < kCols; u++) o[u] = fmaf(wk, r[u], o[u]);
                }
            }
            // every tensor-memory read of this tile is done: its region may take tile n+2
            tc_fence_before_sync();
            mbar_arrive(&s.bar_tfree[sg]);

            // ---- stage the tile in the q/k buffers (every product that read them is
            // complete) for the producer's TMA store; rows past T are clipped by the
            // tensor map
            ConsStage<D> &t = s.st[sg];
            if (sizeof(OutT) == 4) {
                // fp32: D/32 boxes of 32 columns x 128 rows, in q then k
#pragma unroll
                for (int c = 0; c < kCols / 4; c++) {
                    const int cg = part * (kCols / 4) + c;  // 4-float chunk of the row
                    *reinterpret_cast<float4 *>(t.q + f32_stage_off(row, cg)) =
                        make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
                }
            } else {
                // bf16: D/64 blocks of 64 columns
#pragma unroll
                for (int c = 0; c < kCols / 8; c++) {
                    const int cg = part * (kCols / 8) + c;  // 8-element chunk of the row
                    uint4 w4;
                    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&w4);
#pragma unroll
                    for (int u = 0; u < 4; u++) h[u] = __floats2bfloat162_rn(o[8 * c + 2 * u], o[8 * c + 2 * u + 1]);
                    *reinterpret_cast<uint4 *>(t.q + (cg >> 3) * kBlk + sw128_offset(row, cg & 7)) = w4;
                }
            }
            fence_proxy_async_smem();
            epi_sync();
            if (tid == 0) mbar_arrive(&s.bar_staged[sg]);  // the producer stores it
        }
    }
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tm, 512);
}

// Gate sums, in two small launches.  First, a warp per tile: Gam_i in fp64
// from one coalesced float4 load per lane, stored in the P array shifted by
// one (P[i+1] = Gam_i); the consumer's queue counter and the workspace error
// word are reset here too (err is null when the caller passed a word of its
// own, which is never cleared).
// Then one CTA per (batch*head) turns the tile sums into the prefix
// P_i = Gam_0 + ... + Gam_{i-1} in place.
constexpr int kScanThreads = 1024;
__global__ void __launch_bounds__(1024)
lla_tile_gate_sum_kernel(const float *__restrict__ g, double *__restrict__ P, float *__restrict__ gamma,
                         int *__restrict__ err, int *__restrict__ queue, int T, int NT)
{
    grid_launch_dependents();  // the scan may launch now; it waits for this grid
    const long long bh = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tile = blockIdx.x * 32 + warp;
    double *Pb = P + bh * (long long)(NT + 1);
    if (tile < NT) {
        const float *gb = g + bh * (long long)T + (long long)tile * kTile;
        const int n = min(kTile, T - tile * kTile);
        double acc = 0.0;
        // 4 consecutive gates per lane; rows past T count as 0
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (n == kTile) {
            x = reinterpret_cast<const float4 *>(gb)[lane];
        } else {
            const int t = 4 * lane;
            if (t < n) x.x = gb[t];
            if (t + 1 < n) x.y = gb[t + 1];
            if (t + 2 < n) x.z = gb[t + 2];
            if (t + 3 < n) x.w = gb[t + 3];
        }
        acc = (double)x.x + (double)x.y + (double)x.z + (double)x.w;
        // inclusive running sum inside the tile (fp32), the form the kernels use
        const float s1 = x.x, s2 = s1 + x.y, s3 = s2 + x.z, s4 = s3 + x.w;
        float incl = s4;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            float y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        const float ex = incl - s4;
        float *gm = gamma + bh * (long long)NT * kTile + (long long)tile * kTile;
        reinterpret_cast<float4 *>(gm)[lane] = make_float4(ex + s1, ex + s2, ex + s3, ex + s4);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) Pb[tile + 1] = acc;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        Pb[0] = 0.0;
        if (bh == 0) {
            if (err != nullptr) *err = 0;
            *queue = 0;
        }
    }
}

__global__ void __launch_bounds__(kScanThreads)
lla_tile_gate_scan_kernel(double *__restrict__ P, int NT)
{
    grid_dependency_wait();    // the tile sums
    grid_launch_dependents();  // the walkers may launch now; they wait for this grid
    __shared__ double wsum[32];
    __shared__ double carry_sh;
    const long long bh = blockIdx.x;
    double *Pb = P + bh * (long long)(NT + 1);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry_sh = 0.0;
    __syncthreads();
    for (int base = 1; base <= NT; base += kScanThreads) {
        const int idx = base + threadIdx.x;
        const double x = idx <= NT ? Pb[idx] : 0.0;
        double incl = x;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            double y = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += y;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            double w = wsum[lane], wi = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                double y = __shfl_up_sync(0xffffffffu, wi, off);
                if (lane >= off) wi += y;
            }
            wsum[lane] = wi - w;  // exclusive prefix of the warp sums
        }
        __syncthreads();
        const double c = carry_sh;
        if (idx <= NT) Pb[idx] = c + wsum[warp] + incl;
        __syncthreads();
        if (threadIdx.x == kScanThreads - 1) carry_sh = c + wsum[warp] + incl;
        __syncthreads();
    }
}

}  // namespace

// Workspace: [P fp64 BH*(NT+1)] [gamma fp32 BH*NT*128] [err word, queue counter]
// [segment totals fp32] [nodes bf16]
static int nseg_full_of(int NT) { return NT > 1 ? (NT - 1) / kSeg : 0; }
static size_t off_gamma(int BH, int NT) { return align_up((size_t)BH * (NT + 1) * 8, 256); }
static size_t off_err(int BH, int NT) { return off_gamma(BH, NT) + align_up((size_t)BH * NT * kTile * 4, 256); }
static size_t off_queue(int BH, int NT) { return off_err(BH, NT) + 128; }
static size_t off_segtot(int BH, int NT) { return off_err(BH, NT) + 256; }
static size_t off_node16(int BH, int NT, int D)
{
    return off_segtot(BH, NT) + align_up((size_t)BH * nseg_full_of(NT) * D * D * 4, 1024);
}

size_t tc_workspace_bytes(int B, int H, int T, int D)
{
    const int BH = B * H, NT = (T + kTile - 1) / kTile;
    return off_node16(BH, NT, D) + align_up((size_t)BH * NT * D * D * 2, 1024);
}

bool tc_supported(int dk, int dv, lla_dtype in_dt)
{
    return in_dt == LLA_BF16 && dk == dv && (dk == 64 || dk == 128);
}

bool tc_mlp_supported(int dk, int dv, lla_dtype in_dt, int L)
{
    return tc_supported(dk, dv, in_dt) && 2 * L <= kMlpHidden;
}

int tc_launches(int T)
{
    const int NT = (T + kTile - 1) / kTile;
    if (NT <= 1) return 3;                          // gate sum, gate scan, read-out
    return 4 + (nseg_full_of(NT) > 0 ? 1 : 0);      // + walkers (+ segment fix-up)
}

static_assert(sizeof(WalkSmem<128>) + 1024 <= 227 * 1024, "walker must fit the shared memory of an SM");
static_assert(sizeof(WalkSmem<64>) + 1024 <= 113 * 1024, "walker (D = 64) must fit two CTAs per SM");
static_assert(sizeof(ConsSmem<128>) + 1024 <= 227 * 1024, "consumer must fit the shared memory of an SM");
static_assert(MlpLayout<128>::kW2 % 1024 == 0, "the MLP's weight parts are whole swizzle atoms");

// Launch configuration, optionally as a programmatic dependent of the
// previous kernel in the stream (it may start before that one finishes and
// synchronises with griddepcontrol.wait).
static cudaLaunchConfig_t launch_cfg(dim3 grid, dim3 block, size_t smem, cudaStream_t st, bool dependent,
                                     cudaLaunchAttribute *attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    attr->id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr->val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cfg;
}

static int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
        n = 148;
    return n;
}

template <int D, typename OutT>
static cudaError_t launch_consumer(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                                   const CUtensorMap &mn, const CUtensorMap &mo, const TcParams &prm,
                                   int grid, cudaStream_t st, bool dependent)
{
    const size_t smem = sizeof(ConsSmem<D>) + 1024;
    cudaError_t e = cudaFuncSetAttribute(lla_readout_consumer_kernel<D, OutT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr;
    cudaLaunchConfig_t cfg = launch_cfg(dim3(grid), dim3(kConsThreads), smem, st, dependent, &attr);
    return cudaLaunchKernelEx(&cfg, lla_readout_consumer_kernel<D, OutT>, mq, mk, mv, mn, mo, prm);
}

static std::atomic<int> g_withhold_first_product{0};

void tc_set_withhold_first_product(int enable) { g_withhold_first_product.store(enable ? 1 : 0); }

template <int D>
static cudaError_t tc_fwd_d(const TcFwdArgs &A)
{
    const int BH = A.B * A.H, NT = (A.T + kTile - 1) / kTile;
    char *ws = (char *)A.workspace;
    TcParams prm;
    prm.g = A.g;
    prm.lam = A.lam;
    prm.out = A.out;
    prm.P = (const double *)ws;
    int *const ws_err = (int *)(ws + off_err(BH, NT));
    prm.err = A.device_error ? (int *)A.device_error : ws_err;
    prm.queue = (int *)(ws + off_queue(BH, NT));
    prm.gamma = (float *)(ws + off_gamma(BH, NT));
    prm.segtot = (float *)(ws + off_segtot(BH, NT));
    prm.node16 = (__nv_bfloat16 *)(ws + off_node16(BH, NT, D));
    prm.T = A.T;
    prm.NT = NT;
    prm.BH = BH;
    prm.L = A.L;
    prm.nseg_full = nseg_full_of(NT);
    prm.W1 = A.W1;
    prm.W2 = A.W2;
    prm.bmlp = A.bmlp;
    prm.mlp = A.W1 != nullptr ? 1 : 0;
    prm.withhold = g_withhold_first_product.load();
    prm.wait_iters = kWaitIters;
    prm.s_wait_iters = prm.withhold ? kWithheldWaitIters : kWaitIters;
    CUtensorMap mq, mk, mv, mn, mo;
    const bool out32 = A.out_dt == LLA_F32;
    if (!make_map_bf16_3d(&mq, A.q, D, A.T, BH, 64, kTile) ||
        !make_map_bf16_3d(&mk, A.k, D, A.T, BH, 64, kTile) ||
        !make_map_bf16_3d(&mv, A.v, D, A.T, BH, 64, kTile) ||
        !make_map_bf16_3d(&mn, prm.node16, D, D, (uint64_t)BH * NT, 64, D) ||
        !(out32 ? make_map_f32_3d(&mo, A.out, D, A.T, BH, 32, kTile)
                : make_map_bf16_3d(&mo, A.out, D, A.T, BH, 64, kTile)))
        return cudaErrorInvalidValue;
    cudaStream_t st = (cudaStream_t)A.stream;
    lla_tile_gate_sum_kernel<<<dim3((NT + 31) / 32, BH), 1024, 0, st>>>(
        A.g, (double *)prm.P, prm.gamma, A.device_error ? nullptr : ws_err, prm.queue, A.T, NT);
    cudaError_t e;
    {
        // programmatic launches: the scan and then the walkers start while the launch
        // before them finishes, and wait for it before reading its results
        cudaLaunchAttribute attr;
        cudaLaunchConfig_t cfg = launch_cfg(dim3(BH), dim3(kScanThreads), 0, st, true, &attr);
        e = cudaLaunchKernelEx(&cfg, lla_tile_gate_scan_kernel, (double *)prm.P, NT);
        if (e != cudaSuccess) return e;
    }
    if (NT > 1) {
        const size_t wsmem = sizeof(WalkSmem<D>) + 1024;
        e = cudaFuncSetAttribute(lla_node_walker_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)wsmem);
        if (e != cudaSuccess) return e;
        const int nseg = (NT - 1 + kSeg - 1) / kSeg;
        cudaLaunchAttribute attr;
        cudaLaunchConfig_t cfg = launch_cfg(dim3(nseg, BH), dim3(kWalkThreads), wsmem, st, true, &attr);
        e = cudaLaunchKernelEx(&cfg, lla_node_walker_kernel<D>, mk, mv, mn, prm);
        if (e != cudaSuccess) return e;
        if (prm.nseg_full > 0) {
            cudaLaunchAttribute attr;
            cudaLaunchConfig_t cfg = launch_cfg(dim3(D * D / kFixElems, prm.nseg_full, BH), dim3(kFixThreads), 0,
                                                st, true, &attr);
            e = cudaLaunchKernelEx(&cfg, lla_node_fixup_kernel<D>, prm);
            if (e != cudaSuccess) return e;
        }
    }
    // persistent read-out: one CTA per SM (or per tile when there are fewer);
    // with nodes to read it starts in the tail of the node launches
    const long long items = (long long)NT * BH;
    const int grid = (int)(items < sm_count() ? items : sm_count());
    e = out32 ? launch_consumer<D, float>(mq, mk, mv, mn, mo, prm, grid, st, NT > 1)
              : launch_consumer<D, __nv_bfloat16>(mq, mk, mv, mn, mo, prm, grid, st, NT > 1);
    if (e != cudaSuccess) return e;
    return cudaPeekAtLastError();
}

cudaError_t tc_fwd(const TcFwdArgs &A)
{
    if (A.dk == 64) return tc_fwd_d<64>(A);
    return tc_fwd_d<128>(A);
}

}  // namespace lla
