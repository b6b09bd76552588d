// Staging of fp32 128 x 128 tiles as bf16 parts for the tensor cores.
//
// An fp32 value x is written as hi = bf16(x) and lo = bf16(x - hi) (two
// parts, about 16 bits) or with a third part (about 24 bits).  The parts go
// to the 128-byte-swizzled layout TMA writes for a [128 rows][128 columns]
// bf16 tile in two 64-column blocks, which serves as a K-major operand (rows
// = M or N, columns = K) or as an MN-major one (rows = K).  The global reads
// are coalesced: 16 lanes cover one 512-byte row, each lane 8 consecutive
// values (two float4), so every warp instruction reads two whole rows.
#pragma once

#include "lla_common.cuh"
#include "sm100.cuh"

namespace lla {

// Rows [0, 128) of src (row stride ld floats); row r scaled by
// all * scale[r] (scale nullptr: all) and rows >= nrows written as 0.  NPARTS = 2 or 3; part p goes
// to dst[p], its second 64-column block BLK bytes after its first (16 KB:
// the two blocks of one tile back to back; 32 KB: the blocks of two parts
// interleaved, the layout of an N = 256 operand).  NTHREADS threads (a
// multiple of 32) call it together; each issues the loads of GROUP rows
// before converting them.
template <int NPARTS, int NTHREADS, int GROUP = 4, uint32_t BLK = 128 * 128>
__device__ __forceinline__ void stage_split_tile(uint8_t *const *dst, const float *src, long long ld,
                                                 const float *scale, float all, int nrows)
{
    constexpr int kPass = (NTHREADS / 32) * 2;  // rows per pass
    constexpr int kGroup = GROUP;               // passes whose loads are issued together
    const int tid = threadIdx.x;
    const int sub = (tid & 31) >> 4;        // which of the warp's two rows
    const int c8 = (tid & 15) * 8;          // first column of this lane
    const int blk = c8 >> 6, chunk = (c8 & 63) >> 3;
    const int r0 = (tid >> 5) * 2 + sub;
#pragma unroll 1
    for (int g = 0; g < 128 / kPass; g += kGroup) {
        float4 ra[kGroup], rb[kGroup];
#pragma unroll
        for (int q = 0; q < kGroup; q++) {
            const int r = r0 + (g + q) * kPass;
            ra[q] = rb[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (r < nrows) {
                const float4 *s4 = reinterpret_cast<const float4 *>(src + r * ld + c8);
                ra[q] = s4[0];
                rb[q] = s4[1];
            }
        }
#pragma unroll
        for (int q = 0; q < kGroup; q++) {
        const int r = r0 + (g + q) * kPass;
        float x[8];
        {
            const float sc = (r < nrows) ? (scale ? all * scale[r] : all) : 0.f;
            const float4 a = ra[q], b = rb[q];
            x[0] = a.x * sc; x[1] = a.y * sc; x[2] = a.z * sc; x[3] = a.w * sc;
            x[4] = b.x * sc; x[5] = b.y * sc; x[6] = b.z * sc; x[7] = b.w * sc;
        }
        uint4 part[NPARTS];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            float a = x[2 * u], b = x[2 * u + 1];
#pragma unroll
            for (int p = 0; p < NPARTS; p++) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
                reinterpret_cast<__nv_bfloat162 *>(&part[p])[u] = h;
                const float2 f = __bfloat1622float2(h);
                a -= f.x;
                b -= f.y;
            }
        }
        const uint32_t off = blk * BLK + sm100::sw128_offset(r, chunk);
#pragma unroll
        for (int p = 0; p < NPARTS; p++) *reinterpret_cast<uint4 *>(dst[p] + off) = part[p];
        }
    }
}

}  // namespace lla

namespace lla {

// A [128][128] fp32 tile in shared memory (64 KB) on its way to global
// memory: piece j (16 bytes, columns 4j..4j+3) of row r is kept at piece
// j ^ (r & 7) of the row, so a thread writing pieces of its own row and a
// warp reading one whole row both touch every bank once.
__device__ __forceinline__ float4 *out_tile_piece(float *tile, int r, int j)
{
    return reinterpret_cast<float4 *>(tile + r * 128 + ((j ^ (r & 7)) << 2));
}

// The staged tile to rows [0, nrows) of dst (row stride 128 floats), whole
// rows per warp: dst = tile, or dst += tile when ADD (the loads of eight
// pieces per thread are issued before their stores).  NTHREADS threads call
// it together after a barrier that follows the staging.
template <int NTHREADS, bool ADD>
__device__ __forceinline__ void out_tile_store(float *dst, float *tile, int nrows)
{
    constexpr int kPer = 128 * 32 / NTHREADS;  // pieces per thread
    static_assert(kPer % 8 == 0, "whole groups of eight pieces");
#pragma unroll 1
    for (int g0 = 0; g0 < kPer; g0 += 8) {
        float4 o[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int e = threadIdx.x + (g0 + u) * NTHREADS;
            const int r = e >> 5, j = e & 31;
            o[u] = *out_tile_piece(tile, r, j);
            if (ADD && r < nrows) {
                const float4 x = reinterpret_cast<const float4 *>(dst + (long long)r * 128)[j];
                o[u].x += x.x;
                o[u].y += x.y;
                o[u].z += x.z;
                o[u].w += x.w;
            }
        }
#pragma unroll
        for (int u = 0; u < 8; u++) {
            const int e = threadIdx.x + (g0 + u) * NTHREADS;
            const int r = e >> 5, j = e & 31;
            if (r < nrows) reinterpret_cast<float4 *>(dst + (long long)r * 128)[j] = o[u];
        }
    }
}

}  // namespace lla
