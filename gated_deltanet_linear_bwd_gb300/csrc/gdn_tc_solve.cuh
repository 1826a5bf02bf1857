// gdn_tc_solve.cuh -- T = (I + A)^-1 of one chunk on the CUDA cores, and the
// bf16 operand tiles built from it, shared by the prep kernel and the fused
// forward kernel.
//
// A is the chunk's strictly lower-triangular 64 x 64 matrix of the UT
// transform (A = strict_lower(diag(beta) K K^T .* D)), held as A^T rows in
// shared memory: At[j][i] = A[i][j], rows padded to 68 floats.  T is unit
// lower triangular; in 32 x 32 blocks
//   T = [T1 0; T21 T2],  T1 = (I + A11)^-1,  T2 = (I + A22)^-1,  T21 = -T2 A21 T1.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "tc_ptx.cuh"

namespace gdn {
namespace tc {

// Rows I0 .. I0 + N - 1 of Y = T2 X for one column of X (xr = that column): T2
// is unit lower triangular with T2[i][m] = At[32 + m][32 + i].  I0, N multiples of 4.
template <int I0, int N>
__device__ __forceinline__ void t2_times_x(const float (*At)[68], const float *xr, float *y) {
#pragma unroll
    for (int i = 0; i < N; ++i) y[i] = xr[I0 + i];
#pragma unroll
    for (int m = 0; m < I0 + N - 1; ++m) {
        const float xm = xr[m];
        const float4 *tr = reinterpret_cast<const float4 *>(At[32 + m] + 32);
#pragma unroll
        for (int i4 = (m + 1 > I0 ? m + 1 : I0) / 4; i4 < (I0 + N) / 4; ++i4) {
            const float4 a4 = tr[i4];
            if (4 * i4 + 0 > m) y[4 * i4 + 0 - I0] += a4.x * xm;
            if (4 * i4 + 1 > m) y[4 * i4 + 1 - I0] += a4.y * xm;
            if (4 * i4 + 2 > m) y[4 * i4 + 2 - I0] += a4.z * xm;
            if (4 * i4 + 3 > m) y[4 * i4 + 3 - I0] += a4.w * xm;
        }
    }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float *x) {
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        w[e] = *reinterpret_cast<uint32_t *>(&b2);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// T by two warps, thread r = 0..63 of them (lane = r % 32, hi = r / 32); `sync`
// is a barrier over at least those 64 threads.  Warp hi solves T1 (hi = 0) or
// T2 (hi = 1), one column per lane, by right-looking forward substitution
// (column j of A = row j of A^T, read by broadcast); then both form X = A21 T1
// (16 of its 32 rows each) and T21 = -T2 X, with the rows split so that both do
// the same number of products.  Each block goes where the A^T region has gone
// dead:
//   T1 column c -> At[c][0..31]       (A11 part of row c; only warp 0 read it)
//   T2 column m -> At[32 + m][32..63] (A22 part; only warp 1 read it)
//   X column c  -> At[32 + c][0..31]  (upper triangle of A: zero, never read)
// On return the thread holds these pieces of T, as (column, first row, values):
//   hi = 0: (lane, 0, t[0..31]), (lane, 32, y[0..7]), (lane, 56, y[8..15])
//   hi = 1: (32 + lane, 32, t[0..31]), (lane, 40, y[0..15])
// (rows 0-31 of column 32 + lane are zero).  At is clobbered.
template <typename Sync>
__device__ __forceinline__ void solve_unit_lower64(float (*At)[68], int r, float (&t)[32],
                                                   float (&y)[16], Sync sync) {
    const int lane = r & 31, hi = r >> 5, jb = 32 * hi;
#pragma unroll
    for (int i = 0; i < 32; ++i) t[i] = (i == lane) ? 1.f : 0.f;
#pragma unroll
    for (int j = 0; j < 31; ++j) {
        const float tj = t[j];
        const float4 *ar = reinterpret_cast<const float4 *>(At[jb + j] + jb);
#pragma unroll
        for (int i4 = (j + 1) / 4; i4 < 8; ++i4) {
            const float4 a4 = ar[i4];
            if (4 * i4 + 0 > j) t[4 * i4 + 0] -= a4.x * tj;
            if (4 * i4 + 1 > j) t[4 * i4 + 1] -= a4.y * tj;
            if (4 * i4 + 2 > j) t[4 * i4 + 2] -= a4.z * tj;
            if (4 * i4 + 3 > j) t[4 * i4 + 3] -= a4.w * tj;
        }
    }
    __syncwarp();
    {
        float4 *dst = reinterpret_cast<float4 *>(At[jb + lane] + jb);
#pragma unroll
        for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(t[4 * q], t[4 * q + 1], t[4 * q + 2], t[4 * q + 3]);
    }
    sync();
    {
        // X = A21 T1: column `lane`, rows 16 hi .. +15  (A21[m][k] = At[k][32 + m],
        // T1[k][lane] = At[lane][k])
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = 0.f;
        const float4 *t1c = reinterpret_cast<const float4 *>(At[lane]);
#pragma unroll 2
        for (int k4 = 0; k4 < 8; ++k4) {
            const float4 tk = t1c[k4];
            const float tkv[4] = {tk.x, tk.y, tk.z, tk.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float4 *ar = reinterpret_cast<const float4 *>(At[4 * k4 + e] + 32 + 16 * hi);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 a4 = ar[q];
                    x[4 * q + 0] += a4.x * tkv[e];
                    x[4 * q + 1] += a4.y * tkv[e];
                    x[4 * q + 2] += a4.z * tkv[e];
                    x[4 * q + 3] += a4.w * tkv[e];
                }
            }
        }
        float4 *dst = reinterpret_cast<float4 *>(At[32 + lane] + 16 * hi);
#pragma unroll
        for (int q = 0; q < 4; ++q)
            dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    }
    sync();
    // Y = T2 X for column `lane` (T21 = -Y): warp 0 rows 0-7 and 24-31, warp 1 rows 8-23
    {
        float xr[32];
        const float4 *xc = reinterpret_cast<const float4 *>(At[32 + lane]);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 x4 = xc[q];
            xr[4 * q] = x4.x;
            xr[4 * q + 1] = x4.y;
            xr[4 * q + 2] = x4.z;
            xr[4 * q + 3] = x4.w;
        }
        if (hi == 0) {
            t2_times_x<0, 8>(At, xr, y);
            t2_times_x<24, 8>(At, xr, y + 8);
        } else {
            t2_times_x<8, 16>(At, xr, y);
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) y[i] = -y[i];
}

// The W and u operand tiles of the chunk (MN-major B operands, bf16, 64 rows x
// 128 B, 128-byte swizzle): row j holds column j of T scaled by wj (bw) and bj
// (bu).  The thread's pieces are those solve_unit_lower64 left; wo / bo are the
// scales of its own column (32 hi + lane), wl / bl those of column `lane`.
// Every row of both tiles is written in full (rows 0-31 of the columns 32-63
// as zeros).
__device__ __forceinline__ void store_wu_operands(uint8_t *bw, uint8_t *bu, int r,
                                                  const float (&t)[32], const float (&y)[16],
                                                  float wo, float bo, float wl, float bl) {
    const int lane = r & 31, hi = r >> 5, cown = 32 * hi + lane;
    float xs[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = t[8 * q + e] * wo;
        st_row8(bw, cown, 4 * hi + q, xs);
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = t[8 * q + e] * bo;
        st_row8(bu, cown, 4 * hi + q, xs);
    }
    if (hi) {
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            st_row8(bw, cown, q, xs);
            st_row8(bu, cown, q, xs);
        }
    }
#pragma unroll
    for (int p2 = 0; p2 < 2; ++p2) {
        const int piece = hi ? 5 + p2 : 4 + 3 * p2;
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = y[8 * p2 + e] * wl;
        st_row8(bw, lane, piece, xs);
#pragma unroll
        for (int e = 0; e < 8; ++e) xs[e] = y[8 * p2 + e] * bl;
        st_row8(bu, lane, piece, xs);
    }
}

}  // namespace tc
}  // namespace gdn
