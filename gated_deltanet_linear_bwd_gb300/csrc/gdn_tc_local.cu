// gdn_tc_local.cu -- tensor-core chunk-local gradients for bf16 q/k/v with
// K = V = 128 (no q/k L2 normalisation), one (chunk, head) per CTA.
//
// Inputs per chunk: q, k, v, dO (TMA); the workspace's bf16 chunk tiles of
// dU^T, W^T, the chunk start state H0^T and the gradient at its end dHL^T
// (TMA) and u^T; T, gam and beta.  With D = exp(gam_r - gam_s),
// e = exp(gam), f = exp(gam_L - gam), and T = (I + A)^-1 recomputed:
//   U    = u - W H0   (T itself is kept by the recompute's prep kernel)
//   dS   = scale (dO U^T) .* lower_incl .* D
//   dW   = -dU H0^T,  dYw = T^T dW,  dYu = T^T dU
//   dT   = dU (diag(beta) V)^T + dW (diag(beta e) K)^T,  dA = -T^T dT T^T
//   G    = dA .* D .* beta_r (strict lower),  Gs = G + G^T
//   dQ   = scale diag(e) dO H0^T + dS K
//   dK   = dS^T Q + diag(f) U dHL^T + diag(beta e) dYw + Gs K
//   dV   = diag(beta) dYu
//   dbeta_r = <dYu_r, v_r> + e_r <dYw_r, k_r> + sum_s dA_rs (K K^T)_rs D_rs
//   dgam from every exp factor, dg = reverse cumsum of dgam.
// Products with a feature-dimension output run with the feature on the MMA's
// M side (128 lanes); 64 x 64 products put the chunk rows on lanes 0-63 and
// let lanes 64-127 compute throwaway rows.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_ptx.cuh"

namespace gdn {
namespace tc {

namespace {
constexpr int kD = 128;
constexpr int kTile = 8192;
constexpr uint32_t kKK = idesc_bf16(128, 64, false, false);   // A K-major, B K-major
constexpr uint32_t kMK = idesc_bf16(128, 64, true, false);    // A MN-major, B K-major
constexpr uint32_t kKM = idesc_bf16(128, 64, false, true);    // A K-major, B MN-major
constexpr uint32_t kMM = idesc_bf16(128, 64, true, true);     // A MN-major, B MN-major
constexpr uint32_t kKK128 = idesc_bf16(128, 128, false, false);   // N = 128, both K-major

struct LocalSmem {
    uint8_t qk[4 * kTile];     // [dk half][Q rows 0-63, K rows 64-127][128 B]
    uint8_t v[2 * kTile];      // [dv half][64 rows][128 B]
    // dO, du, w, h0T, ds, tt, gs (104 KB, contiguous) stage dq, dk, dv after wave 3
    uint8_t dO[2 * kTile];
    uint8_t du[2 * kTile];     // dU^T: [128 rows v][64 chunk rows]
    uint8_t w[2 * kTile];      // W^T: [128 rows k][64 chunk rows]
    uint8_t h0T[4 * kTile];    // H0^T: [k half][128 rows v][128 B]; after wave 1: uT, dwT
    uint8_t ds[kTile];         // dS rows r
    uint8_t tt[kTile];         // row r = column r of T
    uint8_t gs[kTile];         // Gs rows r
    float xm[64][64];          // dHL^T k half 0 until wave 2 is done; then X = dT T^T
    float fd[64 * 68];         // dHL^T k half 1 (first 16 KB) until wave 2 is done; then
                               // dT^T (stride 68), then dA row-major (stride 65)
    float tf[64][64];          // T, row-major
    float tft[64][64];         // T^T
    float gam[64], bet[64], ee[64], ff[64];
    float red[8][32];
    float zrow[2][64], zprow[2][64], dbA[2][64];
    float zcol[64], rowA[64], yw[64], yu[64], zpp[64];
    float hdot[16];            // [0..3]: per-warp parts of <dHL, H0>; [8..15]: block_sum scratch
    uint64_t tma_bar, mma_bar;
    uint32_t tmem_base;
};

// 256 threads; thread t contributes a[j] to entry 32 * (t / 128) + j.
// dst[i] (+)= the sum of all contributions to entry i (i < 64).  Warp
// butterfly (lane l ends with entry l of its warp), then the four warps of
// each half combine through shared memory.
__device__ __forceinline__ void reduce32(float (&a)[32], float *dst, float (&red)[8][32],
                                         bool accumulate) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#define GDN_BFLY(MASK, HALF)                                                  \
    {                                                                         \
        const bool up = (lane & (MASK)) != 0;                                 \
        _Pragma("unroll") for (int i = 0; i < (HALF); ++i) {                  \
            const float send = up ? a[i] : a[i + (HALF)];                     \
            const float keep = up ? a[i + (HALF)] : a[i];                     \
            a[i] = keep + __shfl_xor_sync(0xffffffffu, send, (MASK));         \
        }                                                                     \
    }
    GDN_BFLY(16, 16)
    GDN_BFLY(8, 8)
    GDN_BFLY(4, 4)
    GDN_BFLY(2, 2)
    GDN_BFLY(1, 1)
#undef GDN_BFLY
    red[warp][lane] = a[0];
    __syncthreads();
    if (threadIdx.x < 64) {
        const int i = threadIdx.x, w0 = 4 * (i >> 5), l = i & 31;
        const float sum = red[w0][l] + red[w0 + 1][l] + red[w0 + 2][l] + red[w0 + 3][l];
        dst[i] = accumulate ? dst[i] + sum : sum;
    }
    __syncthreads();
}

__device__ __forceinline__ float block_sum(float x, float *scratch8) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0) scratch8[threadIdx.x >> 5] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) s += scratch8[w];
    __syncthreads();
    return s;
}

struct TcLocalArgs {
    const float *ws_gam, *tmat;
    const __nv_bfloat16 *ws_u;
    void *dq, *dk, *dv;
    float *dg, *dbeta;
};

template <typename F>
cudaError_t set_smem(F kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
}  // namespace

// 256 threads.  Feature-major results: thread t reads TMEM lane v = t % 128
// (feature v) and the chunk-row half hs = t / 128.  Row-major 64 x 64
// results sit on lanes 0-63 (warps 0, 1, 4, 5: row r = v, column half hs);
// lanes 64-127 of the [Q; K] K^T product hold K K^T (warps 2, 3, 6, 7).
template <typename TG>
__global__ void __launch_bounds__(256, 1)
tc_local_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_du, const __grid_constant__ CUtensorMap tm_w,
                const __grid_constant__ CUtensorMap tm_hc, const __grid_constant__ CUtensorMap tm_dhc,
                Geo g, TcLocalArgs a) {
    extern __shared__ uint8_t smem_raw[];
    LocalSmem &s = *reinterpret_cast<LocalSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, h = blockIdx.y, H = g.H, ci = blockIdx.x;
    const int v = tid & 127, hs = tid >> 7, c0 = 32 * hs;
    ChunkRef cr;
    if (!chunk_ref(g, ci, cr)) return;
    const int L = cr.len;
    const long long bos = cr.bos;
    const float scale = g.scale;
    uint8_t *uT = s.h0T, *dwT = s.h0T + 2 * kTile;   // after wave 1

    if (tid == 0) {
        mbar_init(&s.tma_bar, 1);
        mbar_init(&s.mma_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = s.tmem_base;
    const uint32_t t_u = tb, t_p = tb + 64, t_dw = tb + 128, t_q1 = tb + 192, t_tu = tb + 256,
                   t_qh = tb + 320, t_hd = tb + 384;
    const uint32_t t_dp = tb, t_tw = tb + 128, t_dkh = tb + 448;
    const uint32_t t_q2 = tb, t_dk = tb + 128, t_yw = tb + 320, t_yu = tb + 384;
    if (tid == 0) {
        const int tok0 = (int)bos;
        mbar_arrive_expect_tx(&s.tma_bar, 20 * kTile);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(s.qk + half * 2 * kTile, &tm_q, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.qk + half * 2 * kTile + kTile, &tm_k, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.v + half * kTile, &tm_v, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.dO + half * kTile, &tm_do, &s.tma_bar, half * 64, h, tok0);
        }
        const int trow = (int)(((long long)ci * H + h) * kD);
        tma_load_2d(s.du, &tm_du, &s.tma_bar, 0, trow);
        tma_load_2d(s.w, &tm_w, &s.tma_bar, 0, trow);
        // bf16 H0^T and dHL^T tiles, [k half][128 rows v][64]
        tma_load_2d(s.h0T, &tm_hc, &s.tma_bar, 0, 2 * trow);
        tma_load_2d(s.h0T + 2 * kTile, &tm_hc, &s.tma_bar, 0, 2 * trow + kD);
        tma_load_2d(s.xm, &tm_dhc, &s.tma_bar, 0, 2 * trow);
        tma_load_2d(s.fd, &tm_dhc, &s.tma_bar, 0, 2 * trow + kD);
    }
    if (tid < 64) {
        s.gam[tid] = tid < L ? a.ws_gam[(bos + tid) * H + h] : 0.f;
        s.bet[tid] = tid < L ? g.beta[(bos + tid) * H + h] : 0.f;
    }
    __syncthreads();
    if (tid < 64) {
        s.ee[tid] = tid < L ? __expf(s.gam[tid]) : 0.f;
        s.ff[tid] = tid < L ? __expf(s.gam[L - 1] - s.gam[tid]) : 0.f;
    }
    int mma_n = 0;
    bool tma_pending = true;
    bool ok = mbar_wait(&s.tma_bar, 0, g.spin_limit, g.status);
    if (__syncthreads_or(!ok)) goto bail;
    tma_pending = false;

    // ---------------- wave 1
    ++mma_n;
    if (tid == 0) {
        tc_fence_after();
        const uint32_t qk = smem_u32(s.qk), h0 = smem_u32(s.h0T), w = smem_u32(s.w),
                       du = smem_u32(s.du), vv = smem_u32(s.v), dO = smem_u32(s.dO),
                       dl0 = smem_u32(s.xm), dl1 = smem_u32(s.fd);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t hh = kk >> 2, sub = (kk & 3) * 32;
            const uint64_t aH = desc_sw128(h0 + hh * 2 * kTile + sub, 16, 1024);
            const uint64_t aQK = desc_sw128(qk + hh * 2 * kTile + sub, 16, 1024);
            const uint64_t bK = desc_sw128(qk + hh * 2 * kTile + kTile + sub, 16, 1024);
            mma_bf16(t_u, aH, desc_sw128(w + kk * 2048, 2 * kTile, 1024), kKM, kk > 0);   // W^T, MN-major
            mma_bf16(t_p, aQK, bK, kKK, kk > 0);
            mma_bf16(t_qh, aH, aQK, kKK, kk > 0);
            // dU V^T: A = dU from the dU^T tile (MN-major; lanes 64-127 alias rows 0-63)
            mma_bf16(t_tu, desc_sw128(du + kk * 2048, 0, 1024),
                     desc_sw128(vv + hh * kTile + sub, 16, 1024), kMK, kk > 0);
            const uint64_t aHm = desc_sw128(h0 + kk * 2048, 2 * kTile, 1024);   // H0, MN-major
            mma_bf16(t_dw, aHm, desc_sw128(du + kk * 2048, 2 * kTile, 1024), kMM, kk > 0);
            mma_bf16(t_q1, aHm, desc_sw128(dO + hh * kTile + sub, 16, 1024), kMK, kk > 0);
            // dHL^T H0 (128 x 128): its trace is <dHL, H0>
            mma_bf16(t_hd, desc_sw128((hh ? dl1 : dl0) + sub, 16, 1024), aH, kKK128, kk > 0);
        }
        mma_commit(&s.mma_bar);
    }
    ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
    if (__syncthreads_or(!ok)) goto bail;
    tc_fence_after();
    {
        // U^T (row v, chunk rows c0..c0+31) into uT; -(H0 dU^T) (row k = v) into dwT;
        // partial sums of dO[r][v] (Q H0)[r][v] over v for rowA
        // u^T tile row v, chunk rows c0 .. c0+31: 64 contiguous bytes
        const uint4 *ug = reinterpret_cast<const uint4 *>(
            a.ws_u + (((long long)ci * H + h) * kD + v) * 64 + c0);
        float x[32], y[32];
        tmem_ld32(tmem_addr(t_u, warp, c0), x);
        tmem_ld32(tmem_addr(t_qh, warp, c0), y);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 raw = ug[q];
            const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int jj = 8 * q + e, c = c0 + jj;
                x[jj] = c < L ? __bfloat162float(bv[e]) - x[jj] : 0.f;
                y[jj] = c < L ? ld_bf16(s.dO + (v >> 6) * kTile, c, v & 63) * y[jj] : 0.f;
            }
        }
        st_row32(uT, v, c0, x);
        tmem_ld32(tmem_addr(t_dw, warp, c0), x);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) x[jj] = (c0 + jj) < L ? -x[jj] : 0.f;
        st_row32(dwT, v, c0, x);
        if (hs == 0) {
            // lane v's diagonal entry of dHL^T H0 sits in column v of t_hd
            const int lane = tid & 31;
            tmem_ld32(tmem_addr(t_hd, warp, 32 * warp), x);
            float d = 0.f;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) d = jj == lane ? x[jj] : d;
            for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            if (lane == 0) s.hdot[warp] = d;
        }
        tc_fence_before();
        fence_proxy_async();
        reduce32(y, s.rowA, s.red, false);    // its barriers publish uT, dwT and hdot
    }

    // ---------------- wave 2: dP = dO U^T, dW K^T (lanes 0-63); T from the recompute
    ++mma_n;
    if (tid == 0) {
        tc_fence_after();
        const uint32_t qk = smem_u32(s.qk), dO = smem_u32(s.dO), uTa = smem_u32(uT),
                       dwa = smem_u32(dwT), dl0 = smem_u32(s.xm), dl1 = smem_u32(s.fd);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t hh = kk >> 2, sub = (kk & 3) * 32;
            mma_bf16(t_dp, desc_sw128(dO + hh * kTile + sub, 16, 1024),
                     desc_sw128(uTa + kk * 2048, kTile, 1024), kKM, kk > 0);
            mma_bf16(t_tw, desc_sw128(dwa + kk * 2048, 0, 1024),
                     desc_sw128(qk + hh * 2 * kTile + kTile + sub, 16, 1024), kMK, kk > 0);
            // dHL U^T: A = dHL from the dHL^T tiles (MN-major, k halves dl1 - dl0 apart)
            mma_bf16(t_dkh, desc_sw128(dl0 + kk * 2048, dl1 - dl0, 1024),
                     desc_sw128(uTa + kk * 2048, kTile, 1024), kMM, kk > 0);
        }
        mma_commit(&s.mma_bar);
    }
    if (tid < 64) {
        // column r of T (kept by the prep kernel of the recompute)
        const int r = tid;
        const float4 *src = reinterpret_cast<const float4 *>(
            a.tmat + (((long long)ci * H + h) * 64 + r) * 64);
        float col[64];
#pragma unroll
        for (int i4 = 0; i4 < 16; ++i4) {
            const float4 t4 = r < L ? src[i4] : make_float4(0.f, 0.f, 0.f, 0.f);
            col[4 * i4] = t4.x;
            col[4 * i4 + 1] = t4.y;
            col[4 * i4 + 2] = t4.z;
            col[4 * i4 + 3] = t4.w;
            reinterpret_cast<float4 *>(s.tft[r])[i4] = t4;
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) s.tf[i][r] = col[i];
        st_row64(s.tt, r, col);
    }
    ok = mbar_wait(&s.mma_bar, 1, g.spin_limit, g.status);
    if (__syncthreads_or(!ok)) goto bail;
    tc_fence_after();
    {
        float z[32];
        if (v < 64) {
            // dS row r = v (columns c0..c0+31), z = dS .* Q K^T, and dT^T (columns r)
            const int r = v;
            const float gr = s.gam[r];
            float dp[32], qk[32];
            tmem_ld32(tmem_addr(t_dp, warp, c0), dp);
            tmem_ld32(tmem_addr(t_p, warp, c0), qk);
            float zr = 0.f;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = c0 + jj;
                const float ds = (c <= r && r < L) ? scale * dp[jj] * __expf(gr - s.gam[c]) : 0.f;
                const float zz = ds * qk[jj];
                zr += zz;
                z[jj] = -zz;
                dp[jj] = ds;
            }
            st_row32(s.ds, r, c0, dp);
            s.zrow[hs][r] = zr;
            tmem_ld32(tmem_addr(t_tu, warp, c0), dp);
            tmem_ld32(tmem_addr(t_tw, warp, c0), qk);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = c0 + jj;
                s.fd[c * 68 + r] = (c < r && r < L) ? s.bet[c] * (dp[jj] + s.ee[c] * qk[jj]) : 0.f;
            }
        } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) z[jj] = 0.f;
        }
        reduce32(z, s.zcol, s.red, false);
    }
    // ---------------- X = dT T^T, then dA = -T^T X (strict lower), fp32, 4 x 4 per thread
    {
        const int rb = 4 * (tid >> 4), sb = 4 * (tid & 15);
        float acc[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j2 = 0; j2 < 4; ++j2) acc[i][j2] = 0.f;
#pragma unroll 4
        for (int b = 0; b < 64; ++b) {
            const float4 d4 = *reinterpret_cast<const float4 *>(&s.fd[b * 68 + rb]);
            const float4 t4 = *reinterpret_cast<const float4 *>(&s.tft[b][sb]);
            const float dv4[4] = {d4.x, d4.y, d4.z, d4.w}, tv4[4] = {t4.x, t4.y, t4.z, t4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j2 = 0; j2 < 4; ++j2) acc[i][j2] += dv4[i] * tv4[j2];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
            *reinterpret_cast<float4 *>(&s.xm[rb + i][sb]) =
                make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
        __syncthreads();
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j2 = 0; j2 < 4; ++j2) acc[i][j2] = 0.f;
#pragma unroll 4
        for (int q = 0; q < 64; ++q) {
            const float4 t4 = *reinterpret_cast<const float4 *>(&s.tf[q][rb]);
            const float4 x4 = *reinterpret_cast<const float4 *>(&s.xm[q][sb]);
            const float tv4[4] = {t4.x, t4.y, t4.z, t4.w}, xv4[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j2 = 0; j2 < 4; ++j2) acc[i][j2] += tv4[i] * xv4[j2];
        }
        __syncthreads();                       // every read of dT^T is done: fd becomes dA
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j2 = 0; j2 < 4; ++j2) {
                const int r = rb + i, c = sb + j2;
                s.fd[r * 65 + c] = (c < r && r < L) ? -acc[i][j2] : 0.f;
            }
        __syncthreads();
    }
    {
        // Gs = G + G^T, z' = G .* K K^T and the dA part of dbeta: row r = v - 64
        float zp[32];
        if (v >= 64) {
            const int r = v - 64;
            const float gr = s.gam[r], br = s.bet[r];
            float kk[32], gsv[32];
            tmem_ld32(tmem_addr(t_p, warp, c0), kk);
            float zpr = 0.f, dba = 0.f;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = c0 + jj;
                const bool low = c < r && r < L, up = c > r && c < L;
                const float d_rc = low ? __expf(gr - s.gam[c]) : 0.f;
                const float da_rc = s.fd[r * 65 + c];
                const float g_rc = low ? da_rc * br * d_rc : 0.f;
                const float g_cr = up ? s.fd[c * 65 + r] * s.bet[c] * __expf(s.gam[c] - gr) : 0.f;
                gsv[jj] = g_rc + g_cr;
                const float zz = g_rc * kk[jj];
                zpr += zz;
                zp[jj] = -zz;
                dba += low ? da_rc * kk[jj] * d_rc : 0.f;
            }
            st_row32(s.gs, r, c0, gsv);
            s.zprow[hs][r] = zpr;
            s.dbA[hs][r] = dba;
        } else {
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) zp[jj] = 0.f;
        }
        tc_fence_before();
        fence_proxy_async();
        reduce32(zp, s.zcol, s.red, true);
    }

    // ---------------- wave 3
    ++mma_n;
    if (tid == 0) {
        tc_fence_after();
        const uint32_t qk = smem_u32(s.qk), ds = smem_u32(s.ds), gs = smem_u32(s.gs),
                       tt = smem_u32(s.tt), dwa = smem_u32(dwT), du = smem_u32(s.du);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t aK = desc_sw128(qk + kTile + kk * 2048, 2 * kTile, 1024);   // K, MN-major
            const uint64_t aQ = desc_sw128(qk + kk * 2048, 2 * kTile, 1024);           // Q, MN-major
            mma_bf16(t_q2, aK, desc_sw128(ds + kk * 32, 16, 1024), kMK, kk > 0);
            mma_bf16(t_dk, aQ, desc_sw128(ds + kk * 2048, kTile, 1024), kMM, kk > 0);
            mma_bf16(t_dk, aK, desc_sw128(gs + kk * 32, 16, 1024), kMK, 1);
            mma_bf16(t_yw, desc_sw128(dwa + kk * 32, 16, 1024), desc_sw128(tt + kk * 32, 16, 1024),
                     kKK, kk > 0);
            mma_bf16(t_yu, desc_sw128(du + kk * 32, 16, 1024), desc_sw128(tt + kk * 32, 16, 1024),
                     kKK, kk > 0);   // dU^T, K-major
        }
        mma_commit(&s.mma_bar);
    }
    ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
    if (__syncthreads_or(!ok)) goto bail;
    tc_fence_after();
    {
        // feature v (= k for dq, dk; = v for dv), chunk rows c0 .. c0+31, staged as
        // row-major [3][64 rows][128] in the dead tiles, then written out in 16-byte rows
        TG *stg = reinterpret_cast<TG *>(s.dO);
        const uint8_t *krow = s.qk + (v >> 6) * 2 * kTile + kTile;
        const uint8_t *vrow = s.v + (v >> 6) * kTile;
        float x[32], y[32], pz[32], pw[32];
        tmem_ld32(tmem_addr(t_q1, warp, c0), x);
        tmem_ld32(tmem_addr(t_q2, warp, c0), y);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int c = c0 + jj;
            from_f(stg + c * kD + v, scale * s.ee[c] * x[jj] + y[jj]);
        }
        tmem_ld32(tmem_addr(t_dk, warp, c0), x);
        tmem_ld32(tmem_addr(t_dkh, warp, c0), y);
        tmem_ld32(tmem_addr(t_yw, warp, c0), pw);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int c = c0 + jj;
            const float kv = c < L ? ld_bf16(krow, c, v & 63) : 0.f;
            const float dkh = s.ff[c] * y[jj];
            from_f(stg + (64 + c) * kD + v, x[jj] + dkh + s.bet[c] * s.ee[c] * pw[jj]);
            pz[jj] = dkh * kv;
            pw[jj] *= kv;
        }
        reduce32(pz, s.zpp, s.red, false);
        reduce32(pw, s.yw, s.red, false);
        tmem_ld32(tmem_addr(t_yu, warp, c0), y);
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
            const int c = c0 + jj;
            from_f(stg + (128 + c) * kD + v, s.bet[c] * y[jj]);
            pz[jj] = c < L ? y[jj] * ld_bf16(vrow, c, v & 63) : 0.f;
        }
        reduce32(pz, s.yu, s.red, false);     // its barriers also publish the staged rows
        constexpr int kVec = 16 / sizeof(TG), kPerRow = kD / kVec;
#pragma unroll
        for (int o = 0; o < 3; ++o) {
            TG *out = (TG *)(o == 0 ? a.dq : o == 1 ? a.dk : a.dv) + (bos * H + h) * (long long)kD;
            for (int i = tid; i < L * kPerRow; i += 256) {
                const int r = i / kPerRow, q = i % kPerRow;
                *reinterpret_cast<uint4 *>(out + (long long)r * H * kD + q * kVec) =
                    *reinterpret_cast<const uint4 *>(stg + (o * 64 + r) * kD + q * kVec);
            }
        }
    }
    {
        const float zsum = block_sum(tid < 64 ? s.zpp[tid] : 0.f, s.hdot + 8);
        if (tid < 64) {
            const int r = tid;
            float dgam = 0.f;
            if (r < L) {
                dgam = s.zrow[0][r] + s.zrow[1][r] + s.zprow[0][r] + s.zprow[1][r] + s.zcol[r] +
                       s.bet[r] * s.ee[r] * s.yw[r] + scale * s.ee[r] * s.rowA[r] - s.zpp[r];
                if (r == L - 1)
                    dgam += zsum + s.ee[r] * (s.hdot[0] + s.hdot[1] + s.hdot[2] + s.hdot[3]);
                a.dbeta[(bos + r) * H + h] = s.yu[r] + s.ee[r] * s.yw[r] + s.dbA[0][r] + s.dbA[1][r];
            }
            s.red[r >> 5][r & 31] = dgam;
        }
        __syncthreads();
        if (tid < 64) {
            // dg = reverse cumsum of dgam within the chunk (warp scans over 2 x 32)
            const int lane = tid & 31, w = tid >> 5;
            float x = s.red[1 - w][31 - lane];          // reversed order: position p = 63 - r
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float yv = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += yv;
            }
            s.red[2 + w][lane] = x;
        }
        __syncthreads();
        if (tid < 64) {
            const int pidx = tid;                        // position in reversed order
            const int r = 63 - pidx;
            float x = s.red[2 + (pidx >> 5)][pidx & 31];
            if (pidx >= 32) x += s.red[2][31];
            if (r < L) a.dg[(bos + r) * H + h] = x;
        }
    }
    goto done;
bail:
    if (tid == 0) {
        if (tma_pending) mbar_drain(&s.tma_bar, 0);
        if (mma_n > 0) mbar_drain(&s.mma_bar, (mma_n - 1) & 1);
    }
done:
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t local_grads(const Plan &p, cudaStream_t s) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    const Geo &g = p.g;
    const long long tokens = (long long)g.B * g.T;
    CUtensorMap mq, mk, mv, mdo, mdu, mw, mhc, mdhc;
    if ((e = make_map(&mq, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mk, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mv, g.v, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mdo, p.d_o, tokens, g.H)) != cudaSuccess) return e;
    const long long tile_rows = (long long)p.max_chunks * g.H * kD;
    if ((e = make_map_tiles(&mdu, p.ws.du, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mw, p.ws.w, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mhc, p.ws.hc, 2 * tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mdhc, p.ws.dhc, 2 * tile_rows)) != cudaSuccess) return e;
    TcLocalArgs a{};
    a.ws_gam = p.ws.gam;
    a.tmat = p.ws.tmat;
    a.ws_u = (const __nv_bfloat16 *)p.ws.u;
    a.dq = p.dq;
    a.dk = p.dk;
    a.dv = p.dv;
    a.dg = p.dg;
    a.dbeta = p.dbeta;
    const size_t smem = sizeof(LocalSmem) + 1024;
    const dim3 grid(p.max_chunks, g.H);
    prof_before("tc_local_grad", s);
    if (p.grad_dtype == GDN_BF16) {
        if ((e = set_smem(tc_local_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        tc_local_kernel<__nv_bfloat16><<<grid, 256, smem, s>>>(mq, mk, mv, mdo, mdu, mw, mhc, mdhc, g, a);
    } else {
        if ((e = set_smem(tc_local_kernel<float>, smem)) != cudaSuccess) return e;
        tc_local_kernel<float><<<grid, 256, smem, s>>>(mq, mk, mv, mdo, mdu, mw, mhc, mdhc, g, a);
    }
    prof_after(s);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace gdn
