// gdn_tc_local.cu -- tensor-core chunk-local gradients for bf16 q/k/v with
// K = V = 128 (no q/k L2 normalisation), one (chunk, head) per CTA.
//
// Inputs per chunk: q, k, v, dO (TMA), dU and W (workspace, TMA), u (from
// the workspace), the chunk start state H0 and the gradient at its end dHL
// (workspace, fp32), gam and beta.  With D = exp(gam_r - gam_s),
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

struct LocalSmem {
    uint8_t qk[4 * kTile];     // [dk half][Q rows 0-63, K rows 64-127][128 B]
    uint8_t v[2 * kTile];      // [dv half][64 rows][128 B]
    uint8_t dO[2 * kTile];     // after wave 2: dHL^T half 1
    uint8_t du[2 * kTile];
    uint8_t w[2 * kTile];      // after wave 1: dHL^T half 0
    uint8_t h0T[4 * kTile];    // [k half][128 rows v][128 B]; after wave 1: uT, dwT
    uint8_t ds[kTile];         // dS rows r
    uint8_t tt[kTile];         // row r = column r of T
    uint8_t gs[kTile];         // Gs rows r
    float fa[64][64];          // X = dT T^T
    float tf[64][65];          // T
    float fd[64][65];          // dT, then dA
    float gam[64], bet[64], ee[64], ff[64];
    float red[4][64];
    float zrow[64], zprow[64], zcol[64], rowA[64], dbA[64], yw[64], yu[64], zpp[64];
    float hdot[8];             // [0]: <dHL, H0>; [4..7]: block_sum scratch
    uint64_t tma_bar, mma_bar;
    uint32_t tmem_base;
};

// Sums 64 per-thread values over all 128 threads: dst[i] (+)= sum_t a_t[i].
// Warp butterfly (each lane ends with the sums of entries 2*lane and
// 2*lane + 1), then the four warps combine through shared memory.
__device__ __forceinline__ void reduce64(float (&a)[64], float *dst, float (&red)[4][64],
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
    GDN_BFLY(16, 32)
    GDN_BFLY(8, 16)
    GDN_BFLY(4, 8)
    GDN_BFLY(2, 4)
    GDN_BFLY(1, 2)
#undef GDN_BFLY
    red[warp][2 * lane] = a[0];
    red[warp][2 * lane + 1] = a[1];
    __syncthreads();
    if (threadIdx.x < 64) {
        const int i = threadIdx.x;
        const float sum = red[0][i] + red[1][i] + red[2][i] + red[3][i];
        dst[i] = accumulate ? dst[i] + sum : sum;
    }
    __syncthreads();
}

__device__ __forceinline__ float block_sum(float x, float *scratch4) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0) scratch4[threadIdx.x >> 5] = x;
    __syncthreads();
    const float s = scratch4[0] + scratch4[1] + scratch4[2] + scratch4[3];
    __syncthreads();
    return s;
}

struct TcLocalArgs {
    const float *ws_gam, *hc, *dhc, *tmat;
    const __nv_bfloat16 *ws_u;
    void *dq, *dk, *dv;
    float *dg, *dbeta;
};

template <typename F>
cudaError_t set_smem(F kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
}  // namespace

template <typename TG>
__global__ void __launch_bounds__(128, 1)
tc_local_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                const __grid_constant__ CUtensorMap tm_du, const __grid_constant__ CUtensorMap tm_w,
                Geo g, TcLocalArgs a) {
    extern __shared__ uint8_t smem_raw[];
    LocalSmem &s = *reinterpret_cast<LocalSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, h = blockIdx.y, H = g.H, ci = blockIdx.x;
    ChunkRef cr;
    if (!chunk_ref(g, ci, cr)) return;
    const int L = cr.len, r = tid & 63;
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
                   t_qh = tb + 320;
    const uint32_t t_dp = tb, t_tw = tb + 128;
    const uint32_t t_q2 = tb, t_dk = tb + 128, t_dkh = tb + 256, t_yw = tb + 320, t_yu = tb + 384;
    if (tid == 0) {
        const int tok0 = (int)bos;
        mbar_arrive_expect_tx(&s.tma_bar, 12 * kTile);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(s.qk + half * 2 * kTile, &tm_q, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.qk + half * 2 * kTile + kTile, &tm_k, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.v + half * kTile, &tm_v, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.dO + half * kTile, &tm_do, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.du + half * kTile, &tm_du, &s.tma_bar, half * 64, h, tok0);
            tma_load_3d(s.w + half * kTile, &tm_w, &s.tma_bar, half * 64, h, tok0);
        }
    }
    if (tid < 64) {
        s.gam[r] = r < L ? a.ws_gam[(bos + r) * H + h] : 0.f;
        s.bet[r] = r < L ? g.beta[(bos + r) * H + h] : 0.f;
    }
    const float *H0 = a.hc + ((long long)ci * H + h) * kD * kD;
    const float *dHL = a.dhc + ((long long)ci * H + h) * kD * kD;
    {
        // H0 column tid -> row tid of H0^T (bf16, two k halves)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float x[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) x[i] = H0[(half * 64 + i) * kD + tid];
            st_row64(s.h0T + half * 2 * kTile, tid, x);
        }
    }
    fence_proxy_async();
    __syncthreads();
    if (tid < 64) {
        s.ee[r] = r < L ? __expf(s.gam[r]) : 0.f;
        s.ff[r] = r < L ? __expf(s.gam[L - 1] - s.gam[r]) : 0.f;
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
                       du = smem_u32(s.du), v = smem_u32(s.v), dO = smem_u32(s.dO);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t hs = kk >> 2, sub = (kk & 3) * 32;
            const uint64_t aH = desc_sw128(h0 + hs * 2 * kTile + sub, 16, 1024);
            const uint64_t aQK = desc_sw128(qk + hs * 2 * kTile + sub, 16, 1024);
            const uint64_t bK = desc_sw128(qk + hs * 2 * kTile + kTile + sub, 16, 1024);
            const uint64_t bQ = aQK;
            mma_bf16(t_u, aH, desc_sw128(w + hs * kTile + sub, 16, 1024), kKK, kk > 0);
            mma_bf16(t_p, aQK, bK, kKK, kk > 0);
            mma_bf16(t_qh, aH, bQ, kKK, kk > 0);
            mma_bf16(t_tu, desc_sw128(du + hs * kTile + sub, 16, 1024),
                     desc_sw128(v + hs * kTile + sub, 16, 1024), kKK, kk > 0);
            const uint64_t aHm = desc_sw128(h0 + kk * 2048, 2 * kTile, 1024);   // H0, MN-major
            mma_bf16(t_dw, aHm, desc_sw128(du + hs * kTile + sub, 16, 1024), kMK, kk > 0);
            mma_bf16(t_q1, aHm, desc_sw128(dO + hs * kTile + sub, 16, 1024), kMK, kk > 0);
        }
        mma_commit(&s.mma_bar);
    }
    ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
    if (__syncthreads_or(!ok)) goto bail;
    tc_fence_after();
    {
        // U^T row (thread = v) into uT; partials of sum_v dO[r][v] (Q H0)[r][v]
        const __nv_bfloat16 *ug = a.ws_u + (bos * H + h) * (long long)kD + tid;
        float p[64];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float acc[32], qh[32];
            tmem_ld32(tmem_addr(t_u, warp, q * 32), acc);
            tmem_ld32(tmem_addr(t_qh, warp, q * 32), qh);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = q * 32 + jj;
                acc[jj] = c < L ? __bfloat162float(ug[(long long)c * H * kD]) - acc[jj] : 0.f;
                p[c] = c < L ? ld_bf16(s.dO + (tid >> 6) * kTile, c, tid & 63) * qh[jj] : 0.f;
            }
            st_row32(uT, tid, q * 32, acc);
        }
        // dW^T row (thread = k) = -(H0 dU^T)[k][:]
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float x[32];
            tmem_ld32(tmem_addr(t_dw, warp, q * 32), x);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) x[jj] = (q * 32 + jj) < L ? -x[jj] : 0.f;
            st_row32(dwT, tid, q * 32, x);
        }
        tc_fence_before();
        fence_proxy_async();
        reduce64(p, s.rowA, s.red, false);    // contains the barrier that publishes uT, dwT
    }

    // ---------------- wave 2: dP = dO U^T, dW K^T (lanes 0-63), T on CUDA cores
    ++mma_n;
    if (tid == 0) {
        tc_fence_after();
        const uint32_t qk = smem_u32(s.qk), dO = smem_u32(s.dO), uTa = smem_u32(uT),
                       dwa = smem_u32(dwT);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t hs = kk >> 2, sub = (kk & 3) * 32;
            mma_bf16(t_dp, desc_sw128(dO + hs * kTile + sub, 16, 1024),
                     desc_sw128(uTa + kk * 2048, kTile, 1024), kKM, kk > 0);
            mma_bf16(t_tw, desc_sw128(dwa + kk * 2048, 0, 1024),
                     desc_sw128(qk + hs * 2 * kTile + kTile + sub, 16, 1024), kMK, kk > 0);
        }
        mma_commit(&s.mma_bar);
    }
    if (tid < 64) {
        // column r of T = (I + A)^-1, kept by the prep kernel of the recompute
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
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) s.tf[i][r] = col[i];
        st_row64(s.tt, r, col);
    }
    ok = mbar_wait(&s.mma_bar, 1, g.spin_limit, g.status);
    if (__syncthreads_or(!ok)) goto bail;
    tc_fence_after();
    {
        float z[64];
        if (tid < 64) {
            const float gr = s.gam[r];
            float zr = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float dp[32], qk[32];
                tmem_ld32(tmem_addr(t_dp, warp, q * 32), dp);
                tmem_ld32(tmem_addr(t_p, warp, q * 32), qk);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int c = q * 32 + jj;
                    const float ds = (c <= r && r < L) ? scale * dp[jj] * __expf(gr - s.gam[c]) : 0.f;
                    const float zz = ds * qk[jj];
                    zr += zz;
                    z[c] = -zz;
                    dp[jj] = ds;
                }
                st_row32(s.ds, r, q * 32, dp);
            }
            s.zrow[r] = zr;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float tu[32], tw[32];
                tmem_ld32(tmem_addr(t_tu, warp, q * 32), tu);
                tmem_ld32(tmem_addr(t_tw, warp, q * 32), tw);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int c = q * 32 + jj;
                    s.fd[r][c] = (c < r && r < L) ? s.bet[c] * (tu[jj] + s.ee[c] * tw[jj]) : 0.f;
                }
            }
        } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) z[c] = 0.f;
        }
        // dHL^T rows (thread = v): k half 0 into the dO tile, half 1 into the W tile
        float hd = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            float x[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                const int k = half * 64 + i;
                const float d = dHL[k * kD + tid];
                hd += d * H0[k * kD + tid];
                x[i] = d;
            }
            st_row64(half ? s.w : s.dO, tid, x);
        }
        reduce64(z, s.zcol, s.red, false);
        hd = block_sum(hd, s.hdot + 4);
        if (tid == 0) s.hdot[0] = hd;
    }
    // ---------------- X = dT T^T, dA = -T^T X on CUDA cores (fp32)
    {
        const int s0 = (tid >> 6) * 32;
        for (int c = s0; c < s0 + 32; ++c) {
            float acc = 0.f;
            const int bmax = min(r, c + 1);
            for (int b = 0; b < bmax; ++b) acc += s.fd[r][b] * s.tf[c][b];
            s.fa[r][c] = acc;
        }
        __syncthreads();
        for (int c = s0; c < s0 + 32; ++c) {
            float acc = 0.f;
            if (c < r && r < L)
                for (int q = r; q < 64; ++q) acc += s.tf[q][r] * s.fa[q][c];
            s.fd[r][c] = -acc;
        }
        __syncthreads();
    }
    {
        // Gs = G + G^T, z' = G .* K K^T, and the dA part of dbeta (threads 64-127, row r)
        float zp[64];
        if (tid >= 64) {
            const float gr = s.gam[r], br = s.bet[r];
            float zpr = 0.f, dba = 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float kk[32], gsv[32];
                tmem_ld32(tmem_addr(t_p, warp, q * 32), kk);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int c = q * 32 + jj;
                    const bool low = c < r && r < L, up = c > r && c < L;
                    const float d_rc = low ? __expf(gr - s.gam[c]) : 0.f;
                    const float g_rc = low ? s.fd[r][c] * br * d_rc : 0.f;
                    const float g_cr = up ? s.fd[c][r] * s.bet[c] * __expf(s.gam[c] - gr) : 0.f;
                    gsv[jj] = g_rc + g_cr;
                    const float zz = g_rc * kk[jj];
                    zpr += zz;
                    zp[c] = -zz;
                    dba += low ? s.fd[r][c] * kk[jj] * d_rc : 0.f;
                }
                st_row32(s.gs, r, q * 32, gsv);
            }
            s.zprow[r] = zpr;
            s.dbA[r] = dba;
        } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) zp[c] = 0.f;
        }
        tc_fence_before();
        fence_proxy_async();
        reduce64(zp, s.zcol, s.red, true);
    }

    // ---------------- wave 3
    ++mma_n;
    if (tid == 0) {
        tc_fence_after();
        const uint32_t qk = smem_u32(s.qk), ds = smem_u32(s.ds), gs = smem_u32(s.gs),
                       tt = smem_u32(s.tt), dhL = smem_u32(s.dO), uTa = smem_u32(uT),
                       dwa = smem_u32(dwT), du = smem_u32(s.du);
        const uint32_t dh_lbo = smem_u32(s.w) - smem_u32(s.dO);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint64_t aK = desc_sw128(qk + kTile + kk * 2048, 2 * kTile, 1024);   // K, MN-major
            const uint64_t aQ = desc_sw128(qk + kk * 2048, 2 * kTile, 1024);           // Q, MN-major
            mma_bf16(t_q2, aK, desc_sw128(ds + kk * 32, 16, 1024), kMK, kk > 0);
            mma_bf16(t_dk, aQ, desc_sw128(ds + kk * 2048, kTile, 1024), kMM, kk > 0);
            mma_bf16(t_dk, aK, desc_sw128(gs + kk * 32, 16, 1024), kMK, 1);
            mma_bf16(t_yw, desc_sw128(dwa + kk * 32, 16, 1024), desc_sw128(tt + kk * 32, 16, 1024),
                     kKK, kk > 0);
            mma_bf16(t_yu, desc_sw128(du + kk * 2048, kTile, 1024), desc_sw128(tt + kk * 32, 16, 1024),
                     kMK, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_bf16(t_dkh, desc_sw128(dhL + kk * 2048, dh_lbo, 1024),
                     desc_sw128(uTa + kk * 2048, kTile, 1024), kMM, kk > 0);
        mma_commit(&s.mma_bar);
    }
    ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
    if (__syncthreads_or(!ok)) goto bail;
    tc_fence_after();
    {
        const long long rs = (long long)H * kD;
        TG *dq = (TG *)a.dq + (bos * H + h) * (long long)kD + tid;
        TG *dk = (TG *)a.dk + (bos * H + h) * (long long)kD + tid;
        TG *dv = (TG *)a.dv + (bos * H + h) * (long long)kD + tid;
        const uint8_t *krow = s.qk + (tid >> 6) * 2 * kTile + kTile;
        const uint8_t *vrow = s.v + (tid >> 6) * kTile;
        float pz[64];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float q1[32], q2[32];
            tmem_ld32(tmem_addr(t_q1, warp, q * 32), q1);
            tmem_ld32(tmem_addr(t_q2, warp, q * 32), q2);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = q * 32 + jj;
                if (c < L) from_f(dq + c * rs, scale * s.ee[c] * q1[jj] + q2[jj]);
            }
            float d[32], e[32], y[32];
            tmem_ld32(tmem_addr(t_dk, warp, q * 32), d);
            tmem_ld32(tmem_addr(t_dkh, warp, q * 32), e);
            tmem_ld32(tmem_addr(t_yw, warp, q * 32), y);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = q * 32 + jj;
                const float dkh = s.ff[c] * e[jj];
                if (c < L) from_f(dk + c * rs, d[jj] + dkh + s.bet[c] * s.ee[c] * y[jj]);
                pz[c] = c < L ? dkh * ld_bf16(krow, c, tid & 63) : 0.f;
            }
        }
        reduce64(pz, s.zpp, s.red, false);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float y[32];
            tmem_ld32(tmem_addr(t_yw, warp, q * 32), y);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = q * 32 + jj;
                pz[c] = c < L ? y[jj] * ld_bf16(krow, c, tid & 63) : 0.f;
            }
        }
        reduce64(pz, s.yw, s.red, false);
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float y[32];
            tmem_ld32(tmem_addr(t_yu, warp, q * 32), y);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int c = q * 32 + jj;
                if (c < L) from_f(dv + c * rs, s.bet[c] * y[jj]);
                pz[c] = c < L ? y[jj] * ld_bf16(vrow, c, tid & 63) : 0.f;
            }
        }
        reduce64(pz, s.yu, s.red, false);
    }
    {
        const float zsum = block_sum(tid < 64 ? s.zpp[tid] : 0.f, s.hdot + 4);
        if (tid < 64) {
            float dgam = 0.f, db = 0.f;
            if (r < L) {
                dgam = s.zrow[r] + s.zprow[r] + s.zcol[r] + s.bet[r] * s.ee[r] * s.yw[r] +
                       scale * s.ee[r] * s.rowA[r] - s.zpp[r];
                if (r == L - 1) dgam += zsum + s.ee[r] * s.hdot[0];
                db = s.yu[r] + s.ee[r] * s.yw[r] + s.dbA[r];
                a.dbeta[(bos + r) * H + h] = db;
            }
            s.red[0][r] = dgam;
        }
        __syncthreads();
        if (tid == 0) {
            float acc = 0.f;
            for (int c = L - 1; c >= 0; --c) {
                acc += s.red[0][c];
                a.dg[(bos + c) * H + h] = acc;
            }
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
    CUtensorMap mq, mk, mv, mdo, mdu, mw;
    if ((e = make_map(&mq, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mk, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mv, g.v, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mdo, p.d_o, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mdu, p.ws.du, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mw, p.ws.w, tokens, g.H)) != cudaSuccess) return e;
    TcLocalArgs a{};
    a.ws_gam = p.ws.gam;
    a.hc = p.ws.hc;
    a.dhc = p.ws.dhc;
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
        tc_local_kernel<__nv_bfloat16><<<grid, 128, smem, s>>>(mq, mk, mv, mdo, mdu, mw, g, a);
    } else {
        if ((e = set_smem(tc_local_kernel<float>, smem)) != cudaSuccess) return e;
        tc_local_kernel<float><<<grid, 128, smem, s>>>(mq, mk, mv, mdo, mdu, mw, g, a);
    }
    prof_after(s);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace gdn
