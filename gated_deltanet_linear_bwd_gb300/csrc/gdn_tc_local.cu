// gdn_tc_local.cu -- tensor-core chunk-local gradients for bf16 q/k/v with
// K = V = 128, one (chunk, head) per CTA.  With q, k L2-normalised inside the
// library, the q and k tiles are normalised in shared memory when they land,
// every formula below is taken with q^, k^, and the norm's chain rule
//   dq = (dq^ - q^ <q^, dq^>) / |q|  (per row; likewise dk)
// finishes dq and dk inside the last products and epilogue.
//
// Inputs per chunk, all by TMA: q, k, v, dO and the workspace's bf16 chunk
// tiles of dU^T, W^T, u^T, T, the chunk start state H0^T and the gradient at
// its end dHL^T; gam and beta.  With D = exp(gam_r - gam_s), e = exp(gam),
// f = exp(gam_L - gam):
//   U    = u - W H0
//   dS   = scale (dO U^T) .* lower_incl .* D
//   dW   = -dU H0^T,  dYw = T^T dW,  dYu = T^T dU
//   dA   = -T^T dT T^T with dT = dU (diag(beta) V)^T + dW (diag(beta e) K)^T;
//          since u = T diag(beta) V and W = T diag(beta e) K this is
//          dA = -(dYu u^T + dYw W^T)
//   G    = dA .* D .* beta_r (strict lower)
//   dQ   = scale diag(e) dO H0^T + dS K
//   dK   = dS^T Q + diag(f) U dHL^T + diag(beta e) dYw + (G + G^T) K
//   dV   = diag(beta) dYu
//   dbeta_r = <dYu_r, v_r> + e_r <dYw_r, k_r> + sum_s dA_rs (K K^T)_rs D_rs
//   dgam from every exp factor, dg = reverse cumsum of dgam.
// Products with a feature-dimension output run with the feature on the MMA's
// M side (128 lanes); 64 x 64 products put the chunk rows on lanes 0-63 and
// let lanes 64-127 compute throwaway rows, or (dA) a copy of rows 0-63.
// Epilogues walk their 32 columns in rolled groups of 8 so the code each CTA
// streams through the instruction cache stays small.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

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
    uint8_t dO[2 * kTile];     // [dv half][64 rows][128 B]
    uint8_t du[2 * kTile];     // dU^T: [128 rows v][64 chunk rows]
    uint8_t w[2 * kTile];      // W^T: [128 rows k][64 chunk rows]
    uint8_t ut[2 * kTile];     // u^T: [128 rows v][64 chunk rows]
    uint8_t h0T[4 * kTile];    // H0^T: [k half][128 rows v][64]; after wave 1: U^T, dW^T
    uint8_t dl[4 * kTile];     // dHL^T: [k half][128 rows v][64]; after wave 2: dYu^T, dYw^T
    uint8_t tt[kTile];         // row r = column r of T; q, k normalised here: after wave 2,
                               // diag(-<q^_r, dq^_r>) (the norm's chain rule for dq, wave 3)
    uint8_t ds[kTile];         // dS rows r
    uint8_t gs[kTile];         // G rows r
    float gam[64], bet[64], ee[64], ff[64];
    float dbet[64], dee[64];   // beta and e of the item whose dgam / dbeta are still to come
    float red[16][16], red4[16][16], red5[16][16];
    float zrow[4][64], zprow[4][64], dbA[4][64];   // per column group
    float scan[4][32];         // dg's reverse cumsum
    float zcol[64], rowA[64], yw[64], yu[64], zpp[64];
    float hdot[4];             // per-warp parts of <dHL, H0>
    float bsum[2];             // the zpp sum's two warp parts
    float rq[64], rk[64];      // 1 / |q_r|, 1 / |k_r| (q, k normalised here)
    float dqd[64];             // -<q^_r, dq^_r> (q, k normalised here)
    uint64_t load_bar[3], mma_bar;  // load groups: {dO, dU^T, H0^T (, T)}, {v, W^T, u^T, dHL^T},
                                    // {q, k (, T when q, k are normalised here)}
    uint64_t diag_bar;         // wave 2.5's diagonal products (yw, yu), one phase per item
    uint32_t tmem_base;
};

// Sums over the 512 threads of per-column values, for epilogues that walk 8
// columns at a time: thread t holds 8 values of columns 16 * (t / 128) + 8q
// .. +7 (q = 0, 1).  warp_sum8 adds them over the warp's lanes into
// red[warp][8q .. +7]; quad_sum / red_combine then add the four warps of each
// column group (warps 4 g .. 4 g + 3 cover the 128 TMEM lanes) into dst[0..63].
__device__ __forceinline__ void warp_sum8(float (&x)[8], float *red_row) {
    const int lane = threadIdx.x & 31;
    bool up = (lane & 16) != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = up ? x[i] : x[i + 4], keep = up ? x[i + 4] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
    }
    up = (lane & 8) != 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = up ? x[i] : x[i + 2], keep = up ? x[i + 2] : x[i];
        x[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    up = (lane & 4) != 0;
    {
        const float send = up ? x[0] : x[1], keep = up ? x[1] : x[0];
        x[0] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
    x[0] += __shfl_xor_sync(0xffffffffu, x[0], 2);
    x[0] += __shfl_xor_sync(0xffffffffu, x[0], 1);
    if ((lane & 3) == 0)
        red_row[((lane >> 4) & 1) * 4 + ((lane >> 3) & 1) * 2 + ((lane >> 2) & 1)] = x[0];
}

__device__ __forceinline__ float quad_sum(float (&red)[16][16], int i) {
    const int w0 = 4 * (i >> 4), l = i & 15;
    return red[w0][l] + red[w0 + 1][l] + red[w0 + 2][l] + red[w0 + 3][l];
}

__device__ __forceinline__ void red_combine(float *dst, float (&red)[16][16], bool accumulate) {
    __syncthreads();
    if (threadIdx.x < 64) {
        const float sum = quad_sum(red, threadIdx.x);
        dst[threadIdx.x] = accumulate ? dst[threadIdx.x] + sum : sum;
    }
    __syncthreads();
}

// 8 bf16 of a 128-byte swizzled row: columns 8 * chunk .. +7.
__device__ __forceinline__ void ld_row8(const uint8_t *tile, int row, int chunk, float *x) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(
        tile + row * 128 + (((uint32_t)chunk ^ (uint32_t)(row & 7)) << 4));
    const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] = __bfloat162float(b[e]);
}

// q and k normalised in place (the library's use_qk_l2norm): row r of the
// stacked [Q; K] tile of each dk half is scaled by (|x_r|^2 + 1e-6)^-1/2.  All
// 512 threads take part, four per row: thread t takes row t / 4, dk half
// (t / 2) % 2 and every other 16-byte piece (odd or even: t % 2), the four
// threads' sums of squares joined by shuffles.  At each of the four steps the 8
// threads of a shared-memory phase (two rows, both halves, both parities) visit
// 8 different bank groups.  Every element of a row gets the same factor, so the
// 128-byte swizzle plays no part.  Writes 1 / |q_r| to rq, 1 / |k_r| to rk.
__device__ __forceinline__ void normalise_qk_rows(uint8_t *qk, float *rq, float *rk) {
    const int t = threadIdx.x, r = t >> 2, hh = (t >> 1) & 1, sub = t & 1;
    const int rot = 2 * (r & 1) + hh;
    uint4 *row = reinterpret_cast<uint4 *>(qk + hh * 2 * kTile + r * 128);
    uint4 x[4];
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        x[i] = row[(2 * (i + rot) + sub) & 7];
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&x[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            ss += f.x * f.x + f.y * f.y;
        }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
    const float inv = rsqrtf(ss + 1e-6f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __nv_bfloat162 *b = reinterpret_cast<__nv_bfloat162 *>(&x[i]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            b[j] = __floats2bfloat162_rn(f.x * inv, f.y * inv);
        }
        row[(2 * (i + rot) + sub) & 7] = x[i];
    }
    if ((t & 3) == 0) (r < 64 ? rq : rk)[r & 63] = inv;
}

struct TcLocalArgs {
    const float *ws_gam;
    void *dq, *dk, *dv;
    float *dg, *dbeta;
    int n_items;               // chunk capacity x H; item i = (chunk i / H, head i % H)
};

struct LocalMaps {
    CUtensorMap q, k, v, dO, du, w, u, hc, dhc, t;
};

template <typename F>
cudaError_t set_smem(F kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
}  // namespace

// Persistent: one CTA per SM walks the (chunk, head) items with a stride of
// the grid.  Each item's tiles arrive in three TMA groups that are issued
// while the previous item is still computing, each as soon as the regions it
// fills are dead: {v, dO, dU^T, H0^T, T} after the second epilogue, {W^T, u^T,
// dHL^T} after the dA product, {q, k} after the last product.
//
// 512 threads.  Feature-major results: thread t reads TMEM lane v = t % 128
// (feature v) and the column group cg = t / 128 (chunk columns c0 = 16 cg ..
// +15), so every epilogue is split four ways.  Row-major 64 x 64 results sit
// on lanes 0-63 (warps with warp % 4 < 2: row r = v); lanes 64-127 of the
// [Q; K] K^T product hold K K^T and those of the dA product a second copy of
// dA (warps with warp % 4 >= 2: row r = v - 64).
template <typename TG>
__global__ void __launch_bounds__(512, 1)
tc_local_kernel(const __grid_constant__ LocalMaps m, Geo g, TcLocalArgs a) {
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    LocalSmem &s = *reinterpret_cast<LocalSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = g.H;
    const int v = tid & 127, cg = tid >> 7, c0 = 16 * cg, cq = c0 >> 3;
    const float scale = g.scale;
    const bool tma_thread = tid == 511;
    uint8_t *uT = s.h0T, *dwT = s.h0T + 2 * kTile;    // after wave 1
    uint8_t *dyuT = s.dl, *dywT = s.dl + 2 * kTile;   // after wave 2

    auto item_ref = [&](int i, int &ci, int &hh, ChunkRef &r) -> bool {
        if (i >= a.n_items) return false;
        ci = i / H;
        hh = i % H;
        return chunk_ref(g, ci, r);
    };
    // the three load groups of item (ci, hh) starting at token bos
    auto load_group = [&](int grp, int ci, int hh, long long bos) {
        const int tok0 = (int)bos;
        const int trow = (int)(((long long)ci * H + hh) * kD);
        uint64_t *bar = &s.load_bar[grp];
        // T travels with group 0, or with group 2 when q, k are normalised here (its
        // region then holds a diagonal tile until wave 3 is done)
        const bool t_late = g.l2norm != 0;
        if (grp == 0) {
            mbar_arrive_expect_tx(bar, (t_late ? 8 : 9) * kTile);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tma_load_3d(s.dO + half * kTile, &m.dO, bar, half * 64, hh, tok0);
                tma_load_2d(s.h0T + half * 2 * kTile, &m.hc, bar, 0, 2 * trow + half * kD);
            }
            tma_load_2d(s.du, &m.du, bar, 0, trow);
            if (!t_late) tma_load_2d(s.tt, &m.t, bar, 0, trow / 2);
        } else if (grp == 1) {
            mbar_arrive_expect_tx(bar, 10 * kTile);
#pragma unroll
            for (int half = 0; half < 2; ++half)
                tma_load_3d(s.v + half * kTile, &m.v, bar, half * 64, hh, tok0);
            tma_load_2d(s.w, &m.w, bar, 0, trow);
            tma_load_2d(s.ut, &m.u, bar, 0, trow);
            tma_load_2d(s.dl, &m.dhc, bar, 0, 2 * trow);
            tma_load_2d(s.dl + 2 * kTile, &m.dhc, bar, 0, 2 * trow + kD);
        } else {
            mbar_arrive_expect_tx(bar, (t_late ? 5 : 4) * kTile);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tma_load_3d(s.qk + half * 2 * kTile, &m.q, bar, half * 64, hh, tok0);
                tma_load_3d(s.qk + half * 2 * kTile + kTile, &m.k, bar, half * 64, hh, tok0);
            }
            if (t_late) tma_load_2d(s.tt, &m.t, bar, 0, trow / 2);
        }
    };

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&s.load_bar[i], 1);
        mbar_init(&s.mma_bar, 1);
        mbar_init(&s.diag_bar, 1);
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
    // TMEM columns: wave 1 | wave 2 | wave 2.5 | wave 3 (a column range is
    // reused only after every read of its previous value)
    const uint32_t t_u = tb, t_p = tb + 64, t_dw = tb + 128, t_q1 = tb + 192, t_qh = tb + 256,
                   t_hd = tb + 384;
    const uint32_t t_dp = tb, t_dkh = tb + 128, t_yw = tb + 256, t_yu = tb + 320;
    const uint32_t t_da = tb + 384;
    // diag(dYw K^T) and diag(dYu V^T): yw and yu (columns free from wave 2.5 to wave 3)
    const uint32_t t_dyk = tb + 320, t_dyv = tb + 448;
    const uint32_t t_dk = tb, t_q2 = tb + 448;

    int item = blockIdx.x, ci = 0, h = 0;
    ChunkRef cr;
    bool have = item_ref(item, ci, h, cr);
    int issued[3] = {0, 0, 0};                // loads issued per group (uniform bookkeeping)
    if (have) {
        if (tma_thread)
            for (int grp = 0; grp < 3; ++grp) load_group(grp, ci, h, cr.bos);
        issued[0] = issued[1] = issued[2] = 1;
    }
    // dgam (every exp factor's share) -> dbeta and dg = reverse cumsum of dgam, for
    // the item at token pbos with pL rows and head ph.  Warps 2 and 3 run it (row
    // r = tid - 64), meeting on named barrier 1, while warp 0 issues the next
    // item's first wave and the others wait for it.
    auto dg_tail = [&](long long pbos, int pL, int ph) {
        const int r = tid - 64, w = r >> 5;
        float zs = s.zpp[r];
        for (int o = 16; o > 0; o >>= 1) zs += __shfl_xor_sync(0xffffffffu, zs, o);
        if (lane == 0) s.bsum[w] = zs;
        named_sync(1, 64);
        const float zsum = s.bsum[0] + s.bsum[1];
        float dgam = 0.f;
        if (r < pL) {
            dgam = s.zrow[0][r] + s.zrow[1][r] + s.zrow[2][r] + s.zrow[3][r] +
                   s.zprow[0][r] + s.zprow[1][r] + s.zprow[2][r] + s.zprow[3][r] + s.zcol[r] +
                   s.dbet[r] * s.dee[r] * s.yw[r] + scale * s.dee[r] * s.rowA[r] - s.zpp[r];
            if (r == pL - 1)
                dgam += zsum + s.dee[r] * (s.hdot[0] + s.hdot[1] + s.hdot[2] + s.hdot[3]);
            a.dbeta[(pbos + r) * H + ph] = s.yu[r] + s.dee[r] * s.yw[r] + s.dbA[0][r] +
                                         s.dbA[1][r] + s.dbA[2][r] + s.dbA[3][r];
        }
        s.scan[w][lane] = dgam;
        named_sync(1, 64);
        {
            // dg = reverse cumsum of dgam within the chunk (warp scans over 2 x 32)
            float x = s.scan[1 - w][31 - lane];         // reversed order: position p = 63 - r
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float yv = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += yv;
            }
            s.scan[2 + w][lane] = x;
        }
        named_sync(1, 64);
        {
            const int pidx = r;                          // position in reversed order
            const int rr = 63 - pidx;
            float x = s.scan[2 + (pidx >> 5)][pidx & 31];
            if (pidx >= 32) x += s.scan[2][31];
            if (rr < pL) a.dg[(pbos + rr) * H + ph] = x;
        }
    };
    bool dg_pending = false;
    long long dg_bos = 0;
    int dg_L = 0, dg_h = 0;
    // an item's dq and dk (16 rows each per thread), stored during the next item's
    // first and second waves, where the warps wait anyway: a warp's lanes write 32
    // consecutive features of one row per store
    float dqv[2][8], dkv[2][8];
    bool st_pending = false;
    long long st_bos = 0;
    int st_L = 0, st_h = 0;
    auto store_grad = [&](void *base, float (&x)[2][8]) {
        const long long rs = (long long)H * kD;
        TG *dst = (TG *)base + (st_bos * H + st_h) * (long long)kD + v;
#pragma unroll
        for (int q = 0; q < 2; ++q) store_rows8(dst, rs, x[q], c0 + 8 * q, st_L);
    };
    int it = 0, mma_n = 0, diag_n = 0;
    bool bailed = false;
    float pre_g = 0.f, pre_b = 0.f;           // the next item's gam / beta (threads < 64), read early
    bool pre = false;
    while (have) {
        const int L = cr.len;
        const long long bos = cr.bos;
        int ci_n = 0, h_n = 0;
        ChunkRef cr_n;
        const bool have_next = item_ref(item + (int)gridDim.x, ci_n, h_n, cr_n);
        tc_fence_before();
        __syncthreads();                          // the previous item's last reads are done
        if (tid < 64) {
            s.gam[tid] = pre ? pre_g : (tid < L ? a.ws_gam[(bos + tid) * H + h] : 0.f);
            s.bet[tid] = pre ? pre_b : (tid < L ? g.beta[(bos + tid) * H + h] : 0.f);
        }
        __syncthreads();
        if (tid < 64) {
            s.ee[tid] = tid < L ? __expf(s.gam[tid]) : 0.f;
            s.ff[tid] = tid < L ? __expf(s.gam[L - 1] - s.gam[tid]) : 0.f;
        }
        {
            bool ok = true;
            for (int grp = 0; grp < 3; ++grp)
                ok = mbar_wait(&s.load_bar[grp], it & 1, g.spin_limit, g.status) && ok;
            if (__syncthreads_or(!ok)) { bailed = true; break; }
        }
        if (g.l2norm) {
            // every product and epilogue below then sees q^ = q / |q| and k^ = k / |k|,
            // giving the gradients with respect to q^ and k^; the norm's own chain
            // rule is applied to dq and dk at the end
            normalise_qk_rows(s.qk, s.rq, s.rk);
            fence_proxy_async();
            __syncthreads();
        }
        bool ok;

        // ---------------- wave 1: W H0, [Q; K] K^T, H0^T Q^T, H0 dU^T, H0 dO^T, dHL^T H0
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t qk = smem_u32(s.qk), h0 = smem_u32(s.h0T), w = smem_u32(s.w),
                           du = smem_u32(s.du), dO = smem_u32(s.dO), dl = smem_u32(s.dl);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t hh = kk >> 2, sub = (kk & 3) * 32;
                const uint64_t aH = desc_sw128(h0 + hh * 2 * kTile + sub, 16, 1024);
                const uint64_t aQK = desc_sw128(qk + hh * 2 * kTile + sub, 16, 1024);
                const uint64_t bK = desc_sw128(qk + hh * 2 * kTile + kTile + sub, 16, 1024);
                const uint64_t aHm = desc_sw128(h0 + kk * 2048, 2 * kTile, 1024);   // H0, MN-major
                mma_bf16(t_u, aH, desc_sw128(w + kk * 2048, 2 * kTile, 1024), kKM, kk > 0);
                mma_bf16(t_p, aQK, bK, kKK, kk > 0);
                mma_bf16(t_qh, aH, aQK, kKK, kk > 0);
                mma_bf16(t_dw, aHm, desc_sw128(du + kk * 2048, 2 * kTile, 1024), kMM, kk > 0);
                mma_bf16(t_q1, aHm, desc_sw128(dO + hh * kTile + sub, 16, 1024), kMK, kk > 0);
                // dHL^T H0 (128 x 128): its trace is <dHL, H0>
                mma_bf16(t_hd, desc_sw128(dl + hh * 2 * kTile + sub, 16, 1024), aH, kKK128, kk > 0);
            }
            {
                // T^T dU needs only loaded tiles: with this wave, into columns it leaves free
                const uint32_t tt = smem_u32(s.tt);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(t_yu, desc_sw128(du + kk * 32, 16, 1024), desc_sw128(tt + kk * 32, 16, 1024),
                             kKK, kk > 0);
            }
            mma_commit(&s.mma_bar);
        }
        if (st_pending) store_grad(a.dq, dqv);   // the previous item's dq (its dk: under wave 2)
        if (dg_pending) {
            if (warp == 2 || warp == 3) dg_tail(dg_bos, dg_L, dg_h);   // the previous item's
            dg_pending = false;
        }
        ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tc_fence_after();
        {
            // U^T and dW^T = -(H0 dU^T) rows v into the dead H0^T tile; partial sums
            // of dO[r][v] (Q H0)[r][v] over v for rowA
#pragma unroll 1
            for (int q = 0; q < 2; ++q) {
                float x[8], y[8], uu[8];
                float dw[8];
                tmem_ld8x3(tmem_addr(t_u, warp, c0 + 8 * q), tmem_addr(t_qh, warp, c0 + 8 * q),
                           tmem_addr(t_dw, warp, c0 + 8 * q), x, y, dw);
                ld_row8(s.ut, v, cq + q, uu);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = c0 + 8 * q + e;
                    x[e] = c < L ? uu[e] - x[e] : 0.f;
                    y[e] = c < L ? ld_bf16(s.dO + (v >> 6) * kTile, c, v & 63) * y[e] : 0.f;
                }
                st_row8(uT, v, cq + q, x);
                warp_sum8(y, s.red[warp] + 8 * q);
#pragma unroll
                for (int e = 0; e < 8; ++e) dw[e] = (c0 + 8 * q + e) < L ? -dw[e] : 0.f;
                st_row8(dwT, v, cq + q, dw);
            }
            if (cg == 0) {
                // lane v's diagonal entry of dHL^T H0 sits in column v of t_hd
                float x[32];
                tmem_ld32(tmem_addr(t_hd, warp, 32 * warp), x);
                float d = 0.f;
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) d = jj == lane ? x[jj] : d;
                for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
                if (lane == 0) s.hdot[warp] = d;
            }
            tc_fence_before();
            fence_proxy_async();
            red_combine(s.rowA, s.red, false);    // its barriers publish U^T, dW^T and hdot
        }

        // ---------------- wave 2: dO U^T, dHL U^T, T^T dW (T^T dU went with wave 1)
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t dO = smem_u32(s.dO), uTa = smem_u32(uT), dwa = smem_u32(dwT),
                           dl = smem_u32(s.dl), du = smem_u32(s.du), tt = smem_u32(s.tt);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t hh = kk >> 2, sub = (kk & 3) * 32;
                const uint64_t bU = desc_sw128(uTa + kk * 2048, kTile, 1024);   // U, MN-major
                mma_bf16(t_dp, desc_sw128(dO + hh * kTile + sub, 16, 1024), bU, kKM, kk > 0);
                mma_bf16(t_dkh, desc_sw128(dl + kk * 2048, 2 * kTile, 1024), bU, kMM, kk > 0);
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bT = desc_sw128(tt + kk * 32, 16, 1024);
                mma_bf16(t_yw, desc_sw128(dwa + kk * 32, 16, 1024), bT, kKK, kk > 0);
            }
            mma_commit(&s.mma_bar);
        }
        if (st_pending) {
            store_grad(a.dk, dkv);                // the previous item's dk, under this wave
            st_pending = false;
        }
        ok = mbar_wait(&s.mma_bar, 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tc_fence_after();
        // every feature f = v: dYw^T, dYu^T rows into the dead dHL^T tiles first, so
        // that wave 2.5 can start; the sums over k of (diag(f) U dHL^T) .* K (zpp)
        // follow under it, dV under wave 3 (yu is kept: wave 2.5 overwrites its columns)
        float yuk[16];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            float yw[8];
            tmem_ld8x2(tmem_addr(t_yw, warp, c0 + 8 * q), tmem_addr(t_yu, warp, c0 + 8 * q), yw,
                       yuk + 8 * q);
            st_row8(dywT, v, cq + q, yw);
            st_row8(dyuT, v, cq + q, yuk + 8 * q);
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        // dO, dU^T, the H0^T / U^T / dW^T tile and T are dead: next item's group 0
        if (have_next) {
            if (tma_thread) {
                fence_proxy_async();
                load_group(0, ci_n, h_n, cr_n.bos);
            }
            ++issued[0];
        }

        // ---------------- wave 2.5: dA = -(dYu u^T + dYw W^T), rows duplicated on lanes 64-127;
        // dYw K^T and dYu V^T, whose diagonals are yw_r = <dYw_r, k_r> and yu_r = <dYu_r, v_r>
        ++mma_n;
        ++diag_n;
        // issued by two warps of the dA half, which wait for the dA product anyway:
        // warp 2 the dA product, warp 3 the diagonal products on their own barrier
        // (so that the dA epilogue need not wait for them)
        const uint32_t yu = smem_u32(dyuT), yw = smem_u32(dywT);
        if (warp == 2) {
            tc_fence_after();
            const uint32_t ua = smem_u32(s.ut), wa = smem_u32(s.w);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                mma_bf16(t_da, desc_sw128(yu + kk * 2048, 0, 1024),
                         desc_sw128(ua + kk * 2048, kTile, 1024), kMM, kk > 0);
                mma_bf16(t_da, desc_sw128(yw + kk * 2048, 0, 1024),
                         desc_sw128(wa + kk * 2048, kTile, 1024), kMM, 1);
            }
            mma_commit(&s.mma_bar);
        } else if (warp == 3) {
            tc_fence_after();
            const uint32_t qk = smem_u32(s.qk), va = smem_u32(s.v);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t hh = kk >> 2, sub = (kk & 3) * 32;
                mma_bf16(t_dyk, desc_sw128(yw + kk * 2048, 0, 1024),
                         desc_sw128(qk + hh * 2 * kTile + kTile + sub, 16, 1024), kMK, kk > 0);
                mma_bf16(t_dyv, desc_sw128(yu + kk * 2048, 0, 1024),
                         desc_sw128(va + hh * kTile + sub, 16, 1024), kMK, kk > 0);
            }
            mma_commit(&s.diag_bar);
        }
        tc_fence_after();
        {
            const uint8_t *krow = s.qk + (v >> 6) * 2 * kTile + kTile;
            float pz[16];
            tmem_ld8x2(tmem_addr(t_dkh, warp, c0), tmem_addr(t_dkh, warp, c0 + 8), pz, pz + 8);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float pq[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = c0 + 8 * q + e;
                    const float kv = c < L ? ld_bf16(krow, c, v & 63) : 0.f;
                    pq[e] = pz[8 * q + e] * s.ff[c] * kv;   // (diag(f) U dHL^T) .* K, summed over k
                }
                warp_sum8(pq, s.red4[warp] + 8 * q);
            }
        }
        // While the dA product runs, lanes 0-63 form dS; lanes 64-127 then take
        // the dA epilogue.  Each half reduces into its own array.
        ok = true;
        if (v < 64) {
            // rows r = v: dS and z = dS .* Q K^T (row sums, negated column sums)
            const int r = v;
            const float gr = s.gam[r];
            float zr = 0.f;
#pragma unroll 1
            for (int q = 0; q < 2; ++q) {
                float dp[8], qk[8], zc[8];
                tmem_ld8x2(tmem_addr(t_dp, warp, c0 + 8 * q), tmem_addr(t_p, warp, c0 + 8 * q),
                           dp, qk);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = c0 + 8 * q + e;
                    const float ds =
                        (c <= r && r < L) ? scale * dp[e] * __expf(gr - s.gam[c]) : 0.f;
                    const float zz = ds * qk[e];
                    zr += zz;
                    zc[e] = -zz;
                    dp[e] = ds;
                }
                st_row8(s.ds, r, cq + q, dp);
                warp_sum8(zc, s.red[warp] + 8 * q);
            }
            s.zrow[cg][r] = zr;
            if (lane < 16) s.red5[warp][lane] = 0.f;
            if (cg == 0) {
                // yw_r, yu_r: lane r's diagonal entries (column r) of wave 2.5's products
                ok = mbar_wait(&s.diag_bar, it & 1, g.spin_limit, g.status);
                if (ok) {
                    tc_fence_after();
                    float xk[32], xv[32];
                    tmem_ld32(tmem_addr(t_dyk, warp, 32 * warp), xk);
                    tmem_ld32(tmem_addr(t_dyv, warp, 32 * warp), xv);
                    float dk_ = 0.f, dv_ = 0.f;
#pragma unroll
                    for (int jj = 0; jj < 32; ++jj) {
                        dk_ = jj == lane ? xk[jj] : dk_;
                        dv_ = jj == lane ? xv[jj] : dv_;
                    }
                    s.yw[r] = r < L ? dk_ : 0.f;
                    s.yu[r] = r < L ? dv_ : 0.f;
                }
            }
        } else {
            // rows r = v - 64: G = dA .* D .* beta_r, z' = G .* K K^T and the dA part
            // of dbeta
            if (lane < 16) s.red[warp][lane] = 0.f;
            ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
            if (ok) {
                tc_fence_after();
                const int r = v - 64;
                const float gr = s.gam[r], br = s.bet[r];
                float zpr = 0.f, dba = 0.f;
#pragma unroll 1
                for (int q = 0; q < 2; ++q) {
                    float da[8], kk[8], zc[8];
                    tmem_ld8x2(tmem_addr(t_da, warp, c0 + 8 * q), tmem_addr(t_p, warp, c0 + 8 * q),
                               da, kk);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int c = c0 + 8 * q + e;
                        const bool low = c < r && r < L;
                        const float d_rc = low ? __expf(gr - s.gam[c]) : 0.f;
                        const float dA = -da[e] * d_rc;     // dA .* D on the strict lower part
                        const float g_rc = dA * br;
                        const float zz = g_rc * kk[e];
                        zpr += zz;
                        zc[e] = -zz;
                        dba += dA * kk[e];
                        da[e] = g_rc;
                    }
                    st_row8(s.gs, r, cq + q, da);
                    warp_sum8(zc, s.red5[warp] + 8 * q);
                }
                s.zprow[cg][r] = zpr;
                s.dbA[cg][r] = dba;
            }
        }
        tc_fence_before();
        fence_proxy_async();
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        // wave 2.5 is done (lanes 64-127 saw it): v, W^T, u^T and the dHL^T / dYu^T /
        // dYw^T tiles are dead, the next item's group 1 can come
        if (have_next) {
            if (tma_thread) {
                fence_proxy_async();
                load_group(1, ci_n, h_n, cr_n.bos);
            }
            ++issued[1];
        }
        if (tid < 64) {
            s.zcol[tid] = quad_sum(s.red, tid) + quad_sum(s.red5, tid);
            s.zpp[tid] = quad_sum(s.red4, tid);
        }
        if (g.l2norm) {
            // The norm's chain rule, dx = (dx^ - x^ <x^, dx^>) / |x| per row, joins
            // wave 3.  The row dots are sums already formed above for dgam:
            //   <q^_r, dq^_r> = rows of dS .* Q K^T + scale e_r <dO_r, (Q H0)_r>
            //   <k^_r, dk^_r> = columns of dS .* Q K^T + rows and columns of G .* K K^T
            //                   + f_r <(U dHL^T)_r, k^_r> + beta_r e_r <dYw_r, k^_r>.
            // -<q^, dq^> q^ comes from one more product, Q^T diag(-<q^, dq^>), onto
            // dS K (the diagonal in the dead T tile); -<k^, dk^> k^ from G's diagonal
            // (zero so far), set to -<k^, dk^> / 2, which G K and G^T K each pass on.
            if (tid < 64) {
                const int r = tid;
                const float zr = s.zrow[0][r] + s.zrow[1][r] + s.zrow[2][r] + s.zrow[3][r];
                const float zp = s.zprow[0][r] + s.zprow[1][r] + s.zprow[2][r] + s.zprow[3][r];
                const float dq_dot = zr + scale * s.ee[r] * s.rowA[r];
                const float dk_dot = -s.zcol[r] + s.zpp[r] + s.bet[r] * s.ee[r] * s.yw[r] + zp;
                s.dqd[r] = -dq_dot;
                *reinterpret_cast<__nv_bfloat16 *>(s.gs + sw128_off(r, r)) =
                    __float2bfloat16_rn(-0.5f * dk_dot);
            }
            __syncthreads();
            {
                // the diagonal tile, one 16-byte piece per thread (row tid / 8)
                const int r = tid >> 3, chunk = tid & 7;
                const float d = s.dqd[r];
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = (8 * chunk + e == r) ? d : 0.f;
                st_row8(s.tt, r, chunk, x);
            }
            fence_proxy_async();
            __syncthreads();
        }

        // ---------------- wave 3: dS K, dS^T Q + (G + G^T) K
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t qk = smem_u32(s.qk), ds = smem_u32(s.ds), gs = smem_u32(s.gs);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t aK = desc_sw128(qk + kTile + kk * 2048, 2 * kTile, 1024);   // K, MN-major
                const uint64_t aQ = desc_sw128(qk + kk * 2048, 2 * kTile, 1024);           // Q, MN-major
                mma_bf16(t_q2, aK, desc_sw128(ds + kk * 32, 16, 1024), kMK, kk > 0);
                mma_bf16(t_dk, aQ, desc_sw128(ds + kk * 2048, kTile, 1024), kMM, kk > 0);
                mma_bf16(t_dk, aK, desc_sw128(gs + kk * 32, 16, 1024), kMK, 1);         // G K
                mma_bf16(t_dk, aK, desc_sw128(gs + kk * 2048, kTile, 1024), kMM, 1);    // G^T K
            }
            if (g.l2norm) {
                const uint32_t dq = smem_u32(s.tt);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)      // Q^T diag(-<q^, dq^>)
                    mma_bf16(t_q2, desc_sw128(qk + kk * 2048, 2 * kTile, 1024),
                             desc_sw128(dq + kk * 2048, kTile, 1024), kMM, 1);
            }
            mma_commit(&s.mma_bar);
        }
        {
            // dV = diag(beta) dYu under this wave (yu kept since the second epilogue);
            // a warp's lanes write 32 consecutive features
            TG *dv = (TG *)a.dv + (bos * H + h) * (long long)kD + v;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float dvq[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) dvq[e] = s.bet[c0 + 8 * q + e] * yuk[8 * q + e];
                store_rows8(dv, (long long)H * kD, dvq, c0 + 8 * q, L);
            }
        }
        ok = mbar_wait(&s.mma_bar, 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        // q, k (and the T region) are dead (their last reader was wave 3): next item's group 2
        if (have_next) {
            if (tma_thread) {
                fence_proxy_async();
                load_group(2, ci_n, h_n, cr_n.bos);
            }
            ++issued[2];
            if (tid < 64) {
                pre_g = tid < cr_n.len ? a.ws_gam[(cr_n.bos + tid) * H + h_n] : 0.f;
                pre_b = tid < cr_n.len ? g.beta[(cr_n.bos + tid) * H + h_n] : 0.f;
            }
        }
        pre = have_next;
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            // feature v (= k), chunk rows c0 + 8 q .. +7; kept in registers and stored
            // during the next item's first two waves
            float x[8], y[8], pw[8], x1[8], y1[8];
            tmem_ld8x5(tmem_addr(t_q1, warp, c0 + 8 * q), tmem_addr(t_q2, warp, c0 + 8 * q),
                       tmem_addr(t_dk, warp, c0 + 8 * q), tmem_addr(t_dkh, warp, c0 + 8 * q),
                       tmem_addr(t_yw, warp, c0 + 8 * q), x1, y1, x, y, pw);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int c = c0 + 8 * q + e;
                // with q, k normalised here the products above already hold
                // dx^ - x^ <x^, dx^>; what is left of the norm's chain rule is 1 / |x|
                const float sq = g.l2norm ? s.rq[c] : 1.f, sk = g.l2norm ? s.rk[c] : 1.f;
                dqv[q][e] = sq * (scale * s.ee[c] * x1[e] + y1[e]);
                dkv[q][e] = sk * (x[e] + s.ff[c] * y[e] + s.bet[c] * s.ee[c] * pw[e]);
            }
        }
        st_pending = true;
        st_bos = bos;
        st_L = L;
        st_h = h;
        // dgam, dbeta and dg of this item come during the next item's first wave (they
        // read only this item's row sums, kept until then, and copies of beta and e)
        if (tid < 64) {
            s.dbet[tid] = s.bet[tid];
            s.dee[tid] = s.ee[tid];
        }
        dg_pending = true;
        dg_bos = bos;
        dg_L = L;
        dg_h = h;
        item += (int)gridDim.x;
        ci = ci_n;
        h = h_n;
        cr = cr_n;
        have = have_next;
        ++it;
    }

    // the last item's tail: after a barrier, since its copies of beta and e were
    // written after the item's last one
    __syncthreads();
    if (!bailed && st_pending) {
        store_grad(a.dq, dqv);
        store_grad(a.dk, dkv);
    }
    if (!bailed && dg_pending && (warp == 2 || warp == 3)) dg_tail(dg_bos, dg_L, dg_h);
    if (bailed && tid == 0) {
        // loads of this item (issued, not yet seen) or of the next one, and the last MMA phase
        for (int grp = 0; grp < 3; ++grp)
            if (issued[grp] > 0) mbar_drain(&s.load_bar[grp], (issued[grp] - 1) & 1);
        if (mma_n > 0) mbar_drain(&s.mma_bar, (mma_n - 1) & 1);
        if (diag_n > 0) mbar_drain(&s.diag_bar, (diag_n - 1) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t local_grads(const Plan &p, cudaStream_t s) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    const Geo &g = p.g;
    const long long tokens = (long long)g.B * g.T;
    LocalMaps m;
    const long long tile_rows = (long long)p.max_chunks * g.H * kD;
    if ((e = make_map(&m.q, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&m.k, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&m.v, g.v, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&m.dO, p.d_o, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.du, p.ws.du, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.w, p.ws.w, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.u, p.ws.u, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.hc, p.ws.hc, 2 * tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.dhc, p.ws.dhc, 2 * tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.t, p.ws.tmat, tile_rows / 2, 64)) != cudaSuccess) return e;
    TcLocalArgs a{};
    a.ws_gam = p.ws.gam;
    a.dq = p.dq;
    a.dk = p.dk;
    a.dv = p.dv;
    a.dg = p.dg;
    a.dbeta = p.dbeta;
    a.n_items = p.max_chunks * g.H;
    const size_t smem = sizeof(LocalSmem) + 1024;
    const dim3 grid(std::min(a.n_items, std::max(p.sms, 1)));
    const dim3 block(512);
    prof_before("tc_local_grad", s);
    if (p.grad_dtype == GDN_BF16) {
        if ((e = set_smem(tc_local_kernel<__nv_bfloat16>, smem)) != cudaSuccess) return e;
        if ((e = launch_pdl(tc_local_kernel<__nv_bfloat16>, grid, block, smem, s,
                            m, g, a)) != cudaSuccess)
            return e;
    } else {
        if ((e = set_smem(tc_local_kernel<float>, smem)) != cudaSuccess) return e;
        if ((e = launch_pdl(tc_local_kernel<float>, grid, block, smem, s,
                            m, g, a)) != cudaSuccess)
            return e;
    }
    prof_after(s);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace gdn
