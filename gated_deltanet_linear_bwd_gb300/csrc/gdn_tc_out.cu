// gdn_tc_out.cu -- tensor-core output kernel of the forward for bf16 q/k/v
// with K = V = 128: chunk-parallel over (chunk, head) items, two persistent
// CTAs per SM.  From the chunk start state H0 that the walk stored (bf16 H0^T tile)
// and the prep kernel's W^T and u^T tiles:
//   U^T = u^T - H0^T W^T                           (pseudo-values of the chunk)
//   P   = scale (Q K^T .* lower_incl .* D)          D_rs = exp(gam_r - gam_s)
//   O^T = scale H0^T Q^T diag(e) + U^T P^T          e = exp(gam)
// with q, k replaced by their L2-normalised rows when the caller asks for it
// (the norms scale the rows of P and the columns of H0^T Q^T).
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
constexpr uint32_t kKK64 = idesc_bf16(128, 64, false, false);   // K-major A and B
constexpr uint32_t kKM64 = idesc_bf16(128, 64, false, true);    // B MN-major

struct OutSmem {
    uint8_t qk[4 * kTile];     // [dk half][Q rows 0-63, K rows 64-127][128 B]
    uint8_t w[2 * kTile];      // W^T: [128 rows k][64 chunk rows]
    uint8_t u[2 * kTile];      // u^T: [128 rows v][64 chunk rows]
    uint8_t h0T[4 * kTile];    // H0^T: [k half][128 rows v][64]; after wave 1: U^T
    uint8_t p[kTile];          // P rows r
    float gam[64], er[64], eg[64];   // eg: e^(gam_j - gam_{j-1})
    float rqk[128];            // q, k normalised here: 1 / |q_r| at r, 1 / |k_r| at 64 + r
    float gpre[64];            // the next item's gam, fetched during the current one
    uint64_t load_bar[3], mma_bar;  // loads: {q, k, W^T}, {u^T}, {H0^T}
    uint32_t tmem_base;
};

template <typename F>
cudaError_t set_smem(F kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
}  // namespace

// Persistent over (chunk, head) items with a stride of the grid, two CTAs
// per SM.  Per item, 256 threads: thread t reads TMEM lane v = t % 128 and
// chunk-row half hs = t / 128 (columns 32 hs .. +31); rows r of P sit on
// lanes 0-63.  The next item's tiles are fetched as soon as their regions
// are dead: q, k, W^T after the first MMA wave, u^T after the first
// epilogue, H0^T (whose space holds U^T) after the second wave.
__global__ void __launch_bounds__(256, 2)
tc_out_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
              const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
              const __grid_constant__ CUtensorMap tm_hc, Geo g, const float *ws_gam,
              __nv_bfloat16 *o, int n_items) {
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    OutSmem &s = *reinterpret_cast<OutSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, H = g.H;
    const int v = tid & 127, hs = tid >> 7, c0 = 32 * hs, cq = c0 >> 3;
    uint8_t *uT = s.h0T;                       // after wave 1

    auto item_ref = [&](int i, int &ci, int &hh, ChunkRef &r) -> bool {
        if (i >= n_items) return false;
        ci = i / H;
        hh = i % H;
        return chunk_ref(g, ci, r);
    };
    auto load_group = [&](int grp, int ci, int hh, long long bos) {
        const int trow = (int)(((long long)ci * H + hh) * kD);
        uint64_t *bar = &s.load_bar[grp];
        if (grp == 0) {
            mbar_arrive_expect_tx(bar, 6 * kTile);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                tma_load_3d(s.qk + half * 2 * kTile, &tm_q, bar, half * 64, hh, (int)bos);
                tma_load_3d(s.qk + half * 2 * kTile + kTile, &tm_k, bar, half * 64, hh, (int)bos);
            }
            tma_load_2d(s.w, &tm_w, bar, 0, trow);
        } else if (grp == 1) {
            mbar_arrive_expect_tx(bar, 2 * kTile);
            tma_load_2d(s.u, &tm_u, bar, 0, trow);
        } else {
            mbar_arrive_expect_tx(bar, 4 * kTile);
            tma_load_2d(s.h0T, &tm_hc, bar, 0, 2 * trow);
            tma_load_2d(s.h0T + 2 * kTile, &tm_hc, bar, 0, 2 * trow + kD);
        }
    };

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&s.load_bar[i], 1);
        mbar_init(&s.mma_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 256);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = s.tmem_base;
    const uint32_t t_u = tb, t_p = tb + 64, t_oi = tb + 128, t_oa = tb + 192;

    int item = blockIdx.x, ci = 0, h = 0;
    ChunkRef cr;
    bool have = item_ref(item, ci, h, cr);
    int issued[3] = {0, 0, 0};                // loads issued per group (uniform bookkeeping)
    if (have) {
        if (tid == 0)
            for (int grp = 0; grp < 3; ++grp) load_group(grp, ci, h, cr.bos);
        issued[0] = issued[1] = issued[2] = 1;
    }
    int it = 0, mma_n = 0;
    bool bailed = false;
    while (have) {
        const int L = cr.len;
        const long long bos = cr.bos;
        int ci_n = 0, h_n = 0;
        ChunkRef cr_n;
        const bool have_next = item_ref(item + (int)gridDim.x, ci_n, h_n, cr_n);
        tc_fence_before();
        __syncthreads();                      // the previous item's last reads are done
        if (tid < 64) {
            // gam of this item: fetched during the previous one (cp.async), else now
            if (it > 0) cp_async_wait_all();
            s.gam[tid] = it > 0 ? s.gpre[tid] : (tid < L ? ws_gam[(bos + tid) * H + h] : 0.f);
        }
        bool ok = mbar_wait(&s.load_bar[0], it & 1, g.spin_limit, g.status);
        ok = mbar_wait(&s.load_bar[2], it & 1, g.spin_limit, g.status) && ok;
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        // every thread is past the copy of gpre above: the next item's gam can come
        if (tid < 64 && have_next)
            cp_async4(&s.gpre[tid], ws_gam + (cr_n.bos + min(tid, cr_n.len - 1)) * H + h_n,
                      tid < cr_n.len);
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t qk = smem_u32(s.qk), wt = smem_u32(s.w), h0 = smem_u32(s.h0T);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
                const uint64_t ah = desc_sw128(h0 + half * 2 * kTile + sub, 16, 1024);
                const uint64_t aq = desc_sw128(qk + half * 2 * kTile + sub, 16, 1024);
                const uint64_t bk = desc_sw128(qk + half * 2 * kTile + kTile + sub, 16, 1024);
                mma_bf16(t_u, ah, desc_sw128(wt + kk * 2048, 2 * kTile, 1024), kKM64, kk > 0);
                mma_bf16(t_p, aq, bk, kKK64, kk > 0);       // rows 0-63: Q K^T
                mma_bf16(t_oi, ah, aq, kKK64, kk > 0);      // H0^T Q^T
            }
            mma_commit(&s.mma_bar);
        }
        if (g.l2norm) {
            // 1 / |q_r| (stacked rows 0-63) and 1 / |k_r| (rows 64-127)
            row_inv_norms(s.qk, 2 * kTile, 128, s.rqk);
            __syncthreads();
        }
        if (tid < 64) {
            s.er[tid] = tid < L ? __expf(s.gam[tid]) * (g.l2norm ? s.rqk[tid] : 1.f) : 0.f;
            s.eg[tid] = tid > 0 ? __expf(s.gam[tid] - s.gam[tid - 1]) : 1.f;
        }
        ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
        ok = mbar_wait(&s.load_bar[1], it & 1, g.spin_limit, g.status) && ok;
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        // q, k and W^T are dead (the first wave and the norms were their last readers)
        if (tid == 0 && have_next) {
            fence_proxy_async();
            load_group(0, ci_n, h_n, cr_n.bos);
        }
        if (have_next) ++issued[0];
        tc_fence_after();
        {
            // U^T rows v into the dead H0^T tile; P rows r = v < 64
            float xs[32];
            tmem_ld32(tmem_addr(t_u, warp, c0), xs);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float *x = xs + 8 * q;
                const uint4 raw = *reinterpret_cast<const uint4 *>(
                    s.u + v * 128 + (((cq + q) ^ (v & 7)) << 4));
                const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = c0 + 8 * q + e;
                    x[e] = r < L ? __bfloat162float(bv[e]) - x[e] : 0.f;
                }
                st_row8(uT, v, cq + q, x);
            }
            if (v < 64) {
                const int r = v;
                const float sr = g.l2norm ? s.rqk[r] : 1.f;
                float dd[32];
                tmem_ld32(tmem_addr(t_p, warp, c0), xs);
                row_decays32(s.gam, s.eg, r, c0, dd);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float *x = xs + 8 * q;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int c = c0 + 8 * q + e;
                        x[e] = (c <= r && r < L)
                                   ? x[e] * dd[8 * q + e] * sr * (g.l2norm ? s.rqk[64 + c] : 1.f)
                                   : 0.f;
                    }
                    st_row8(s.p, r, cq + q, x);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        // u^T is dead: the next item's
        if (tid == 0 && have_next) load_group(1, ci_n, h_n, cr_n.bos);
        if (have_next) ++issued[1];
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t ua = smem_u32(uT), pp = smem_u32(s.p);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(t_oa, desc_sw128(ua + kk * 32, 16, 1024),
                         desc_sw128(pp + kk * 32, 16, 1024), kKK64, kk > 0);
            mma_commit(&s.mma_bar);
        }
        ok = mbar_wait(&s.mma_bar, 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        // the H0^T / U^T tile is dead: the next item's H0^T
        if (tid == 0 && have_next) {
            fence_proxy_async();
            load_group(2, ci_n, h_n, cr_n.bos);
        }
        if (have_next) ++issued[2];
        tc_fence_after();
        {
            // O rows r, feature v; each group of 8 rows leaves as 8-byte row pieces
            // (four features) after a quad transpose
            __nv_bfloat16 *dst = o + (bos * H + h) * (long long)kD + v;
            float oi[32], oa[32];
            tmem_ld32x2(tmem_addr(t_oi, warp, c0), tmem_addr(t_oa, warp, c0), oi, oa);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float x[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = c0 + 8 * q + e;
                    x[e] = g.scale * (oi[8 * q + e] * s.er[r] + oa[8 * q + e]);
                }
                store_rows8(dst, (long long)H * kD, x, c0 + 8 * q, L);
            }
        }
        item += (int)gridDim.x;
        ci = ci_n;
        h = h_n;
        cr = cr_n;
        have = have_next;
        ++it;
    }
    if (bailed && tid == 0) {
        for (int grp = 0; grp < 3; ++grp)
            if (issued[grp] > 0) mbar_drain(&s.load_bar[grp], (issued[grp] - 1) & 1);
        if (mma_n > 0) mbar_drain(&s.mma_bar, (mma_n - 1) & 1);
    }
    if (tid < 64) cp_async_wait_all();        // a prefetch still in flight after a bail
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 256);
}

cudaError_t output(const Plan &p, cudaStream_t s) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    const Geo &g = p.g;
    const long long tokens = (long long)g.B * g.T;
    const long long tile_rows = (long long)p.max_chunks * g.H * kD;
    CUtensorMap mq, mk, mw, mu, mhc;
    if ((e = make_map(&mq, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mk, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mw, p.ws.w, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mu, p.ws.u, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mhc, p.ws.hc, 2 * tile_rows)) != cudaSuccess) return e;
    const size_t smem = sizeof(OutSmem) + 1024;
    if ((e = set_smem(tc_out_kernel, smem)) != cudaSuccess) return e;
    prof_before("tc_out", s);
    const int n_items = p.max_chunks * g.H;
    if ((e = launch_pdl(tc_out_kernel, dim3(std::min(n_items, 2 * std::max(p.sms, 1))), dim3(256),
                        smem, s, mq, mk, mw, mu, mhc, g, p.ws.gam, (__nv_bfloat16 *)p.o,
                        n_items)) != cudaSuccess)
        return e;
    prof_after(s);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace gdn
