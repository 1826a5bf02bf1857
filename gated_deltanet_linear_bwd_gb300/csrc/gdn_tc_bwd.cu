// gdn_tc_bwd.cu -- tensor-core (tcgen05 + TMA) backward pieces for bf16
// q/k/v with K = V = 128.
//
// Reverse walk of the state gradient, per (sequence or segment, head),
// chunks last to first.  With dH the gradient at a chunk's end, held as
// dH^T (V rows x K columns, one row per thread, fp32 registers):
//   X^T  = dH^T K^T                      (K dH)^T
//   Y^T  = dO^T P,  P = scale (Q K^T .* lower_incl .* D)
//   dU^T = Y^T + X^T diag(f),            f = exp(gam_L - gam)
//   dH^T <- exp(gam_L) dH^T + dO^T (diag(scale e^gam) Q) - dU^T W
// The segment map of this walk ([A' | B'], A' the transpose of the forward
// map) is walked the same way with dO = 0 on its A' columns.
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

// kind::f16 descriptor with A negated (bit 13).
constexpr uint32_t idesc_neg_a(uint32_t d) { return d | (1u << 13); }

constexpr uint32_t kIdKK64 = idesc_bf16(128, 64, false, false);   // K-major A, K-major B
constexpr uint32_t kIdMM64 = idesc_bf16(128, 64, true, true);     // MN-major A and B, N = 64
constexpr uint32_t kIdMM128 = idesc_bf16(128, 128, true, true);   // MN-major A and B, N = 128
constexpr uint32_t kIdKK128Neg = idesc_neg_a(idesc_bf16(128, 128, false, false));

struct DWalkSmem {
    uint8_t qk[2][4 * kTile];      // per stage: [dk half][Q rows 0-63, K rows 64-127][128 B]
    uint8_t w[2][2 * kTile];       // per stage: W^T, [128 rows k][64 chunk rows]  K-major B
    uint8_t dO[2][2 * kTile];      // per stage: [dv half][64 rows][128 B]
    uint8_t dhT[4 * kTile];        // [dk half][128 rows (v)][128 B]      K-major A
    uint8_t qs[2 * kTile];         // diag(scale e^gam) Q: [dk half][64 rows r][128 B], MN-major B
    uint8_t duT[2 * kTile];        // [128 rows (v)][64 c]                 K-major A
    uint8_t p[kTile];              // [64 rows r][64 c], includes scale    MN-major B
    float gam[2][64];
    float fr[64];                  // exp(gam_L - gam_r) (x rk_r), 0 past L
    float rq[64], rk[64];
    uint64_t tma_bar[2], mma_bar;
    uint32_t tmem_base;
};

struct TcDWalkArgs {
    const float *ws_gam;
    const float *dht;         // [N, H, K, V] nullable
    const float *seg_end;     // [segs, H, K, V] (CP): gradient at each segment's end
    float *dh0;               // [N, H, K, V] nullable
    __nv_bfloat16 *dhc;       // gradient at every chunk's end (kOut), bf16 dH^T tiles
                              // [chunk][H][k half][v][64]
    __nv_bfloat16 *du;        // [chunk][H][V][64] dU^T tiles (kOut), nullable
    float *maps;              // [segs, H, K, K+V] (kMap)
    int cp;
};

enum { kDOut = 0, kDMap = 1 };

template <typename F>
cudaError_t set_smem(F kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
}  // namespace

// 256 threads: thread t owns row v = t % 128 of dH^T (TMEM lane v) and the
// column half hs = t / 128; warps w and w + 4 split each epilogue's columns.
template <int MODE>
__global__ void __launch_bounds__(256, 1)
tc_dwalk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_do,
                Geo g, TcDWalkArgs a) {
    extern __shared__ uint8_t smem_raw[];
    DWalkSmem &s = *reinterpret_cast<DWalkSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, h = blockIdx.y, cb = blockIdx.z, H = g.H;
    const int v = tid & 127, hs = tid >> 7;
    int n, j = 0, nseg = 1;
    if (a.cp) {
        if (!seg_ref(g, blockIdx.x, n, j)) return;
        nseg = seq_nsegs(g, n);
    } else {
        n = blockIdx.x;
        if (n >= g.N) return;
    }
    if (MODE == kDMap && j == 0) return;                 // segment 0 needs no map
    const bool a_cols = MODE == kDMap && cb == 0;        // A' columns: start I, dO = 0
    const bool use_do = !a_cols;
    const int nc = seq_nchunks(g, n);
    const int c0 = min(nc, j * g.seg_chunks), c1 = min(nc, (j + 1) * g.seg_chunks);
    const int cbase = seq_chunk_base(g, n);
    long long sbos;
    int slen;
    seq_range(g, n, sbos, slen);

    if (tid == 0) {
        mbar_init(&s.tma_bar[0], 1);
        mbar_init(&s.tma_bar[1], 1);
        mbar_init(&s.mma_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    float dH[64];     // dk half hs of row v of dH^T (= column v of dH)
    {
        const float *src = nullptr;
        if (MODE == kDOut) {
            if (a.cp && j < nseg - 1)
                src = a.seg_end + ((long long)(seq_seg_base(g, n) + j) * H + h) * kD * kD;
            else if (a.dht)
                src = a.dht + ((long long)n * H + h) * kD * kD;
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const int k = 64 * hs + i;
            dH[i] = src ? src[k * kD + v] : ((a_cols && k == v) ? 1.f : 0.f);
        }
    }
    st_row64(s.dhT + hs * 2 * kTile, v, dH);
    if (tid < 64 && c1 > c0) {
        const int Lf = min(kChunk, slen - (c1 - 1) * kChunk);
        s.gam[0][tid] = tid < Lf ? a.ws_gam[(sbos + (long long)(c1 - 1) * kChunk + tid) * H + h] : 0.f;
    }
    fence_proxy_async();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;
    const uint32_t t_p = tbase, t_x = tbase + 64, t_y = tbase + 128, t_z = tbase + 256;

    auto issue_tma = [&](int st, int c) {
        const int tok0 = (int)(sbos + (long long)c * kChunk);
        mbar_arrive_expect_tx(&s.tma_bar[st], 8 * kTile);   // 2 halves x (q, k, w, dO)
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(s.qk[st] + half * 2 * kTile, &tm_q, &s.tma_bar[st], half * 64, h, tok0);
            tma_load_3d(s.qk[st] + half * 2 * kTile + kTile, &tm_k, &s.tma_bar[st], half * 64, h, tok0);
            tma_load_3d(s.dO[st] + half * kTile, &tm_do, &s.tma_bar[st], half * 64, h, tok0);
        }
        tma_load_2d(s.w[st], &tm_w, &s.tma_bar[st], 0, (int)(((long long)(cbase + c) * H + h) * kD));
    };

    int it = 0, mma_n = 0, tma_pending = 0;
    bool bailed = false;
    if (c1 > c0) {
        if (tid == 0) issue_tma(0, c1 - 1);
        tma_pending |= 1;
    }
    for (int c = c1 - 1; c >= c0; --c, ++it) {
        const int st = it & 1;
        const long long bos = sbos + (long long)c * kChunk;
        const int L = min(kChunk, slen - c * kChunk);
        float gnext = 0.f;                     // gam of chunk c - 1, stored at the end
        if (c - 1 >= c0) {
            if (tid == 0) {
                fence_proxy_async();
                issue_tma(st ^ 1, c - 1);
            }
            tma_pending |= 1 << (st ^ 1);
            if (tid < 64) gnext = a.ws_gam[(bos - kChunk + tid) * H + h];   // a full chunk
        }
        if (MODE == kDOut) {
            // row v, k half hs of dH^T: 128 contiguous bytes of the chunk's tile
            uint4 *dst = reinterpret_cast<uint4 *>(
                a.dhc + ((((long long)(cbase + c) * H + h) * 2 + hs) * kD + v) * 64);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                uint32_t w4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    __nv_bfloat162 b2 = __floats2bfloat162_rn(dH[8 * q + 2 * e], dH[8 * q + 2 * e + 1]);
                    w4[e] = *reinterpret_cast<uint32_t *>(&b2);
                }
                dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
        }
        bool ok = mbar_wait(&s.tma_bar[st], (it >> 1) & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tma_pending &= ~(1 << st);
        if (g.l2norm && tid < 128) {
            const int r = tid & 63;
            const uint8_t *base = s.qk[st] + (tid >= 64 ? kTile : 0);
            float ss = 0.f;
#pragma unroll
            for (int half = 0; half < 2; ++half)
#pragma unroll 8
                for (int col = 0; col < 64; ++col) {
                    const float x = ld_bf16(base + half * 2 * kTile, r, col);
                    ss += x * x;
                }
            (tid >= 64 ? s.rk : s.rq)[r] = rsqrtf(ss + 1e-6f);
        }
        // group 1: P (rows of [Q; K] K^T) and X^T = dH^T K^T
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t qk = smem_u32(s.qk[st]), dhT = smem_u32(s.dhT);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
                const uint64_t bk = desc_sw128(qk + half * 2 * kTile + kTile + sub, 16, 1024);
                const uint64_t ad = desc_sw128(dhT + half * 2 * kTile + sub, 16, 1024);
                mma_bf16(t_x, ad, bk, kIdKK64, kk > 0);
                if (use_do) {
                    const uint64_t aq = desc_sw128(qk + half * 2 * kTile + sub, 16, 1024);
                    mma_bf16(t_p, aq, bk, kIdKK64, kk > 0);
                }
            }
            mma_commit(&s.mma_bar);
        }
        if (g.l2norm) __syncthreads();
        if (tid < 64) {
            const float gl = s.gam[st][L - 1];
            s.fr[tid] = tid < L ? __expf(gl - s.gam[st][tid]) * (g.l2norm ? s.rk[tid] : 1.f) : 0.f;
        }
        if (use_do && v >= 64) {
            // row r of diag(scale e^gam) Q, dk half hs (the Q tile is already in place)
            const int r = v - 64;
            const float f = r < L ? g.scale * __expf(s.gam[st][r]) * (g.l2norm ? s.rq[r] : 1.f) : 0.f;
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float x[32];
#pragma unroll
                for (int jj = 0; jj < 32; ++jj)
                    x[jj] = f * ld_bf16(s.qk[st] + hs * 2 * kTile, r, q * 32 + jj);
                st_row32(s.qs + hs * kTile, r, q * 32, x);
            }
        }
        ok = mbar_wait(&s.mma_bar, (mma_n - 1) & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tc_fence_after();
        if (use_do) {
            if (v < 64) {
                // P row r = v, columns 32*hs .. +31, scale included
                const int r = v;
                const float gr = s.gam[st][r];
                const float sr = g.l2norm ? s.rq[r] : 1.f;
                float x[32];
                tmem_ld32(tmem_addr(t_p, warp, 32 * hs), x);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) {
                    const int c2 = 32 * hs + jj;
                    x[jj] = (c2 <= r && r < L)
                                ? g.scale * x[jj] * __expf(gr - s.gam[st][c2]) * sr *
                                      (g.l2norm ? s.rk[c2] : 1.f)
                                : 0.f;
                }
                st_row32(s.p, r, 32 * hs, x);
            }
            tc_fence_before();
            fence_proxy_async();
            __syncthreads();
            ++mma_n;
            if (warp == 0) {
                tc_fence_after();
                const uint32_t dO = smem_u32(s.dO[st]), pp = smem_u32(s.p);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ao = desc_sw128(dO + kk * 2048, kTile, 1024);   // dO^T, MN-major
                    const uint64_t bp = desc_sw128(pp + kk * 2048, kTile, 1024);   // P, MN-major
                    mma_bf16(t_y, ao, bp, kIdMM64, kk > 0);
                }
                mma_commit(&s.mma_bar);
            }
            ok = mbar_wait(&s.mma_bar, (mma_n - 1) & 1, g.spin_limit, g.status);
            if (__syncthreads_or(!ok)) { bailed = true; break; }
            tc_fence_after();
        }
        {
            // dU^T row v, chunk rows 32*hs .. +31: Y^T + X^T diag(f)
            float x[32], y[32];
            tmem_ld32(tmem_addr(t_x, warp, 32 * hs), x);
            if (use_do) tmem_ld32(tmem_addr(t_y, warp, 32 * hs), y);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
                const int r = 32 * hs + jj;
                x[jj] = r < L ? (use_do ? y[jj] : 0.f) + s.fr[r] * x[jj] : 0.f;
            }
            st_row32(s.duT, v, 32 * hs, x);
            if (MODE == kDOut && a.du) {
                // 32 chunk rows of dU^T row v: 64 contiguous bytes of the chunk tile
                uint4 *dst = reinterpret_cast<uint4 *>(
                    a.du + (((long long)(cbase + c) * H + h) * kD + v) * 64 + 32 * hs);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w4[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        __nv_bfloat162 b2 = __floats2bfloat162_rn(x[8 * q + 2 * e], x[8 * q + 2 * e + 1]);
                        w4[e] = *reinterpret_cast<uint32_t *>(&b2);
                    }
                    dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                }
            }
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        // group 3: Z^T = dO^T (diag(scale e^gam) Q) - dU^T W
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t dO = smem_u32(s.dO[st]), qs = smem_u32(s.qs), du = smem_u32(s.duT),
                           wt = smem_u32(s.w[st]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (use_do) {
                    const uint64_t ao = desc_sw128(dO + kk * 2048, kTile, 1024);
                    const uint64_t bq = desc_sw128(qs + kk * 2048, kTile, 1024);
                    mma_bf16(t_z, ao, bq, kIdMM128, kk > 0);
                }
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t au = desc_sw128(du + kk * 32, 16, 1024);
                const uint64_t bw = desc_sw128(wt + kk * 32, 16, 1024);   // W^T, K-major
                mma_bf16(t_z, au, bw, kIdKK128Neg, (use_do || kk > 0) ? 1u : 0u);
            }
            mma_commit(&s.mma_bar);
        }
        ok = mbar_wait(&s.mma_bar, (mma_n - 1) & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tc_fence_after();
        {
            const float el = __expf(s.gam[st][L - 1]);
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                float z[32];
                tmem_ld32(tmem_addr(t_z, warp, 64 * hs + 32 * q), z);
#pragma unroll
                for (int jj = 0; jj < 32; ++jj) dH[32 * q + jj] = el * dH[32 * q + jj] + z[jj];
            }
        }
        st_row64(s.dhT + hs * 2 * kTile, v, dH);
        if (tid < 64) s.gam[st ^ 1][tid] = gnext;
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
    }

    if (bailed) {
        if (tid == 0) {
            for (int st = 0; st < 2; ++st)
                if (tma_pending & (1 << st))
                    mbar_drain(&s.tma_bar[st], ((it + (st != (it & 1))) >> 1) & 1);
            if (mma_n > 0) mbar_drain(&s.mma_bar, (mma_n - 1) & 1);
        }
    } else if (MODE == kDMap) {
        float *dst = a.maps + ((long long)(seq_seg_base(g, n) + j) * H + h) * kD * (2 * kD);
#pragma unroll
        for (int i = 0; i < 64; ++i) dst[(64 * hs + i) * (2 * kD) + cb * kD + v] = dH[i];
    } else if (a.dh0 && j == 0) {
        float *dst = a.dh0 + ((long long)n * H + h) * kD * kD;
#pragma unroll
        for (int i = 0; i < 64; ++i) dst[(64 * hs + i) * kD + v] = dH[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 512);
}

// ------------------------------------------------------------------ host side
cudaError_t backward(const Plan &p, cudaStream_t s, bool have_ctx) {
    cudaError_t e = simt::tables(p, s);
    if (e != cudaSuccess) return e;
    if (!have_ctx && (e = recompute_states(p, s)) != cudaSuccess) return e;
    const Geo &g = p.g;
    const long long tokens = (long long)g.B * g.T;
    CUtensorMap mq, mk, mw, mdo;
    if ((e = make_map(&mq, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mk, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mw, p.ws.w, (long long)p.max_chunks * g.H * kD)) != cudaSuccess)
        return e;
    if ((e = make_map(&mdo, p.d_o, tokens, g.H)) != cudaSuccess) return e;
    const size_t smem = sizeof(DWalkSmem) + 1024;
    if ((e = set_smem(tc_dwalk_kernel<kDOut>, smem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_dwalk_kernel<kDMap>, smem)) != cudaSuccess) return e;
    TcDWalkArgs a{};
    a.ws_gam = p.ws.gam;
    a.dht = p.dht;
    a.dh0 = p.dh0;
    a.dhc = (__nv_bfloat16 *)p.ws.dhc;
    a.du = (__nv_bfloat16 *)p.ws.du;
    if (p.cp) {
        a.cp = 1;
        a.maps = p.ws.maps;
        a.seg_end = p.ws.seg_state;
        prof_before("tc_dwalk_map", s);
        tc_dwalk_kernel<kDMap><<<dim3(p.max_segs, g.H, 2), 256, smem, s>>>(mq, mk, mw, mdo, g, a);
        prof_after(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = simt::cp_rscan(p, s)) != cudaSuccess) return e;
        prof_before("tc_dwalk_out", s);
        tc_dwalk_kernel<kDOut><<<dim3(p.max_segs, g.H, 1), 256, smem, s>>>(mq, mk, mw, mdo, g, a);
        prof_after(s);
    } else {
        prof_before("tc_dwalk_out", s);
        tc_dwalk_kernel<kDOut><<<dim3(g.N, g.H, 1), 256, smem, s>>>(mq, mk, mw, mdo, g, a);
        prof_after(s);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return g.l2norm ? simt::local_grads(p, s, true) : local_grads(p, s);
}

}  // namespace tc
}  // namespace gdn
