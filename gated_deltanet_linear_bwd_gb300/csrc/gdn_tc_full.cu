// gdn_tc_full.cu -- the whole forward in one kernel (bf16 q/k/v, K = V = 128),
// for batches whose (sequence, head) pairs fill the GPU without sequence
// parallelism and when no context is kept for the backward.
//
// One CTA per (sequence, head) walks its chunks.  For each chunk it does the
// chunk-local preparation that the split path runs as a kernel of its own,
//   gam = cumsum(g),  A = strict_lower(diag(beta) K K^T .* D),  T = (I + A)^-1,
//   W = T diag(beta e) K,  u = T diag(beta) V,
// and then the walk step with its output,
//   U = u - W H,  H <- exp(gam_L) H + K^T diag(f) U,
//   O = scale (diag(e) Q H + (Q K^T .* lower_incl .* D) U),
// so that gam, W and u never leave the SM.  K K^T is the lower half of the
// [Q; K] K^T product that P needs anyway.  The layout and the state recurrence
// are those of the fused walk in gdn_tc_fwd.cu; T comes from the same blocked
// solve as the prep kernel's (gdn_tc_solve.cuh), run by warps 0-1.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "gdn_tc_solve.cuh"
#include "tc_ptx.cuh"

namespace gdn {
namespace tc {

namespace {
constexpr int kD = 128;
constexpr int kTile = 8192;
constexpr uint32_t kIdDH = idesc_bf16(128, 128, false, true);     // B MN-major, N = 128
constexpr uint32_t kIdKM64 = idesc_bf16(128, 64, false, true);    // B MN-major, N = 64
constexpr uint32_t kIdKK64 = idesc_bf16(128, 64, false, false);   // both K-major, N = 64
constexpr uint32_t kIdMM64 = idesc_bf16(128, 64, true, true);     // both MN-major, N = 64

struct FullSmem {
    uint8_t qk[2][4 * kTile];   // per stage: [dk half][Q rows 0-63, K rows 64-127][128 B]
    uint8_t v[2][2 * kTile];    // per stage: [dv half][64 rows][128 B]
    uint8_t w[2 * kTile];       // W^T of the chunk: [128 rows k][64 chunk rows]
    uint8_t u[2 * kTile];       // u^T: [128 rows v][64 chunk rows]
    float A[64][68];            // A^T rows (row j = column j of A), then T's blocks; after
                                // the solve the W and u B operands (bf16, 8 KB each)
    uint8_t hT[4 * kTile];      // [dk half][128 state rows][128 B] (A operand)
    uint8_t uTs[2 * kTile];     // U^T diag(f) (A operand)
    uint8_t uT[2 * kTile];      // U^T (A operand of U^T P^T)
    uint8_t p[kTile];           // P rows r
    float graw[2][64], braw[2][64];   // g and beta per stage
    float gam[2][64];           // per chunk parity
    alignas(16) float fr[64];   // exp(gam_L - gam_r) / |k_r|; 0 past L
    alignas(16) float er[2][64];   // exp(gam_r) / |q_r| per chunk parity; 0 past L
    float egw[2][64];           // exp(gam_j - gam_{j-1}) per chunk parity
    float eb[64], bt[64];       // beta_j e_j / |k_j| (W's scale) and beta_j (u's); 0 past L
    float rqk[128];             // 1 / |q_r| at r, 1 / |k_r| at 64 + r (1 without the norm)
    float wsum[2];
    uint64_t tma_bar[2], bar_q, bar_w, bar_u, bar_dh;
    uint32_t tmem_base;
};

struct FullArgs {
    const float *h0;            // [N, H, K, V] nullable
    float *final_state;         // nullable
    __nv_bfloat16 *o;           // [tokens, H, V]
};
}  // namespace

// 256 threads, as in the fused walk: thread t owns state row v = t % 128 (TMEM
// lane v) and the column half hs = t / 128.  TMEM: U (0-63), [Q; K] K^T
// (64-127: Q K^T on lanes 0-63, K K^T on lanes 64-127), the state update
// (128-255, which first holds W^T and u^T), H^T Q^T and U^T P^T per chunk
// parity (256 + 128 b, 320 + 128 b).  Per chunk:
//   1. [Q; K] K^T; gam; the norms; the previous chunk's O
//   2. A^T rows (lanes 64-127) and P (lanes 0-63)
//   3. T by warps 0-1, then the W / u operands
//   4. W^T = K^T (T diag(beta e / |k|))^T, u^T = V^T (T diag(beta))^T into TMEM,
//      then into shared memory as bf16
//   5. the walk step: U, U^T diag(f), K^T diag(f) U, U^T P^T and H^T Q^T, the state
//      update
__global__ void __launch_bounds__(256, 1)
tc_full_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_v, Geo g, FullArgs a) {
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    FullSmem &s = *reinterpret_cast<FullSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, H = g.H;
    const int v = tid & 127, hs = tid >> 7;
    int n, h;
    walk_unit(g, blockIdx.x, n, h);
    if (n >= g.N) return;
    const int nc = seq_nchunks(g, n);
    long long sbos;
    int slen;
    seq_range(g, n, sbos, slen);
    const bool tma_thread = tid == 255;

    auto issue_tma = [&](int st, int c) {
        const int tok0 = (int)(sbos + (long long)c * kChunk);
        mbar_arrive_expect_tx(&s.tma_bar[st], 6 * kTile);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(s.qk[st] + half * 2 * kTile, &tm_q, &s.tma_bar[st], 64 * half, h, tok0);
            tma_load_3d(s.qk[st] + half * 2 * kTile + kTile, &tm_k, &s.tma_bar[st], 64 * half, h,
                        tok0);
            tma_load_3d(s.v[st] + half * kTile, &tm_v, &s.tma_bar[st], 64 * half, h, tok0);
        }
    };
    // g and beta of chunk c into stage st (threads 0-63, zero past the sequence)
    auto fetch_gb = [&](int st, int c) {
        const int Lc = min(kChunk, slen - c * kChunk);
        const bool ok = tid < Lc;
        const long long i = ok ? (sbos + (long long)c * kChunk + tid) * H + h : 0;
        cp_async4(&s.graw[st][tid], g.g + i, ok);
        cp_async4(&s.braw[st][tid], g.beta + i, ok);
    };

    if (tid == 0) {
        mbar_init(&s.tma_bar[0], 1);
        mbar_init(&s.tma_bar[1], 1);
        mbar_init(&s.bar_q, 1);
        mbar_init(&s.bar_w, 1);
        mbar_init(&s.bar_u, 1);
        mbar_init(&s.bar_dh, 1);
        fence_barrier_init();
        if (nc > 0) issue_tma(0, 0);          // the thread that set up the barrier
    }
    if (tid < 64 && nc > 0) fetch_gb(0, 0);
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
        tc_fence_before();
    }
    // start state: this thread's half (dk 64 hs ..) of column v of H
    float Hr[64];
    {
        const float *src = a.h0 ? a.h0 + ((long long)n * H + h) * kD * kD : nullptr;
#pragma unroll
        for (int i = 0; i < 64; ++i) Hr[i] = src ? src[(64 * hs + i) * kD + v] : 0.f;
    }
    st_row64(s.hT + hs * 2 * kTile, v, Hr);
    fence_proxy_async();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = s.tmem_base;
    const uint32_t t_u = tb, t_p = tb + 64, t_dh = tb + 128, t_w = tb + 128, t_uu = tb + 192;
    auto t_qh = [&](int b) { return tb + 256 + 128 * b; };
    auto t_pu = [&](int b) { return tb + 320 + 128 * b; };
    uint8_t *bw = reinterpret_cast<uint8_t *>(&s.A[0][0]);
    uint8_t *bu = bw + kTile;

    long long pbos = 0;
    int pL = 0;
    // O rows 32 hs .. +31 of the chunk at token pbos (parity b), feature v:
    // scale (e_c (H^T Q^T) + U^T P^T)
    auto out_epilogue = [&](int b) {
        float qh[32], pu[32];
        tmem_ld32x2(tmem_addr(t_qh(b), warp, 32 * hs), tmem_addr(t_pu(b), warp, 32 * hs), qh, pu);
        __nv_bfloat16 *dst = a.o + (pbos * H + h) * (long long)kD + v;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 e0 = reinterpret_cast<const float4 *>(s.er[b])[8 * hs + 2 * q];
            const float4 e1 = reinterpret_cast<const float4 *>(s.er[b])[8 * hs + 2 * q + 1];
            const float eq[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = g.scale * (eq[e] * qh[8 * q + e] + pu[8 * q + e]);
            store_rows8(dst, (long long)H * kD, x, 32 * hs + 8 * q, pL);
        }
    };

    // uniform bookkeeping for the bail-out path: the stages whose latest load has
    // not been waited for, and the MMA groups committed but not yet waited for
    int tma_pending = nc > 0 ? 1 : 0, pend = 0, it = 0;
    bool bailed = false;
    for (int c = 0; c < nc; ++c, ++it) {
        const int st = it & 1, gb = it & 1;
        const uint32_t par = it & 1;
        const long long bos = sbos + (long long)c * kChunk;
        const int L = min(kChunk, slen - c * kChunk);
        if (tid < 64) cp_async_wait_all();      // this chunk's g and beta
        bool ok = mbar_wait(&s.tma_bar[st], (it >> 1) & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tma_pending &= ~(1 << st);

        // ---- 1. [Q; K] K^T (H^T Q^T goes with the state update's group)
        if (warp == 0) {
            tc_fence_after();
            const uint32_t qk = smem_u32(s.qk[st]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 2 * kTile + (kk & 3) * 32;
                const uint64_t aq = desc_sw128(qk + off, 16, 1024);              // [Q; K]
                mma_bf16(t_p, aq, desc_sw128(qk + kTile + off, 16, 1024), kIdKK64, kk > 0);
            }
            mma_commit(&s.bar_q);
        }
        pend = 1;
        // the next chunk's tiles into the other stage (its last reader was the
        // previous chunk's state update), and its g and beta
        if (c + 1 < nc) {
            if (tma_thread) {
                fence_proxy_async();
                issue_tma(st ^ 1, c + 1);
            }
            tma_pending |= 1 << (st ^ 1);
            if (tid < 64) fetch_gb(st ^ 1, c + 1);
        }
        // gam = cumsum of the log decay within the chunk (warps 0-1)
        if (tid < 64) {
            const float gr = tid < L ? decay_of(g, s.graw[st][tid], h) : 0.f;
            float x = gr;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane == 31) s.wsum[warp] = x;
            named_sync(1, 64);
            if (warp == 1) x += s.wsum[0];
            s.gam[gb][tid] = x;
        }
        if (g.l2norm) row_inv_norms(s.qk[st], 2 * kTile, 128, s.rqk);
        else if (tid < 128) s.rqk[tid] = 1.f;
        __syncthreads();
        if (tid < 64) {
            const int r = tid;
            const float gl = s.gam[gb][L - 1], gr = s.gam[gb][r];
            const bool in = r < L;
            const float e = __expf(gr), rk = s.rqk[64 + r], b = in ? s.braw[st][r] : 0.f;
            s.fr[r] = in ? __expf(gl - gr) * rk : 0.f;
            s.er[gb][r] = in ? e * s.rqk[r] : 0.f;
            s.egw[gb][r] = r > 0 ? __expf(gr - s.gam[gb][r - 1]) : 1.f;
            s.eb[r] = b * e * rk;
            s.bt[r] = b;
        }
        if (c > 0) {
            tc_fence_after();
            out_epilogue(gb ^ 1);                 // the previous chunk's O
        }
        ok = mbar_wait(&s.bar_q, par, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        pend = 0;
        tc_fence_after();

        // ---- 2. A^T rows from K K^T (lanes 64-127), P from Q K^T (lanes 0-63)
        if (v >= 64) {
            // row r = v - 64 of A^T = column r of A:
            //   A[i][r] = beta_i (k^_i . k^_r) exp(gam_i - gam_r) for r < i < L
            const int r = v - 64;
            float kk[32];
            tmem_ld32(tmem_addr(t_p, warp, 32 * hs), kk);
            const float gr = s.gam[gb][r], rr = s.rqk[64 + r];
            float4 *arow = reinterpret_cast<float4 *>(s.A[r]) + 8 * hs;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 32 * hs + 4 * q + e;
                    x[e] = (i > r && i < L)
                               ? s.bt[i] * s.rqk[64 + i] * rr * kk[4 * q + e] * __expf(s.gam[gb][i] - gr)
                               : 0.f;
                }
                arow[q] = make_float4(x[0], x[1], x[2], x[3]);
            }
        } else {
            // row r = v of P: Q K^T masked to c <= r < L, times D_rc / (|q_r| |k_c|)
            const int r = v;
            float xp[32], dd[32];
            tmem_ld32(tmem_addr(t_p, warp, 32 * hs), xp);
            row_decays32(s.gam[gb], s.egw[gb], r, 32 * hs, dd);
            const float sr = s.rqk[r];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float *x = xp + 8 * q;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int cc = 32 * hs + 8 * q + e;
                    x[e] = (cc <= r && r < L) ? x[e] * dd[8 * q + e] * sr * s.rqk[64 + cc] : 0.f;
                }
                st_row8(s.p, r, 4 * hs + q, x);
            }
        }
        tc_fence_before();
        __syncthreads();

        // ---- 3. T = (I + A)^-1 by warps 0-1, then the W / u operands over A's space
        float t[32], y[16];
        if (tid < 64) solve_unit_lower64(s.A, tid, t, y, [] { named_sync(1, 64); });
        __syncthreads();
        if (tid < 64) {
            const int cown = 32 * (tid >> 5) + lane;
            store_wu_operands(bw, bu, tid, t, y, s.eb[cown], s.bt[cown], s.eb[lane], s.bt[lane]);
        }
        fence_proxy_async();
        __syncthreads();

        // ---- 4. W^T and u^T (feature rows on the MMA's M side)
        if (warp == 0) {
            tc_fence_after();
            const uint32_t kt = smem_u32(s.qk[st]) + kTile, vt = smem_u32(s.v[st]);
            const uint32_t bwa = smem_u32(bw), bua = smem_u32(bu);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                mma_bf16(t_w, desc_sw128(kt + kk * 2048, 2 * kTile, 1024),   // K^T, MN-major
                         desc_sw128(bwa + kk * 2048, kTile, 1024), kIdMM64, kk > 0);
                mma_bf16(t_uu, desc_sw128(vt + kk * 2048, kTile, 1024),      // V^T, MN-major
                         desc_sw128(bua + kk * 2048, kTile, 1024), kIdMM64, kk > 0);
            }
            mma_commit(&s.bar_w);
        }
        pend = 2;
        ok = mbar_wait(&s.bar_w, par, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        pend = 0;
        tc_fence_after();
        {
            // row v of W^T and u^T, chunk rows 32 hs .. +31 (zero past L)
            float xw[32], xv[32];
            tmem_ld32x2(tmem_addr(t_w, warp, 32 * hs), tmem_addr(t_uu, warp, 32 * hs), xw, xv);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const bool in = 32 * hs + 8 * q + e < L;
                    xw[8 * q + e] = in ? xw[8 * q + e] : 0.f;
                    xv[8 * q + e] = in ? xv[8 * q + e] : 0.f;
                }
                st_row8(s.w, v, 4 * hs + q, xw + 8 * q);
                st_row8(s.u, v, 4 * hs + q, xv + 8 * q);
            }
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();

        // ---- 5. the walk step
        if (warp == 0) {
            tc_fence_after();
            const uint32_t wt = smem_u32(s.w), hT = smem_u32(s.hT);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ah = desc_sw128(hT + (kk >> 2) * 2 * kTile + (kk & 3) * 32, 16, 1024);
                mma_bf16(t_u, ah, desc_sw128(wt + kk * 2048, 2 * kTile, 1024), kIdKM64, kk > 0);
            }
            mma_commit(&s.bar_u);
        }
        pend = 4;
        ok = mbar_wait(&s.bar_u, par, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        pend = 0;
        tc_fence_after();
        {
            // U^T = u^T - H^T W^T and U^T diag(f), rows v, chunk rows 32 hs .. +31
            float xu[32];
            tmem_ld32(tmem_addr(t_u, warp, 32 * hs), xu);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float *x = xu + 8 * q, uu[8];
                const int chunk = 4 * hs + q;
                const uint4 raw =
                    *reinterpret_cast<const uint4 *>(s.u + v * 128 + ((chunk ^ (v & 7)) << 4));
                const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(&raw);
                const float4 f0 = reinterpret_cast<const float4 *>(s.fr)[2 * chunk];
                const float4 f1 = reinterpret_cast<const float4 *>(s.fr)[2 * chunk + 1];
                const float fq[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int r = 8 * chunk + e;
                    x[e] = r < L ? __bfloat162float(bv[e]) - x[e] : 0.f;
                    uu[e] = x[e] * fq[e];
                }
                st_row8(s.uTs, v, chunk, uu);
                st_row8(s.uT, v, chunk, x);
            }
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        if (warp == 0) {
            tc_fence_after();
            const uint32_t uTs = smem_u32(s.uTs), kt = smem_u32(s.qk[st]) + kTile;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(t_dh, desc_sw128(uTs + kk * 32, 16, 1024),
                         desc_sw128(kt + kk * 2048, 2 * kTile, 1024), kIdDH, kk > 0);   // K, MN-major
            const uint32_t ua = smem_u32(s.uT), pp = smem_u32(s.p);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(t_pu(gb), desc_sw128(ua + kk * 32, 16, 1024),
                         desc_sw128(pp + kk * 32, 16, 1024), kIdKK64, kk > 0);
            // H^T Q^T from this chunk's start state, which the update below overwrites
            // only after this group completes
            const uint32_t hT = smem_u32(s.hT), qk = smem_u32(s.qk[st]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 2 * kTile + (kk & 3) * 32;
                mma_bf16(t_qh(gb), desc_sw128(hT + off, 16, 1024), desc_sw128(qk + off, 16, 1024),
                         kIdKK64, kk > 0);
            }
            mma_commit(&s.bar_dh);
        }
        pend = 8;
        ok = mbar_wait(&s.bar_dh, par, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        pend = 0;
        tc_fence_after();
        {
            const float el = __expf(s.gam[gb][L - 1]);
            float d[64];
            tmem_ld32x2(tmem_addr(t_dh, warp, 64 * hs), tmem_addr(t_dh, warp, 64 * hs + 32), d,
                        d + 32);
#pragma unroll
            for (int jj = 0; jj < 64; ++jj) Hr[jj] = el * Hr[jj] + d[jj];
        }
        st_row64(s.hT + hs * 2 * kTile, v, Hr);
        pbos = bos;
        pL = L;
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
    }
    if (!bailed && nc > 0) {
        tc_fence_after();
        out_epilogue((it - 1) & 1);               // the last chunk's O
    }
    if (tid < 64) cp_async_wait_all();          // a g / beta prefetch still in flight after a bail
    if (bailed) {
        if (tid == 0) {
            for (int st = 0; st < 2; ++st)
                if (tma_pending & (1 << st))
                    mbar_drain(&s.tma_bar[st], ((it + (st != (it & 1))) >> 1) & 1);
            if (pend & 1) mbar_drain(&s.bar_q, it & 1);
            if (pend & 2) mbar_drain(&s.bar_w, it & 1);
            if (pend & 4) mbar_drain(&s.bar_u, it & 1);
            if (pend & 8) mbar_drain(&s.bar_dh, it & 1);
        }
    } else if (a.final_state) {
        float *dst = a.final_state + ((long long)n * H + h) * kD * kD;
#pragma unroll
        for (int i = 0; i < 64; ++i) dst[(64 * hs + i) * kD + v] = Hr[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

bool full_forward_fits(const Plan &p) {
    return !p.cp && (long long)p.g.N * p.g.H * 4 >= 3ll * std::max(p.sms, 1);
}

cudaError_t full_forward(const Plan &p, cudaStream_t s) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    const Geo &g = p.g;
    const long long tokens = (long long)g.B * g.T;
    CUtensorMap mq, mk, mv;
    if ((e = make_map(&mq, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mk, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mv, g.v, tokens, g.H)) != cudaSuccess) return e;
    const size_t smem = sizeof(FullSmem) + 1024;
    if ((e = cudaFuncSetAttribute(tc_full_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)smem)) != cudaSuccess)
        return e;
    FullArgs a{};
    a.h0 = p.h0;
    a.final_state = p.final_state;
    a.o = (__nv_bfloat16 *)p.o;
    prof_before("tc_full_fwd", s);
    if ((e = launch_pdl(tc_full_kernel, dim3(g.N * g.H, 1, 1), dim3(256), smem, s, mq, mk, mv, g,
                        a)) != cudaSuccess)
        return e;
    prof_after(s);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace gdn
