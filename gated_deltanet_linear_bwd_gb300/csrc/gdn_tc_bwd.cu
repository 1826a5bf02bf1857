// gdn_tc_bwd.cu -- tensor-core (tcgen05 + TMA) backward pieces for bf16
// q/k/v with K = V = 128.
//
// Reverse walk of the state gradient, per (sequence or segment, head),
// chunks last to first.  With dH the gradient at a chunk's end, held as
// dH^T (V rows x K columns, one row per thread, fp32 registers):
//   X^T  = dH^T K^T                      (K dH)^T
//   dU^T = Y^T + X^T diag(f),            f = exp(gam_L - gam)
//   dH^T <- exp(gam_L) dH^T + dO^T Qs - dU^T W
// where the parts that do not depend on dH come from the chunk-parallel
// intra kernel run first, or, without CP when the walk's CTAs fill the GPU,
// are formed inside the walk's own loop (its fused variant):
//   P    = scale (Q K^T .* lower_incl .* D),  Y^T = dO^T P
//   Qs   = diag(scale e^gam) Q
// The segment map of the walk ([A' | B'], A' the transpose of the forward
// map) is walked the same way with dO = 0 on its A' columns.
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

// kind::f16 descriptor with A negated (bit 13).
constexpr uint32_t idesc_neg_a(uint32_t d) { return d | (1u << 13); }

constexpr uint32_t kIdKK64 = idesc_bf16(128, 64, false, false);   // K-major A, K-major B
constexpr uint32_t kIdMM64 = idesc_bf16(128, 64, true, true);     // MN-major A and B, N = 64
constexpr uint32_t kIdMM128 = idesc_bf16(128, 128, true, true);   // MN-major A and B, N = 128
constexpr uint32_t kIdKK128Neg = idesc_neg_a(idesc_bf16(128, 128, false, false));

template <typename F>
cudaError_t set_smem(F kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

// ------------------------------------------------------------------ intra kernel
struct IntraSmem {
    uint8_t qk[4 * kTile];         // [dk half][Q rows 0-63, K rows 64-127][128 B]
    uint8_t dO[2 * kTile];         // [dv half][64 rows][128 B]
    uint8_t qs[2 * kTile];         // Qs, [dk half][64 rows][128 B]
    uint8_t yT[2 * kTile];         // Y^T, [128 rows v][64 chunk rows]
    uint8_t p[kTile];              // P rows r (scale included)
    float gam[64];
    float rqk[128];            // q, k normalised here: 1 / |q_r| at r, 1 / |k_r| at 64 + r
    float gpre[64];            // the next item's gam, fetched during the current one
    float eg[64];              // e^(gam_j - gam_{j-1})
    uint64_t load_bar[2], mma_bar; // loads: {q, k}, {dO}
    uint32_t tmem_base;
};
}  // namespace

// Persistent over (chunk, head) items with a stride of the grid, two CTAs
// per SM.  Per item, 256 threads: P on lanes 0-63 (row r = v), Qs rows by
// threads 128-191, then Y^T = dO^T P feature-major (thread: row v, column
// half hs); Qs and Y^T leave by TMA from shared memory.  The next item's
// q, k are fetched as soon as P and Qs are done with them, its dO once
// Y^T's product has read the current one.
__global__ void __launch_bounds__(256, 2)
tc_bwd_intra_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_qs,
                    const __grid_constant__ CUtensorMap tm_y, Geo g, const float *ws_gam,
                    int n_items) {
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    IntraSmem &s = *reinterpret_cast<IntraSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, H = g.H;
    const int v = tid & 127, hs = tid >> 7, c0 = 32 * hs, cq = c0 >> 3;

    auto item_ref = [&](int i, int &ci, int &hh, ChunkRef &r) -> bool {
        if (i >= n_items) return false;
        ci = i / H;
        hh = i % H;
        return chunk_ref(g, ci, r);
    };
    auto load_qk = [&](int hh, long long bos) {
        mbar_arrive_expect_tx(&s.load_bar[0], 4 * kTile);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(s.qk + half * 2 * kTile, &tm_q, &s.load_bar[0], half * 64, hh, (int)bos);
            tma_load_3d(s.qk + half * 2 * kTile + kTile, &tm_k, &s.load_bar[0], half * 64, hh,
                        (int)bos);
        }
    };
    auto load_do = [&](int hh, long long bos) {
        mbar_arrive_expect_tx(&s.load_bar[1], 2 * kTile);
        tma_load_3d(s.dO, &tm_do, &s.load_bar[1], 0, hh, (int)bos);
        tma_load_3d(s.dO + kTile, &tm_do, &s.load_bar[1], 64, hh, (int)bos);
    };

    if (tid == 0) {
        mbar_init(&s.load_bar[0], 1);
        mbar_init(&s.load_bar[1], 1);
        mbar_init(&s.mma_bar, 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, 128);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = s.tmem_base;
    const uint32_t t_p = tb, t_y = tb + 64;

    int item = blockIdx.x, ci = 0, h = 0;
    ChunkRef cr;
    bool have = item_ref(item, ci, h, cr);
    int issued[2] = {0, 0};                   // loads issued per group (uniform bookkeeping)
    if (have) {
        if (tid == 0) {
            load_qk(h, cr.bos);
            load_do(h, cr.bos);
        }
        issued[0] = issued[1] = 1;
    }
    int it = 0, mma_n = 0;
    bool bailed = false;
    while (have) {
        const int L = cr.len;
        const long long bos = cr.bos;
        int ci_n = 0, h_n = 0;
        ChunkRef cr_n;
        const bool have_next = item_ref(item + (int)gridDim.x, ci_n, h_n, cr_n);
        if (tid == 0) bulk_wait_read_but_newest();   // the previous item's Qs store has read Qs
        tc_fence_before();
        __syncthreads();
        if (tid < 64) {
            // gam of this item: fetched during the previous one (cp.async), else now
            if (it > 0) cp_async_wait_all();
            s.gam[tid] = it > 0 ? s.gpre[tid] : (tid < L ? ws_gam[(bos + tid) * H + h] : 0.f);
        }
        bool ok = mbar_wait(&s.load_bar[0], it & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        ++mma_n;
        if (tid >= 192) {
            const int j = tid - 192;
            s.eg[j] = j > 0 ? __expf(s.gam[j] - s.gam[j - 1]) : 1.f;
        }
        // every thread is past the copy of gpre above: the next item's gam can come
        if (tid < 64 && have_next)
            cp_async4(&s.gpre[tid], ws_gam + (cr_n.bos + min(tid, cr_n.len - 1)) * H + h_n,
                      tid < cr_n.len);
        if (warp == 0) {
            tc_fence_after();
            const uint32_t qk = smem_u32(s.qk);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
                mma_bf16(t_p, desc_sw128(qk + half * 2 * kTile + sub, 16, 1024),
                         desc_sw128(qk + half * 2 * kTile + kTile + sub, 16, 1024), kIdKK64, kk > 0);
            }
            mma_commit(&s.mma_bar);
        }
        if (g.l2norm) {
            // 1 / |q_r| (stacked rows 0-63) and 1 / |k_r| (rows 64-127)
            row_inv_norms(s.qk, 2 * kTile, 128, s.rqk);
            __syncthreads();
        }
        if (tid >= 128 && tid < 192) {
            // row r of Qs = diag(scale e^gam (x 1/|q_r|)) Q, both dk halves
            const int r = tid - 128;
            const float f = r < L ? g.scale * __expf(s.gam[r]) * (g.l2norm ? s.rqk[r] : 1.f) : 0.f;
#pragma unroll 1
            for (int q = 0; q < 16; ++q) {
                const int half = q >> 3, chunk = q & 7;
                float x[8];
                const uint4 raw = *reinterpret_cast<const uint4 *>(
                    s.qk + half * 2 * kTile + r * 128 + ((chunk ^ (r & 7)) << 4));
                const __nv_bfloat16 *bb = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[e] = f * __bfloat162float(bb[e]);
                st_row8(s.qs + half * kTile, r, chunk, x);
            }
        }
        ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tc_fence_after();
        if (v < 64) {
            // P row r = v, columns c0 .. c0+31, scale included
            const int r = v;
            const float sr = g.l2norm ? s.rqk[r] : 1.f;
            float xs[32], dd[32];
            tmem_ld32(tmem_addr(t_p, warp, c0), xs);
            row_decays32(s.gam, s.eg, r, c0, dd);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float *x = xs + 8 * q;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = c0 + 8 * q + e;
                    x[e] = (c <= r && r < L) ? g.scale * x[e] * dd[8 * q + e] * sr *
                                                   (g.l2norm ? s.rqk[64 + c] : 1.f)
                                             : 0.f;
                }
                st_row8(s.p, r, cq + q, x);
            }
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            // Qs is complete: store it while Y^T is computed; q, k are free for the next item
            const int row = (int)(((long long)ci * H + h) * 2 * 64);
            tma_store_2d(&tm_qs, s.qs, 0, row);
            tma_store_2d(&tm_qs, s.qs + kTile, 0, row + 64);
            bulk_commit();
            if (have_next) load_qk(h_n, cr_n.bos);
        }
        if (have_next) ++issued[0];
        ok = mbar_wait(&s.load_bar[1], it & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t dO = smem_u32(s.dO), pp = smem_u32(s.p);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(t_y, desc_sw128(dO + kk * 2048, kTile, 1024),    // dO^T, MN-major
                         desc_sw128(pp + kk * 2048, kTile, 1024), kIdMM64, kk > 0);   // P, MN-major
            mma_commit(&s.mma_bar);
        }
        // the previous item's Y^T store (older than this item's Qs store) has read Y^T
        if (tid == 0) bulk_wait_read_but_newest();
        ok = mbar_wait(&s.mma_bar, 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        if (tid == 0 && have_next) {
            fence_proxy_async();
            load_do(h_n, cr_n.bos);           // dO's last reader was the product above
        }
        if (have_next) ++issued[1];
        tc_fence_after();
        {
            float xs[32];
            tmem_ld32(tmem_addr(t_y, warp, c0), xs);
#pragma unroll
            for (int q = 0; q < 4; ++q) st_row8(s.yT, v, cq + q, xs + 8 * q);
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            tma_store_2d(&tm_y, s.yT, 0, (int)(((long long)ci * H + h) * kD));
            bulk_commit();
        }
        item += (int)gridDim.x;
        ci = ci_n;
        h = h_n;
        cr = cr_n;
        have = have_next;
        ++it;
    }
    if (bailed && tid == 0) {
        for (int grp = 0; grp < 2; ++grp)
            if (issued[grp] > 0) mbar_drain(&s.load_bar[grp], (issued[grp] - 1) & 1);
        if (mma_n > 0) mbar_drain(&s.mma_bar, (mma_n - 1) & 1);
    }
    if (tid < 64) cp_async_wait_all();        // a prefetch still in flight after a bail
    if (tid == 0) bulk_wait_read();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 128);
}

// ------------------------------------------------------------------ reverse walk
namespace {
// kDOut: the reverse walk (gradient states, dU); kDMap: segment maps;
// kDFused: the reverse walk that forms the chunk's P, Qs and Y^T = dO^T P
// itself from q, k, dO instead of reading the intra kernel's tiles.
enum { kDOut = 0, kDMap = 1, kDFused = 2 };

template <int MODE>
struct DWalkSmem {
    static constexpr bool kF = MODE == kDFused;
    uint8_t k[2][kF ? 4 * kTile : 2 * kTile];   // per stage: K, [dk half][64 rows][128 B];
                                                 // fused: [dk half][Q rows | K rows][128 B]
    uint8_t w[2][2 * kTile];       // per stage: W^T, [128 rows k][64 chunk rows]  K-major B
    uint8_t dO[2][2 * kTile];      // per stage: dO, [dv half][64 rows][128 B]
    uint8_t qs[kF ? 1 : 2][2 * kTile];           // per stage: Qs, [dk half][64 rows][128 B]
    uint8_t y[kF ? 1 : 2][kF ? 1024 : 2 * kTile];   // per stage: Y^T, [128 rows v][64 chunk rows]
    uint8_t p[kF ? kTile : 1024];   // P rows r (fused)
    uint8_t dhT[4 * kTile];        // dH^T: [k half][128 rows v][128 B]   K-major A
    uint8_t duT[2 * kTile];        // dU^T: [128 rows v][64 chunk rows]    K-major A
    float gam[2][64];
    alignas(16) float fr[64];      // exp(gam_L - gam_r) (x 1/|k_r|), 0 past L
    float rqk[128];                // q, k normalised here: 1 / |q_r| at r (fused walk),
                                   // 1 / |k_r| at 64 + r
    float egd[64];                 // exp(gam_j - gam_{j-1}) of the current chunk (fused)
    uint64_t tma_bar[2], bar_x, bar_z, bar_q, bar_y;
    uint32_t tmem_base;
};

struct TcDWalkArgs {
    const float *ws_gam;
    const float *dht;         // [N, H, K, V] nullable
    const float *seg_end;     // [segs, H, K, V] (CP): gradient at each segment's end
    float *dh0;               // [N, H, K, V] nullable
    float *maps;              // [segs, H, K, K+V] (kDMap)
    int cb_base;              // kDMap: 1 = only the B' columns (A' comes from the forward's maps)
    int cp;
};

struct DWalkMaps {
    CUtensorMap q, k, w, dO, qs, y, dhc, du;
};
}  // namespace

// 256 threads: thread t owns row v = t % 128 of dH^T (TMEM lane v) and the
// column half hs = t / 128; warps w and w + 4 split each epilogue's columns.
// Per chunk: X^T = dH^T K^T (first MMA group; dO^T Qs is issued behind it
// into the state-update accumulator), dU^T = Y^T + X^T diag(f), then
// -dU^T W onto that accumulator (second group) and the dH^T update.  The
// gradient at each chunk's end (bf16 dH^T) and dU^T leave by TMA stores.
template <int MODE>
__global__ void __launch_bounds__(256, 1)
tc_dwalk_kernel(const __grid_constant__ DWalkMaps m, Geo g, TcDWalkArgs a) {
    pdl_enter();
    typedef DWalkSmem<MODE> S;
    constexpr bool fused = MODE == kDFused;
    constexpr bool kOut = MODE != kDMap;                 // a gradient-state walk
    constexpr int kKOff = fused ? kTile : 0;             // K rows inside a dk half block
    constexpr uint32_t kKHalf = fused ? 2 * kTile : kTile;
    extern __shared__ uint8_t smem_raw[];
    S &s = *reinterpret_cast<S *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, cb = blockIdx.z + a.cb_base, H = g.H;
    int h = blockIdx.y;
    const int v = tid & 127, hs = tid >> 7;
    int n, j = 0, nseg = 1;
    if (a.cp) {
        if (!seg_ref(g, blockIdx.x, n, j)) return;
        nseg = seq_nsegs(g, n);
    } else {
        walk_unit(g, blockIdx.x, n, h);
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
    const bool tma_thread = tid == 255;

    auto issue_tma = [&](int st, int c) {
        const int tok0 = (int)(sbos + (long long)c * kChunk);
        const int trow = (int)(((long long)(cbase + c) * H + h) * kD);
        mbar_arrive_expect_tx(&s.tma_bar[st], (fused ? 8 : use_do ? 10 : 4) * kTile);
        tma_load_3d(s.k[st] + kKOff, &m.k, &s.tma_bar[st], 0, h, tok0);
        tma_load_3d(s.k[st] + kKOff + kKHalf, &m.k, &s.tma_bar[st], 64, h, tok0);
        tma_load_2d(s.w[st], &m.w, &s.tma_bar[st], 0, trow);
        if (use_do) {
            tma_load_3d(s.dO[st], &m.dO, &s.tma_bar[st], 0, h, tok0);
            tma_load_3d(s.dO[st] + kTile, &m.dO, &s.tma_bar[st], 64, h, tok0);
        }
        if (fused) {
            tma_load_3d(s.k[st], &m.q, &s.tma_bar[st], 0, h, tok0);
            tma_load_3d(s.k[st] + kKHalf, &m.q, &s.tma_bar[st], 64, h, tok0);
        } else if (use_do) {
            tma_load_2d(s.qs[st], &m.qs, &s.tma_bar[st], 0, trow);
            tma_load_2d(s.qs[st] + kTile, &m.qs, &s.tma_bar[st], 0, trow + 64);
            tma_load_2d(s.y[st], &m.y, &s.tma_bar[st], 0, trow);
        }
    };

    // the first chunk's tiles are requested at once, so that their latency
    // overlaps the start gradient's load
    if (tid == 0) {
        mbar_init(&s.tma_bar[0], 1);
        mbar_init(&s.tma_bar[1], 1);
        mbar_init(&s.bar_x, 1);
        mbar_init(&s.bar_z, 1);
        mbar_init(&s.bar_q, 1);
        mbar_init(&s.bar_y, 1);
        fence_barrier_init();
        if (c1 > c0) issue_tma(0, c1 - 1);
    }
    constexpr uint32_t kTmemCols = fused ? 512 : 256;
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    float dH[64];     // dk half hs of row v of dH^T (= column v of dH)
    {
        const float *src = nullptr;
        if (kOut) {
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
    const uint32_t t_x = tbase, t_z = tbase + 128;
    const uint32_t t_p = tbase + 64, t_y = tbase + 256;      // fused: P, Y^T

    // one commit per barrier per chunk: every barrier's parity is the chunk
    // iteration's; `pend` marks groups committed in this iteration, not yet waited
    int it = 0, tma_pending = 0, pend = 0;
    bool bailed = false;
    if (c1 > c0) tma_pending |= 1;            // issued above
    for (int c = c1 - 1; c >= c0; --c, ++it) {
        const int st = it & 1;
        const uint32_t par = it & 1;
        const long long bos = sbos + (long long)c * kChunk;
        const int L = min(kChunk, slen - c * kChunk);
        const int trow = (int)(((long long)(cbase + c) * H + h) * kD);
        pend = 0;
        // gam of chunk c - 1 (a full chunk) into the other buffer, asynchronously
        if (c - 1 >= c0 && tid < 64)
            cp_async4(&s.gam[st ^ 1][tid], a.ws_gam + (bos - kChunk + tid) * H + h, true);
        bool ok = mbar_wait(&s.tma_bar[st], (it >> 1) & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tma_pending &= ~(1 << st);
        if (warp == 0) {
            tc_fence_after();
            const uint32_t kt = smem_u32(s.k[st]), dhT = smem_u32(s.dhT);
            if (fused) {
                // [Q; K] K^T first, on its own barrier: the P epilogue that reads it
                // comes before X^T's, which then completes under it
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kKHalf + (kk & 3) * 32;
                    mma_bf16(t_p, desc_sw128(kt + off, 16, 1024),
                             desc_sw128(kt + kKOff + off, 16, 1024), kIdKK64, kk > 0);
                }
                mma_commit(&s.bar_q);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t half = kk >> 2, sub = (kk & 3) * 32;
                mma_bf16(t_x, desc_sw128(dhT + half * 2 * kTile + sub, 16, 1024),
                         desc_sw128(kt + kKOff + half * kKHalf + sub, 16, 1024), kIdKK64, kk > 0);
            }
            mma_commit(&s.bar_x);
            if (!fused && use_do) {
                const uint32_t dO = smem_u32(s.dO[st]), qs = smem_u32(s.qs[st]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(t_z, desc_sw128(dO + kk * 2048, kTile, 1024),   // dO^T, MN-major
                             desc_sw128(qs + kk * 2048, kTile, 1024), kIdMM128, kk > 0);
            }
        }
        pend = fused ? 5 : 1;
        // while the products run, the last warp requests chunk c - 1 (into the
        // stage the previous chunk used) and stores the gradient at this chunk's end
        if (c - 1 >= c0) {
            if (tma_thread) {
                fence_proxy_async();
                issue_tma(st ^ 1, c - 1);
            }
            tma_pending |= 1 << (st ^ 1);
        }
        if (kOut && tma_thread) {
            // the bf16 dH^T tile, by TMA
            tma_store_2d(&m.dhc, s.dhT, 0, 2 * trow);
            tma_store_2d(&m.dhc, s.dhT + 2 * kTile, 0, 2 * trow + kD);
            bulk_commit();
        }
        if (g.l2norm) {
            // 1 / |k_r| (and, in the fused walk, whose stage stacks Q rows 0-63
            // over K rows 64-127, 1 / |q_r|) from the stage's rows
            if (fused)
                row_inv_norms(s.k[st], kKHalf, 128, s.rqk);
            else
                row_inv_norms(s.k[st] + kKOff, kKHalf, 64, s.rqk + 64);
            __syncthreads();
        }
        if (tid < 64) {
            const float gl = s.gam[st][L - 1];
            s.fr[tid] = tid < L ? __expf(gl - s.gam[st][tid]) * (g.l2norm ? s.rqk[64 + tid] : 1.f) : 0.f;
            if (fused) s.egd[tid] = tid > 0 ? __expf(s.gam[st][tid] - s.gam[st][tid - 1]) : 1.f;
        }
        if (fused) {
            ok = mbar_wait(&s.bar_q, par, g.spin_limit, g.status);
            if (__syncthreads_or(!ok)) { bailed = true; break; }
            pend &= ~4;
            tc_fence_after();
            if (v < 64) {
                // P row r = v, columns 32 hs .. +31: scale Q K^T D, masked to c <= r < L
                // (and 1 / (|q_r| |k_c|) when q, k are normalised here)
                const int r = v;
                float xp[32], dd[32];
                tmem_ld32(tmem_addr(t_p, warp, 32 * hs), xp);
                row_decays32(s.gam[st], s.egd, r, 32 * hs, dd);
                const float sr = g.scale * (g.l2norm ? s.rqk[r] : 1.f);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float *x = xp + 8 * q;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int c = 32 * hs + 8 * q + e;
                        const float sc = g.l2norm ? sr * s.rqk[64 + c] : sr;
                        x[e] = (c <= r && r < L) ? sc * x[e] * dd[8 * q + e] : 0.f;
                    }
                    st_row8(s.p, r, 4 * hs + q, x);
                }
            } else {
                // meanwhile the other warps form Qs = diag(scale e^gam) Q (zero past L)
                // from the Q rows of the stage: thread u = 0..127 scales eight 16-byte
                // pieces of row u % 64
                const int u = (tid & 63) + 64 * (tid >> 7), r = u & 63;
                const float f = r < L ? g.scale * __expf(s.gam[st][r]) * (g.l2norm ? s.rqk[r] : 1.f)
                                      : 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int pc = 8 * (u >> 6) + i, half = pc >> 3, chunk = pc & 7;
                    const uint4 raw = *reinterpret_cast<const uint4 *>(
                        s.k[st] + half * kKHalf + r * 128 + ((chunk ^ (r & 7)) << 4));
                    const __nv_bfloat16 *bb = reinterpret_cast<const __nv_bfloat16 *>(&raw);
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = f * __bfloat162float(bb[e]);
                    st_row8(s.qs[0] + half * kTile, r, chunk, x);
                }
            }
            tc_fence_before();
            fence_proxy_async();
            __syncthreads();
            if (warp == 0) {
                // Y^T = dO^T P, and dO^T Qs into the update accumulator
                tc_fence_after();
                const uint32_t dO = smem_u32(s.dO[st]), pp = smem_u32(s.p), qs = smem_u32(s.qs[0]);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    mma_bf16(t_y, desc_sw128(dO + kk * 2048, kTile, 1024),    // dO^T, MN-major
                             desc_sw128(pp + kk * 2048, kTile, 1024), kIdMM64, kk > 0);   // P, MN-major
                    mma_bf16(t_z, desc_sw128(dO + kk * 2048, kTile, 1024),
                             desc_sw128(qs + kk * 2048, kTile, 1024), kIdMM128, kk > 0);
                }
                mma_commit(&s.bar_y);
            }
            pend |= 8;
        }
        // the previous chunk's dU^T store has read its tile (this chunk's dH^T store,
        // the newest group, may go on)
        if (tma_thread) bulk_wait_read_but_newest();
        ok = mbar_wait(&s.bar_x, par, g.spin_limit, g.status);
        if (fused) ok = mbar_wait(&s.bar_y, par, g.spin_limit, g.status) && ok;
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        pend = 0;
        tc_fence_after();
        // dU^T row v, chunk rows 32*hs .. +31 (one TMEM load, groups of 8): Y^T + X^T diag(f)
        float xs[32], ys[32];
        if (fused)
            tmem_ld32x2(tmem_addr(t_x, warp, 32 * hs), tmem_addr(t_y, warp, 32 * hs), xs, ys);
        else
            tmem_ld32(tmem_addr(t_x, warp, 32 * hs), xs);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float *x = xs + 8 * q;
            const int chunk = 4 * hs + q;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (use_do && !fused)
                raw = *reinterpret_cast<const uint4 *>(s.y[st] + v * 128 + ((chunk ^ (v & 7)) << 4));
            const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(&raw);
            // f of rows 8 chunk .. +7 as two 16-byte broadcast reads
            const float4 f0 = reinterpret_cast<const float4 *>(s.fr)[2 * chunk];
            const float4 f1 = reinterpret_cast<const float4 *>(s.fr)[2 * chunk + 1];
            const float fq[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = 8 * chunk + e;
                const float y = fused ? ys[8 * q + e] : __bfloat162float(bv[e]);
                x[e] = r < L ? y + fq[e] * x[e] : 0.f;
            }
            st_row8(s.duT, v, chunk, x);
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        if (kOut && tma_thread) {
            tma_store_2d(&m.du, s.duT, 0, trow);
            bulk_commit();
        }
        if (warp == 0) {
            tc_fence_after();
            const uint32_t du = smem_u32(s.duT), wt = smem_u32(s.w[st]);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
                mma_bf16(t_z, desc_sw128(du + kk * 32, 16, 1024),
                         desc_sw128(wt + kk * 32, 16, 1024),             // W^T, K-major
                         kIdKK128Neg, (use_do || kk > 0) ? 1u : 0u);
            mma_commit(&s.bar_z);
        }
        pend = 2;
        // the dH^T store has read its tile (the dU^T store, the newest group, may
        // go on until the next chunk's dU epilogue)
        if (tma_thread) bulk_wait_read_but_newest();
        ok = mbar_wait(&s.bar_z, par, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        pend = 0;
        tc_fence_after();
        {
            const float el = __expf(s.gam[st][L - 1]);
            float z[64];
            tmem_ld32x2(tmem_addr(t_z, warp, 64 * hs), tmem_addr(t_z, warp, 64 * hs + 32), z,
                        z + 32);
#pragma unroll
            for (int jj = 0; jj < 64; ++jj) dH[jj] = el * dH[jj] + z[jj];
        }
        st_row64(s.dhT + hs * 2 * kTile, v, dH);
        if (tid < 64) cp_async_wait_all();
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
    }

    if (tma_thread) bulk_wait_read();
    if (tid < 64) cp_async_wait_all();    // a gam prefetch may still be in flight after a bail
    if (bailed) {
        if (tid == 0) {
            for (int st = 0; st < 2; ++st)
                if (tma_pending & (1 << st))
                    mbar_drain(&s.tma_bar[st], ((it + (st != (it & 1))) >> 1) & 1);
            if (pend & 1) mbar_drain(&s.bar_x, it & 1);
            if (pend & 4) mbar_drain(&s.bar_q, it & 1);
            if (pend & 8) mbar_drain(&s.bar_y, it & 1);
            if (pend & 2) mbar_drain(&s.bar_z, it & 1);
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
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// ------------------------------------------------------------------ host side
cudaError_t backward(const Plan &p, cudaStream_t s, bool have_ctx) {
    cudaError_t e = simt::tables(p, s);
    if (e != cudaSuccess) return e;
    if (!have_ctx && (e = recompute_states(p, s)) != cudaSuccess) return e;
    if ((e = encoder()) != cudaSuccess) return e;
    const Geo &g = p.g;
    const long long tokens = (long long)g.B * g.T;
    const long long tile_rows = (long long)p.max_chunks * g.H * kD;
    DWalkMaps m;
    if ((e = make_map(&m.q, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&m.k, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&m.dO, p.d_o, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.w, p.ws.w, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.qs, p.ws.qs, tile_rows, 64)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.y, p.ws.yt, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.dhc, p.ws.dhc, 2 * tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&m.du, p.ws.du, tile_rows)) != cudaSuccess) return e;

    // Without CP, when the reverse walk's CTAs fill at least three quarters of
    // the SMs, the walk forms P, Qs and Y^T itself and the chunk-parallel intra
    // kernel is skipped: its work then costs the walk less than the separate
    // pass (the rule of the forward's fused output walk).
    const bool fuse_intra = !p.cp && 4 * g.N * g.H >= 3 * std::max(p.sms, 1);
    if (!fuse_intra) {
        const size_t ismem = sizeof(IntraSmem) + 1024;
        if ((e = set_smem(tc_bwd_intra_kernel, ismem)) != cudaSuccess) return e;
        prof_before("tc_bwd_intra", s);
        const int n_items = p.max_chunks * g.H;
        if ((e = launch_pdl(tc_bwd_intra_kernel, dim3(std::min(n_items, 2 * std::max(p.sms, 1))),
                            dim3(256), ismem, s, m.q, m.k, m.dO, m.qs, m.y, g, p.ws.gam,
                            n_items)) != cudaSuccess)
            return e;
        prof_after(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }

    const size_t smem = sizeof(DWalkSmem<kDOut>) + 1024;
    const size_t map_smem = sizeof(DWalkSmem<kDMap>) + 1024;
    const size_t fused_smem = sizeof(DWalkSmem<kDFused>) + 1024;
    if ((e = set_smem(tc_dwalk_kernel<kDOut>, smem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_dwalk_kernel<kDMap>, map_smem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_dwalk_kernel<kDFused>, fused_smem)) != cudaSuccess) return e;
    TcDWalkArgs a{};
    a.ws_gam = p.ws.gam;
    a.dht = p.dht;
    a.dh0 = p.dh0;
    if (p.cp) {
        a.cp = 1;
        a.maps = p.ws.maps;
        a.seg_end = p.ws.seg_state;
        // with the forward's A maps saved, A'_j = A_j^T and only the B' half runs
        const bool fwd_a = have_ctx && p.ws.fwd_maps != nullptr;
        a.cb_base = fwd_a ? 1 : 0;
        prof_before("tc_dwalk_map", s);
        if ((e = launch_pdl(tc_dwalk_kernel<kDMap>, dim3(p.max_segs, g.H, fwd_a ? 1 : 2), dim3(256),
                            map_smem, s, m, g, a)) != cudaSuccess)
            return e;
        prof_after(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        a.cb_base = 0;
        if ((e = simt::cp_rscan(p, s, fwd_a ? p.ws.fwd_maps : nullptr)) != cudaSuccess) return e;
        prof_before("tc_dwalk_out", s);
        if ((e = launch_pdl(tc_dwalk_kernel<kDOut>, dim3(p.max_segs, g.H, 1), dim3(256), smem, s,
                            m, g, a)) != cudaSuccess)
            return e;
        prof_after(s);
    } else if (fuse_intra) {
        prof_before("tc_dwalk_fused", s);
        if ((e = launch_pdl(tc_dwalk_kernel<kDFused>, dim3(g.N * g.H, 1, 1), dim3(256), fused_smem, s,
                            m, g, a)) != cudaSuccess)
            return e;
        prof_after(s);
    } else {
        prof_before("tc_dwalk_out", s);
        if ((e = launch_pdl(tc_dwalk_kernel<kDOut>, dim3(g.N * g.H, 1, 1), dim3(256), smem, s,
                            m, g, a)) != cudaSuccess)
            return e;
        prof_after(s);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return local_grads(p, s);
}

}  // namespace tc
}  // namespace gdn
