// gdn_tc_fwd.cu -- tensor-core (tcgen05 + TMA) forward kernels for bf16
// q/k/v with K = V = 128.
//
// Orientation: every product is issued with M = 128 by putting the feature
// dimension (K or V) on the MMA's M side and the 64 chunk rows on N.  The
// walking state is held as H^T (V rows x K columns), one row per thread, in
// fp32 registers; its bf16 copy in shared memory is the A operand of the
// state products.  TMEM lane t is thread t's row.
//
// Prep kernel (chunk-parallel, two chunks per CTA):
//   [Ka; Kb] [Ka; Kb]^T                -> the two 64x64 K K^T blocks
//   A = strict_lower(diag(beta) K K^T .* D),  T = (I + A)^-1 (CUDA cores,
//   in 32 x 32 blocks)
//   W^T = K^T (diag(beta e) T^T),  u^T = V^T (diag(beta) T^T)
// Walk kernel (per sequence or segment, sequential over chunks; the state
// recurrence, every chunk's start state stored for the output kernel):
//   U^T = u^T - H^T W^T                 (state product)
//   dH^T = (U^T diag(f)) K              H <- exp(gam_L) H + dH,  f = exp(gam_L - gam)
// Its fused variant also forms each chunk's O inside the loop, so that no
// output pass runs, when the walk's CTAs fill the GPU (host side, below).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>

#include "gdn_common.cuh"
#include "gdn_internal.h"
#include "tc_ptx.cuh"
#include "gdn_tc_solve.cuh"

namespace gdn {
namespace tc {

constexpr int kD = 128;           // K = V = 128 on this path
constexpr int kTile = 8192;       // one 64-row x 128-byte swizzled box
constexpr uint32_t kIdescKK = idesc_bf16(128, 128, false, false);
constexpr uint32_t kIdescPrepMN = idesc_bf16(128, 64, true, true);

// ------------------------------------------------------------------ prep
struct PrepSmem {
    uint8_t k[4 * kTile];          // [dk half][rows 0-63 chunk a, 64-127 chunk b][128 B]
    uint8_t v[4 * kTile];          // same for v
    float A[2][64][68];            // A^T per chunk (row j = column j of strict-lower A); rows padded
                                   // to 272 bytes so that 32 threads writing their own rows hit
                                   // every bank; reused for bw/bu below
    alignas(16) float gam[2][64], bet[2][64], brk[2][64], eg[2][64], wsum[4];   // eg: e^(g_i)
    float gpre[2][64], bpre[2][64];  // g and beta of the item, fetched during the previous one
    uint64_t k_bar, v_bar, mma_bar;
    uint32_t tmem_base;
};

// Inclusive cumsum of 64 values held one per thread by two consecutive warps.
__device__ __forceinline__ float scan64(float x, float *wsum) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp & 1) x += wsum[warp - 1];
    return x;
}

// Persistent over (chunk pair, head) items with a stride of the grid, two
// CTAs per SM.  The next item's K tile is fetched as soon as the W/u products
// have read the current one, its V tile at the start of its turn; W^T and u^T
// leave by TMA store from the dead A region and the dead V tile.
__global__ void __launch_bounds__(128, 2)
tc_prep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
               const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
               Geo g, float *ws_gam, __nv_bfloat16 *ws_t, int n_items) {
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    PrepSmem &s = *reinterpret_cast<PrepSmem *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, H = g.H;
    const int ch = tid >> 6, r = tid & 63;
    uint8_t *stage = reinterpret_cast<uint8_t *>(&s.A[0][0][0]);   // 32 KB after the W/u products

    // item i: chunks 2 (i / H) and 2 (i / H) + 1 of head i % H
    auto item_ref = [&](int i, int &pair, int &hh, ChunkRef &ra, ChunkRef &rb, bool &hb) -> bool {
        if (i >= n_items) return false;
        pair = i / H;
        hh = i % H;
        if (!chunk_ref(g, 2 * pair, ra)) return false;
        hb = chunk_ref(g, 2 * pair + 1, rb);
        if (!hb) rb = ra;
        return true;
    };
    // K and V of an item land on their own barriers: V's tile doubles as the u^T
    // staging area of the previous item, so its load waits until those stores
    // have read it
    auto load_x = [&](const CUtensorMap *map, uint8_t *dst, uint64_t *bar, int hh,
                      const ChunkRef &ra, const ChunkRef &rb) {
        mbar_arrive_expect_tx(bar, 4 * kTile);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            tma_load_3d(dst + half * 2 * kTile, map, bar, half * 64, hh, (int)ra.bos);
            tma_load_3d(dst + half * 2 * kTile + kTile, map, bar, half * 64, hh, (int)rb.bos);
        }
    };

    // g and beta of this thread's token in an item, fetched asynchronously (a plain
    // load would be waited for by the fences between here and its use)
    auto fetch_gb = [&](int hh, const ChunkRef &rc, bool valid_chunk) {
        const bool ok = valid_chunk && r < rc.len;
        const long long i = ok ? (rc.bos + r) * H + hh : 0;
        cp_async4(&s.gpre[ch][r], g.g + i, ok);
        cp_async4(&s.bpre[ch][r], g.beta + i, ok);
    };

    if (tid == 0) {
        mbar_init(&s.k_bar, 1);
        mbar_init(&s.v_bar, 1);
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
    const uint32_t tbase = s.tmem_base;

    int item = blockIdx.x, pair = 0, h = 0;
    ChunkRef ra, rb;
    bool has_b = false;
    bool have = item_ref(item, pair, h, ra, rb, has_b);
    if (have && tid == 0) load_x(&tm_k, s.k, &s.k_bar, h, ra, rb);
    if (have) fetch_gb(h, ch ? rb : ra, !ch || has_b);
    int k_loads = have ? 1 : 0, v_loads = 0;  // TMA loads issued (uniform bookkeeping)
    int it = 0, mma_n = 0;
    bool bailed = false;
    while (have) {
        int pair_n = 0, h_n = 0;
        ChunkRef ra_n, rb_n;
        bool has_b_n = false;
        const bool have_next = item_ref(item + (int)gridDim.x, pair_n, h_n, ra_n, rb_n, has_b_n);
        const ChunkRef &mine = ch ? rb : ra;
        const int L = (ch && !has_b) ? 0 : mine.len;
        if (tid == 0) {
            bulk_wait_read();                 // the previous item's W^T / u^T stores have read
            load_x(&tm_v, s.v, &s.v_bar, h, ra, rb);   // the A region and the V tile
        }
        ++v_loads;
        tc_fence_before();
        __syncthreads();
        // gam = cumsum(g), beta (zero beyond the chunk)
        const long long tok = mine.bos + r;
        cp_async_wait_all();
        const float graw = r < L ? decay_of(g, s.gpre[ch][r], h) : 0.f;
        const float gam = scan64(graw, s.wsum);
        s.gam[ch][r] = gam;
        s.eg[ch][r] = r < L ? __expf(graw) : 0.f;
        s.bet[ch][r] = r < L ? s.bpre[ch][r] : 0.f;
        if (r < L) ws_gam[tok * H + h] = gam;

        bool ok = mbar_wait(&s.k_bar, it & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t kb = smem_u32(s.k);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint32_t off = (kk >> 2) * 2 * kTile + (kk & 3) * 32;
                const uint64_t d = desc_sw128(kb + off, 16, 1024);
                mma_bf16(tbase, d, d, kIdescKK, kk > 0);
            }
            mma_commit(&s.mma_bar);
        }
        ok = mbar_wait(&s.mma_bar, 0, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tc_fence_after();
        {
            // row r of this chunk's K K^T block
            float kk[64];
            tmem_ld32x2(tmem_addr(tbase, warp, ch * 64), tmem_addr(tbase, warp, ch * 64 + 32), kk,
                        kk + 32);
            float nrm = 0.f;
#pragma unroll
            for (int c = 0; c < 64; ++c) nrm = (c == r) ? kk[c] : nrm;
            const float rk = (r < L) ? (g.l2norm ? rsqrtf(nrm + 1e-6f) : 1.f) : 0.f;
            s.brk[ch][r] = s.bet[ch][r] * rk;
            tc_fence_before();
            __syncthreads();
            // K K^T is symmetric, so this row is also column r: thread r writes
            // A[i][r] = beta_i (k_i . k_r) e^(gamma_i - gamma_r) for i > r, i.e. row r of A^T.
            // The decay is a running product: e^(gamma_i - gamma_r) = prod_{r<j<=i} e^(g_j),
            // one exponential per token for the whole chunk instead of one per entry.
            float4 *arow = reinterpret_cast<float4 *>(s.A[ch][r]);
            const float4 *brk4 = reinterpret_cast<const float4 *>(s.brk[ch]);
            const float4 *eg4 = reinterpret_cast<const float4 *>(s.eg[ch]);
            float dec = 1.f;
#pragma unroll
            for (int i4 = 0; i4 < 16; ++i4) {
                const float4 b4 = brk4[i4], g4 = eg4[i4];
                const float bb[4] = {b4.x, b4.y, b4.z, b4.w}, ge[4] = {g4.x, g4.y, g4.z, g4.w};
                float x[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int i = 4 * i4 + e;
                    dec = i > r ? dec * ge[e] : 1.f;
                    x[e] = (i > r && i < L) ? bb[e] * kk[i] * rk * dec : 0.f;
                }
                arow[i4] = make_float4(x[0], x[1], x[2], x[3]);
            }
        }
        __syncthreads();
        {
            // T = (I + A)^-1 by both warps of the chunk (32 x 32 blocks)
            float (*At)[68] = s.A[ch];
            const int lane = r & 31, hi = r >> 5, jb = 32 * hi;
            float t[32], y[16];
            solve_unit_lower64(At, r, t, y, [] { __syncthreads(); });
            const int cown = jb + lane;               // column of t
            const bool own_ok = cown < L, low_ok = lane < L;
            if (ws_t && (!ch || has_b)) {
                // the backward keeps T as bf16: row c of the tile [chunk][h][64][64] is
                // column c of this chunk's T (zero past the chunk's end)
                __nv_bfloat16 *tt = ws_t + ((long long)(2 * pair + ch) * H + h) * 64 * 64;
                uint4 *own = reinterpret_cast<uint4 *>(tt + cown * 64);
                uint4 *low = reinterpret_cast<uint4 *>(tt + lane * 64);
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    own[4 * hi + q] = own_ok ? pack_bf16x8(t + 8 * q) : z;
                    if (hi) own[q] = z;
                }
                if (hi == 0) {
                    low[4] = low_ok ? pack_bf16x8(y) : z;
                    low[7] = low_ok ? pack_bf16x8(y + 8) : z;
                } else {
                    low[5] = low_ok ? pack_bf16x8(y) : z;
                    low[6] = low_ok ? pack_bf16x8(y + 8) : z;
                }
            }
            __syncthreads();  // every block done: A's space becomes bw / bu
            // MN-major B operands: row j holds column j of T scaled by beta_j e_j rk_j (W)
            // and by beta_j (u); both scales are zero past the chunk's end.
            store_wu_operands(stage + ch * kTile, stage + 2 * kTile + ch * kTile, r, t, y,
                              __expf(s.gam[ch][cown]) * s.brk[ch][cown], s.bet[ch][cown],
                              __expf(s.gam[ch][lane]) * s.brk[ch][lane], s.bet[ch][lane]);
        }
        fence_proxy_async();
        ok = mbar_wait(&s.v_bar, it & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        ++mma_n;
        if (warp == 0) {
            tc_fence_after();
            const uint32_t kb = smem_u32(s.k), vb = smem_u32(s.v);
            const uint32_t bw = smem_u32(stage), bu = bw + 2 * kTile;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t bdw = desc_sw128(bw + c * kTile + kk * 2048, kTile, 1024);
                    const uint64_t bdu = desc_sw128(bu + c * kTile + kk * 2048, kTile, 1024);
                    const uint64_t ak = desc_sw128(kb + c * kTile + kk * 2048, 2 * kTile, 1024);
                    const uint64_t av = desc_sw128(vb + c * kTile + kk * 2048, 2 * kTile, 1024);
                    mma_bf16(tbase + c * 64, ak, bdw, kIdescPrepMN, kk > 0);
                    mma_bf16(tbase + 128 + c * 64, av, bdu, kIdescPrepMN, kk > 0);
                }
            }
            mma_commit(&s.mma_bar);
        }
        ok = mbar_wait(&s.mma_bar, 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        // K is dead: the next item's (its V follows once the u^T stores below have
        // read the V tile)
        if (tid == 0 && have_next) {
            fence_proxy_async();
            load_x(&tm_k, s.k, &s.k_bar, h_n, ra_n, rb_n);
        }
        if (have_next) {
            ++k_loads;
            fetch_gb(h_n, ch ? rb_n : ra_n, !ch || has_b_n);
        }
        tc_fence_after();
        // thread t = feature index (dk for W, dv for u): its 64 chunk rows form row t
        // of the W^T / u^T tile, staged swizzled (two tiles of [128 rows][128 B] each)
        // in the dead A region (W^T) and the dead V tile (u^T), and stored by TMA
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            uint8_t *base = pass ? s.v : stage;
#pragma unroll 1
            for (int c = 0; c < 2; ++c) {
                const int Lc = (c && !has_b) ? 0 : (c ? rb.len : ra.len);
                float x[64];    // both halves of the row with one wait
                tmem_ld32x2(tmem_addr(tbase, warp, 128 * pass + c * 64),
                            tmem_addr(tbase, warp, 128 * pass + c * 64 + 32), x, x + 32);
#pragma unroll
                for (int j = 0; j < 64; ++j) x[j] = j < Lc ? x[j] : 0.f;
                st_row64(base + c * 2 * kTile, tid, x);
            }
        }
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            for (int pass = 0; pass < 2; ++pass)
                for (int c = 0; c < (has_b ? 2 : 1); ++c) {
                    const int row = (int)(((long long)(2 * pair + c) * H + h) * kD);
                    tma_store_2d(pass ? &tm_u : &tm_w, (pass ? s.v : stage) + c * 2 * kTile, 0, row);
                }
            bulk_commit();
        }
        item += (int)gridDim.x;
        pair = pair_n;
        h = h_n;
        ra = ra_n;
        rb = rb_n;
        has_b = has_b_n;
        have = have_next;
        ++it;
    }
    if (bailed && tid == 0) {
        if (k_loads > 0) mbar_drain(&s.k_bar, (k_loads - 1) & 1);
        if (v_loads > 0) mbar_drain(&s.v_bar, (v_loads - 1) & 1);
        if (mma_n > 0) mbar_drain(&s.mma_bar, (mma_n - 1) & 1);
    }
    if (tid == 0) bulk_wait_read();
    cp_async_wait_all();                      // a prefetch still in flight after a bail
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}

// ------------------------------------------------------------------ walk
// kWalkOut: the state walk (start states stored; O from the output pass).
// kWalkMap: segment maps.  kWalkFused: the state walk that also forms each
// chunk's O inside its loop -- the start state, U and the decay are at hand
// there -- so that no output pass runs:
//   P = Q K^T .* lower_incl .* D,   O^T = scale (H^T Q^T diag(e) + U^T P^T).
// Its stages carry Q stacked over K ([Q rows | K rows] per dk half) and it
// keeps one chunk in flight ahead of the current one; the others keep two.
enum { kWalkOut = 0, kWalkMap = 1, kWalkFused = 2 };

template <int MODE>
struct WalkSmem {
    static constexpr int kStages = MODE == kWalkFused ? 2 : 3;
    static constexpr int kKBytes = MODE == kWalkFused ? 4 * kTile : 2 * kTile;
    uint8_t k[kStages][kKBytes];   // per stage: [dk half][(Q rows 0-63,) K rows][128 B]
    uint8_t w[kStages][2 * kTile];   // per stage: W^T, [128 rows k][64 chunk rows]
    uint8_t u[kStages][2 * kTile];   // per stage: u^T, [128 rows v][64 chunk rows]
    uint8_t hT[4 * kTile];         // [dk half][128 state rows][128 B]  (A operand)
    uint8_t uTs[2 * kTile];        // U^T diag(f): [128 state rows][64 chunk rows] (A operand)
    uint8_t uT[MODE == kWalkFused ? 2 * kTile : 1024];   // U^T (fused walk)
    uint8_t p[MODE == kWalkFused ? kTile : 1024];        // P rows r (fused walk)
    float gam[2][64];
    alignas(16) float fr[64];      // exp(gam_L - gam_r) (x 1/|k_r|); 0 past L
    alignas(16) float er[2][64];   // exp(gam_r) per chunk parity (output walk); 0 past L
    float egw[2][64];              // exp(gam_j - gam_{j-1}) per chunk parity (output walk)
    float rqk[128];                // q, k normalised here: 1 / |q_r| at r (output walk),
                                   // 1 / |k_r| at 64 + r
    uint64_t tma_bar[kStages], bar_u, bar_q, bar_dh;
    uint32_t tmem_base;
};

struct TcWalkArgs {
    const float *ws_gam;
    const float *h0;          // [N, H, K, V] nullable
    const float *seg_start;   // [segs, H, K, V] (CP)
    const int32_t *warm;      // [N, H] (CP warmup)
    int warm_chunks;
    float *final_state;       // nullable
    __nv_bfloat16 *hc;        // chunk start states as bf16 H^T tiles [chunk][H][k half][v][64], nullable
    float *maps;              // [segs, H, K, K+V] (kWalkMap)
    float *maps_a;            // nullable: A columns to [segs, H, K, K] here instead (a saved context)
    __nv_bfloat16 *o;         // [tokens, H, V]: formed inside the output walk when set
    int cp;
};

constexpr uint32_t kIdescDH = idesc_bf16(128, 128, false, true);      // B MN-major
constexpr uint32_t kIdescKM64 = idesc_bf16(128, 64, false, true);     // B MN-major, N = 64
constexpr uint32_t kIdescKK64 = idesc_bf16(128, 64, false, false);    // both K-major, N = 64

// 256 threads: thread t owns state row v = t % 128 (TMEM lane v) and the
// column half hs = t / 128; warps w and w + 4 share a TMEM lane quarter and
// split every epilogue's columns between them.  Per chunk: U = u - W H (one
// MMA group), U^T diag(f) into shared memory, K^T diag(f) U (second group),
// H <- exp(gam_L) H + that.  The output walk adds [Q; K] K^T and H^T Q^T to
// the first group, P (rows r on lanes 0-63) and U^T to shared memory, U^T P^T
// to the second group, and O after it.
template <int MODE>
__global__ void __launch_bounds__(256, 1)
tc_walk_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
               const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_u,
               const __grid_constant__ CUtensorMap tm_hc, Geo g, TcWalkArgs a) {
    pdl_enter();
    typedef WalkSmem<MODE> S;
    constexpr int kWalkStages = S::kStages;
    extern __shared__ uint8_t smem_raw[];
    S &s = *reinterpret_cast<S *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int tid = threadIdx.x, warp = tid >> 5, cb = blockIdx.z, H = g.H;
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
    const bool a_cols = MODE == kWalkMap && cb == 0;   // A columns: start I, u = 0
    // the forward scan needs no map of the last segment; the backward's reverse
    // scan does need that segment's A part when it takes it from a saved context
    if (MODE == kWalkMap &&
        ((j == nseg - 1 && !(a_cols && a.maps_a)) || (a.warm && a.warm[n * H + h])))
        return;
    constexpr bool kState = MODE != kWalkMap;         // a state walk (start states, O)
    constexpr bool fused = MODE == kWalkFused;        // O formed here
    const bool states = kState && a.hc != nullptr;
    // byte offset of K's dk half hh inside a stage, and the stride between the halves
    constexpr int kKOff = fused ? kTile : 0;
    constexpr uint32_t kKHalf = fused ? 2 * kTile : kTile;
    const int nc = seq_nchunks(g, n);
    const int c0 = min(nc, j * g.seg_chunks), c1 = min(nc, (j + 1) * g.seg_chunks);
    const int cbase = seq_chunk_base(g, n);
    long long sbos;
    int slen;
    seq_range(g, n, sbos, slen);
    bool warm = false;
    int cstart = c0;
    if (kState && a.cp && j > 0 && a.warm && a.warm[n * H + h]) {
        warm = true;
        cstart = max(0, c0 - a.warm_chunks);
    }

    auto issue_tma = [&](int st, int c) {
        const int tok0 = (int)(sbos + (long long)c * kChunk);
        // K (2 halves), W^T, u^T (and Q's 2 halves above K's in the output walk)
        mbar_arrive_expect_tx(&s.tma_bar[st], (fused ? 8 : 6) * kTile);
        tma_load_3d(s.k[st] + kKOff, &tm_k, &s.tma_bar[st], 0, h, tok0);
        tma_load_3d(s.k[st] + kKOff + kKHalf, &tm_k, &s.tma_bar[st], 64, h, tok0);
        if (fused) {
            tma_load_3d(s.k[st], &tm_q, &s.tma_bar[st], 0, h, tok0);
            tma_load_3d(s.k[st] + kKHalf, &tm_q, &s.tma_bar[st], 64, h, tok0);
        }
        const int trow = (int)(((long long)(cbase + c) * H + h) * kD);
        tma_load_2d(s.w[st], &tm_w, &s.tma_bar[st], 0, trow);
        tma_load_2d(s.u[st], &tm_u, &s.tma_bar[st], 0, trow);
    };

    // the first chunks' tiles are requested at once, so that their latency
    // overlaps the start state's load
    if (tid == 0) {
        for (int i = 0; i < kWalkStages; ++i) mbar_init(&s.tma_bar[i], 1);
        mbar_init(&s.bar_u, 1);
        mbar_init(&s.bar_q, 1);
        mbar_init(&s.bar_dh, 1);
        fence_barrier_init();
        for (int i = 0; i < kWalkStages - 1 && cstart + i < c1; ++i) issue_tma(i, cstart + i);
    }
    constexpr uint32_t kTmemCols = fused ? 512 : 256;
    if (warp == 0) {
        tmem_alloc(&s.tmem_base, kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    // start state: this thread's half (dk 64*hs ..) of column v of H
    float Hr[64];
    {
        const float *src = nullptr;
        if (kState && !warm) {
            if (a.cp && j > 0)
                src = a.seg_start + ((long long)(seq_seg_base(g, n) + j) * H + h) * kD * kD;
            else if (a.h0)
                src = a.h0 + ((long long)n * H + h) * kD * kD;
        }
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const int k = 64 * hs + i;
            Hr[i] = src ? src[k * kD + v] : ((a_cols && k == v) ? 1.f : 0.f);
        }
    }
    st_row64(s.hT + hs * 2 * kTile, v, Hr);
    if (tid < 64 && cstart < c1) {
        const int L0 = min(kChunk, slen - cstart * kChunk);
        s.gam[0][tid] = tid < L0 ? a.ws_gam[(sbos + (long long)cstart * kChunk + tid) * H + h] : 0.f;
    }
    fence_proxy_async();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s.tmem_base;
    const uint32_t t_u = tbase, t_dh = tbase + 128;
    // output walk: P, and H^T Q^T / U^T P^T per chunk parity (a chunk's O is formed
    // while the next chunk's first products run)
    const uint32_t t_p = tbase + 64;
    auto t_qh = [&](int b) { return tbase + 256 + 128 * b; };
    auto t_pu = [&](int b) { return tbase + 320 + 128 * b; };
    long long pbos = 0;
    int pL = 0, pc = -1;                       // the previous chunk (output walk)
    // O rows c = 32 hs .. +31 of the chunk at token pbos (parity b), feature v:
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

    // one commit per barrier per chunk: every barrier's parity is the chunk
    // iteration's; `pend` marks groups committed in this iteration, not yet waited
    // uniform bookkeeping for the bail-out path: loads issued per stage, and
    // the stages whose latest load has not been waited for
    int it = 0, tma_pending = 0, pend = 0;
    unsigned loaded = 0, ld_par = 0;   // per stage: loaded at least once; parity of its latest load
    auto note_load = [&](int sn) {
        if (loaded & (1u << sn)) ld_par ^= 1u << sn;
        loaded |= 1u << sn;
        tma_pending |= 1 << sn;
    };
    bool bailed = false;
    // the last warp issues the loads, away from warp 0 (MMA issue) and the
    // threads that read gam
    const bool tma_thread = tid == 255;
    for (int i = 0; i < kWalkStages - 1 && cstart + i < c1; ++i) note_load(i);   // issued above
    for (int c = cstart; c < c1; ++c, ++it) {
        const int st = it % kWalkStages, gb = it & 1;
        const uint32_t par = it & 1;
        const long long bos = sbos + (long long)c * kChunk;
        const int L = min(kChunk, slen - c * kChunk);
        pend = 0;
        if (c + 1 < c1) {
            const int Ln = min(kChunk, slen - (c + 1) * kChunk);
            // gam of the next chunk into the other buffer, asynchronously
            if (tid < 64)
                cp_async4(&s.gam[gb ^ 1][tid], a.ws_gam + (bos + kChunk + min(tid, Ln - 1)) * H + h,
                          tid < Ln);
        }
        bool ok = mbar_wait(&s.tma_bar[st], (it / kWalkStages) & 1, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        tma_pending &= ~(1 << st);
        if (warp == 0) {
            tc_fence_after();
            const uint32_t wt = smem_u32(s.w[st]), hT = smem_u32(s.hT), qk = smem_u32(s.k[st]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ah = desc_sw128(hT + (kk >> 2) * 2 * kTile + (kk & 3) * 32, 16, 1024);
                const uint64_t bw = desc_sw128(wt + kk * 2048, 2 * kTile, 1024);   // W^T, MN-major
                mma_bf16(t_u, ah, bw, kIdescKM64, kk > 0);
            }
            mma_commit(&s.bar_u);
            if (fused) {
                // behind U on their own barrier: the U epilogue need not wait for them
                // (H^T Q^T, read only by the next chunk's O, goes with the second group)
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kKHalf + (kk & 3) * 32;
                    const uint64_t aq = desc_sw128(qk + off, 16, 1024);           // [Q; K], K-major
                    const uint64_t bk = desc_sw128(qk + kKOff + off, 16, 1024);   // K, K-major
                    mma_bf16(t_p, aq, bk, kIdescKK64, kk > 0);       // rows 0-63: Q K^T
                }
                mma_commit(&s.bar_q);
            }
        }
        pend = fused ? 5 : 1;
        // while the product runs, the last warp requests the next chunk(s) (into
        // the stage the previous chunk used) and stores this chunk's start state
        if (c + kWalkStages - 1 < c1) {
            const int sn = (it + kWalkStages - 1) % kWalkStages;
            if (tma_thread) {
                fence_proxy_async();
                issue_tma(sn, c + kWalkStages - 1);
            }
            note_load(sn);
        }
        if (states && c >= c0 && tma_thread) {
            // the bf16 H^T tile in shared memory, by TMA
            const int row = (int)(((long long)(cbase + c) * H + h) * 2 * kD);
            tma_store_2d(&tm_hc, s.hT, 0, row);
            tma_store_2d(&tm_hc, s.hT + 2 * kTile, 0, row + kD);
            bulk_commit();
        }
        if (fused && pc >= c0) {
            tc_fence_after();
            out_epilogue(gb ^ 1);                 // the previous chunk's O
        }
        if (g.l2norm) {
            // 1 / |k_r| (and, in the output walk, whose stage stacks Q rows 0-63
            // over K rows 64-127, 1 / |q_r|) from the stage's rows
            if (fused)
                row_inv_norms(s.k[st], kKHalf, 128, s.rqk);
            else
                row_inv_norms(s.k[st] + kKOff, kKHalf, 64, s.rqk + 64);
            __syncthreads();
        }
        if (tid < 64) {
            const float gl = s.gam[gb][L - 1], gr = s.gam[gb][tid];
            s.fr[tid] = tid < L ? __expf(gl - gr) * (g.l2norm ? s.rqk[64 + tid] : 1.f) : 0.f;
            if (fused) {
                s.er[gb][tid] = tid < L ? __expf(gr) * (g.l2norm ? s.rqk[tid] : 1.f) : 0.f;
                s.egw[gb][tid] = tid > 0 ? __expf(gr - s.gam[gb][tid - 1]) : 1.f;
            }
        }
        ok = mbar_wait(&s.bar_u, par, g.spin_limit, g.status);
        if (__syncthreads_or(!ok)) { bailed = true; break; }
        pend &= ~1;
        tc_fence_after();
        // U^T diag(f) rows v, chunk rows 32*hs .. +31 (one TMEM load, groups of 8)
        float xu[32];
        tmem_ld32(tmem_addr(t_u, warp, 32 * hs), xu);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float *x = xu + 8 * q, uu[8];
            const int chunk = 4 * hs + q;
            uint4 raw = make_uint4(0u, 0u, 0u, 0u);
            if (!a_cols)
                raw = *reinterpret_cast<const uint4 *>(s.u[st] + v * 128 + ((chunk ^ (v & 7)) << 4));
            const __nv_bfloat16 *bv = reinterpret_cast<const __nv_bfloat16 *>(&raw);
            // f of rows 8 chunk .. +7 as two 16-byte broadcast reads
            const float4 f0 = reinterpret_cast<const float4 *>(s.fr)[2 * chunk];
            const float4 f1 = reinterpret_cast<const float4 *>(s.fr)[2 * chunk + 1];
            const float fq[8] = {f0.x, f0.y, f0.z, f0.w, f1.x, f1.y, f1.z, f1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int r = 8 * chunk + e;
                x[e] = r < L ? __bfloat162float(bv[e]) - x[e] : 0.f;   // U^T
                uu[e] = x[e] * fq[e];
            }
            st_row8(s.uTs, v, chunk, uu);
            if (fused) st_row8(s.uT, v, chunk, x);
        }
        // The state update's product Uᵀdiag(f) K and (fused) H^T Q^T need only the U
        // epilogue's tiles: in the output walk warp 2, which has no P rows, issues
        // them at once, so that they run under the P epilogue, and U^T P^T after it,
        // all on bar_dh; otherwise warp 0 issues the product after the barrier.
        if (fused) {
            tc_fence_before();
            fence_proxy_async();                  // the U epilogue's tiles, for the products
            ok = mbar_wait(&s.bar_q, par, g.spin_limit, g.status);
            if (__syncthreads_or(!ok)) { bailed = true; break; }
            pend &= ~4;
            tc_fence_after();
            if (warp == 2) {
                const uint32_t uTs = smem_u32(s.uTs), kt = smem_u32(s.k[st]) + kKOff;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(t_dh, desc_sw128(uTs + kk * 32, 16, 1024),
                             desc_sw128(kt + kk * 2048, kKHalf, 1024), kIdescDH, kk > 0);
                // H^T Q^T (this chunk's start state, which the state update
                // overwrites only after bar_dh)
                const uint32_t hT = smem_u32(s.hT), qk = smem_u32(s.k[st]);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t off = (kk >> 2) * kKHalf + (kk & 3) * 32;
                    mma_bf16(t_qh(gb), desc_sw128(hT + (kk >> 2) * 2 * kTile + (kk & 3) * 32, 16, 1024),
                             desc_sw128(qk + off, 16, 1024), kIdescKK64, kk > 0);
                }
            }
        }
        if (fused && v < 64) {
            // row r = v of P: Q K^T on lanes 0-63, masked to c <= r < L, times D_rc
            // (and 1 / (|q_r| |k_c|) when q, k are normalised here)
            const int r = v;
            float xp[32], dd[32];
            tmem_ld32(tmem_addr(t_p, warp, 32 * hs), xp);
            row_decays32(s.gam[gb], s.egw[gb], r, 32 * hs, dd);
            const float sr = g.l2norm ? s.rqk[r] : 1.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float *x = xp + 8 * q;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int c = 32 * hs + 8 * q + e;
                    const float sc = g.l2norm ? sr * s.rqk[64 + c] : 1.f;
                    x[e] = (c <= r && r < L) ? x[e] * dd[8 * q + e] * sc : 0.f;
                }
                st_row8(s.p, r, 4 * hs + q, x);
            }
        }
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
        if (warp == (fused ? 2 : 0)) {
            tc_fence_after();
            if (fused) {
                // U^T P^T: both operands K-major over the chunk rows
                const uint32_t ua = smem_u32(s.uT), pp = smem_u32(s.p);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(t_pu(gb), desc_sw128(ua + kk * 32, 16, 1024),
                             desc_sw128(pp + kk * 32, 16, 1024), kIdescKK64, kk > 0);
            } else {
                const uint32_t uTs = smem_u32(s.uTs), kt = smem_u32(s.k[st]) + kKOff;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    mma_bf16(t_dh, desc_sw128(uTs + kk * 32, 16, 1024),
                             desc_sw128(kt + kk * 2048, kKHalf, 1024), kIdescDH, kk > 0);
            }
            mma_commit(&s.bar_dh);
        }
        pend |= 2;
        if (tma_thread) bulk_wait_read();     // the state store has read H^T
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
        pc = c;
        if (tid < 64) cp_async_wait_all();
        tc_fence_before();
        fence_proxy_async();
        __syncthreads();
    }
    if (fused && !bailed && pc >= c0) {
        tc_fence_after();
        out_epilogue((it - 1) & 1);              // the last chunk's O
    }

    if (tma_thread) bulk_wait_read();
    if (tid < 64) cp_async_wait_all();    // a gam prefetch may still be in flight after a bail
    if (bailed) {
        if (tid == 0) {
            for (int st = 0; st < kWalkStages; ++st)
                if (tma_pending & (1 << st)) mbar_drain(&s.tma_bar[st], (ld_par >> st) & 1u);
            if (pend & 1) mbar_drain(&s.bar_u, it & 1);
            if (pend & 4) mbar_drain(&s.bar_q, it & 1);
            if (pend & 2) mbar_drain(&s.bar_dh, it & 1);
        }
    } else if (MODE == kWalkMap) {
        const long long sh = (long long)(seq_seg_base(g, n) + j) * H + h;
        if (a_cols && a.maps_a) {
            float *dst = a.maps_a + sh * kD * kD;
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(64 * hs + i) * kD + v] = Hr[i];
        } else {
            float *dst = a.maps + sh * kD * (2 * kD);
#pragma unroll
            for (int i = 0; i < 64; ++i) dst[(64 * hs + i) * (2 * kD) + cb * kD + v] = Hr[i];
        }
    } else if (a.final_state && j == nseg - 1) {
        float *dst = a.final_state + ((long long)n * H + h) * kD * kD;
#pragma unroll
        for (int i = 0; i < 64; ++i) dst[(64 * hs + i) * kD + v] = Hr[i];
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, kTmemCols);
}

// ------------------------------------------------------------------ host side
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

template <typename F>
cudaError_t set_smem(F kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}
}  // namespace

cudaError_t encoder() {
    if (g_encode) return cudaSuccess;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return e;
    if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorSymbolNotFound;
    g_encode = (EncodeTiledFn)fn;
    return cudaSuccess;
}

// [tokens, H, 128] bf16 viewed as 3-D (feature, head, token); 64 x 1 x 64 boxes
// with the 128-byte swizzle.  Rows past the last token read as zeros.
cudaError_t make_map(CUtensorMap *m, const void *base, long long tokens, int H) {
    const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)tokens};
    const cuuint64_t strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)H * kD * 2};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t es[3] = {1, 1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base),
                                dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Chunk-major tiles of 64 bf16 columns ([chunk][H][box_rows][64], e.g. the
// transposed [128 features][64 rows] tiles) viewed as 2-D (64, rows_total);
// one 64 x box_rows box = one (chunk, head) tile.
cudaError_t make_map_tiles(CUtensorMap *m, const void *base, long long rows_total, int box_rows) {
    const cuuint64_t dims[2] = {64, (cuuint64_t)rows_total};
    const cuuint64_t strides[1] = {64 * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t es[2] = {1, 1};
    const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                                dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

bool supported(const Plan &p) {
    // TMA row coordinates are 32-bit ints: the largest, of the chunk-state tiles
    // (two 128-row halves per (chunk, head)), is 2 (chunk * H + head) * 128 + 128
    return p.dtype == GDN_BF16 && p.g.K == kD && p.g.V == kD && (long long)p.g.B * p.g.T > 0 &&
           (long long)p.max_chunks * p.g.H * 2 * kD + kD < (1ll << 31);
}

// Prep, then the walk: with output (states_only = false) or storing every
// chunk's start state into p.ws.hc (states_only = true, for the backward).
// save (with output): also keep T and the chunk start states for the backward.
static cudaError_t run_forward(const Plan &p, cudaStream_t s, bool states_only, bool save) {
    cudaError_t e = encoder();
    if (e != cudaSuccess) return e;
    const Geo &g = p.g;
    const long long tokens = (long long)g.B * g.T;
    CUtensorMap mq, mk, mv, mw, mu;
    if ((e = make_map(&mq, g.q, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mk, g.k, tokens, g.H)) != cudaSuccess) return e;
    if ((e = make_map(&mv, g.v, tokens, g.H)) != cudaSuccess) return e;
    const long long tile_rows = (long long)p.max_chunks * g.H * kD;
    if ((e = make_map_tiles(&mw, p.ws.w, tile_rows)) != cudaSuccess) return e;
    if ((e = make_map_tiles(&mu, p.ws.u, tile_rows)) != cudaSuccess) return e;
    CUtensorMap mhc;
    if ((e = make_map_tiles(&mhc, p.ws.hc, 2 * tile_rows)) != cudaSuccess) return e;

    const size_t prep_smem = sizeof(PrepSmem) + 1024;
    const size_t out_smem = sizeof(WalkSmem<kWalkOut>) + 1024;
    const size_t fused_smem = sizeof(WalkSmem<kWalkFused>) + 1024;
    const size_t map_smem = sizeof(WalkSmem<kWalkMap>) + 1024;
    if ((e = set_smem(tc_prep_kernel, prep_smem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_walk_kernel<kWalkOut>, out_smem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_walk_kernel<kWalkFused>, fused_smem)) != cudaSuccess) return e;
    if ((e = set_smem(tc_walk_kernel<kWalkMap>, map_smem)) != cudaSuccess) return e;

    prof_before("tc_prep", s);
    const int prep_items = (p.max_chunks + 1) / 2 * g.H;
    if ((e = launch_pdl(tc_prep_kernel, dim3(std::min(prep_items, 2 * std::max(p.sms, 1))),
                        dim3(128), prep_smem, s, mk, mv, mw, mu, g, p.ws.gam,
                        (states_only || save) ? (__nv_bfloat16 *)p.ws.tmat : nullptr,
                        prep_items)) != cudaSuccess)
        return e;
    prof_after(s);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    // the walk stores every chunk's start state: the output kernel and the
    // backward read them
    TcWalkArgs a{};
    a.ws_gam = p.ws.gam;
    a.h0 = p.h0;
    a.final_state = states_only ? nullptr : p.final_state;
    a.hc = (__nv_bfloat16 *)p.ws.hc;
    // The walk forms O itself when its CTAs fill at least three quarters of the
    // SMs: each chunk then costs the walk about 4.3K more cycles, against about
    // 6.6K SM-cycles of the chunk-parallel output pass (GB300 measurements on
    // the four workloads; with fewer walk CTAs the output pass, spread over
    // every SM, is cheaper).
    const int walk_ctas = (p.cp ? p.max_segs : g.N) * g.H;
    const bool fuse_out = !states_only && 4 * walk_ctas >= 3 * std::max(p.sms, 1);
    a.o = fuse_out ? (__nv_bfloat16 *)p.o : nullptr;
    auto walk_kernel = fuse_out ? tc_walk_kernel<kWalkFused> : tc_walk_kernel<kWalkOut>;
    const char *out_name = states_only ? "tc_walk_states" : fuse_out ? "tc_walk_fused" : "tc_walk";
    const size_t walk_smem = fuse_out ? fused_smem : out_smem;
    const dim3 walk_block(256);
    if (p.cp) {
        a.cp = 1;
        a.maps = p.ws.maps;
        a.maps_a = p.ws.fwd_maps;
        a.seg_start = p.ws.seg_state;
        if (p.warm_chunks > 0 && !states_only) {
            if ((e = simt::warm_decide(p, s)) != cudaSuccess) return e;
            a.warm = p.ws.warm;
            a.warm_chunks = p.warm_chunks;
        }
        prof_before("tc_walk_map", s);
        if ((e = launch_pdl(tc_walk_kernel<kWalkMap>, dim3(p.max_segs, g.H, 2), dim3(256), map_smem, s,
                            mq, mk, mw, mu, mhc, g, a)) != cudaSuccess)
            return e;
        prof_after(s);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        if ((e = simt::cp_scan(p, a.warm, s)) != cudaSuccess) return e;
        prof_before(out_name, s);
        if ((e = launch_pdl(walk_kernel, dim3(p.max_segs, g.H, 1), walk_block, walk_smem, s,
                            mq, mk, mw, mu, mhc, g, a)) != cudaSuccess)
            return e;
        prof_after(s);
    } else {
        prof_before(out_name, s);
        if ((e = launch_pdl(walk_kernel, dim3(g.N * g.H, 1, 1), walk_block, walk_smem, s,
                            mq, mk, mw, mu, mhc, g, a)) != cudaSuccess)
            return e;
        prof_after(s);
    }
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    return (states_only || fuse_out) ? cudaSuccess : output(p, s);
}

cudaError_t forward(const Plan &p, cudaStream_t s, bool save) {
    cudaError_t e = simt::tables(p, s);
    if (e != cudaSuccess) return e;
    // asked for, and without a context to keep: the one-kernel forward (prep
    // inside the walk) for pairs that fill the GPU
    if (p.fuse_prep && !save && full_forward_fits(p)) return full_forward(p, s);
    return run_forward(p, s, false, save);
}

cudaError_t recompute_states(const Plan &p, cudaStream_t s) { return run_forward(p, s, true, false); }

}  // namespace tc
}  // namespace gdn
