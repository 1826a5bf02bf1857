// gdn_simt.cu -- fp32 CUDA-core kernels for GDN chunked prefill.
//
// This is the general path: any supported shape (K, V in {64, 128}), fp32 or
// bf16 inputs, all arithmetic in fp32.  It is the only path for fp32 inputs
// (a bf16 tensor-core operand cannot meet fp32 accuracy) and serves bf16
// shapes the tcgen05 kernels do not cover.
//
// Chunk form (per (sequence, head), chunk rows r = 0..L-1, state H = S^T of
// shape K x V at the chunk start, gam = within-chunk cumsum of g,
// D[r][s] = exp(gam_r - gam_s)):
//   A = strict_lower(diag(beta) K K^T .* D),  T = (I + A)^-1
//   W = T diag(beta exp(gam)) K,  u = T diag(beta) V,  U = u - W H
//   O = scale (diag(exp(gam)) Q H + (Q K^T .* lower_incl .* D) U)
//   H <- exp(gam_L) H + K^T diag(exp(gam_L - gam)) U
// The pages split the work into a chunk-local kernel and a walking kernel
// with a sequence-parallel preprocessing step between them, rather than one
// fully fused kernel (traeai.com page, announcement text; ollai.cn page,
// "FlashQLA的技术原理", last item); this file follows that split.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace simt {

constexpr int kThreads = 256;
constexpr int kBV = 32;  // state columns per walking CTA

// Loads `L` rows of a [tokens, H, D] tensor into smem rows of stride `ld`,
// optionally scaling each row to unit L2 norm ((|x|^2 + eps)^-1/2).  One warp
// per row.  `rnorm` (nullable) receives the scale factor per row.
template <typename TI>
__device__ void load_rows(float *dst, int ld, const TI *src, long long bos, int L, int H, int h,
                          int D, bool normalise, float *rnorm) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int r = warp; r < L; r += nw) {
        const TI *row = src + ((bos + r) * H + h) * (long long)D;
        float ss = 0.f;
        for (int i = lane; i < D; i += 32) {
            const float x = to_f(row[i]);
            dst[r * ld + i] = x;
            ss += x * x;
        }
        float s = 1.f;
        if (normalise) {
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            s = rsqrtf(ss + 1e-6f);
            for (int i = lane; i < D; i += 32) dst[r * ld + i] *= s;
        }
        if (rnorm && lane == 0) rnorm[r] = s;
    }
}

// gam = inclusive cumsum of g over the chunk (thread 0; 64 adds).
__device__ void chunk_cumsum(float *gam, const Geo &g, long long bos, int L, int H, int h) {
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int r = 0; r < L; ++r) {
            s += decay_at(g, (bos + r) * H + h, h);
            gam[r] = s;
        }
    }
}

// T = (I + A)^-1 for strictly lower A (L x L, stride 65), by forward
// substitution over columns of the elimination: after step s row s is final.
__device__ void unit_lower_inverse(float *Tm, const float *A, int L) {
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) {
        const int r = idx / kChunk, c = idx % kChunk;
        Tm[r * 65 + c] = (r == c) ? 1.f : 0.f;
    }
    __syncthreads();
    for (int s = 0; s + 1 < L; ++s) {
        const int width = s + 1, rows = L - 1 - s;
        for (int idx = threadIdx.x; idx < rows * width; idx += blockDim.x) {
            const int r = s + 1 + idx / width, j = idx % width;
            Tm[r * 65 + j] -= A[r * 65 + s] * Tm[s * 65 + j];
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- prep
// Per (chunk, head): gam, W = T diag(beta e^gam) K, u = T diag(beta) V.
// Writes gam [tokens, H], W [tokens, H, K], u [tokens, H, V] (fp32).
template <typename TI>
__global__ void __launch_bounds__(kThreads)
prep_kernel(Geo g, float *ws_gam, float *ws_w, float *ws_u) {
    ChunkRef cr;
    if (!chunk_ref(g, blockIdx.x, cr)) return;
    const int h = blockIdx.y, L = cr.len, K = g.K, V = g.V, H = g.H;
    extern __shared__ float sm[];
    float *Ks = sm;                       // [64][K+1]
    float *Vs = Ks + kChunk * (K + 1);    // [64][V+1]
    float *A = Vs + kChunk * (V + 1);     // [64][65]
    float *Tm = A + kChunk * 65;          // [64][65]
    float *gam = Tm + kChunk * 65;        // [64]
    float *bet = gam + kChunk;            // [64]
    load_rows(Ks, K + 1, (const TI *)g.k, cr.bos, L, H, h, K, g.l2norm, nullptr);
    load_rows(Vs, V + 1, (const TI *)g.v, cr.bos, L, H, h, V, false, nullptr);
    chunk_cumsum(gam, g, cr.bos, L, H, h);
    for (int r = threadIdx.x; r < L; r += blockDim.x) bet[r] = g.beta[(cr.bos + r) * H + h];
    __syncthreads();
    for (int r = threadIdx.x; r < L; r += blockDim.x) ws_gam[(cr.bos + r) * H + h] = gam[r];
    for (int idx = threadIdx.x; idx < kChunk * kChunk; idx += blockDim.x) {
        const int r = idx / kChunk, s = idx % kChunk;
        float a = 0.f;
        if (r < L && s < r) {
            float d = 0.f;
            for (int i = 0; i < K; ++i) d += Ks[r * (K + 1) + i] * Ks[s * (K + 1) + i];
            a = bet[r] * d * expf(gam[r] - gam[s]);
        }
        A[r * 65 + s] = a;
    }
    __syncthreads();
    unit_lower_inverse(Tm, A, L);
    for (int idx = threadIdx.x; idx < L * (K + V); idx += blockDim.x) {
        const int r = idx / (K + V), c = idx % (K + V);
        float acc = 0.f;
        if (c < K) {
            for (int s = 0; s <= r; ++s)
                acc += Tm[r * 65 + s] * bet[s] * expf(gam[s]) * Ks[s * (K + 1) + c];
            ws_w[((cr.bos + r) * H + h) * (long long)K + c] = acc;
        } else {
            const int j = c - K;
            for (int s = 0; s <= r; ++s) acc += Tm[r * 65 + s] * bet[s] * Vs[s * (V + 1) + j];
            ws_u[((cr.bos + r) * H + h) * (long long)V + j] = acc;
        }
    }
}

// ---------------------------------------------------------------- walk
// Walks one (item, head, column block) over its chunks.
//   mode kOut : item = sequence (no CP) or segment (CP).  Writes O columns,
//               optional per-chunk start states, final state on the last item.
//   mode kMap : item = segment; the walked state is the segment's affine map
//               [A | B] (K x (K+V)), started from [I | 0], with u = 0 on the
//               A columns; written to `maps` for non-final segments.
struct WalkArgs {
    const float *ws_gam, *ws_w, *ws_u;
    const float *h0;          // [N, H, K, V] nullable
    const float *seg_start;   // [segs, H, K, V] (CP, kOut) nullable
    const int32_t *warm;      // [N, H] 1 = this head uses the warmup start (CP only)
    int warm_chunks;
    void *o;                  // [tokens, H, V]
    float *final_state;       // [N, H, K, V] nullable
    float *hc;                // [chunks, H, K, V] start state of every chunk, nullable
    float *maps;              // [segs, H, K, K+V] (kMap)
    int cp;                   // items are segments
};
enum { kOut = 0, kMap = 1 };

template <typename TI, int MODE>
__global__ void __launch_bounds__(kThreads)
walk_kernel(Geo g, WalkArgs a) {
    const int h = blockIdx.y, cb = blockIdx.z, K = g.K, V = g.V, H = g.H;
    const int tid = threadIdx.x;
    int n, j = 0, nseg = 1;
    if (a.cp) {
        if (!seg_ref(g, blockIdx.x, n, j)) return;
        nseg = seq_nsegs(g, n);
    } else {
        n = blockIdx.x;
        if (n >= g.N) return;
    }
    if (MODE == kMap && j == nseg - 1) return;           // the last segment needs no map
    if (MODE == kMap && a.warm && a.warm[n * g.H + h]) return;  // warmup heads skip the maps
    const int ncols = (MODE == kMap) ? K + V : V;
    const int col0 = cb * kBV;
    if (col0 >= ncols) return;
    const bool a_cols = (MODE == kMap) && col0 < K;      // columns of A (u = 0, start I)
    const int nc = seq_nchunks(g, n);
    const int c0 = min(nc, j * g.seg_chunks), c1 = min(nc, (j + 1) * g.seg_chunks);
    const int cbase = seq_chunk_base(g, n);
    long long sbos;
    int slen;
    seq_range(g, n, sbos, slen);

    extern __shared__ float sm[];
    float *Hs = sm;                            // [K][kBV]
    float *Qs = Hs + K * kBV;                  // [64][K+1]
    float *Ks = Qs + kChunk * (K + 1);         // [64][K+1]
    float *Ws = Ks + kChunk * (K + 1);         // [64][K+1]
    float *Us = Ws + kChunk * (K + 1);         // [64][kBV+1]
    float *Ps = Us + kChunk * (kBV + 1);       // [64][65]
    float *gam = Ps + kChunk * 65;             // [64]

    // Start state.
    int cstart = c0;
    bool warm = false;
    if (MODE == kOut && a.cp && j > 0 && a.warm && a.warm[n * H + h]) {
        warm = true;
        cstart = max(0, c0 - a.warm_chunks);
    }
    for (int idx = tid; idx < K * kBV; idx += blockDim.x) {
        const int i = idx / kBV, c = col0 + idx % kBV;
        float x = 0.f;
        if (MODE == kMap) {
            x = (a_cols && i == c) ? 1.f : 0.f;
        } else if (warm) {
            x = 0.f;
        } else if (a.cp && j > 0) {
            x = a.seg_start[(((long long)(seq_seg_base(g, n) + j) * H + h) * K + i) * V + c];
        } else if (a.h0) {
            x = a.h0[(((long long)n * H + h) * K + i) * V + c];
        }
        Hs[idx] = x;
    }
    __syncthreads();

    for (int c = cstart; c < c1; ++c) {
        const bool emit = (MODE == kOut) && a.o && c >= c0;
        const long long bos = sbos + (long long)c * kChunk;
        const int L = min(kChunk, slen - c * kChunk);
        if (emit) load_rows(Qs, K + 1, (const TI *)g.q, bos, L, H, h, K, g.l2norm, nullptr);
        load_rows(Ks, K + 1, (const TI *)g.k, bos, L, H, h, K, g.l2norm, nullptr);
        for (int idx = tid; idx < L * K; idx += blockDim.x) {
            const int r = idx / K, i = idx % K;
            Ws[r * (K + 1) + i] = a.ws_w[((bos + r) * H + h) * (long long)K + i];
        }
        for (int r = tid; r < L; r += blockDim.x) gam[r] = a.ws_gam[(bos + r) * H + h];
        __syncthreads();
        // U = u - W H
        for (int idx = tid; idx < L * kBV; idx += blockDim.x) {
            const int r = idx / kBV, jj = idx % kBV;
            float acc = 0.f;
            if (!a_cols) {
                const int vc = (MODE == kMap) ? col0 - K + jj : col0 + jj;
                acc = a.ws_u[((bos + r) * H + h) * (long long)V + vc];
            }
            for (int i = 0; i < K; ++i) acc -= Ws[r * (K + 1) + i] * Hs[i * kBV + jj];
            Us[r * (kBV + 1) + jj] = acc;
        }
        if (emit) {
            for (int idx = tid; idx < L * L; idx += blockDim.x) {
                const int r = idx / L, s = idx % L;
                float p = 0.f;
                if (s <= r) {
                    for (int i = 0; i < K; ++i) p += Qs[r * (K + 1) + i] * Ks[s * (K + 1) + i];
                    p *= expf(gam[r] - gam[s]);
                }
                Ps[r * 65 + s] = p;
            }
        }
        if (MODE == kOut && a.hc && c >= c0) {
            float *dst = a.hc + ((long long)(cbase + c) * H + h) * K * V;
            for (int idx = tid; idx < K * kBV; idx += blockDim.x)
                dst[(idx / kBV) * V + col0 + idx % kBV] = Hs[idx];
        }
        __syncthreads();
        if (emit) {
            TI *o = (TI *)a.o;
            for (int idx = tid; idx < L * kBV; idx += blockDim.x) {
                const int r = idx / kBV, jj = idx % kBV;
                float inter = 0.f, intra = 0.f;
                for (int i = 0; i < K; ++i) inter += Qs[r * (K + 1) + i] * Hs[i * kBV + jj];
                for (int s = 0; s <= r; ++s) intra += Ps[r * 65 + s] * Us[s * (kBV + 1) + jj];
                from_f(o + ((bos + r) * H + h) * (long long)V + col0 + jj,
                       g.scale * (expf(gam[r]) * inter + intra));
            }
        }
        __syncthreads();
        const float gl = gam[L - 1];
        for (int idx = tid; idx < K * kBV; idx += blockDim.x) {
            const int i = idx / kBV, jj = idx % kBV;
            float acc = expf(gl) * Hs[idx];
            for (int r = 0; r < L; ++r)
                acc += Ks[r * (K + 1) + i] * expf(gl - gam[r]) * Us[r * (kBV + 1) + jj];
            Hs[idx] = acc;
        }
        __syncthreads();
    }

    if (MODE == kMap) {
        float *dst = a.maps + ((long long)(seq_seg_base(g, n) + j) * H + h) * K * (K + V);
        for (int idx = tid; idx < K * kBV; idx += blockDim.x)
            dst[(idx / kBV) * (K + V) + col0 + idx % kBV] = Hs[idx];
    } else if (a.final_state && j == nseg - 1) {
        float *dst = a.final_state + ((long long)n * H + h) * K * V;
        for (int idx = tid; idx < K * kBV; idx += blockDim.x)
            dst[(idx / kBV) * V + col0 + idx % kBV] = Hs[idx];
    }
}

// ---------------------------------------------------------------- CP scans
// Exclusive scan of segment maps S -> A S + B over one (sequence, head,
// block of kSB state columns).  Forward (reverse = 0): start[0] = h0 and
// start[j+1] = A_j start[j] + B_j.  Backward (reverse = 1): end[nseg-1] =
// d(final state) and end[j-1] = A'_j end[j] + B'_j.  The maps of the next
// two steps are copied into shared memory (cp.async, three buffers, rows
// padded by 4 floats against bank conflicts) while the current step
// computes.  Thread t owns four of the kSB columns of rows r and r + 64
// (r = (t % 128) / 2) over one half of the contraction index (t / 128); the
// halves meet in shared memory, so each 16-byte read of A or S feeds more FMAs.
constexpr int kSB = 8;
constexpr int kScanStages = 3;

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(
                     (uint32_t)__cvta_generic_to_shared(smem)),
                 "l"(gmem)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// maps_a holds the A parts, K rows of lda floats per (segment, head) (maps
// itself with lda = K + V, or a separate [segs, H, K, K] array with lda = K).
// TA: apply the transpose of each A instead (the backward with a saved forward
// context, whose forward A maps are the reverse ones transposed).
template <int K, bool TA>
__global__ void __launch_bounds__(256)
map_scan_kernel(Geo g, const float *maps, const float *maps_a, int lda, const float *init,
                const int32_t *warm, float *out, int reverse) {
    pdl_enter();
    const int n = blockIdx.x, h = blockIdx.y, col0 = blockIdx.z * kSB, V = g.V, H = g.H;
    if (n >= g.N || col0 >= V) return;
    if (warm && warm[n * H + h]) return;
    const int nseg = seq_nsegs(g, n), sbase = seq_seg_base(g, n);
    extern __shared__ __align__(16) float sm[];
    const int ld = K + 4;                        // padded row stride of the A buffers
    float *Abuf = sm;                            // [kScanStages][K][ld]
    float *Bbuf = Abuf + kScanStages * K * ld;   // [kScanStages][K][kSB]
    float *S = Bbuf + kScanStages * K * kSB;     // [K][kSB]
    float *X = S + K * kSB;                      // [K][kSB] upper-half partial sums
    constexpr int R = K / 64;                    // rows per thread
    const int t = threadIdx.x, kh = t >> 7, r2 = (t & 127) >> 1, jq = (t & 1) * 4;
    auto stage = [&](int step, int buf) {
        const int j = reverse ? nseg - 1 - step : step;
        const long long sh = (long long)(sbase + j) * H + h;
        const float *M = maps + sh * K * (K + V), *MA = maps_a + sh * K * lda;
        float *A = Abuf + buf * K * ld, *Bm = Bbuf + buf * K * kSB;
        constexpr int per_row = K / 4;
#pragma unroll
        for (int m = 0; m < K * per_row / 256; ++m) {
            const int idx = t + 256 * m, row = idx / per_row, c4 = idx % per_row;
            cp_async16(A + row * ld + 4 * c4, MA + (long long)row * lda + 4 * c4);
        }
        if (t < K * (kSB / 4)) {
            const int row = t / (kSB / 4), c4 = t % (kSB / 4);
            cp_async16(Bm + row * kSB + 4 * c4, M + (long long)row * (K + V) + K + col0 + 4 * c4);
        }
        cp_async_commit();
    };
    for (int idx = t; idx < K * kSB; idx += blockDim.x) {
        const int r = idx / kSB, c = col0 + idx % kSB;
        S[idx] = init ? init[(((long long)n * H + h) * K + r) * V + c] : 0.f;
    }
    const int steps = nseg - 1;
    for (int st = 0; st < kScanStages - 1 && st < steps; ++st) stage(st, st);
    for (int step = 0; step < steps; ++step) {
        const int buf = step % kScanStages;
        // the buffer of step - 1 (every thread is past its reads) takes step + 2
        if (step + 2 < steps) {
            stage(step + 2, (step + 2) % kScanStages);
            cp_async_wait<2>();
        } else if (step + 1 < steps) {
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const int j = reverse ? nseg - 1 - step : step;      // map applied
        const int jo = reverse ? j - 1 : j + 1;              // segment that receives the state
        float4 acc[R];
#pragma unroll
        for (int m = 0; m < R; ++m) acc[m] = make_float4(0.f, 0.f, 0.f, 0.f);
        {
            const float *A = Abuf + buf * K * ld;
            const int l0 = kh * (K / 2);
#pragma unroll 4
            for (int l4 = 0; l4 < K / 8; ++l4) {
                const int l = l0 + 4 * l4;
                float4 s4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    s4[e] = *reinterpret_cast<const float4 *>(&S[(l + e) * kSB + jq]);
#pragma unroll
                for (int m = 0; m < R; ++m) {
                    float av[4];
                    if (TA) {            // A^T[row][l + e] = A[l + e][row]
#pragma unroll
                        for (int e = 0; e < 4; ++e) av[e] = A[(l + e) * ld + r2 + 64 * m];
                    } else {
                        const float4 a4 = *reinterpret_cast<const float4 *>(A + (r2 + 64 * m) * ld + l);
                        av[0] = a4.x; av[1] = a4.y; av[2] = a4.z; av[3] = a4.w;
                    }
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[m].x += av[e] * s4[e].x;
                        acc[m].y += av[e] * s4[e].y;
                        acc[m].z += av[e] * s4[e].z;
                        acc[m].w += av[e] * s4[e].w;
                    }
                }
            }
        }
        if (kh == 1) {
#pragma unroll
            for (int m = 0; m < R; ++m)
                *reinterpret_cast<float4 *>(&X[(r2 + 64 * m) * kSB + jq]) = acc[m];
        } else {
            // B now: the next step's prefetch may refill this buffer once all
            // threads are past the barrier below
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const float4 b = *reinterpret_cast<const float4 *>(Bbuf + buf * K * kSB +
                                                                   (r2 + 64 * m) * kSB + jq);
                acc[m] = make_float4(acc[m].x + b.x, acc[m].y + b.y, acc[m].z + b.z, acc[m].w + b.w);
            }
        }
        __syncthreads();
        if (kh == 0) {
#pragma unroll
            for (int m = 0; m < R; ++m) {
                const int i = r2 + 64 * m;
                const float4 x = *reinterpret_cast<const float4 *>(&X[i * kSB + jq]);
                const float4 r = make_float4(acc[m].x + x.x, acc[m].y + x.y, acc[m].z + x.z,
                                             acc[m].w + x.w);
                *reinterpret_cast<float4 *>(&S[i * kSB + jq]) = r;
                float *dst = out + (((long long)(sbase + jo) * H + h) * K + i) * V + col0 + jq;
                *reinterpret_cast<float4 *>(dst) = r;
            }
        }
    }
}

static size_t map_scan_smem(int K) {
    // K in {64, 128}; the kernel is instantiated for both
    return sizeof(float) * (kScanStages * K * (K + 4) + kScanStages * K * kSB + 2 * K * kSB);
}

// Warmup shortcut decision per (sequence, head): every segment j > 0 must
// see its preceding `wc` chunks decay by less than tau, i.e.
// exp(sum of g over those chunks) < tau; then the state entering the
// segment is dominated by the last wc chunks (each step I - beta k k^T has
// norm <= 1 for unit keys and beta in [0, 1]).  Sliding-window warmup as on
// the ollai.cn page ("FlashQLA的技术原理", third item).
// One CTA per (sequence, head); warp w sums the windows of segments
// j = 1 + w, 1 + w + warps, ... and the CTA takes the AND over all of them.
__global__ void warm_decide_kernel(Geo g, int wc, float tau, int32_t *warm, int32_t *stats) {
    const int n = blockIdx.x / g.H, h = blockIdx.x % g.H;
    if (n >= g.N) return;
    long long bos;
    int len;
    seq_range(g, n, bos, len);
    const int nseg = seq_nsegs(g, n);
    const float lt = logf(tau);
    const int lane = threadIdx.x & 31, warps = blockDim.x >> 5;
    int ok = nseg > 1;
    for (int j = 1 + (threadIdx.x >> 5); j < nseg && ok; j += warps) {
        const int t1 = min(len, j * g.seg_chunks * kChunk);
        const int t0 = max(0, t1 - wc * kChunk);
        float s = 0.f;
        for (int t = t0 + lane; t < t1; t += 32) s += decay_at(g, (bos + t) * g.H + h, h);
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        ok = s < lt;
    }
    ok = __syncthreads_and(ok);
    if (threadIdx.x == 0) {
        warm[n * g.H + h] = ok;
        if (stats) {
            if (ok) atomicAdd(stats, 1);
            atomicAdd(stats + 1, 1);
        }
    }
}

// ---------------------------------------------------------------- backward walk
// Reverse walk of the state gradient over one (item, head, column block).
// With dH the gradient at a chunk's end:
//   dU = scale P^T dO + diag(exp(gam_L - gam)) K dH
//   dH <- scale (diag(exp(gam)) Q)^T dO + exp(gam_L) dH - W^T dU
// kOut stores dH at every chunk end (dhc) and d(initial_state) on segment 0;
// kMap walks [A' | B'] (A' = the transposed forward map, dO = 0 on its
// columns) for segments j > 0.
struct DWalkArgs {
    const float *ws_gam, *ws_w;
    const void *d_o;
    const float *dht;        // [N, H, K, V] nullable
    const float *seg_end;    // [segs, H, K, V] (CP, kOut)
    float *dh0;              // nullable
    float *dhc;              // [chunks, H, K, V]
    float *maps;             // [segs, H, K, K+V]
    int cp;
};

template <typename TI, int MODE>
__global__ void __launch_bounds__(kThreads)
dwalk_kernel(Geo g, DWalkArgs a) {
    const int h = blockIdx.y, cb = blockIdx.z, K = g.K, V = g.V, H = g.H, tid = threadIdx.x;
    int n, j = 0, nseg = 1;
    if (a.cp) {
        if (!seg_ref(g, blockIdx.x, n, j)) return;
        nseg = seq_nsegs(g, n);
    } else {
        n = blockIdx.x;
        if (n >= g.N) return;
    }
    if (MODE == kMap && j == 0) return;
    const int ncols = (MODE == kMap) ? K + V : V;
    const int col0 = cb * kBV;
    if (col0 >= ncols) return;
    const bool a_cols = (MODE == kMap) && col0 < K;
    const bool use_do = !a_cols;
    const int vc0 = (MODE == kMap) ? col0 - K : col0;
    const int nc = seq_nchunks(g, n);
    const int c0 = min(nc, j * g.seg_chunks), c1 = min(nc, (j + 1) * g.seg_chunks);
    const int cbase = seq_chunk_base(g, n);
    long long sbos;
    int slen;
    seq_range(g, n, sbos, slen);

    extern __shared__ float sm[];
    float *dH = sm;                            // [K][kBV]
    float *Qs = dH + K * kBV;                  // [64][K+1]
    float *Ks = Qs + kChunk * (K + 1);
    float *Ws = Ks + kChunk * (K + 1);
    float *dO = Ws + kChunk * (K + 1);         // [64][kBV+1]
    float *dU = dO + kChunk * (kBV + 1);       // [64][kBV+1]
    float *Ps = dU + kChunk * (kBV + 1);       // [64][65]
    float *gam = Ps + kChunk * 65;

    for (int idx = tid; idx < K * kBV; idx += blockDim.x) {
        const int i = idx / kBV, c = col0 + idx % kBV;
        float x = 0.f;
        if (MODE == kMap) {
            x = (a_cols && i == c) ? 1.f : 0.f;
        } else if (a.cp && j < nseg - 1) {
            x = a.seg_end[(((long long)(seq_seg_base(g, n) + j) * H + h) * K + i) * V + c];
        } else if (a.dht) {
            x = a.dht[(((long long)n * H + h) * K + i) * V + c];
        }
        dH[idx] = x;
    }
    __syncthreads();

    for (int c = c1 - 1; c >= c0; --c) {
        const long long bos = sbos + (long long)c * kChunk;
        const int L = min(kChunk, slen - c * kChunk);
        if (use_do) load_rows(Qs, K + 1, (const TI *)g.q, bos, L, H, h, K, g.l2norm, nullptr);
        load_rows(Ks, K + 1, (const TI *)g.k, bos, L, H, h, K, g.l2norm, nullptr);
        for (int idx = tid; idx < L * K; idx += blockDim.x) {
            const int r = idx / K, i = idx % K;
            Ws[r * (K + 1) + i] = a.ws_w[((bos + r) * H + h) * (long long)K + i];
        }
        if (use_do) {
            const TI *src = (const TI *)a.d_o;
            for (int idx = tid; idx < L * kBV; idx += blockDim.x) {
                const int r = idx / kBV, jj = idx % kBV;
                dO[r * (kBV + 1) + jj] = to_f(src[((bos + r) * H + h) * (long long)V + vc0 + jj]);
            }
        }
        for (int r = tid; r < L; r += blockDim.x) gam[r] = a.ws_gam[(bos + r) * H + h];
        if (MODE == kOut) {
            float *dst = a.dhc + ((long long)(cbase + c) * H + h) * K * V;
            for (int idx = tid; idx < K * kBV; idx += blockDim.x)
                dst[(idx / kBV) * V + col0 + idx % kBV] = dH[idx];
        }
        __syncthreads();
        if (use_do) {
            for (int idx = tid; idx < L * L; idx += blockDim.x) {
                const int r = idx / L, s = idx % L;
                float p = 0.f;
                if (s <= r) {
                    for (int i = 0; i < K; ++i) p += Qs[r * (K + 1) + i] * Ks[s * (K + 1) + i];
                    p *= expf(gam[r] - gam[s]);
                }
                Ps[r * 65 + s] = p;
            }
        }
        __syncthreads();
        const float gl = gam[L - 1];
        for (int idx = tid; idx < L * kBV; idx += blockDim.x) {
            const int r = idx / kBV, jj = idx % kBV;
            float acc = 0.f;
            if (use_do) {
                for (int rr = r; rr < L; ++rr) acc += Ps[rr * 65 + r] * dO[rr * (kBV + 1) + jj];
                acc *= g.scale;
            }
            float kd = 0.f;
            for (int i = 0; i < K; ++i) kd += Ks[r * (K + 1) + i] * dH[i * kBV + jj];
            dU[r * (kBV + 1) + jj] = acc + expf(gl - gam[r]) * kd;
        }
        __syncthreads();
        for (int idx = tid; idx < K * kBV; idx += blockDim.x) {
            const int i = idx / kBV, jj = idx % kBV;
            float acc = expf(gl) * dH[idx];
            for (int r = 0; r < L; ++r) {
                if (use_do) acc += g.scale * Qs[r * (K + 1) + i] * expf(gam[r]) * dO[r * (kBV + 1) + jj];
                acc -= Ws[r * (K + 1) + i] * dU[r * (kBV + 1) + jj];
            }
            dH[idx] = acc;
        }
        __syncthreads();
    }

    if (MODE == kMap) {
        float *dst = a.maps + ((long long)(seq_seg_base(g, n) + j) * H + h) * K * (K + V);
        for (int idx = tid; idx < K * kBV; idx += blockDim.x)
            dst[(idx / kBV) * (K + V) + col0 + idx % kBV] = dH[idx];
    } else if (a.dh0 && j == 0) {
        float *dst = a.dh0 + ((long long)n * H + h) * K * V;
        for (int idx = tid; idx < K * kBV; idx += blockDim.x)
            dst[(idx / kBV) * V + col0 + idx % kBV] = dH[idx];
    }
}

// ---------------------------------------------------------------- local gradients
// Per (chunk, head), from the chunk's start state H0 (hc) and the gradient
// at its end dHL (dhc); chain rule through the chunk form above:
//   dU  = scale P^T dO + diag(f) K dHL            (f_r = exp(gam_L - gam_r))
//   dS  = scale (dO U^T) .* lower_incl .* D        (gradient of Q K^T)
//   dW  = -dU H0^T,  dYw = T^T dW,  dYu = T^T dU
//   dT  = dU (diag(beta) V)^T + dW (diag(beta e) K)^T,  dA = -T^T dT T^T (strict lower)
//   G   = dA .* D .* beta_r                        (gradient of K K^T)
//   dQ  = scale diag(e) dO H0^T + dS K
//   dK  = dS^T Q + diag(f) U dHL^T + diag(beta e) dYw + (G + G^T) K
//   dV  = diag(beta) dYu
//   dbeta_r = <dYu_r, v_r> + e_r <dYw_r, k_r> + sum_s dA_rs (K K^T)_rs D_rs
//   dgam from every exp(gam ...) factor; dg = reverse cumsum of dgam in the chunk
// followed by the L2-norm backward when q, k were normalised.
struct LocalArgs {
    const float *ws_gam, *hc, *dhc;
    const void *ws_w, *ws_u;         // fp32 or bf16 (template TW)
    const void *d_o;
    void *dq, *dk, *dv;
    float *dg, *dbeta;
    float *scratch;          // per CTA: 64 * (3V + 2K) floats
    int n_items;             // chunk capacity * H
};

template <typename TI, typename TG, typename TW>
__global__ void __launch_bounds__(kThreads)
local_grad_kernel(Geo g, LocalArgs a) {
    const int K = g.K, V = g.V, H = g.H, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const float scale = g.scale;
    extern __shared__ float sm[];
    float *Qs = sm;                          // [64][K+1] normalised q
    float *Ks = Qs + kChunk * (K + 1);       // [64][K+1] normalised k
    float *QK = Ks + kChunk * (K + 1);       // [64][65]
    float *KK = QK + kChunk * 65;
    float *Tm = KK + kChunk * 65;
    float *Dm = Tm + kChunk * 65;            // D on lower_incl, 0 above
    float *M1 = Dm + kChunk * 65;            // A, then dS
    float *M2 = M1 + kChunk * 65;            // dT, then dA
    float *M3 = M2 + kChunk * 65;            // dT T^T, then G
    float *gam = M3 + kChunk * 65;
    float *e = gam + kChunk, *f = e + kChunk, *bet = f + kChunk;
    float *rq = bet + kChunk, *rk = rq + kChunk;
    float *rowA = rk + kChunk, *rowB = rowA + kChunk;   // heavy per-row dgam terms
    float *red = rowB + kChunk;                         // [32]
    float *U = a.scratch + (long long)blockIdx.x * kChunk * (3 * V + 2 * K);
    float *dU = U + kChunk * V, *dYu = dU + kChunk * V, *dW = dYu + kChunk * V,
          *dYw = dW + kChunk * K;
    const TI *vin = (const TI *)g.v;
    const TI *dOin = (const TI *)a.d_o;

    for (int item = blockIdx.x; item < a.n_items; item += gridDim.x) {
        const int ci = item / H, h = item % H;
        ChunkRef cr;
        if (!chunk_ref(g, ci, cr)) break;
        const int L = cr.len;
        const long long bos = cr.bos;
        // chunk states: fp32 [K][V] from the CUDA-core walks, bf16 transposed tiles
        // [k half][v][64] from the tensor-core walks (K = V = 128 there)
        const long long hoff = ((long long)ci * H + h) * K * V;
        const float *hc32 = a.hc + hoff, *dhc32 = a.dhc + hoff;
        const __nv_bfloat16 *hc16 = (const __nv_bfloat16 *)a.hc + hoff,
                            *dhc16 = (const __nv_bfloat16 *)a.dhc + hoff;
        auto tile_at = [&](int i, int j) { return ((i >> 6) * V + j) * 64 + (i & 63); };
        auto H0at = [&](int i, int j) {
            return sizeof(TW) == 4 ? hc32[i * V + j] : __bfloat162float(hc16[tile_at(i, j)]);
        };
        auto dHLat = [&](int i, int j) {
            return sizeof(TW) == 4 ? dhc32[i * V + j] : __bfloat162float(dhc16[tile_at(i, j)]);
        };
        auto dOat = [&](int r, int j) { return to_f(dOin[((bos + r) * H + h) * (long long)V + j]); };
        auto Vat = [&](int r, int j) { return to_f(vin[((bos + r) * H + h) * (long long)V + j]); };

        load_rows(Qs, K + 1, (const TI *)g.q, bos, L, H, h, K, g.l2norm, rq);
        load_rows(Ks, K + 1, (const TI *)g.k, bos, L, H, h, K, g.l2norm, rk);
        for (int r = tid; r < L; r += blockDim.x) {
            gam[r] = a.ws_gam[(bos + r) * H + h];
            bet[r] = g.beta[(bos + r) * H + h];
        }
        __syncthreads();
        for (int r = tid; r < L; r += blockDim.x) {
            e[r] = expf(gam[r]);
            f[r] = expf(gam[L - 1] - gam[r]);
        }
        for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
            const int r = idx / kChunk, s = idx % kChunk;
            float qk = 0.f, kk = 0.f, d = 0.f;
            if (r < L && s < L) {
                for (int i = 0; i < K; ++i) {
                    qk += Qs[r * (K + 1) + i] * Ks[s * (K + 1) + i];
                    kk += Ks[r * (K + 1) + i] * Ks[s * (K + 1) + i];
                }
                if (s <= r) d = expf(gam[r] - gam[s]);
            }
            QK[r * 65 + s] = qk;
            KK[r * 65 + s] = kk;
            Dm[r * 65 + s] = d;
        }
        __syncthreads();
        for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
            const int r = idx / kChunk, s = idx % kChunk;
            M1[r * 65 + s] = (s < r) ? bet[r] * KK[r * 65 + s] * Dm[r * 65 + s] : 0.f;
        }
        __syncthreads();
        unit_lower_inverse(Tm, M1, L);

        // W and u: fp32 token rows from the CUDA-core forward, bf16 transposed
        // chunk tiles [chunk][H][feature][64 rows] from the tensor-core forward
        const TW *wsw = (const TW *)a.ws_w, *wsu = (const TW *)a.ws_u;
        auto Wat = [&](int r, int i) {
            return sizeof(TW) == 4 ? to_f(wsw[((bos + r) * H + h) * (long long)K + i])
                                   : to_f(wsw[(((long long)ci * H + h) * K + i) * kChunk + r]);
        };
        auto uat = [&](int r, int j) {
            return sizeof(TW) == 4 ? to_f(wsu[((bos + r) * H + h) * (long long)V + j])
                                   : to_f(wsu[(((long long)ci * H + h) * V + j) * kChunk + r]);
        };
        // U = u - W H0 ; dU = scale P^T dO + diag(f) K dHL
        for (int idx = tid; idx < L * V; idx += blockDim.x) {
            const int r = idx / V, j = idx % V;
            float u = uat(r, j);
            float kd = 0.f;
            for (int i = 0; i < K; ++i) {
                u -= Wat(r, i) * H0at(i, j);
                kd += Ks[r * (K + 1) + i] * dHLat(i, j);
            }
            float pd = 0.f;
            for (int rr = r; rr < L; ++rr) pd += QK[rr * 65 + r] * Dm[rr * 65 + r] * dOat(rr, j);
            U[r * V + j] = u;
            dU[r * V + j] = scale * pd + f[r] * kd;
        }
        __syncthreads();
        // dS ; dW
        for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
            const int r = idx / kChunk, s = idx % kChunk;
            float ds = 0.f;
            if (r < L && s <= r) {
                for (int j = 0; j < V; ++j) ds += dOat(r, j) * U[s * V + j];
                ds *= scale * Dm[r * 65 + s];
            }
            M1[r * 65 + s] = ds;
        }
        for (int idx = tid; idx < L * K; idx += blockDim.x) {
            const int r = idx / K, i = idx % K;
            float acc = 0.f;
            for (int j = 0; j < V; ++j) acc += dU[r * V + j] * H0at(i, j);
            dW[r * K + i] = -acc;
        }
        __syncthreads();
        // dYw = T^T dW ; dYu = T^T dU ; dT (strict lower)
        for (int idx = tid; idx < L * K; idx += blockDim.x) {
            const int s = idx / K, i = idx % K;
            float acc = 0.f;
            for (int r = s; r < L; ++r) acc += Tm[r * 65 + s] * dW[r * K + i];
            dYw[s * K + i] = acc;
        }
        for (int idx = tid; idx < L * V; idx += blockDim.x) {
            const int s = idx / V, j = idx % V;
            float acc = 0.f;
            for (int r = s; r < L; ++r) acc += Tm[r * 65 + s] * dU[r * V + j];
            dYu[s * V + j] = acc;
        }
        for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
            const int r = idx / kChunk, s = idx % kChunk;
            float dt = 0.f;
            if (r < L && s < r) {
                float a1 = 0.f, a2 = 0.f;
                for (int j = 0; j < V; ++j) a1 += dU[r * V + j] * Vat(s, j);
                for (int i = 0; i < K; ++i) a2 += dW[r * K + i] * Ks[s * (K + 1) + i];
                dt = bet[s] * (a1 + e[s] * a2);
            }
            M2[r * 65 + s] = dt;
        }
        __syncthreads();
        // X = dT T^T (into M3), then dA = -T^T X (into M2, strict lower)
        for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
            const int r = idx / kChunk, s = idx % kChunk;
            float acc = 0.f;
            if (r < L && s < L)
                for (int b = 0; b <= s; ++b) acc += M2[r * 65 + b] * Tm[s * 65 + b];
            M3[r * 65 + s] = acc;
        }
        __syncthreads();
        for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
            const int r = idx / kChunk, s = idx % kChunk;
            float acc = 0.f;
            if (r < L && s < r)
                for (int q = r; q < L; ++q) acc += Tm[q * 65 + r] * M3[q * 65 + s];
            M2[r * 65 + s] = -acc;
        }
        __syncthreads();
        for (int idx = tid; idx < kChunk * kChunk; idx += blockDim.x) {
            const int r = idx / kChunk, s = idx % kChunk;
            M3[r * 65 + s] = (s < r) ? M2[r * 65 + s] * bet[r] * Dm[r * 65 + s] : 0.f;
        }
        // heavy per-row terms: rowA = scale e_r <dO_r, H0^T q_r>, rowB = f_r <k_r, dHL U_r>
        for (int r = warp; r < L; r += nw) {
            float sa = 0.f, sb = 0.f;
            for (int j = lane; j < V; j += 32) {
                float qh = 0.f, kd = 0.f;
                for (int i = 0; i < K; ++i) {
                    qh += Qs[r * (K + 1) + i] * H0at(i, j);
                    kd += Ks[r * (K + 1) + i] * dHLat(i, j);
                }
                sa += dOat(r, j) * qh;
                sb += kd * U[r * V + j];
            }
            for (int o = 16; o > 0; o >>= 1) {
                sa += __shfl_xor_sync(0xffffffffu, sa, o);
                sb += __shfl_xor_sync(0xffffffffu, sb, o);
            }
            if (lane == 0) {
                rowA[r] = scale * e[r] * sa;
                rowB[r] = f[r] * sb;
            }
        }
        // <dHL, H0>
        float part = 0.f;
        for (int idx = tid; idx < K * V; idx += blockDim.x)
            part += dHLat(idx / V, idx % V) * H0at(idx / V, idx % V);
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) red[warp] = part;
        __syncthreads();
        // per-row dbeta and dgam (thread r), then the reverse cumsum
        if (tid < L) {
            const int r = tid;
            float yu = 0.f, yw = 0.f;
            for (int j = 0; j < V; ++j) yu += dYu[r * V + j] * Vat(r, j);
            for (int i = 0; i < K; ++i) yw += dYw[r * K + i] * Ks[r * (K + 1) + i];
            float db = yu + e[r] * yw, dgm = bet[r] * e[r] * yw + rowA[r] - rowB[r];
            for (int s = 0; s < L; ++s) {
                if (s <= r) dgm += M1[r * 65 + s] * QK[r * 65 + s];     // z row
                if (s >= r) dgm -= M1[s * 65 + r] * QK[s * 65 + r];     // z column
                if (s < r) {
                    db += M2[r * 65 + s] * KK[r * 65 + s] * Dm[r * 65 + s];
                    dgm += M3[r * 65 + s] * KK[r * 65 + s];             // z' row
                }
                if (s > r) dgm -= M3[s * 65 + r] * KK[s * 65 + r];      // z' column
            }
            rowA[r] = dgm;
            a.dbeta[(bos + r) * H + h] = db;
        }
        __syncthreads();
        if (tid == 0) {
            float tail = 0.f, zsum = 0.f;
            for (int w = 0; w < nw; ++w) tail += red[w];
            for (int r = 0; r < L; ++r) zsum += rowB[r];
            rowA[L - 1] += expf(gam[L - 1]) * tail + zsum;
            float acc = 0.f;
            for (int r = L - 1; r >= 0; --r) {
                acc += rowA[r];
                a.dg[(bos + r) * H + h] = acc;
            }
        }
        // dQ, dK (warp per row, with the L2-norm backward), dV
        TG *dq = (TG *)a.dq, *dk = (TG *)a.dk, *dv = (TG *)a.dv;
        for (int r = warp; r < L; r += nw) {
            float gq[4], gk[4];                 // K <= 128: 4 per lane
            float pq = 0.f, pk = 0.f;
            for (int t = 0; t < K / 32; ++t) {
                const int i = lane + 32 * t;
                float aq = 0.f, ak = 0.f;
                for (int j = 0; j < V; ++j) {
                    aq += dOat(r, j) * H0at(i, j);
                    ak += U[r * V + j] * dHLat(i, j);
                }
                aq *= scale * e[r];
                ak = f[r] * ak + bet[r] * e[r] * dYw[r * K + i];
                for (int s = 0; s <= r; ++s) aq += M1[r * 65 + s] * Ks[s * (K + 1) + i];
                for (int s = r; s < L; ++s) ak += M1[s * 65 + r] * Qs[s * (K + 1) + i];
                for (int s = 0; s < L; ++s)
                    ak += (M3[r * 65 + s] + M3[s * 65 + r]) * Ks[s * (K + 1) + i];
                gq[t] = aq;
                gk[t] = ak;
                pq += aq * Qs[r * (K + 1) + i];
                pk += ak * Ks[r * (K + 1) + i];
            }
            if (g.l2norm) {
                for (int o = 16; o > 0; o >>= 1) {
                    pq += __shfl_xor_sync(0xffffffffu, pq, o);
                    pk += __shfl_xor_sync(0xffffffffu, pk, o);
                }
            }
            for (int t = 0; t < K / 32; ++t) {
                const int i = lane + 32 * t;
                float xq = gq[t], xk = gk[t];
                if (g.l2norm) {
                    xq = (xq - Qs[r * (K + 1) + i] * pq) * rq[r];
                    xk = (xk - Ks[r * (K + 1) + i] * pk) * rk[r];
                }
                from_f(dq + ((bos + r) * H + h) * (long long)K + i, xq);
                from_f(dk + ((bos + r) * H + h) * (long long)K + i, xk);
            }
        }
        for (int idx = tid; idx < L * V; idx += blockDim.x) {
            const int r = idx / V, j = idx % V;
            from_f(dv + ((bos + r) * H + h) * (long long)V + j, bet[r] * dYu[r * V + j]);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- tables
// Validates cu_seqlens and writes chunk offsets (and segment offsets when
// seg_chunks > 0).  One CTA; a serial pass over N sequences.
__global__ void tables_kernel(const int32_t *cu, int N, int T, int seg_chunks,
                              int32_t *chunk_off, int32_t *seg_off, int *status) {
    if (threadIdx.x != 0) return;
    int bad = cu[0] != 0 || cu[N] != T;
    int co = 0, so = 0;
    chunk_off[0] = 0;
    if (seg_off) seg_off[0] = 0;
    for (int n = 0; n < N; ++n) {
        const int len = cu[n + 1] - cu[n];
        if (len < 0) bad = 1;
        const int nc = len > 0 ? (len + kChunk - 1) / kChunk : 0;
        co += nc;
        chunk_off[n + 1] = co;
        if (seg_off) {
            so += nc > 0 ? (nc + seg_chunks - 1) / seg_chunks : 1;
            seg_off[n + 1] = so;
        }
    }
    if (bad) {
        set_status(status, GDN_ERR_BAD_SEQLENS);
        // leave an empty problem so that every later kernel exits at once
        for (int n = 0; n <= N; ++n) {
            chunk_off[n] = 0;
            if (seg_off) seg_off[n] = 0;
        }
    }
}

// Sequences ranked by chunk count, longest first (ties by index): thread n
// counts the sequences that go before it and writes n at that rank.  O(N^2)
// work, so beyond kOrderMax sequences the order is left as given.
constexpr int kOrderMax = 8192;
__global__ void order_kernel(const int32_t *chunk_off, int N, int32_t *order) {
    const int n = blockIdx.x * blockDim.x + threadIdx.x;
    if (n >= N) return;
    if (N > kOrderMax) {
        order[n] = n;
        return;
    }
    const int mine = chunk_off[n + 1] - chunk_off[n];
    int rank = 0;
    for (int m = 0; m < N; ++m) {
        const int other = chunk_off[m + 1] - chunk_off[m];
        rank += (other > mine || (other == mine && m < n)) ? 1 : 0;
    }
    order[rank] = n;
}

}  // namespace simt

// ---------------------------------------------------------------- launchers
namespace simt {

size_t scratch_floats_per_cta(int K, int V) { return (size_t)kChunk * (3 * V + 2 * K); }

static size_t prep_smem(int K, int V) {
    return sizeof(float) * (kChunk * (K + 1) + kChunk * (V + 1) + 2 * kChunk * 65 + 2 * kChunk);
}
static size_t walk_smem(int K) {
    return sizeof(float) * (K * kBV + 3 * kChunk * (K + 1) + kChunk * (kBV + 1) + kChunk * 65 +
                            kChunk);
}
static size_t dwalk_smem(int K) {
    return sizeof(float) * (K * kBV + 3 * kChunk * (K + 1) + 2 * kChunk * (kBV + 1) +
                            kChunk * 65 + kChunk);
}
static size_t local_smem(int K) {
    return sizeof(float) * (2 * kChunk * (K + 1) + 7 * kChunk * 65 + 8 * kChunk + 32);
}

#define GDN_LAUNCH(name, kernel, grid, smem, stream, ...)                                    \
    do {                                                                                     \
        cudaError_t e_ = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                              (int)(smem));                                  \
        if (e_ != cudaSuccess) return e_;                                                    \
        if ((grid).x > 0 && (grid).y > 0 && (grid).z > 0) {                                   \
            prof_before(name, stream);                                                       \
            kernel<<<(grid), kThreads, (smem), (stream)>>>(__VA_ARGS__);                     \
            prof_after(stream);                                                              \
        }                                                                                    \
        e_ = cudaGetLastError();                                                             \
        if (e_ != cudaSuccess) return e_;                                                    \
    } while (0)

// Same with programmatic stream serialization, for kernels that begin with pdl_enter().
#define GDN_LAUNCH_PDL(name, kernel, grid, smem, stream, ...)                                \
    do {                                                                                     \
        cudaError_t e_ = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, \
                                              (int)(smem));                                  \
        if (e_ != cudaSuccess) return e_;                                                    \
        if ((grid).x > 0 && (grid).y > 0 && (grid).z > 0) {                                   \
            prof_before(name, stream);                                                       \
            e_ = launch_pdl(kernel, (grid), dim3(kThreads), (size_t)(smem), (stream), __VA_ARGS__); \
            if (e_ != cudaSuccess) return e_;                                                \
            prof_after(stream);                                                              \
        }                                                                                    \
    } while (0)

cudaError_t tables(const Plan &p, cudaStream_t s) {
    if (!p.g.cu) return cudaSuccess;
    prof_before("tables", s);
    tables_kernel<<<1, 32, 0, s>>>(p.g.cu, p.g.N, p.g.T, p.cp ? p.g.seg_chunks : 0,
                                   p.ws.chunk_off, p.cp ? p.ws.seg_off : nullptr, p.g.status);
    if (p.ws.order)
        order_kernel<<<(p.g.N + 255) / 256, 256, 0, s>>>(p.ws.chunk_off, p.g.N, p.ws.order);
    prof_after(s);
    return cudaGetLastError();
}

template <typename TI>
static cudaError_t forward_t(const Plan &p, cudaStream_t s, bool states_only) {
    const Geo &g = p.g;
    const int H = g.H, K = g.K, V = g.V;
    GDN_LAUNCH("simt_prep", prep_kernel<TI>, dim3(p.max_chunks, H, 1), prep_smem(K, V), s, g, p.ws.gam,
               (float *)p.ws.w, (float *)p.ws.u);
    WalkArgs a{};
    a.ws_gam = p.ws.gam;
    a.ws_w = (const float *)p.ws.w;
    a.ws_u = (const float *)p.ws.u;
    a.h0 = p.h0;
    a.o = states_only ? nullptr : p.o;
    a.final_state = states_only ? nullptr : p.final_state;
    a.hc = states_only ? p.ws.hc : nullptr;
    if (p.cp) {
        a.cp = 1;
        a.maps = p.ws.maps;
        a.seg_start = p.ws.seg_state;
        if (p.warm_chunks > 0 && !states_only) {
            prof_before("warm_decide", s);
            warm_decide_kernel<<<g.N * g.H, 128, 0, s>>>(g, p.warm_chunks, p.warm_tau, p.ws.warm,
                                                 p.cp_stats);
            prof_after(s);
            cudaError_t e = cudaGetLastError();
            if (e != cudaSuccess) return e;
            a.warm = p.ws.warm;
            a.warm_chunks = p.warm_chunks;
        }
        GDN_LAUNCH("simt_walk_map", (walk_kernel<TI, kMap>), dim3(p.max_segs, H, (K + V) / kBV), walk_smem(K), s,
                   g, a);
        GDN_LAUNCH_PDL("map_scan", (K == 128 ? map_scan_kernel<128, false> : map_scan_kernel<64, false>), dim3(g.N, H, V / kSB), map_scan_smem(K), s, g,
                   (const float *)p.ws.maps, (const float *)p.ws.maps, K + V, p.h0, (const int32_t *)a.warm, p.ws.seg_state, 0);
        GDN_LAUNCH(states_only ? "simt_walk_states" : "simt_walk_out", (walk_kernel<TI, kOut>), dim3(p.max_segs, H, V / kBV), walk_smem(K), s, g, a);
    } else {
        GDN_LAUNCH(states_only ? "simt_walk_states" : "simt_walk_out", (walk_kernel<TI, kOut>), dim3(g.N, H, V / kBV), walk_smem(K), s, g, a);
    }
    return cudaSuccess;
}

// Gate backward over every token of head h (one CTA per head): with the log
// decay -a_h softplus(x), dx = dg * (-a_h sigmoid(x)) replaces dg, and
// d a_h = sum over tokens of dg * (-softplus(x)) (a fixed-order block sum).
__global__ void __launch_bounds__(256)
gate_bwd_kernel(const float *x, const float *a, float *dg, float *da, long long tokens, int H) {
    const int h = blockIdx.x;
    __shared__ float part[256];
    float acc = 0.f;
    for (long long t = threadIdx.x; t < tokens; t += blockDim.x) {
        const long long i = t * H + h;
        const float xv = x[i], d = dg[i];
        const float sp = xv > 0.f ? xv + log1pf(expf(-xv)) : log1pf(expf(xv));
        dg[i] = -a[h] * d / (1.f + expf(-xv));
        acc -= d * sp;
    }
    part[threadIdx.x] = acc;
    __syncthreads();
    for (int o = 128; o > 0; o >>= 1) {
        if ((int)threadIdx.x < o) part[threadIdx.x] += part[threadIdx.x + o];
        __syncthreads();
    }
    if (threadIdx.x == 0 && da) da[h] = part[0];
}

cudaError_t gate_bwd(const Plan &p, const float *gate_scale, float *d_gate_scale, cudaStream_t s) {
    const long long tokens = (long long)p.g.B * p.g.T;
    if (tokens <= 0 || p.g.H <= 0) {
        if (d_gate_scale && p.g.H > 0) return cudaMemsetAsync(d_gate_scale, 0, sizeof(float) * p.g.H, s);
        return cudaSuccess;
    }
    prof_before("gate_bwd", s);
    gate_bwd_kernel<<<p.g.H, 256, 0, s>>>(p.g.g, gate_scale, p.dg, d_gate_scale, tokens, p.g.H);
    prof_after(s);
    return cudaGetLastError();
}

cudaError_t warm_decide(const Plan &p, cudaStream_t s) {
    prof_before("warm_decide", s);
    warm_decide_kernel<<<p.g.N * p.g.H, 128, 0, s>>>(p.g, p.warm_chunks, p.warm_tau, p.ws.warm,
                                             p.cp_stats);
    prof_after(s);
    return cudaGetLastError();
}

cudaError_t cp_scan(const Plan &p, const int32_t *warm, cudaStream_t s) {
    const Geo &g = p.g;
    GDN_LAUNCH_PDL("map_scan", (g.K == 128 ? map_scan_kernel<128, false> : map_scan_kernel<64, false>), dim3(g.N, g.H, g.V / kSB), map_scan_smem(g.K), s, g,
               (const float *)p.ws.maps,
               (const float *)(p.ws.fwd_maps ? p.ws.fwd_maps : p.ws.maps),
               p.ws.fwd_maps ? g.K : g.K + g.V, p.h0, warm, p.ws.seg_state, 0);
    return cudaSuccess;
}

cudaError_t forward(const Plan &p, cudaStream_t s) {
    cudaError_t e = tables(p, s);
    if (e != cudaSuccess) return e;
    return p.dtype == GDN_BF16 ? forward_t<__nv_bfloat16>(p, s, false)
                               : forward_t<float>(p, s, false);
}

template <typename TI, typename TG, typename TW>
static cudaError_t local_grads_t(const Plan &p, cudaStream_t s) {
    const Geo &g = p.g;
    LocalArgs l{};
    l.ws_gam = p.ws.gam;
    l.ws_w = p.ws.w;
    l.ws_u = p.ws.u;
    l.hc = p.ws.hc;
    l.dhc = p.ws.dhc;
    l.d_o = p.d_o;
    l.dq = p.dq;
    l.dk = p.dk;
    l.dv = p.dv;
    l.dg = p.dg;
    l.dbeta = p.dbeta;
    l.scratch = p.ws.scratch;
    l.n_items = p.max_chunks * g.H;
    const int grid = l.n_items < p.scratch_ctas ? l.n_items : p.scratch_ctas;
    GDN_LAUNCH("simt_local_grad", (local_grad_kernel<TI, TG, TW>), dim3(grid, 1, 1),
               local_smem(g.K), s, g, l);
    return cudaSuccess;
}

template <typename TI, typename TG>
static cudaError_t backward_t(const Plan &p, cudaStream_t s) {
    cudaError_t e = forward_t<TI>(p, s, true);   // recompute W, u, gam and chunk start states
    if (e != cudaSuccess) return e;
    const Geo &g = p.g;
    const int H = g.H, K = g.K, V = g.V;
    DWalkArgs d{};
    d.ws_gam = p.ws.gam;
    d.ws_w = (const float *)p.ws.w;
    d.d_o = p.d_o;
    d.dht = p.dht;
    d.dh0 = p.dh0;
    d.dhc = p.ws.dhc;
    d.maps = p.ws.maps;
    d.seg_end = p.ws.seg_state;
    if (p.cp) {
        d.cp = 1;
        GDN_LAUNCH("simt_dwalk_map", (dwalk_kernel<TI, kMap>), dim3(p.max_segs, H, (K + V) / kBV), dwalk_smem(K), s,
                   g, d);
        GDN_LAUNCH_PDL("map_rscan", (K == 128 ? map_scan_kernel<128, false> : map_scan_kernel<64, false>), dim3(g.N, H, V / kSB), map_scan_smem(K), s, g,
                   (const float *)p.ws.maps, (const float *)p.ws.maps, K + V, p.dht, (const int32_t *)nullptr, p.ws.seg_state, 1);
        GDN_LAUNCH("simt_dwalk_out", (dwalk_kernel<TI, kOut>), dim3(p.max_segs, H, V / kBV), dwalk_smem(K), s, g,
                   d);
    } else {
        GDN_LAUNCH("simt_dwalk_out", (dwalk_kernel<TI, kOut>), dim3(g.N, H, V / kBV), dwalk_smem(K), s, g, d);
    }
    return local_grads_t<TI, TG, float>(p, s);
}

cudaError_t cp_rscan(const Plan &p, cudaStream_t s, const float *fwd_maps) {
    const Geo &g = p.g;
    if (fwd_maps) {
        // A'_j = A_j^T from the forward's A maps ([segs, H, K, K]); B'_j from this
        // backward's walk
        GDN_LAUNCH_PDL("map_rscan", (g.K == 128 ? map_scan_kernel<128, true> : map_scan_kernel<64, true>), dim3(g.N, g.H, g.V / kSB), map_scan_smem(g.K), s, g,
                   (const float *)p.ws.maps, fwd_maps, g.K, p.dht, (const int32_t *)nullptr, p.ws.seg_state, 1);
    } else {
        GDN_LAUNCH_PDL("map_rscan", (g.K == 128 ? map_scan_kernel<128, false> : map_scan_kernel<64, false>), dim3(g.N, g.H, g.V / kSB), map_scan_smem(g.K), s, g,
                   (const float *)p.ws.maps, (const float *)p.ws.maps, g.K + g.V, p.dht, (const int32_t *)nullptr, p.ws.seg_state, 1);
    }
    return cudaSuccess;
}

cudaError_t backward(const Plan &p, cudaStream_t s) {
    cudaError_t e = tables(p, s);
    if (e != cudaSuccess) return e;
    if (p.dtype == GDN_BF16)
        return p.grad_dtype == GDN_BF16 ? backward_t<__nv_bfloat16, __nv_bfloat16>(p, s)
                                        : backward_t<__nv_bfloat16, float>(p, s);
    return p.grad_dtype == GDN_BF16 ? backward_t<float, __nv_bfloat16>(p, s)
                                    : backward_t<float, float>(p, s);
}

}  // namespace simt
}  // namespace gdn
