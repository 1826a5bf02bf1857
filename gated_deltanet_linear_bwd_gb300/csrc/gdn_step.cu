// gdn_step.cu -- one decode step of the gated delta rule per (sequence, head),
// the state updated in place.  It reads and writes the K x V fp32 state once,
// so it is bound by HBM.  Every warp works alone, with no CTA barrier: it
// takes (sequence, head, 16-column slice) items in turn, holds the slice's
// K x 16 block in registers (16-byte pieces of 64-byte row runs), reduces the
// column sums Hbar^T k and H^T q over its lanes by shuffles, and writes the
// new block back in place.  The eight warps of a CTA take adjacent slices (the
// eight of one (sequence, head) when V = 128), so the state's rows are read
// whole at about the same time; the warps of the persistent grid share the
// items to within one.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"

namespace gdn {
namespace step {

namespace {
struct StepArgs {
    const void *q, *k, *v;
    const float *g, *beta, *gate_a;
    float *state;
    void *o;
    int N, H;
    float scale;
    int l2norm;
};

constexpr int kWarps = 8;  // per CTA
constexpr int kSlice = 16; // state columns per item

// `n` consecutive elements from `p + i` (n = 2 or 4, 16-byte aligned for
// fp32 and 8-byte for bf16 at the offsets used here).
template <typename T, int n>
__device__ __forceinline__ void ld_vec(const void *p, long long i, float *x) {
    const T *s = reinterpret_cast<const T *>(p) + i;
    if constexpr (sizeof(T) == 4) {
        if constexpr (n == 4) {
            const float4 a = *reinterpret_cast<const float4 *>(s);
            x[0] = a.x, x[1] = a.y, x[2] = a.z, x[3] = a.w;
        } else {
            const float2 a = *reinterpret_cast<const float2 *>(s);
            x[0] = a.x, x[1] = a.y;
        }
    } else {
        if constexpr (n == 4) {
            const uint2 a = *reinterpret_cast<const uint2 *>(s);
            const __nv_bfloat162 b0 = *reinterpret_cast<const __nv_bfloat162 *>(&a.x);
            const __nv_bfloat162 b1 = *reinterpret_cast<const __nv_bfloat162 *>(&a.y);
            x[0] = __low2float(b0), x[1] = __high2float(b0);
            x[2] = __low2float(b1), x[3] = __high2float(b1);
        } else {
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(s);
            x[0] = __low2float(b), x[1] = __high2float(b);
        }
    }
}

__device__ __forceinline__ void store4(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 x) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(x.x, x.y), hi = __floats2bfloat162_rn(x.z, x.w);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t *>(&lo);
    w.y = *reinterpret_cast<uint32_t *>(&hi);
    *reinterpret_cast<uint2 *>(p) = w;
}

// Sum over the eight lanes that share lane % 4 (the row blocks of one column group).
__device__ __forceinline__ float4 sum_row_blocks(float4 x) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
        x.x += __shfl_xor_sync(0xffffffffu, x.x, o);
        x.y += __shfl_xor_sync(0xffffffffu, x.y, o);
        x.z += __shfl_xor_sync(0xffffffffu, x.z, o);
        x.w += __shfl_xor_sync(0xffffffffu, x.w, o);
    }
    return x;
}
}  // namespace

// Item w covers state columns cb .. cb + 15 of unit u = w / (V / 16),
// cb = 16 (w % (V / 16)).  Lane l owns columns cb + c .. cb + c + 3, c = 4 (l % 4),
// of rows RL (l / 4) .. RL (l / 4) + RL - 1, RL = K / 8.
template <typename T, int K, int V>
__global__ void __launch_bounds__(32 * kWarps, 2)
step_kernel(StepArgs a) {
    constexpr int NSL = V / kSlice, RL = K / 8, KL = K / 32;
    __shared__ __align__(16) float kq[kWarps][2][K];  // each warp's normalised k and q
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = 4 * (lane & 3), r0 = RL * (lane >> 2);
    float *kb = kq[warp][0], *qb = kq[warp][1];
    const long long n_items = (long long)a.N * a.H * NSL;
    const long long stride = (long long)gridDim.x * kWarps;
    for (long long w = (long long)blockIdx.x * kWarps + warp; w < n_items; w += stride) {
        const long long u = w / NSL;
        const int cb = kSlice * (int)(w % NSL), h = (int)(u % a.H);
        float *S = a.state + u * K * V + cb + c;
        float4 hr[RL];
#pragma unroll
        for (int i = 0; i < RL; ++i)
            hr[i] = *reinterpret_cast<const float4 *>(S + (long long)(r0 + i) * V);
        float kx[KL], qx[KL], vx[4];
        ld_vec<T, KL>(a.k, u * K + KL * lane, kx);
        ld_vec<T, KL>(a.q, u * K + KL * lane, qx);
        ld_vec<T, 4>(a.v, u * V + cb + c, vx);
        const float gx = a.g[u], beta = a.beta[u];
        if (a.l2norm) {
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int i = 0; i < KL; ++i) sk += kx[i] * kx[i], sq += qx[i] * qx[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, o);
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
            }
            const float ik = rsqrtf(sk + 1e-6f), iq = rsqrtf(sq + 1e-6f);
#pragma unroll
            for (int i = 0; i < KL; ++i) kx[i] *= ik, qx[i] *= iq;
        }
        __syncwarp();  // the previous item's reads of kb, qb are done
#pragma unroll
        for (int i = 0; i < KL; ++i) kb[KL * lane + i] = kx[i], qb[KL * lane + i] = qx[i];
        __syncwarp();
        const float gl = a.gate_a ? -a.gate_a[h] * (gx > 0.f ? gx + log1pf(expf(-gx))
                                                           : log1pf(expf(gx)))
                                  : gx;
        const float alpha = expf(gl);

        // Hbar = alpha H; (Hbar^T k) over the lane's rows, then over the warp
        float4 dot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RL; ++i) {
            const float kr = kb[r0 + i];
            hr[i] = make_float4(alpha * hr[i].x, alpha * hr[i].y, alpha * hr[i].z, alpha * hr[i].w);
            dot.x += hr[i].x * kr;
            dot.y += hr[i].y * kr;
            dot.z += hr[i].z * kr;
            dot.w += hr[i].w * kr;
        }
        dot = sum_row_blocks(dot);
        const float4 rr = make_float4(vx[0] - dot.x, vx[1] - dot.y, vx[2] - dot.z, vx[3] - dot.w);

        // H = Hbar + beta k r^T, written back; H^T q likewise
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RL; ++i) {
            const float bk = beta * kb[r0 + i], qr = qb[r0 + i];
            const float4 hn = make_float4(hr[i].x + bk * rr.x, hr[i].y + bk * rr.y,
                                          hr[i].z + bk * rr.z, hr[i].w + bk * rr.w);
            *reinterpret_cast<float4 *>(S + (long long)(r0 + i) * V) = hn;
            o.x += hn.x * qr;
            o.y += hn.y * qr;
            o.z += hn.z * qr;
            o.w += hn.w * qr;
        }
        o = sum_row_blocks(o);
        if (lane < 4)
            store4(reinterpret_cast<T *>(a.o) + u * V + cb + c,
                   make_float4(a.scale * o.x, a.scale * o.y, a.scale * o.z, a.scale * o.w));
    }
}

template <typename T, int K, int V>
static cudaError_t launch_kv(const StepArgs &a, int sms, cudaStream_t st) {
    // resident CTAs per SM, asked once per instantiation (the library runs on
    // sm_103a only, so the answer is the same on every device)
    static int per_sm = 0;
    if (per_sm == 0) {
        int n = 0;
        const cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, step_kernel<T, K, V>, 32 * kWarps, 0);
        if (e != cudaSuccess) return e;
        per_sm = n > 0 ? n : 1;
    }
    const long long ctas = ((long long)a.N * a.H * (V / kSlice) + kWarps - 1) / kWarps;
    const int grid = (int)(ctas < (long long)sms * per_sm ? ctas : (long long)sms * per_sm);
    step_kernel<T, K, V><<<grid, 32 * kWarps, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t launch(const StepArgs &a, int K, int V, int sms, cudaStream_t s) {
    prof_before("recurrent_step", s);
    cudaError_t e;
    if (K == 128 && V == 128) e = launch_kv<T, 128, 128>(a, sms, s);
    else if (K == 128 && V == 64) e = launch_kv<T, 128, 64>(a, sms, s);
    else if (K == 64 && V == 128) e = launch_kv<T, 64, 128>(a, sms, s);
    else e = launch_kv<T, 64, 64>(a, sms, s);
    prof_after(s);
    return e;
}

cudaError_t run(const gdn_step_args *p, int sms, cudaStream_t s) {
    StepArgs a{p->q, p->k, p->v, p->g, p->beta, p->gate_scale, p->state, p->o, p->N, p->H,
               p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->K), p->use_qk_l2norm ? 1 : 0};
    return p->dtype == GDN_BF16 ? launch<__nv_bfloat16>(a, p->K, p->V, sms, s)
                                : launch<float>(a, p->K, p->V, sms, s);
}

}  // namespace step
}  // namespace gdn
