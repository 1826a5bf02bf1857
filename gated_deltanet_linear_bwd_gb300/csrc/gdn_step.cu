// gdn_step.cu -- one decode step of the gated delta rule per (sequence, head),
// the state updated in place.  It reads and writes the K x V fp32 state once,
// so it is bound by HBM: each CTA streams one state through registers in
// 16-byte, coalesced pieces and needs no shared-memory tiles beyond the vectors.
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

template <typename T>
__device__ __forceinline__ float ld(const void *p, long long i) {
    return to_f(reinterpret_cast<const T *>(p)[i]);
}

// Sum over the CTA of one value per thread (KV threads in warps of 32).
template <int NT>
__device__ __forceinline__ float cta_sum(float x, float *red) {
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) s += red[w];
    __syncthreads();
    return s;
}
}  // namespace

// One CTA per (sequence, head), 2V threads.  Thread t owns state columns
// 4 (t % (V/4)) .. +3 and the key rows of row group t / (V/4) (8 groups of K/8
// rows), so that every state access is a 16-byte, fully coalesced piece; the
// groups' partial sums meet in shared memory.
template <int V>
__device__ __forceinline__ float4 sum_groups(const float (*part)[V], int c) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
        const float4 p = *reinterpret_cast<const float4 *>(&part[g][c]);
        s.x += p.x;
        s.y += p.y;
        s.z += p.z;
        s.w += p.w;
    }
    return s;
}

__device__ __forceinline__ void store4(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 x) {
    __nv_bfloat162 a = __floats2bfloat162_rn(x.x, x.y), b = __floats2bfloat162_rn(x.z, x.w);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

template <typename T, int K, int V>
__global__ void __launch_bounds__(2 * V)
step_kernel(StepArgs a) {
    constexpr int NT = 2 * V, NCG = V / 4, RG = K / 8;   // column groups, rows per group
    static_assert(NT / NCG == 8, "eight row groups");
    __shared__ float kv[K], qv[K], red[NT / 32];
    __shared__ __align__(16) float part[8][V];
    const int u = blockIdx.x, h = u % a.H, t = threadIdx.x;
    const int c = 4 * (t % NCG), r0 = (t / NCG) * RG;
    const long long qk0 = (long long)u * K, v0 = (long long)u * V;
    // inputs of the token: k, q (optionally L2-normalised), decay, beta
    float kk = 0.f, qq = 0.f;
    if (t < K) {
        kk = ld<T>(a.k, qk0 + t);
        qq = ld<T>(a.q, qk0 + t);
    }
    if (a.l2norm) {
        const float sk = cta_sum<NT>(kk * kk, red), sq = cta_sum<NT>(qq * qq, red);
        kk *= rsqrtf(sk + 1e-6f);
        qq *= rsqrtf(sq + 1e-6f);
    }
    if (t < K) {
        kv[t] = kk;
        qv[t] = qq;
    }
    const float x = a.g[u];
    const float gl = a.gate_a ? -a.gate_a[h] * (x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x)))
                              : x;
    const float alpha = expf(gl), beta = a.beta[u];
    __syncthreads();
    // Hbar = alpha H (this thread's rows and columns), partial (Hbar^T k)_c
    float *S = a.state + (long long)u * K * V;
    float4 hr[RG];
    float4 dot = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RG; ++i) {
        const float4 x4 = *reinterpret_cast<const float4 *>(S + (long long)(r0 + i) * V + c);
        const float kr = kv[r0 + i];
        hr[i] = make_float4(alpha * x4.x, alpha * x4.y, alpha * x4.z, alpha * x4.w);
        dot.x += hr[i].x * kr;
        dot.y += hr[i].y * kr;
        dot.z += hr[i].z * kr;
        dot.w += hr[i].w * kr;
    }
    *reinterpret_cast<float4 *>(&part[t / NCG][c]) = dot;
    __syncthreads();
    const float4 kh = sum_groups<V>(part, c);
    const float4 rr = make_float4(ld<T>(a.v, v0 + c) - kh.x, ld<T>(a.v, v0 + c + 1) - kh.y,
                                  ld<T>(a.v, v0 + c + 2) - kh.z, ld<T>(a.v, v0 + c + 3) - kh.w);
    // H = Hbar + beta k r^T, written back; partial (H^T q)_c
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < RG; ++i) {
        const float bk = beta * kv[r0 + i], qr = qv[r0 + i];
        const float4 hn = make_float4(hr[i].x + bk * rr.x, hr[i].y + bk * rr.y,
                                      hr[i].z + bk * rr.z, hr[i].w + bk * rr.w);
        *reinterpret_cast<float4 *>(S + (long long)(r0 + i) * V + c) = hn;
        o.x += hn.x * qr;
        o.y += hn.y * qr;
        o.z += hn.z * qr;
        o.w += hn.w * qr;
    }
    __syncthreads();                          // every group has read part[] above
    *reinterpret_cast<float4 *>(&part[t / NCG][c]) = o;
    __syncthreads();
    if (t < NCG) {
        const float4 os = sum_groups<V>(part, c);
        store4(reinterpret_cast<T *>(a.o) + v0 + c,
               make_float4(a.scale * os.x, a.scale * os.y, a.scale * os.z, a.scale * os.w));
    }
}

template <typename T>
static cudaError_t launch(const StepArgs &a, int K, int V, cudaStream_t s) {
    const int n = a.N * a.H;
    prof_before("recurrent_step", s);
    if (K == 128 && V == 128) step_kernel<T, 128, 128><<<n, 256, 0, s>>>(a);
    else if (K == 128 && V == 64) step_kernel<T, 128, 64><<<n, 128, 0, s>>>(a);
    else if (K == 64 && V == 128) step_kernel<T, 64, 128><<<n, 256, 0, s>>>(a);
    else step_kernel<T, 64, 64><<<n, 128, 0, s>>>(a);
    prof_after(s);
    return cudaGetLastError();
}

cudaError_t run(const gdn_step_args *p, cudaStream_t s) {
    StepArgs a{p->q, p->k, p->v, p->g, p->beta, p->gate_scale, p->state, p->o, p->N, p->H,
               p->scale > 0.f ? p->scale : 1.0f / sqrtf((float)p->K), p->use_qk_l2norm ? 1 : 0};
    return p->dtype == GDN_BF16 ? launch<__nv_bfloat16>(a, p->K, p->V, s)
                                : launch<float>(a, p->K, p->V, s);
}

}  // namespace step
}  // namespace gdn
