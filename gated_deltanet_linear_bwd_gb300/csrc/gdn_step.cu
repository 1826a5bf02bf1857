// gdn_step.cu -- one decode step of the gated delta rule per (sequence, head),
// the state updated in place.  It reads and writes the K x V fp32 state once,
// so it is bound by HBM: each CTA streams one state through registers with
// coalesced row accesses and needs no shared-memory tiles beyond the vectors.
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

// One CTA per (sequence, head), 2V threads: thread t owns state column
// v = t % V and the key rows kr = (t / V) * K/2 .. +K/2.  The partial sums of
// the two row halves meet in shared memory.
template <typename T, int K, int V>
__global__ void __launch_bounds__(2 * V)
step_kernel(StepArgs a) {
    constexpr int NT = 2 * V, KH = K / 2;
    __shared__ float kv[K], qv[K], part[2][V], red[NT / 32];
    const int u = blockIdx.x, h = u % a.H, t = threadIdx.x, v = t % V, half = t / V;
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
    // Hbar = alpha H (rows of this half), partial (Hbar^T k)_v
    float *S = a.state + (long long)u * K * V;
    float hr[KH];
    float dot = 0.f;
#pragma unroll
    for (int i = 0; i < KH; ++i) {
        hr[i] = alpha * S[(long long)(half * KH + i) * V + v];
        dot += hr[i] * kv[half * KH + i];
    }
    part[half][v] = dot;
    __syncthreads();
    const float r = ld<T>(a.v, v0 + v) - (part[0][v] + part[1][v]);
    // H = Hbar + beta k r^T, written back; partial (H^T q)_v
    float o = 0.f;
#pragma unroll
    for (int i = 0; i < KH; ++i) {
        const float hn = hr[i] + beta * kv[half * KH + i] * r;
        S[(long long)(half * KH + i) * V + v] = hn;
        o += hn * qv[half * KH + i];
    }
    __syncthreads();                          // both halves have read part[] above
    part[half][v] = o;
    __syncthreads();
    if (half == 0) from_f(reinterpret_cast<T *>(a.o) + v0 + v, a.scale * (part[0][v] + part[1][v]));
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
