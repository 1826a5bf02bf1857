// gdn_internal.h -- host-side plan shared by the C-ABI layer (gdn_api.cu)
// and the kernel launchers.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gdn_common.cuh"

namespace gdn {

// Device pointers carved out of the caller's workspace.
struct Ws {
    float *gam = nullptr;        // [tokens, H] within-chunk cumsum of g
    void *w = nullptr;           // W: fp32 [tokens, H, K] (CUDA cores) or bf16 W^T tiles
                                 // [chunk][H][K][64] (tensor cores)
    void *u = nullptr;           // u: likewise ([tokens, H, V] or [chunk][H][V][64])
    int32_t *chunk_off = nullptr;  // [N+1] (varlen)
    int32_t *seg_off = nullptr;    // [N+1] (varlen + CP)
    int32_t *order = nullptr;      // [N] sequences by chunk count, longest first (varlen)
    int32_t *warm = nullptr;       // [N, H] warmup decision
    float *maps = nullptr;         // [segs, H, K, K+V] affine maps
    float *fwd_maps = nullptr;     // [segs, H, K, K] A parts of the forward's segment maps kept in
                                   // a saved context (sequence parallelism forced, fixed length)
    float *seg_state = nullptr;    // [segs, H, K, V] segment start states / end gradients
    float *hc = nullptr;           // chunk start states (bwd): fp32 [chunks, H, K, V] (CUDA
                                   // cores) or bf16 H^T tiles [chunk][H][k half][v][64] (tensor cores)
    float *dhc = nullptr;          // chunk end gradients (bwd): likewise, dH^T tiles on tensor cores
    void *du = nullptr;            // [chunk][H][V][64] bf16 dU^T of the reverse walk (bwd, tensor cores)
    void *qs = nullptr;            // [chunk][H][dk half][64][64] bf16 diag(scale e^gam) Q (bwd, tensor cores)
    void *yt = nullptr;            // [chunk][H][V][64] bf16 (dO^T P) tiles (bwd, tensor cores)
    void *tmat = nullptr;          // [chunks, H, 64, 64] bf16 T = (I + A)^-1 by column (bwd, tensor cores)
    float *scratch = nullptr;      // per-CTA scratch (bwd, CUDA-core path)
};

struct Plan {
    Geo g;
    Ws ws;
    int dtype = GDN_FP32;
    int path = 0;               // kPathSimt / kPathTc
    int max_chunks = 0;         // chunk capacity (>= actual)
    int max_segs = 0;           // segment capacity under CP
    int cp = 0;
    int cp_forced = 0;          // cp_mode == GDN_CP_FORCE (device independent)
    int seg_chunks_arg = 0;     // cp_segment_chunks as given (0: chosen here)
    int warm_chunks = 0;
    bool fuse_prep = false;     // the one-kernel forward where it applies
    float warm_tau = 0.f;
    int sms = 0;
    int scratch_ctas = 0;
    // forward
    const float *h0 = nullptr;
    void *o = nullptr;
    float *final_state = nullptr;
    int32_t *cp_stats = nullptr;
    // backward
    const void *d_o = nullptr;
    const float *dht = nullptr;
    int grad_dtype = GDN_FP32;
    void *dq = nullptr, *dk = nullptr, *dv = nullptr;
    float *dg = nullptr, *dbeta = nullptr, *dh0 = nullptr;
};

enum { kPathSimt = 0, kPathTc = 1 };

// Tracing hooks around every launch (no-ops unless gdn_profile_begin ran).
void prof_before(const char *name, cudaStream_t s);
void prof_after(cudaStream_t s);

// Launches `kernel` with programmatic stream serialization: it may start while
// the previous kernel on the stream is finishing.  Only for kernels that call
// pdl_enter() before their first global memory access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

namespace step {
// One decode step per (sequence, head), the state updated in place, on a
// device with `sms` SMs.
cudaError_t run(const gdn_step_args *args, int sms, cudaStream_t s);
}  // namespace step

namespace simt {
// Per-CTA scratch floats of the local-gradient kernel.
size_t scratch_floats_per_cta(int K, int V);
cudaError_t tables(const Plan &p, cudaStream_t s);
cudaError_t forward(const Plan &p, cudaStream_t s);
cudaError_t backward(const Plan &p, cudaStream_t s);
cudaError_t warm_decide(const Plan &p, cudaStream_t s);
cudaError_t cp_scan(const Plan &p, const int32_t *warm, cudaStream_t s);
// fwd_maps: NULL, or the A parts of the forward's segment maps ([segs, H, K,
// K], from a saved context); their transposes are the reverse maps' A'.
cudaError_t cp_rscan(const Plan &p, cudaStream_t s, const float *fwd_maps = nullptr);
// Gate backward: dg (with respect to the log decay) becomes the gradient with
// respect to the logits in place; d_gate_scale [H] (nullable) gets its sum.
cudaError_t gate_bwd(const Plan &p, const float *gate_scale, float *d_gate_scale, cudaStream_t s);
}  // namespace simt

namespace tc {
// bf16 q/k/v with K = V = 128 and at least one token.
bool supported(const Plan &p);
// save: also keep T (p.ws.tmat) and every chunk's start state (p.ws.hc).
cudaError_t forward(const Plan &p, cudaStream_t s, bool save);
// The whole forward in one kernel (gdn_tc_full.cu): no sequence parallelism,
// no saved context, and enough (sequence, head) pairs to fill the GPU.
bool full_forward_fits(const Plan &p);
cudaError_t full_forward(const Plan &p, cudaStream_t s);
// Backward pieces: prep + walk storing chunk start states (p.ws.hc).
cudaError_t recompute_states(const Plan &p, cudaStream_t s);
// Chunk-parallel outputs O from the stored chunk start states (after the walk).
cudaError_t output(const Plan &p, cudaStream_t s);
// have_ctx: gam, W, u, T and the chunk start states are already in p.ws.
cudaError_t backward(const Plan &p, cudaStream_t s, bool have_ctx);
// Chunk-local gradients on tensor cores (q, k normalised inside or not).
cudaError_t local_grads(const Plan &p, cudaStream_t s);
// TMA descriptors of [tokens, H, 128] bf16 tensors (64 x 1 x 64 boxes, 128B swizzle).
cudaError_t encoder();
cudaError_t make_map(CUtensorMap *m, const void *base, long long tokens, int H);
// Chunk-major transposed tiles [chunk][H][128][64] bf16 (W^T, u^T, dU^T): one box per tile.
cudaError_t make_map_tiles(CUtensorMap *m, const void *base, long long rows_total,
                           int box_rows = 128);
}  // namespace tc

}  // namespace gdn
