// gdn_common.cuh -- problem geometry, chunk / segment mapping and element
// access shared by the kernels of libgdn.so.
//
// Chunking: every sequence is cut into chunks of kChunk = 64 tokens (the last
// one may be shorter); chunks never cross a sequence boundary.  Chunk-parallel
// kernels index chunks globally; walk kernels follow one (sequence, head).
// Under intra-card sequence parallelism a sequence's chunks are grouped into
// segments of `seg_chunks` chunks.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

constexpr int kChunk = 64;

// Kernels launched with programmatic stream serialization start while the
// previous kernel on the stream is still running: each lets its own
// dependents launch at once, then waits for its predecessor's grid (and its
// memory) before touching anything in global memory.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Everything a kernel needs to locate a sequence, chunk or segment and to
// read the inputs.  Passed by value.
struct Geo {
    const void *q, *k, *v;
    const float *g, *beta;
    const float *gate_a;        // nullable: g holds gate logits x, the log decay is -a_h softplus(x)
    const int32_t *cu;          // nullable: fixed-length rows
    const int32_t *chunk_off;   // [N+1] chunk offsets (varlen only)
    const int32_t *seg_off;     // [N+1] segment offsets (varlen + CP only)
    const int32_t *order;       // [N] sequences by chunk count, longest first (varlen), or null
    int B, T, H, K, V, N;
    int nc_fixed;               // chunks per row when cu == nullptr
    int seg_chunks;             // chunks per segment (CP), else huge
    int nseg_fixed;             // segments per row when cu == nullptr
    int l2norm;
    float scale;
    int *status;                // device status word
    long long spin_limit;       // bounded waits
};

// Log decay of token row i (index of [tokens, H]) and head h: g itself, or
// -a_h softplus(x) from a gate logit.
__device__ __forceinline__ float decay_of(const Geo &g, float x, int h) {
    if (!g.gate_a) return x;
    const float sp = x > 0.f ? x + log1pf(expf(-x)) : log1pf(expf(x));
    return -g.gate_a[h] * sp;
}
__device__ __forceinline__ float decay_at(const Geo &g, long long i, int h) {
    return decay_of(g, g.g[i], h);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ void from_f(float *p, float x) { *p = x; }
__device__ __forceinline__ void from_f(__nv_bfloat16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Token range of sequence n.
__device__ __forceinline__ void seq_range(const Geo &g, int n, long long &bos, int &len) {
    if (g.cu) {
        bos = g.cu[n];
        len = g.cu[n + 1] - g.cu[n];
    } else {
        bos = (long long)n * g.T;
        len = g.T;
    }
}

__device__ __forceinline__ int seq_nchunks(const Geo &g, int n) {
    if (!g.cu) return g.nc_fixed;
    return g.chunk_off[n + 1] - g.chunk_off[n];
}

// Global index of sequence n's first chunk.
__device__ __forceinline__ int seq_chunk_base(const Geo &g, int n) {
    return g.cu ? g.chunk_off[n] : n * g.nc_fixed;
}

// Largest n with off[n] <= x (off non-decreasing, off[0] = 0).
__device__ __forceinline__ int upper_index(const int32_t *off, int N, int x) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (off[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

struct ChunkRef {
    int n;            // sequence
    int c;            // chunk index within the sequence
    long long bos;    // first token (global token index)
    int len;          // rows in this chunk (1..64)
};

// Maps a global chunk index to its sequence; false when past the end.
__device__ __forceinline__ bool chunk_ref(const Geo &g, int ci, ChunkRef &r) {
    int n, c;
    if (g.cu) {
        if (ci >= g.chunk_off[g.N]) return false;
        // the largest n with chunk_off[n] <= ci also has chunk_off[n+1] > ci,
        // so empty sequences (equal offsets) are stepped over
        n = upper_index(g.chunk_off, g.N, ci);
        c = ci - g.chunk_off[n];
    } else {
        if (ci >= g.B * g.nc_fixed) return false;
        n = ci / g.nc_fixed;
        c = ci - n * g.nc_fixed;
    }
    long long bos;
    int L;
    seq_range(g, n, bos, L);
    r.n = n;
    r.c = c;
    r.bos = bos + (long long)c * kChunk;
    r.len = min(kChunk, L - c * kChunk);
    return true;
}

__device__ __forceinline__ int seq_nsegs(const Geo &g, int n) {
    if (!g.cu) return g.nseg_fixed;
    return g.seg_off[n + 1] - g.seg_off[n];
}
__device__ __forceinline__ int seq_seg_base(const Geo &g, int n) {
    return g.cu ? g.seg_off[n] : n * g.nseg_fixed;
}

// Sequence and head walked by block b of a walk launched without sequence
// parallelism as a 1-D grid of N x H blocks: the blocks go out in index
// order, so rank-major numbering (every head of the longest sequence first)
// lets the longest walks start first.
__device__ __forceinline__ void walk_unit(const Geo &g, int b, int &n, int &h) {
    const int rank = b / g.H;
    h = b - rank * g.H;
    n = g.order ? g.order[rank] : rank;
}

// Maps a global segment index to (sequence, segment-in-sequence).
__device__ __forceinline__ bool seg_ref(const Geo &g, int si, int &n, int &j) {
    if (g.cu) {
        if (si >= g.seg_off[g.N]) return false;
        n = upper_index(g.seg_off, g.N, si);
        j = si - g.seg_off[n];
    } else {
        if (si >= g.B * g.nseg_fixed) return false;
        n = si / g.nseg_fixed;
        j = si - n * g.nseg_fixed;
    }
    return true;
}

// Records the first non-OK device status (sticky until read by the host).
__device__ __forceinline__ void set_status(int *status, int code) {
    if (status) atomicCAS(status, 0, code);
}

}  // namespace gdn
