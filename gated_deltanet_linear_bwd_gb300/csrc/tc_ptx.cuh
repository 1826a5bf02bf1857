// tc_ptx.cuh -- thin inline-PTX wrappers for the Blackwell (sm_103a) data
// path used by the tensor-core kernels: mbarriers, TMA tiled loads,
// tcgen05 MMA with TMEM accumulators, TMEM loads, and the shared-memory /
// instruction descriptors those MMAs take.
//
// Shared-memory operand tiles are written in the canonical 128-byte-swizzle
// layout (the layout TMA produces with CU_TENSOR_MAP_SWIZZLE_128B): rows of
// 128 bytes, 8-row atoms of 1024 bytes, the 16-byte chunk index of a row
// XORed with (row % 8).  Every tile base is 1024-byte aligned.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gdn_common.cuh"

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: gives up after `limit` polls, records GDN_ERR_TIMEOUT in the
// status word and returns false.  Callers then skip the rest of their work.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, long long limit,
                                          int *status) {
    for (long long i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    set_status(status, GDN_ERR_TIMEOUT);
    return false;
}
// After a wait gave up: waits (with a fixed limit, independent of the
// testing hook) for the last phase still in flight on `bar`, so that no
// asynchronous write lands after the CTA has released its TMEM and exited.
__device__ __forceinline__ void mbar_drain(uint64_t *bar, uint32_t parity) {
    for (long long i = 0; i < (1ll << 22); ++i)
        if (mbar_try_wait(bar, parity)) return;
}

// ------------------------------------------------------------------ TMA
// 3-D tiled load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1, int c2) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
        : "memory");
}
// 2-D tiled load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar,
                                            int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}
// 2-D tiled store from shared memory (coordinates innermost first, never
// negative), tracked by the issuing thread's bulk-async group.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int c0,
                                             int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(smem_u32(src)), "r"(c0), "r"(c1)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until the issuing thread's bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Waits until every bulk store group of the issuing thread but the newest one
// has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_but_newest() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// 4-byte asynchronous global -> shared copy (zero-filled when !valid; the
// source address must still be a valid one).  Unlike a plain load it does not
// hold up the thread at the next barrier; cp_async_wait_all completes it.
__device__ __forceinline__ void cp_async4(void *dst, const void *src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(dst)), "l"(src),
                 "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}
// Named barrier `id` (1-15) over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ TMEM / tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t ncols) {  // one full warp
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {  // same warp
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulation.
// Warp-collective: the whole (converged) warp calls it with the same
// operands and one lane, chosen by elect.sync, issues the MMA.  Issuing from
// a full warp keeps the descriptors warp-uniform, which the single-thread
// form does not, and issues several times faster.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n"
        ".reg .pred p, e;\n"
        "setp.ne.b32 p, %4, 0;\n"
        "elect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
        "}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrives on `bar` once every MMA issued so far by this warp has completed.
// Warp-collective like mma_bf16 (the elected lane commits).
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile(
        "{\n"
        ".reg .pred e;\n"
        "elect.sync _|e, 0xffffffff;\n"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n"
        "}\n" ::"r"(smem_u32(bar))
        : "memory");
}

// Loads 32 consecutive fp32 columns of this thread's TMEM lane (32x32b
// shape: warp w reads lanes 32*(w%4) .. +31) and waits for them in the same
// asm block, so no use of the registers can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Two 32-column loads (from two TMEM addresses of this warp's lanes) behind
// one wait, so that the second load's latency overlaps the first's.
__device__ __forceinline__ void tmem_ld32x2(uint32_t a0, uint32_t a1, float *v0, float *v1) {
    uint32_t r[64];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n"
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]),
          "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]),
          "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]),
          "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]),
          "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]),
          "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
        : "r"(a0), "r"(a1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(r[32 + i]);
    }
}

// Two or three 8-column loads from different TMEM addresses, one wait: the
// loads overlap instead of each paying the full TMEM latency.
__device__ __forceinline__ void tmem_ld8x2(uint32_t a0, uint32_t a1, float *v0, float *v1) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(a0), "r"(a1)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(r[8 + i]);
    }
}
__device__ __forceinline__ void tmem_ld8x3(uint32_t a0, uint32_t a1, uint32_t a2, float *v0,
                                           float *v1, float *v2) {
    uint32_t r[24];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%24];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%25];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%26];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
        : "r"(a0), "r"(a1), "r"(a2)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(r[8 + i]);
        v2[i] = __uint_as_float(r[16 + i]);
    }
}

__device__ __forceinline__ void tmem_ld8x5(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                           uint32_t a4, float *v0, float *v1, float *v2,
                                           float *v3, float *v4) {
    uint32_t r[40];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%40];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%41];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%42];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%43];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%32,%33,%34,%35,%36,%37,%38,%39}, [%44];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]),
          "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(a4)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v0[i] = __uint_as_float(r[i]);
        v1[i] = __uint_as_float(r[8 + i]);
        v2[i] = __uint_as_float(r[16 + i]);
        v3[i] = __uint_as_float(r[24 + i]);
        v4[i] = __uint_as_float(r[32 + i]);
    }
}

// Writes 8 bf16 values (columns 8 * chunk .. +7) of a 128-byte swizzled row.
__device__ __forceinline__ void st_row8(uint8_t *tile, int row, int chunk, const float *x) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        __nv_bfloat162 b = __floats2bfloat162_rn(x[2 * j], x[2 * j + 1]);
        w[j] = *reinterpret_cast<uint32_t *>(&b);
    }
    const uint32_t c = (uint32_t)chunk ^ (uint32_t)(row & 7);
    *reinterpret_cast<uint4 *>(tile + row * 128 + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
}

// TMEM address of (lane base of this warp, column col).
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int warp, int col) {
    return base + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)col;
}

// ------------------------------------------------------------------ descriptors
// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format:
// start >> 4 in bits 0-13, leading byte offset >> 4 in 16-29, stride byte
// offset >> 4 in 32-45, version 1 in bits 46-47, layout SWIZZLE_128B = 2 in
// bits 61-63).  K-major tiles: sbo = 1024 (8-row groups), lbo unused.
// MN-major tiles: lbo = stride between 64-element MN blocks, sbo = stride
// between 8-row groups along K.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16: bf16 A and B, fp32 D; a_mn / b_mn
// select MN-major (transposed) operands.  N >> 3 in bits 17-22, M >> 4 in
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Byte offset of element (row, col) of a bf16 tile with 128-byte rows in the
// 128-byte swizzle layout (the tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
    const uint32_t chunk = (uint32_t)(col >> 3) ^ (uint32_t)(row & 7);
    return (uint32_t)row * 128u + (chunk << 4) + (uint32_t)(col & 7) * 2u;
}

// Writes 32 bf16 values (columns col0 .. col0+31, col0 in {0, 32}) of a
// 128-byte swizzled row (4 x 16-byte stores).
__device__ __forceinline__ void st_row32(uint8_t *tile, int row, int col0, const float *x) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __nv_bfloat162 b = __floats2bfloat162_rn(x[8 * c + 2 * j], x[8 * c + 2 * j + 1]);
            w[j] = *reinterpret_cast<uint32_t *>(&b);
        }
        const uint32_t chunk = (uint32_t)((col0 >> 3) + c) ^ (uint32_t)(row & 7);
        *reinterpret_cast<uint4 *>(tile + row * 128 + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// Writes 64 bf16 values as one whole 128-byte swizzled row.
__device__ __forceinline__ void st_row64(uint8_t *tile, int row, const float *x) {
    st_row32(tile, row, 0, x);
    st_row32(tile, row, 32, x + 32);
}

// 4 x 4 transpose inside each quad of lanes: lane 4j + f holds a[e] = M[f][e]
// on entry and a[f'] = M[f'][f] on return (two exchange rounds).
__device__ __forceinline__ void quad_transpose4(float *a) {
    const int f = threadIdx.x & 3;
    const bool up2 = (f & 2) != 0, up1 = (f & 1) != 0;
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const float r = __shfl_xor_sync(0xffffffffu, up2 ? a[k] : a[k + 2], 2);
        if (up2) a[k] = r; else a[k + 2] = r;
    }
#pragma unroll
    for (int k = 0; k < 4; k += 2) {
        const float r = __shfl_xor_sync(0xffffffffu, up1 ? a[k] : a[k + 1], 1);
        if (up1) a[k] = r; else a[k + 1] = r;
    }
}

__device__ __forceinline__ void st4(float *p, const float *a) {
    *reinterpret_cast<float4 *>(p) = make_float4(a[0], a[1], a[2], a[3]);
}
__device__ __forceinline__ void st4(__nv_bfloat16 *p, const float *a) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(a[0], a[1]), hi = __floats2bfloat162_rn(a[2], a[3]);
    *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<uint32_t *>(&lo),
                                              *reinterpret_cast<uint32_t *>(&hi));
}

// Feature-major results to a row-major [rows][features] tensor: lane l holds
// feature l of the warp's 32 at rows r0 .. r0+7 (x[e] is row r0 + e; `col`
// points at row 0, feature l; rows are rs elements apart).  After a quad
// transpose lane 4j + f writes features 4j .. 4j+3 of rows r0 + f and r0 + 4 + f
// as one 16-byte (fp32) or 8-byte (bf16) store each; rows >= L are skipped.
template <typename TG>
__device__ __forceinline__ void store_rows8(TG *col, long long rs, float (&x)[8], int r0, int L) {
    const int f = threadIdx.x & 3;
    quad_transpose4(x);
    quad_transpose4(x + 4);
    TG *p = col - f + (long long)(r0 + f) * rs;
    if (r0 + f < L) st4(p, x);
    if (r0 + 4 + f < L) st4(p + 4 * rs, x + 4);
}

// Decay factors D_rc = e^(gam_r - gam_c) of row r for the 32 columns c = c_lo ..
// c_lo + 31, valid where c <= r (the caller masks the rest).  They are formed as
// a running product downward from c = min(r, c_lo + 31), using
// e^(gam_r - gam_c) = e^(gam_r - gam_{c+1}) e^(gam_{c+1} - gam_c) with
// eg[j] = e^(gam_j - gam_{j-1}): every factor multiplied in is a decay of one
// token, so at most one exponential per row (when r lies past the block).
__device__ __forceinline__ void row_decays32(const float *gam, const float *eg, int r, int c_lo,
                                             float (&d)[32]) {
    const int top = c_lo + 31;
    float x = r > top ? __expf(gam[r] - gam[top]) : 1.f;
#pragma unroll
    for (int k = 31; k >= 0; --k) {
        const int c = c_lo + k;
        if (k < 31) x = c < r ? x * eg[c + 1] : 1.f;
        d[k] = x;
    }
}

// 1 / |x_r| = (sum of squares + 1e-6)^-1/2 of rows r = 0 .. nrows-1 of a bf16
// tile stored as two dk halves of 128-byte rows, the second half_stride bytes
// after the first (the q / k normalisation inside the library).  Thread t <
// 2 nrows reads row t / 2, half t % 2, as 16-byte pieces (starting at piece
// r + 4 (t % 2), so the 8 threads of a shared-memory phase hit 8 different
// bank groups; the swizzle does not matter for a sum over the row); the two
// halves meet by a shuffle and the even thread writes out[r].  Threads
// t >= 2 nrows do nothing; a warp is either wholly in or wholly out.
__device__ __forceinline__ void row_inv_norms(const uint8_t *base, uint32_t half_stride,
                                              int nrows, float *out) {
    const int t = threadIdx.x, r = t >> 1, hh = t & 1;
    if (r >= nrows) return;
    const uint4 *row = reinterpret_cast<const uint4 *>(base + hh * half_stride + r * 128);
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint4 x = row[(i + r + 4 * hh) & 7];
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&x);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(b[j]);
            ss += f.x * f.x + f.y * f.y;
        }
    }
    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
    if (hh == 0) out[r] = rsqrtf(ss + 1e-6f);
}

__device__ __forceinline__ float ld_bf16(const uint8_t *tile, int row, int col) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_off(row, col)));
}

}  // namespace tc
}  // namespace gdn
