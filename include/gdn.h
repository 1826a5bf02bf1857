/*
 * gdn.h -- C ABI of libgdn.so: Gated DeltaNet (GDN) chunked prefill,
 * forward and backward, on one NVIDIA GB300 (sm_103a).
 *
 * The operation (the pages name it "GDN Chunked Prefill" -- "FlashQLA是什么"
 * on ollai.cn, sections "FlashQLA的主要功能" and "如何使用FlashQLA" -- and
 * describe its call as chunk_gated_delta_rule(q, k, v, g, beta,
 * initial_state, cu_seqlens) returning O and the final state, with separate
 * low-level fwd / bwd entry points) is the gated delta rule of Yang, Kautz
 * and Hatamizadeh ("Gated Delta Networks", ICLR 2025), per (sequence, head):
 *
 *     S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *     o_t = S_t (scale * q_t)
 *
 * evaluated chunk by chunk (64 tokens).  States cross the ABI as H = S^T,
 * i.e. [K, V] with the key index first.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor pointer is a DEVICE pointer on the current CUDA device,
 *   contiguous, row-major, in the layout stated for it.  The caller owns
 *   all memory: the library never allocates or frees device memory and
 *   never synchronises the stream (except gdn_sync_status).
 * - `stream` is a cudaStream_t passed as void*; NULL means the legacy
 *   default stream.  Calls are asynchronous on it.
 * - `workspace` is caller-allocated device memory of at least the size the
 *   matching *_workspace_size function returns, 256-byte aligned.  It holds
 *   per-call intermediates only; nothing persists between calls.
 * - Errors: host-detectable argument problems return a non-zero gdn_status
 *   before anything is launched, and gdn_last_error() describes them.
 *   Problems only the device can see (bad cu_seqlens contents, a bounded
 *   wait that ran out) are recorded in a per-device status word that
 *   gdn_sync_status() reads and clears.
 * - Shapes: B batch, T tokens per batch row, H heads, K key dim, V value
 *   dim.  K and V must each be 64 or 128.  T may be 0.
 */
#ifndef GDN_H_
#define GDN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define GDN_ABI_VERSION 4

typedef int32_t gdn_status;
enum {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1,  /* null required pointer, bad sizes, misalignment */
    GDN_ERR_UNSUPPORTED = 2,  /* dtype / shape / device not supported */
    GDN_ERR_WORKSPACE = 3,    /* workspace smaller than *_workspace_size */
    GDN_ERR_CUDA = 4,         /* a CUDA runtime call failed; message has its text */
    GDN_ERR_TIMEOUT = 5,      /* a bounded device-side wait ran out (gdn_sync_status) */
    GDN_ERR_BAD_SEQLENS = 6   /* cu_seqlens not 0 = c0 <= c1 <= ... <= cN = T (device check) */
};

/* Element type of q, k, v, o and d_o (and of dq/dk/dv when chosen). */
enum { GDN_FP32 = 0, GDN_BF16 = 1 };

/* Intra-card sequence parallelism ("AutoCP", ollai.cn page, sections
 * "FlashQLA的技术原理" and "FlashQLA的核心优势"): each (sequence, head) is
 * cut into segments walked on separate SMs.  Exact mode reduces every
 * segment to an affine state map S -> A S + B and joins the maps with a
 * prefix scan; results equal the serial walk up to rounding order. */
enum { GDN_CP_AUTO = 0, GDN_CP_OFF = 1, GDN_CP_FORCE = 2 };

typedef struct gdn_fwd_args {
    /* inputs */
    const void *q;              /* [B, T, H, K], dtype                              */
    const void *k;              /* [B, T, H, K], dtype                              */
    const void *v;              /* [B, T, H, V], dtype                              */
    const float *g;             /* [B, T, H] log decay (g <= 0 expected)            */
    const float *beta;          /* [B, T, H] write strength                         */
    const float *initial_state; /* [N, H, K, V] fp32, NULL = zeros                  */
    const int32_t *cu_seqlens;  /* [N + 1] int32, NULL = B separate rows of length T.
                                   When given, B must be 1 and sequence n covers
                                   tokens cu_seqlens[n] .. cu_seqlens[n+1]-1.        */
    int32_t B, T, H, K, V;
    int32_t N;                  /* number of sequences when cu_seqlens != NULL      */
    int32_t dtype;              /* GDN_FP32 or GDN_BF16                              */
    float scale;                /* <= 0 means K^-1/2                                */
    int32_t use_qk_l2norm;      /* 1: q, k scaled to unit norm, (|x|^2 + 1e-6)^-1/2 */
    int32_t cp_mode;            /* GDN_CP_*                                          */
    int32_t cp_segment_chunks;  /* chunks per segment under CP; 0 = chosen here     */
    int32_t cp_warmup_chunks;   /* 0 = exact CP.  W > 0: a segment whose preceding W
                                   chunks decay by less than cp_warmup_tau starts
                                   from a W-chunk walk from zero instead of the
                                   exact map (approximate; off by default)           */
    float cp_warmup_tau;        /* threshold on exp(sum of g over the W chunks)      */
    /* outputs */
    void *o;                    /* [B, T, H, V], dtype                              */
    float *final_state;         /* [N, H, K, V] fp32, NULL = not written            */
    int32_t *cp_stats;          /* NULL, or 2 device int32: heads that took the warmup
                                   shortcut, heads walked under CP (accumulated)     */
    void *ctx;                  /* NULL, or a saved-context buffer of
                                   gdn_fwd_ctx_size() bytes (256-byte aligned): the
                                   forward also keeps what the backward would
                                   otherwise recompute (see gdn_fwd_ctx_size)        */
    /* gate preprocessing (the pages' "gate preprocessing" ahead of the kernels,
       aivizor, FLA-flow paragraph) */
    const float *gate_scale;    /* NULL: g is the log decay itself.  Else [H] fp32,
                                   a_h > 0, and g holds raw gate logits x: the log
                                   decay is -a_h * softplus(x), softplus(x) = log(1 + e^x) */
    /* the one-kernel forward ("FlashQLA是什么", ollai.cn, "FlashQLA的核心优势", first
       item: a fully fused kernel against the split one at large batch) */
    int32_t fuse_prep;          /* 0 (default): the chunk-local preparation (gam, A,
                                   T = (I + A)^-1, W, u) and the state walk run as two
                                   kernels, W and u passing through the workspace.
                                   1: where the forward keeps no ctx, runs without
                                   sequence parallelism, and its (sequence, head)
                                   pairs fill at least three quarters of the SMs
                                   (bf16, K = V = 128), one kernel does both, so that
                                   W, u and gam never reach HBM; elsewhere ignored.
                                   Same results up to rounding; on GB300 the two-kernel
                                   form is the faster one (the preparation then runs
                                   beside another CTA's instead of in line with the
                                   walk).  Other values: GDN_ERR_INVALID_ARG.       */
} gdn_fwd_args;

typedef struct gdn_bwd_args {
    /* the forward's inputs, same meaning and layout as in gdn_fwd_args */
    const void *q, *k, *v;
    const float *g, *beta;
    const float *initial_state;
    const int32_t *cu_seqlens;
    int32_t B, T, H, K, V, N;
    int32_t dtype;
    float scale;
    int32_t use_qk_l2norm;
    int32_t cp_mode;
    int32_t cp_segment_chunks;
    /* incoming gradients */
    const void *d_o;            /* [B, T, H, V], dtype                              */
    const float *d_final_state; /* [N, H, K, V] fp32, NULL = zeros                  */
    /* outputs (every one written in full) */
    int32_t grad_dtype;         /* element type of dq, dk, dv (GDN_FP32 or GDN_BF16) */
    void *dq;                   /* [B, T, H, K]                                     */
    void *dk;                   /* [B, T, H, K]                                     */
    void *dv;                   /* [B, T, H, V]                                     */
    float *dg;                  /* [B, T, H]                                        */
    float *dbeta;               /* [B, T, H]                                        */
    float *d_initial_state;     /* [N, H, K, V] fp32, NULL = not written            */
    const void *ctx;            /* NULL, or the buffer a gdn_chunk_fwd call with the same
                                   inputs and sizes filled: the backward then skips
                                   recomputing the forward's per-chunk quantities   */
    const float *gate_scale;    /* as in gdn_fwd_args.  When given, dg receives the
                                   gradient with respect to the logits x            */
    float *d_gate_scale;        /* [H] fp32 gradient with respect to gate_scale;
                                   NULL = not written (ignored without gate_scale)  */
} gdn_bwd_args;

/* GDN_ABI_VERSION of the loaded library. */
int32_t gdn_abi_version(void);

/* Bytes of workspace gdn_chunk_fwd needs for these arguments: at least 256
 * for any valid arguments (an empty problem included), 0 when the arguments
 * are invalid (gdn_last_error then says why). */
size_t gdn_fwd_workspace_size(const gdn_fwd_args *args);

/* Forward: O and (optionally) the final state, in chunked form: per chunk a UT transform T = (I + strict_lower(diag(beta)
 * K K^T * decay))^-1 gives w and u, the state walks chunk to chunk, and O is
 * the inter-chunk term plus the masked intra-chunk term. */
gdn_status gdn_chunk_fwd(const gdn_fwd_args *args, void *workspace, size_t workspace_bytes,
                         void *stream);

/* Bytes of the saved forward context for these arguments: 0 when the path
 * keeps none (then gdn_chunk_fwd ignores args->ctx and gdn_chunk_bwd
 * recomputes).  The tensor-core path (bf16, K = V = 128) keeps the
 * within-chunk cumsum of g and, in bf16, W, u, each chunk's (I + A)^-1 and
 * each chunk's start state: about 2 K V / 64 + 2 (K + V) + 132 bytes per
 * token and head.
 * The contents are only meaningful to a gdn_chunk_bwd call with the same
 * inputs, sizes and flags; the library cannot check that. */
size_t gdn_fwd_ctx_size(const gdn_fwd_args *args);

/* Bytes of workspace gdn_chunk_bwd needs (at least 256 for valid arguments,
 * 0 for invalid ones, as gdn_fwd_workspace_size). */
size_t gdn_bwd_workspace_size(const gdn_bwd_args *args);

/* Backward (which the traeai.com page, announcement text, singles out as the
 * most difficult piece to make fast): given
 * dO and d(final_state), writes dq, dk, dv, dg, dbeta and d(initial_state).
 * Without args->ctx the forward's per-chunk quantities (W, u, (I + A)^-1 and
 * the chunk start states) are recomputed here; with a ctx that a gdn_chunk_fwd
 * call on the same inputs filled, they are read from it instead.  The result
 * depends on neither choice, nor on cp_mode, beyond rounding. */
gdn_status gdn_chunk_bwd(const gdn_bwd_args *args, void *workspace, size_t workspace_bytes,
                         void *stream);

/* Forward for callers that cannot allocate device memory.  No counterpart
 * on the pages: this is a library-usage addition.  Some callers cannot call
 * cudaMalloc -- for example a plugin running inside a host framework that
 * owns every device allocation, or a latency-critical server thread that
 * must never hit cudaMalloc's implicit device synchronisation -- so they
 * cannot hand gdn_chunk_fwd a workspace.  This entry point takes the same
 * arguments without a workspace and uses a fixed scratch area built into
 * the library instead: GDN_STATIC_SCRATCH_BYTES (64 MiB) of device memory
 * that every GPU which loads the library holds until the process exits.
 *
 * - The caller still allocates and passes every input and output.
 * - Problems whose gdn_fwd_workspace_size exceeds GDN_STATIC_SCRATCH_BYTES
 *   are rejected with GDN_ERR_WORKSPACE before any work is queued.
 * - The first call on a device looks up the scratch area's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture on the device.  The address is kept for the
 *   life of the process, one per device index: it belongs to the device's
 *   primary context (the CUDA runtime's), so do not call this entry point
 *   with another driver-API context current, nor after cudaDeviceReset on
 *   that device.  The per-device status word every entry point reports
 *   through (gdn_sync_status) is located and kept the same way.
 * - Every call on a device shares the one scratch area, which keeps the
 *   last call's contents; the forward writes every scratch byte it reads,
 *   so nothing needs clearing between calls.  Calls whose work overlaps on
 *   the GPU (other streams, other host threads) race on the scratch area:
 *   order them, for example on one stream.
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
#define GDN_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
gdn_status gdn_chunk_fwd_static(const gdn_fwd_args *args, void *stream);

/* One decode step: the recurrence advanced by a single token per (sequence,
 * head), the state updated in place.  The pages target prefill ("FlashQLA是什么"
 * on ollai.cn, section "FlashQLA的主要功能"); this entry point carries the same
 * gated delta rule to token-by-token generation, so that a model prefilled with
 * gdn_chunk_fwd can continue from its final state:
 *     Hbar = exp(g) H;  r = v - Hbar^T k;  H <- Hbar + beta k r^T;  o = scale H^T q
 * (H = S^T, [K, V]).  Steps taken one after another equal the prefill over
 * the same tokens up to rounding. */
typedef struct gdn_step_args {
    const void *q;              /* [N, H, K], dtype                                 */
    const void *k;              /* [N, H, K], dtype                                 */
    const void *v;              /* [N, H, V], dtype                                 */
    const float *g;             /* [N, H] log decay, or gate logits (gate_scale)    */
    const float *beta;          /* [N, H]                                           */
    const float *gate_scale;    /* NULL, or [H]: the log decay is -a_h softplus(g)  */
    float *state;               /* [N, H, K, V] fp32, read and overwritten          */
    int32_t N, H, K, V;         /* K, V in {64, 128}                                */
    int32_t dtype;              /* GDN_FP32 or GDN_BF16                              */
    float scale;                /* <= 0 means K^-1/2                                */
    int32_t use_qk_l2norm;      /* as in gdn_fwd_args                                */
    void *o;                    /* [N, H, V], dtype                                 */
} gdn_step_args;

/* Asynchronous on `stream`; needs no workspace.  Every pointer 16-byte
 * aligned.  GDN_ERR_INVALID_ARG / GDN_ERR_UNSUPPORTED for bad arguments
 * (nothing is launched), GDN_ERR_CUDA for a launch failure. */
gdn_status gdn_recurrent_step(const gdn_step_args *args, void *stream);

/* Synchronises `stream`, then reads and clears this device's status word:
 * GDN_OK, GDN_ERR_BAD_SEQLENS, GDN_ERR_TIMEOUT or GDN_ERR_CUDA. */
gdn_status gdn_sync_status(void *stream);

/* Message for the last non-OK status returned on this host thread. */
const char *gdn_last_error(void);

/* Testing hook: iteration limit of every bounded device-side wait (default
 * 1 << 21 polls; a negative value restores the default).  A limit of 0 makes
 * every wait give up at once: the kernel records GDN_ERR_TIMEOUT, waits for
 * its own copies and MMAs still in flight, frees its tensor memory and
 * returns without finishing its outputs.  Takes effect for later calls. */
void gdn_set_spin_limit(int64_t polls);

/* Per-kernel tracing.  Between gdn_profile_begin() and gdn_profile_end()
 * every kernel launch of this library (on any stream, any device) is
 * bracketed by a pair of CUDA events recorded on its launching stream.
 * gdn_profile_end() waits for those events, then fills up to `max` entries
 * of `out` (one per kernel name, in first-launch order) and returns the
 * number of distinct kernels (which may exceed `max`).  Off by default;
 * when off, launches carry no extra events. */
typedef struct gdn_kernel_stat {
    char name[64];
    int32_t launches;
    double total_ms;
} gdn_kernel_stat;

gdn_status gdn_profile_begin(void);
int32_t gdn_profile_end(gdn_kernel_stat *out, int32_t max);

#ifdef __cplusplus
}
#endif
#endif /* GDN_H_ */
