// gdn_api.cu -- the C ABI of libgdn.so (declared in include/gdn.h):
// argument validation, the intra-card sequence-parallel decision, workspace
// layout and launch sequencing.  All device work goes on the caller's stream;
// nothing here allocates device memory.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "gdn.h"
#include "gdn_internal.h"

namespace gdn {

// One sticky status word per device (module memory, not an allocation).
static __device__ int g_status_word;

static thread_local std::string t_last_error;
static constexpr long long kDefaultSpinLimit = 1ll << 21;
static std::atomic<long long> g_spin_limit{kDefaultSpinLimit};

static gdn_status fail(gdn_status code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_last_error = buf;
    return code;
}

static gdn_status cuda_fail(cudaError_t e, const char *what) {
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

struct DeviceInfo {
    int *status = nullptr;
    int sms = 0;
    int major = 0, minor = 0;
    bool ready = false;
};
static DeviceInfo g_dev[64];
static std::mutex g_dev_mu;

// Per-device set-up on first use: the status word's device address and the
// SM count.  Runs with the target device current.
static gdn_status device_info(DeviceInfo **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(GDN_ERR_UNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceInfo &d = g_dev[dev];
    if (!d.ready) {
        e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
        if (d.major != 10 || d.minor != 3)
            return fail(GDN_ERR_UNSUPPORTED, "libgdn is built for sm_103a; device %d is sm_%d%d",
                        dev, d.major, d.minor);
        e = cudaGetSymbolAddress((void **)&d.status, g_status_word);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(status word)");
        d.ready = true;
    }
    *out = &d;
    return GDN_OK;
}

// Fields the forward and backward share.
struct Common {
    const void *q, *k, *v;
    const float *g, *beta, *h0;
    const int32_t *cu;
    int B, T, H, K, V, N, dtype, l2, cp_mode, seg_chunks;
    float scale;
    const float *gate_scale;
};

static constexpr size_t kAlign = 256;
static constexpr int kScratchCtas = 256;  // CTAs of the CUDA-core local-gradient kernel

static bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

static bool has_tokens(const Common &c) { return (long long)c.B * c.T > 0; }

static gdn_status validate(const Common &c) {
    // empty inputs (T == 0) may come with null pointers
    if (has_tokens(c) && (!c.q || !c.k || !c.v || !c.g || !c.beta))
        return fail(GDN_ERR_INVALID_ARG, "q, k, v, g and beta are required");
    if (c.B < 1 || c.T < 0 || c.H < 1)
        return fail(GDN_ERR_INVALID_ARG, "bad sizes B=%d T=%d H=%d", c.B, c.T, c.H);
    if ((c.K != 64 && c.K != 128) || (c.V != 64 && c.V != 128))
        return fail(GDN_ERR_INVALID_ARG, "K and V must each be 64 or 128 (K=%d V=%d)", c.K, c.V);
    if (c.dtype != GDN_FP32 && c.dtype != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "dtype %d is not GDN_FP32 or GDN_BF16", c.dtype);
    if (c.cu && (c.B != 1 || c.N < 1))
        return fail(GDN_ERR_INVALID_ARG, "cu_seqlens needs B == 1 and N >= 1 (B=%d N=%d)", c.B, c.N);
    if (c.cp_mode < GDN_CP_AUTO || c.cp_mode > GDN_CP_FORCE)
        return fail(GDN_ERR_INVALID_ARG, "cp_mode %d", c.cp_mode);
    if (c.seg_chunks < 0) return fail(GDN_ERR_INVALID_ARG, "cp_segment_chunks < 0");
    if (!aligned16(c.q) || !aligned16(c.k) || !aligned16(c.v) || !aligned16(c.g) ||
        !aligned16(c.beta) || (c.h0 && !aligned16(c.h0)) || (c.cu && !aligned16(c.cu)) ||
        (c.gate_scale && !aligned16(c.gate_scale)))
        return fail(GDN_ERR_INVALID_ARG, "every tensor must be 16-byte aligned");
    const long long tokens = (long long)c.B * c.T;
    if (tokens * c.H * (long long)(c.K > c.V ? c.K : c.V) >= (1ll << 40) ||
        (long long)(c.cu ? c.N : c.B) * c.H >= (1ll << 31))
        return fail(GDN_ERR_INVALID_ARG, "problem too large");
    return GDN_OK;
}

// The pages' AutoCP rule (ollai.cn page, "FlashQLA的核心优势", second item):
// on when batch x heads <= 40, or <= 56 with seq_len >= 8192, tuned on an
// H200 with 132 SMs.  Rescaled here by this GPU's SM count.
static bool cp_auto(long long units, long long avg_len, int sms) {
    return units * 132 <= 40ll * sms || (units * 132 <= 56ll * sms && avg_len >= 8192);
}

// Segments per sequence for the tensor-core path: the P minimising a cost
// model in units of one chunk step of a walk.  The map walk runs 2 (P - 1)
// CTAs per unit (its last segment needs no map), the output walk P, each
// over G = ceil(nc / P) chunks, in waves of one CTA per SM; the scan takes
// P - 1 dependent steps of about 1.6 chunk steps per wave of its 16 column
// blocks per unit.
static long long tc_segments(long long units, int nc, int sms) {
    auto waves = [&](long long ctas) { return (ctas + sms - 1) / sms; };
    long long best_p = 2;
    double best = 1e300;
    for (long long P = 2; P <= 64 && P <= nc; ++P) {
        const long long G = (nc + P - 1) / P;
        const double cost = (double)(waves(2 * (P - 1) * units) + waves(P * units)) * (double)G +
                            1.6 * (double)(P - 1) * (double)waves(16 * units);
        if (cost < best) {
            best = cost;
            best_p = P;
        }
    }
    return best_p;
}

static gdn_status make_plan(const Common &c, bool bwd, int sms, Plan &p) {
    gdn_status st = validate(c);
    if (st != GDN_OK) return st;
    Geo &g = p.g;
    g = Geo{};
    g.q = c.q; g.k = c.k; g.v = c.v; g.g = c.g; g.beta = c.beta; g.cu = c.cu;
    g.gate_a = c.gate_scale;
    g.B = c.B; g.T = c.T; g.H = c.H; g.K = c.K; g.V = c.V;
    g.N = c.cu ? c.N : c.B;
    g.nc_fixed = (c.T + kChunk - 1) / kChunk;
    g.l2norm = c.l2 ? 1 : 0;
    g.scale = c.scale > 0.f ? c.scale : 1.0f / sqrtf((float)c.K);
    g.spin_limit = g_spin_limit.load();
    p.dtype = c.dtype;
    p.path = kPathSimt;
    p.h0 = c.h0;
    p.max_chunks = c.cu ? (c.T + kChunk - 1) / kChunk + c.N : c.B * g.nc_fixed;
    const long long units = (long long)g.N * c.H;
    const long long avg_len = c.cu ? (c.T + c.N - 1) / c.N : c.T;
    const int nc_avg = (int)((avg_len + kChunk - 1) / kChunk);
    p.cp = c.cp_mode == GDN_CP_FORCE || (c.cp_mode == GDN_CP_AUTO && sms > 0 &&
                                         cp_auto(units, avg_len, sms));
    p.cp_forced = c.cp_mode == GDN_CP_FORCE;
    p.seg_chunks_arg = c.seg_chunks;
    if (p.cp) {
        int G = c.seg_chunks;
        if (G <= 0) {
            long long P = sms > 0 ? (sms + units - 1) / units : 2;
            if (c.dtype == GDN_BF16 && c.K == 128 && c.V == 128 && sms > 0)
                P = tc_segments(units, nc_avg, sms);
            if (P < 2) P = 2;
            if (P > nc_avg) P = nc_avg > 0 ? nc_avg : 1;
            G = (int)((nc_avg + P - 1) / P);
            if (G < 1) G = 1;
        }
        g.seg_chunks = G;
        g.nseg_fixed = g.nc_fixed > 0 ? (g.nc_fixed + G - 1) / G : 1;
        p.max_segs = c.cu ? p.max_chunks + c.N : c.B * g.nseg_fixed;  // <= seg_capacity
    } else {
        g.seg_chunks = 1 << 30;
        g.nseg_fixed = 1;
        p.max_segs = 0;
    }
    p.scratch_ctas = bwd ? kScratchCtas : 0;
    p.sms = sms;
    return GDN_OK;
}

// Carves the workspace; with base == nullptr only sizes it.
static size_t layout(Plan &p, bool bwd, char *base) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> char * {
        char *ptr = base ? base + off : nullptr;
        off += (bytes + kAlign - 1) / kAlign * kAlign;
        return ptr;
    };
    const Geo &g = p.g;
    const size_t th = (size_t)g.B * g.T * g.H;
    Ws &w = p.ws;
    w = Ws{};
    w.gam = (float *)take(th * sizeof(float));
    // CUDA cores keep fp32 token rows, tensor cores bf16 chunk tiles of 64 rows
    const size_t tiles = (size_t)p.max_chunks * g.H * 64 * 2;
    w.w = take(std::max(th * g.K * sizeof(float), tiles * g.K));
    w.u = take(std::max(th * g.V * sizeof(float), tiles * g.V));
    if (g.cu) {
        w.chunk_off = (int32_t *)take((g.N + 1) * sizeof(int32_t));
        w.seg_off = (int32_t *)take((g.N + 1) * sizeof(int32_t));
        w.order = (int32_t *)take(g.N * sizeof(int32_t));
    }
    if (p.cp) {
        w.warm = (int32_t *)take((size_t)g.N * g.H * sizeof(int32_t));
        w.maps = (float *)take((size_t)p.max_segs * g.H * g.K * (g.K + g.V) * sizeof(float));
        w.seg_state = (float *)take((size_t)p.max_segs * g.H * g.K * g.V * sizeof(float));
    }
    if (!bwd) {
        // chunk start states (bf16 tiles) the tensor-core walk hands to the output kernel
        w.hc = (float *)take((size_t)p.max_chunks * g.H * g.K * g.V * 2);
    }
    if (bwd) {
        const size_t st = (size_t)p.max_chunks * g.H * g.K * g.V * sizeof(float);
        w.hc = (float *)take(st);
        w.dhc = (float *)take(st);
        w.du = take(tiles * g.V);
        w.qs = take(tiles * g.K);
        w.yt = take(tiles * g.V);
        w.tmat = take((size_t)p.max_chunks * g.H * 64 * 64 * 2);
        w.scratch = (float *)take((size_t)p.scratch_ctas *
                                  simt::scratch_floats_per_cta(g.K, g.V) * sizeof(float));
    }
    // never 0 for valid arguments (an empty problem included): the size
    // queries return 0 only for invalid ones
    return std::max(off, kAlign);
}

// Upper bound on segments under CP for any segment length: every segment
// holds at least one chunk, except the single segment of an empty sequence.
static int seg_capacity(const Common &c, int max_chunks) {
    return c.cu ? max_chunks + c.N : (max_chunks > c.B ? max_chunks : c.B);
}

// Saved forward context (tensor-core path): gam, W, u, T, chunk start states,
// and, for fixed-length batches with sequence parallelism forced, the A parts
// of the forward's segment maps (the backward's reverse maps are their
// transposes, so it then walks only the other half).  Every size here follows
// from the arguments alone, not from the device: the maps region is sized for
// the most segments the forward can choose (64 per sequence, or the count
// cp_segment_chunks fixes).
static size_t ctx_layout(Plan &p, char *base) {
    size_t off = 0;
    auto take = [&](size_t bytes) -> char * {
        char *ptr = base ? base + off : nullptr;
        off += (bytes + kAlign - 1) / kAlign * kAlign;
        return ptr;
    };
    const Geo &g = p.g;
    const size_t th = (size_t)g.B * g.T * g.H;
    float *gam = (float *)take(th * sizeof(float));
    const size_t tiles = (size_t)p.max_chunks * g.H * 64 * 2;   // bf16 chunk tiles
    void *w = take(tiles * g.K);
    void *u = take(tiles * g.V);
    void *tm = take((size_t)p.max_chunks * g.H * 64 * 64 * 2);
    float *hc = (float *)take((size_t)p.max_chunks * g.H * g.K * g.V * 2);   // bf16 tiles
    float *fm = nullptr;
    if (p.cp && p.cp_forced && !g.cu) {
        const int nc = std::max(g.nc_fixed, 1);
        const long long segs =
            (long long)g.B * (p.seg_chunks_arg > 0 ? (nc + p.seg_chunks_arg - 1) / p.seg_chunks_arg
                                                   : std::min(64, nc));
        fm = (float *)take((size_t)segs * g.H * g.K * g.K * sizeof(float));
    }
    if (base) {
        p.ws.fwd_maps = fm;
        p.ws.gam = gam;
        p.ws.w = w;
        p.ws.u = u;
        p.ws.tmat = tm;
        p.ws.hc = hc;
    }
    return off;
}

static Common common_of(const gdn_fwd_args *a) {
    return Common{a->q, a->k, a->v, a->g, a->beta, a->initial_state, a->cu_seqlens,
                  a->B, a->T, a->H, a->K, a->V, a->N, a->dtype, a->use_qk_l2norm,
                  a->cp_mode, a->cp_segment_chunks, a->scale, a->gate_scale};
}
static Common common_of(const gdn_bwd_args *a) {
    return Common{a->q, a->k, a->v, a->g, a->beta, a->initial_state, a->cu_seqlens,
                  a->B, a->T, a->H, a->K, a->V, a->N, a->dtype, a->use_qk_l2norm,
                  a->cp_mode, a->cp_segment_chunks, a->scale, a->gate_scale};
}

}  // namespace gdn

using namespace gdn;

extern "C" {

int32_t gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char *gdn_last_error(void) { return t_last_error.c_str(); }

void gdn_set_spin_limit(int64_t polls) { g_spin_limit.store(polls < 0 ? kDefaultSpinLimit : polls); }

size_t gdn_fwd_workspace_size(const gdn_fwd_args *a) {
    if (!a) { fail(GDN_ERR_INVALID_ARG, "null args"); return 0; }
    Plan p;
    // sizes are device independent: CP capacities use upper bounds
    if (make_plan(common_of(a), false, 0, p) != GDN_OK) return 0;
    if (a->cp_mode != GDN_CP_OFF) {  // room for CP whether or not AUTO picks it
        p.cp = 1;
        p.max_segs = seg_capacity(common_of(a), p.max_chunks);
    }
    return layout(p, false, nullptr);
}

size_t gdn_fwd_ctx_size(const gdn_fwd_args *a) {
    if (!a) { fail(GDN_ERR_INVALID_ARG, "null args"); return 0; }
    Plan p;
    if (make_plan(common_of(a), false, 0, p) != GDN_OK) return 0;
    if (!tc::supported(p)) return 0;
    return ctx_layout(p, nullptr);
}

size_t gdn_bwd_workspace_size(const gdn_bwd_args *a) {
    if (!a) { fail(GDN_ERR_INVALID_ARG, "null args"); return 0; }
    Plan p;
    if (make_plan(common_of(a), true, 0, p) != GDN_OK) return 0;
    if (a->cp_mode != GDN_CP_OFF) {
        p.cp = 1;
        p.max_segs = seg_capacity(common_of(a), p.max_chunks);
    }
    return layout(p, true, nullptr);
}

static gdn_status prepare(const Common &c, bool bwd, void *ws, size_t ws_bytes, Plan &p) {
    gdn_status st = validate(c);  // host-side checks first: they need no device
    if (st != GDN_OK) return st;
    DeviceInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != GDN_OK) return st;
    st = make_plan(c, bwd, dev->sms, p);
    if (st != GDN_OK) return st;
    p.g.status = dev->status;
    const size_t need = layout(p, bwd, nullptr);
    if (!ws && need > 0) return fail(GDN_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
    if (ws_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", ws_bytes, need);
    if (((uintptr_t)ws & (kAlign - 1)) != 0)
        return fail(GDN_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    layout(p, bwd, (char *)ws);
    p.g.chunk_off = p.ws.chunk_off;
    p.g.seg_off = p.ws.seg_off;
    p.g.order = p.ws.order;
    return GDN_OK;
}

gdn_status gdn_chunk_fwd(const gdn_fwd_args *a, void *ws, size_t ws_bytes, void *stream) {
    if (!a) return fail(GDN_ERR_INVALID_ARG, "null args");
    if (!a->o && (long long)a->B * a->T > 0) return fail(GDN_ERR_INVALID_ARG, "o is required");
    if (!aligned16(a->o) || (a->final_state && !aligned16(a->final_state)))
        return fail(GDN_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
    if (a->cp_warmup_chunks < 0 || (a->cp_warmup_chunks > 0 && !(a->cp_warmup_tau > 0.f)))
        return fail(GDN_ERR_INVALID_ARG, "cp_warmup_chunks < 0 or cp_warmup_tau <= 0");
    if (a->fuse_prep != 0 && a->fuse_prep != 1)
        return fail(GDN_ERR_INVALID_ARG, "fuse_prep must be 0 or 1");
    Plan p;
    gdn_status st = prepare(common_of(a), false, ws, ws_bytes, p);
    if (st != GDN_OK) return st;
    p.o = a->o;
    p.final_state = a->final_state;
    p.cp_stats = a->cp_stats;
    p.warm_chunks = p.cp ? a->cp_warmup_chunks : 0;
    p.warm_tau = a->cp_warmup_tau;
    p.fuse_prep = a->fuse_prep == 1;
    const bool save = a->ctx && tc::supported(p);
    if (save && p.warm_chunks > 0)
        return fail(GDN_ERR_INVALID_ARG,
                    "ctx cannot be saved under the warmup shortcut (its states are approximate)");
    if (save) {
        if (((uintptr_t)a->ctx & (kAlign - 1)) != 0)
            return fail(GDN_ERR_INVALID_ARG, "ctx must be 256-byte aligned");
        ctx_layout(p, (char *)a->ctx);
    }
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = tc::supported(p) ? tc::forward(p, s, save) : simt::forward(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "forward launch");
    return GDN_OK;
}

gdn_status gdn_recurrent_step(const gdn_step_args *a, void *stream) {
    if (!a) return fail(GDN_ERR_INVALID_ARG, "null args");
    if (a->N < 0 || a->H < 0) return fail(GDN_ERR_INVALID_ARG, "N and H must be >= 0");
    if ((a->K != 64 && a->K != 128) || (a->V != 64 && a->V != 128))
        return fail(GDN_ERR_UNSUPPORTED, "K = %d, V = %d (64 or 128 supported)", a->K, a->V);
    if (a->dtype != GDN_FP32 && a->dtype != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "dtype %d", a->dtype);
    if ((long long)a->N * a->H == 0) return GDN_OK;
    if (!a->q || !a->k || !a->v || !a->g || !a->beta || !a->state || !a->o)
        return fail(GDN_ERR_INVALID_ARG, "q, k, v, g, beta, state and o are required");
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->g) ||
        !aligned16(a->beta) || !aligned16(a->state) || !aligned16(a->o) ||
        (a->gate_scale && !aligned16(a->gate_scale)))
        return fail(GDN_ERR_INVALID_ARG, "every tensor must be 16-byte aligned");
    DeviceInfo *dev = nullptr;
    gdn_status st = device_info(&dev);
    if (st != GDN_OK) return st;
    const cudaError_t e = step::run(a, dev->sms, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "recurrent step launch");
    return GDN_OK;
}

gdn_status gdn_chunk_bwd(const gdn_bwd_args *a, void *ws, size_t ws_bytes, void *stream) {
    if (!a) return fail(GDN_ERR_INVALID_ARG, "null args");
    if ((long long)a->B * a->T > 0 && (!a->d_o || !a->dq || !a->dk || !a->dv || !a->dg || !a->dbeta))
        return fail(GDN_ERR_INVALID_ARG, "d_o, dq, dk, dv, dg and dbeta are required");
    if (a->grad_dtype != GDN_FP32 && a->grad_dtype != GDN_BF16)
        return fail(GDN_ERR_UNSUPPORTED, "grad_dtype %d", a->grad_dtype);
    if (!aligned16(a->d_o) || !aligned16(a->dq) || !aligned16(a->dk) || !aligned16(a->dv) ||
        !aligned16(a->dg) || !aligned16(a->dbeta) ||
        (a->d_final_state && !aligned16(a->d_final_state)) ||
        (a->d_initial_state && !aligned16(a->d_initial_state)) ||
        (a->d_gate_scale && !aligned16(a->d_gate_scale)))
        return fail(GDN_ERR_INVALID_ARG, "tensors must be 16-byte aligned");
    Plan p;
    gdn_status st = prepare(common_of(a), true, ws, ws_bytes, p);
    if (st != GDN_OK) return st;
    p.d_o = a->d_o;
    p.dht = a->d_final_state;
    p.grad_dtype = a->grad_dtype;
    p.dq = a->dq; p.dk = a->dk; p.dv = a->dv;
    p.dg = a->dg; p.dbeta = a->dbeta; p.dh0 = a->d_initial_state;
    const bool have_ctx = a->ctx && tc::supported(p);
    if (have_ctx) {
        if (((uintptr_t)a->ctx & (kAlign - 1)) != 0)
            return fail(GDN_ERR_INVALID_ARG, "ctx must be 256-byte aligned");
        ctx_layout(p, (char *)const_cast<void *>(a->ctx));
    }
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = tc::supported(p) ? tc::backward(p, s, have_ctx) : simt::backward(p, s);
    if (e == cudaSuccess && a->gate_scale)
        e = simt::gate_bwd(p, a->gate_scale, a->d_gate_scale, s);
    if (e != cudaSuccess) return cuda_fail(e, "backward launch");
    return GDN_OK;
}

gdn_status gdn_sync_status(void *stream) {
    DeviceInfo *dev = nullptr;
    gdn_status st = device_info(&dev);
    if (st != GDN_OK) return st;
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int word = 0;
    e = cudaMemcpy(&word, dev->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the status word");
    if (word != 0) {
        const int zero = 0;
        e = cudaMemcpy(dev->status, &zero, sizeof(int), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return cuda_fail(e, "clearing the status word");
        if (word == GDN_ERR_BAD_SEQLENS)
            return fail(GDN_ERR_BAD_SEQLENS, "cu_seqlens is not 0 = c0 <= ... <= cN = T");
        if (word == GDN_ERR_TIMEOUT)
            return fail(GDN_ERR_TIMEOUT, "a bounded device-side wait ran out");
        return fail(word, "device status %d", word);
    }
    return GDN_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- tracing
namespace gdn {
namespace {
struct ProfRec {
    const char *name;
    cudaEvent_t a, b;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;
std::vector<cudaEvent_t> g_ev_pool;
size_t g_ev_used = 0;
ProfRec *g_open = nullptr;

cudaEvent_t next_event() {
    if (g_ev_used == g_ev_pool.size()) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        g_ev_pool.push_back(e);
    }
    return g_ev_pool[g_ev_used++];
}
}  // namespace

void prof_before(const char *name, cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (!g_prof_on) return;
    cudaEvent_t a = next_event(), b = next_event();
    if (!a || !b) return;
    cudaEventRecord(a, s);
    g_prof.push_back(ProfRec{name, a, b});
    g_open = &g_prof.back();
}

void prof_after(cudaStream_t s) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    if (!g_prof_on || !g_open) return;
    cudaEventRecord(g_open->b, s);
    g_open = nullptr;
}
}  // namespace gdn

extern "C" {

gdn_status gdn_profile_begin(void) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof.clear();
    g_ev_used = 0;
    g_open = nullptr;
    g_prof_on = true;
    return GDN_OK;
}

int32_t gdn_profile_end(gdn_kernel_stat *out, int32_t max) {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    g_prof_on = false;
    std::vector<gdn_kernel_stat> acc;
    for (const ProfRec &r : g_prof) {
        if (cudaEventSynchronize(r.b) != cudaSuccess) continue;
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess) continue;
        gdn_kernel_stat *st = nullptr;
        for (auto &x : acc)
            if (strncmp(x.name, r.name, sizeof x.name - 1) == 0) st = &x;
        if (!st) {
            acc.push_back(gdn_kernel_stat{});
            st = &acc.back();
            strncpy(st->name, r.name, sizeof st->name - 1);
        }
        st->launches += 1;
        st->total_ms += ms;
    }
    g_prof.clear();
    g_ev_used = 0;
    for (int32_t i = 0; i < (int32_t)acc.size() && i < max && out; ++i) out[i] = acc[i];
    return (int32_t)acc.size();
}

}  // extern "C"

// ---------------------------------------------------------------- static-scratch forward
// The allocation-free forward keeps its workspace in this file-scope array.
// In host code `g_static_scratch` names a host-side stand-in, not device
// memory, so its device address is looked up once per device with
// cudaGetSymbolAddress and only that address is handed to the kernels.
namespace gdn {
static __device__ __align__(256) unsigned char g_static_scratch[GDN_STATIC_SCRATCH_BYTES];
static void *g_static_ptr[64];
static std::mutex g_static_mu;
}  // namespace gdn

extern "C" gdn_status gdn_chunk_fwd_static(const gdn_fwd_args *a, void *stream) {
    if (!a) return fail(GDN_ERR_INVALID_ARG, "null args");
    // the same host-side checks, in the same order, as gdn_chunk_fwd's, so that
    // both entry points return the same status for the same bad arguments
    gdn_status st = validate(common_of(a));
    if (st != GDN_OK) return st;
    DeviceInfo *dev_info = nullptr;
    st = device_info(&dev_info);          // sm_103a check before any symbol lookup
    if (st != GDN_OK) return st;
    const size_t need = gdn_fwd_workspace_size(a);
    if (need == 0) return GDN_ERR_INVALID_ARG;     // gdn_last_error already says why
    if (need > GDN_STATIC_SCRATCH_BYTES)
        return fail(GDN_ERR_WORKSPACE,
                    "gdn_chunk_fwd_static: this problem needs %zu bytes of scratch, more than "
                    "the %zu-byte static scratch area; call gdn_chunk_fwd with a workspace",
                    need, (size_t)GDN_STATIC_SCRATCH_BYTES);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_static_mu);
        if (!g_static_ptr[dev]) {
            e = cudaGetSymbolAddress(&g_static_ptr[dev], g_static_scratch);
            if (e != cudaSuccess) {
                g_static_ptr[dev] = nullptr;
                return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
            }
        }
        scratch = g_static_ptr[dev];
    }
    return gdn_chunk_fwd(a, scratch, GDN_STATIC_SCRATCH_BYTES, stream);
}
