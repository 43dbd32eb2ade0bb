// The C ABI of slmoe.h: argument validation, the workspace layout, and the sequencing of
// the kernels of one call on the caller's stream.  Nothing here synchronises the host.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <mutex>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "internal.h"
#include "tc_gemm.h"

namespace slmoe {

static thread_local char g_err[512];
static thread_local void **g_events = nullptr;
static thread_local int g_nevents = 0;
static std::atomic<long long> g_launches{0};

void stage_event(int i, cudaStream_t st) {
    if (g_events && i < g_nevents && g_events[i])
        cudaEventRecord(static_cast<cudaEvent_t>(g_events[i]), st);
}

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

int check_launch(const char *what) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SLMOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
    return SLMOE_OK;
}

int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

static size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int validate_config(const slmoe_config *c) {
    if (!c) return fail(SLMOE_EINVAL, "config is NULL");
    if (c->dtype != SLMOE_F32 && c->dtype != SLMOE_BF16 && c->dtype != SLMOE_MXFP4)
        return fail(SLMOE_EINVAL, "dtype %d is not SLMOE_F32, SLMOE_BF16 or SLMOE_MXFP4", c->dtype);
    if (c->T < 0) return fail(SLMOE_EINVAL, "T = %d < 0", c->T);
    if (c->E < 1 || c->E > 4096) return fail(SLMOE_EINVAL, "E = %d outside [1, 4096]", c->E);
    if (c->k < 1 || c->k > c->E || c->k > 32)
        return fail(SLMOE_EINVAL, "k = %d outside [1, min(E, 32)]", c->k);
    if (c->nbins < 1 || c->nbins > 1024) return fail(SLMOE_EINVAL, "nbins = %d outside [1, 1024]", c->nbins);
    if (c->n_shared < 0 || c->n_shared > 3) return fail(SLMOE_EINVAL, "n_shared = %d outside [0, 3]", c->n_shared);
    const int m = c->dtype != SLMOE_F32 ? 64 : 8;
    if (c->d < m || c->d % m) return fail(SLMOE_EINVAL, "d = %d is not a positive multiple of %d", c->d, m);
    if (c->d_latent < m || c->d_latent % m)
        return fail(SLMOE_EINVAL, "d_latent = %d is not a positive multiple of %d", c->d_latent, m);
    if (c->I < m || c->I % m) return fail(SLMOE_EINVAL, "I = %d is not a positive multiple of %d", c->I, m);
    if (c->n_shared > 0 && (c->I_shared < m || c->I_shared % m))
        return fail(SLMOE_EINVAL, "I_shared = %d is not a positive multiple of %d", c->I_shared, m);
    if (c->dtype == SLMOE_MXFP4 && (c->d_latent % 128 || c->I % 128))
        return fail(SLMOE_EINVAL, "SLMOE_MXFP4 needs d_latent and I multiples of 128 (%d, %d)", c->d_latent, c->I);
    if (!(c->beta1 > 0.f) || !(c->beta2 > 0.f) || !(c->eps >= 0.f))
        return fail(SLMOE_EINVAL, "beta1, beta2 must be > 0 and eps >= 0");
    if ((int64_t)c->T * c->k > (int64_t)INT32_MAX / 2)
        return fail(SLMOE_EUNSUPPORTED, "T * k = %lld too large", (long long)c->T * c->k);
    return SLMOE_OK;
}

int make_layout(const slmoe_config *c, Layout *L) {
    int rc = validate_config(c);
    if (rc) return rc;
    const size_t T = c->T, E = c->E, k = c->k, es = c->dtype != SLMOE_F32 ? 2 : 4;
    const size_t nchunks = (T + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + (bytes ? bytes : 1), 256);
        return at;
    };
    memset(L, 0, sizeof(*L));
    L->nchunks = nchunks;
    L->pub.scores = take(T * E * 4);
    L->pub.topk_idx = take(T * k * 4);
    L->pub.topk_w = take(T * k * 4);
    L->pub.counts = take(E * 4);
    L->pub.offsets = take((E + 1) * 4);
    L->pub.perm = take(T * k * 4);
    L->pub.slot_pos = take(T * k * 4);
    L->chunk_counts = take(nchunks * E * 4);
    L->pub.x_lat = take(T * c->d_latent * es);
    L->pub.h = take(T * k * c->I * es);
    L->pub.y_e = take(T * k * c->d_latent * es);
    L->pub.z = take(T * c->d_latent * es);
    L->pub.h_s = take(T * (size_t)c->n_shared * c->I_shared * es);
    L->pub.status = take(16);
    L->wr_split = c->dtype != SLMOE_F32 ? take(3 * E * c->d * 2) : 0;
    L->counters = take(16 * 4);
    if (c->dtype != SLMOE_F32) {
        // work items: nfb feature blocks x (one pass per expert + one per full pass of tokens)
        const size_t Tk = T * k;
        const size_t nfb1 = (c->I + 127) / 128, nfb2 = (c->d_latent + down_block(c) - 1) / down_block(c);
        // per feature block at most E + ceil(T k / pass) passes (sum of ceil(n_e / pass))
        const size_t pass = grouped_pass(c);
        L->items1 = take(nfb1 * (E + (Tk + pass - 1) / pass) * 16);
        L->items2 = take(nfb2 * (E + (Tk + pass - 1) / pass) * 16);
    }
    if (c->dtype != SLMOE_F32 && T <= (size_t)ROUTER_SPLITK_MAX_M)
        L->rt_split = take(ROUTER_SPLITK_MAX * T * E * 4);
    L->pub.total = off;
    return SLMOE_OK;
}

static bool misaligned(const void *p) { return ((uintptr_t)p & 15u) != 0; }

#define REQ(p, name)                                                                    \
    do {                                                                                \
        if (!(p)) return fail(SLMOE_EINVAL, "%s is NULL", name);                        \
        if (misaligned(p)) return fail(SLMOE_EINVAL, "%s is not 16-byte aligned", name); \
    } while (0)
#define OPT(p, name)                                                                    \
    do {                                                                                \
        if ((p) && misaligned(p)) return fail(SLMOE_EINVAL, "%s is not 16-byte aligned", name); \
    } while (0)

struct Routing {
    float *scores;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *counts, *offsets, *perm, *slot_pos, *chunk_counts;
    int *counters;          // zeroed tile counters; [0] is the router's
};

// One auxiliary stream (lowest priority) and a fork/join event pair per device, created on
// first use and kept until the process exits.  The bf16 forward runs the parts of the layer
// that need only x there, concurrently with routing on the caller's stream.
struct AuxStreams {
    cudaStream_t aux = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
constexpr int MAX_DEVICES = 64;
static AuxStreams g_aux[MAX_DEVICES];
static std::mutex g_aux_mu;

static int aux_streams(AuxStreams **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return fail(SLMOE_ECUDA, "no current device");
    std::lock_guard<std::mutex> lock(g_aux_mu);
    AuxStreams &a = g_aux[dev];
    if (!a.aux) {
        int least = 0, greatest = 0;
        if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
            cudaStreamCreateWithPriority(&a.aux, cudaStreamNonBlocking, least) != cudaSuccess ||
            cudaEventCreateWithFlags(&a.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&a.join, cudaEventDisableTiming) != cudaSuccess)
            return check_launch("auxiliary stream");
    }
    *out = &a;
    return SLMOE_OK;
}

// Router scores, top-k and permutation.  (苏神复盘 Kimi K3 §01-§02.)
static int route_impl(const slmoe_config *c, const Layout &L, char *ws, const void *x,
                      const float *W_r, const float *bias, const float *mu, const Routing &R,
                      uint32_t *hist, int32_t *status, cudaStream_t st) {
    int rc;
    if (c->dtype != SLMOE_F32) {
        rc = tc_router_scores(c, x, W_r, mu, reinterpret_cast<__nv_bfloat16 *>(ws + L.wr_split),
                              R.scores, status, R.counters,
                              L.rt_split ? reinterpret_cast<float *>(ws + L.rt_split) : nullptr, st);
    } else {
        SimtGemm g = {};
        g.seg[0] = {x, W_r, c->d, c->d, c->d, 0};
        g.nseg = 1;
        g.groups = 1;
        g.M = c->T;
        g.N = c->E;
        g.C = R.scores;
        g.ldc = c->E;
        g.mu = mu;
        g.epi = SIMT_SIGMOID;
        g.a_type = DT_F32;
        g.b_type = DT_F32;
        g.c_type = DT_F32;
        rc = launch_simt_gemm(g, st);
    }
    if (rc) return rc;
    stage_event(1, st);
    if ((rc = launch_topk(R.scores, bias, c->T, c->E, c->k, R.topk_idx, R.topk_w, R.chunk_counts,
                          status, st)))
        return rc;
    if ((rc = launch_scan(R.chunk_counts, (int)L.nchunks, c->E, R.counts, st))) return rc;
    if ((rc = launch_scatter(R.topk_idx, R.chunk_counts, R.counts, c->T, c->E, c->k, R.offsets, R.perm,
                             R.slot_pos, st)))
        return rc;
    if (hist) {
        if ((rc = launch_qb_histogram(R.scores, c->T, c->E, c->nbins, hist, status, st))) return rc;
    }
    stage_event(2, st);
    return SLMOE_OK;
}

// The fp32 layer type: every contraction on CUDA cores in fp32.
static int forward_f32(const slmoe_config *c, const Layout &L, char *ws, const void *x,
                       const slmoe_weights *w, const Routing &R, void *y, cudaStream_t st) {
    const int T = c->T, d = c->d, dl = c->d_latent, E = c->E, k = c->k, I = c->I;
    const int ns = c->n_shared, Is = c->I_shared;
    float *x_lat = reinterpret_cast<float *>(ws + L.pub.x_lat);
    float *h = reinterpret_cast<float *>(ws + L.pub.h);
    float *y_e = reinterpret_cast<float *>(ws + L.pub.y_e);
    float *z = reinterpret_cast<float *>(ws + L.pub.z);
    float *h_s = reinterpret_cast<float *>(ws + L.pub.h_s);
    int rc;
    auto base = [&]() {
        SimtGemm g = {};
        g.nseg = 1;
        g.groups = 1;
        g.beta1 = c->beta1;
        g.beta2 = c->beta2;
        g.a_type = g.b_type = g.c_type = DT_F32;
        return g;
    };
    {   // latent down-projection
        SimtGemm g = base();
        g.seg[0] = {x, w->W_in, d, d, d, 0};
        g.M = T; g.N = dl; g.C = x_lat; g.ldc = dl; g.epi = SIMT_STORE;
        if ((rc = launch_simt_gemm(g, st))) return rc;
    }
    stage_event(3, st);
    {   // expert gate|up with SiTU-GLU, rows gathered by perm, grouped by expert
        SimtGemm g = base();
        g.seg[0] = {x_lat, w->W13, dl, dl, dl, (int64_t)2 * I * dl};
        g.a_index = R.perm; g.group_offsets = R.offsets; g.groups = E;
        g.M = T; g.N = I; g.glu_up_row = I; g.C = h; g.ldc = I; g.epi = SIMT_GLU;
        if ((rc = launch_simt_gemm(g, st))) return rc;
    }
    stage_event(4, st);
    {   // expert down-projection
        SimtGemm g = base();
        g.seg[0] = {h, w->W2, I, I, I, (int64_t)dl * I};
        g.group_offsets = R.offsets; g.groups = E;
        g.M = T; g.N = dl; g.C = y_e; g.ldc = dl; g.epi = SIMT_STORE;
        if ((rc = launch_simt_gemm(g, st))) return rc;
    }
    stage_event(5, st);
    if ((rc = launch_combine_rmsnorm(DT_F32, y_e, R.topk_w, R.slot_pos, w->gamma, T, dl, k, c->eps,
                                     z, st)))
        return rc;
    stage_event(6, st);
    for (int s = 0; s < ns; ++s) {   // shared experts: gate|up with SiTU-GLU
        SimtGemm g = base();
        g.seg[0] = {x, static_cast<const float *>(w->W13_s) + (size_t)s * 2 * Is * d, d, d, d, 0};
        g.M = T; g.N = Is; g.glu_up_row = Is; g.C = h_s + (size_t)s * Is; g.ldc = (int64_t)ns * Is;
        g.epi = SIMT_GLU;
        if ((rc = launch_simt_gemm(g, st))) return rc;
    }
    stage_event(7, st);
    {   // y = z W_out^T + sum_s h_s W2_s^T in one K-segmented product
        SimtGemm g = base();
        g.seg[0] = {z, w->W_out, dl, dl, dl, 0};
        for (int s = 0; s < ns; ++s)
            g.seg[1 + s] = {h_s + (size_t)s * Is, static_cast<const float *>(w->W2_s) + (size_t)s * d * Is,
                            (int64_t)ns * Is, Is, Is, 0};
        g.nseg = 1 + ns;
        g.M = T; g.N = d; g.C = y; g.ldc = d; g.epi = SIMT_STORE;
        if ((rc = launch_simt_gemm(g, st))) return rc;
    }
    stage_event(8, st);
    (void)E;
    return SLMOE_OK;
}

}  // namespace slmoe

using namespace slmoe;

extern "C" {

const char *slmoe_last_error(void) { return g_err; }

int slmoe_set_stage_events(void **events, int n) {
    g_events = n > 0 ? events : nullptr;
    g_nevents = n > 0 ? n : 0;
    return SLMOE_OK;
}

long long slmoe_launch_count(void) { return g_launches.load(); }

int slmoe_device_sm_count(void) { return sm_count(); }

size_t slmoe_workspace_size(const slmoe_config *cfg) {
    Layout L;
    if (make_layout(cfg, &L)) return 0;
    return L.pub.total;
}

int slmoe_workspace_layout_get(const slmoe_config *cfg, slmoe_workspace_layout *out) {
    if (!out) return fail(SLMOE_EINVAL, "out is NULL");
    Layout L;
    int rc = make_layout(cfg, &L);
    if (rc) return rc;
    *out = L.pub;
    return SLMOE_OK;
}

int slmoe_route(const slmoe_config *cfg, const void *x, const float *W_r, const float *bias,
                const float *logit_offset, int32_t *topk_idx, float *topk_w, float *scores,
                int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos,
                uint32_t *hist, int32_t *status, void *workspace, size_t workspace_bytes,
                void *stream) {
    g_err[0] = 0;
    Layout L;
    int rc = make_layout(cfg, &L);
    if (rc) return rc;
    REQ(workspace, "workspace");
    if (workspace_bytes < L.pub.total)
        return fail(SLMOE_ENOSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, L.pub.total);
    REQ(counts, "counts");
    REQ(offsets, "offsets");
    if (cfg->T > 0) {
        REQ(x, "x"); REQ(W_r, "W_r"); REQ(bias, "bias"); OPT(logit_offset, "logit_offset");
        REQ(topk_idx, "topk_idx"); REQ(topk_w, "topk_w"); REQ(perm, "perm"); REQ(slot_pos, "slot_pos");
        OPT(scores, "scores"); OPT(hist, "hist");
    }
    OPT(status, "status");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    if (cfg->T == 0) {
        if (cudaMemsetAsync(counts, 0, cfg->E * 4, st) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, (cfg->E + 1) * 4, st) != cudaSuccess)
            return check_launch("memset");
        return SLMOE_OK;
    }
    Routing R = {scores ? scores : reinterpret_cast<float *>(ws + L.pub.scores), topk_idx, topk_w,
                 counts, offsets, perm, slot_pos, reinterpret_cast<int32_t *>(ws + L.chunk_counts),
                 reinterpret_cast<int *>(ws + L.counters)};
    if (cudaMemsetAsync(R.counters, 0, 16 * sizeof(int), st) != cudaSuccess) return check_launch("memset");
    stage_event(0, st);
    return route_impl(cfg, L, ws, x, W_r, bias, logit_offset, R, hist, status, st);
}

int slmoe_qb_histogram(const float *scores, int64_t T, int32_t E, int32_t nbins, uint32_t *hist,
                       int32_t *status, void *stream) {
    g_err[0] = 0;
    if (T < 0 || T > INT32_MAX) return fail(SLMOE_EINVAL, "T outside [0, 2^31 - 1]");
    if (E < 1) return fail(SLMOE_EINVAL, "E < 1");
    if (nbins < 1 || nbins > 1024) return fail(SLMOE_EINVAL, "nbins outside [1, 1024]");
    if (!hist) return fail(SLMOE_EINVAL, "hist is NULL");
    if (T > 0 && !scores) return fail(SLMOE_EINVAL, "scores is NULL");
    if (((uintptr_t)scores & 3u) || ((uintptr_t)hist & 3u) || ((uintptr_t)status & 3u))
        return fail(SLMOE_EINVAL, "scores, hist and status must be 4-byte aligned");
    return launch_qb_histogram(scores, T, E, nbins, hist, status, static_cast<cudaStream_t>(stream));
}

int slmoe_qb_update(const uint32_t *hist, int32_t E, int32_t nbins, int32_t k, float *q_out,
                    float *bias, void *stream) {
    g_err[0] = 0;
    if (E < 1 || E > 8192) return fail(SLMOE_EINVAL, "E outside [1, 8192]");
    if (k < 1 || k > E) return fail(SLMOE_EINVAL, "k outside [1, E]");
    if (nbins < 1 || nbins > 1024) return fail(SLMOE_EINVAL, "nbins outside [1, 1024]");
    if (!hist || !bias) return fail(SLMOE_EINVAL, "hist and bias are required");
    if (((uintptr_t)hist & 3u) || ((uintptr_t)bias & 3u) || ((uintptr_t)q_out & 3u))
        return fail(SLMOE_EINVAL, "hist, bias and q_out must be 4-byte aligned");
    return launch_qb_update(hist, E, nbins, k, q_out, bias, static_cast<cudaStream_t>(stream));
}

int slmoe_signsgd_update(const int32_t *counts, int32_t E, float step, float *bias, void *stream) {
    g_err[0] = 0;
    if (E < 1 || E > 65536) return fail(SLMOE_EINVAL, "E outside [1, 65536]");
    if (!std::isfinite(step) || !(step > 0.0f)) return fail(SLMOE_EINVAL, "step must be finite and > 0");
    if (!counts || !bias) return fail(SLMOE_EINVAL, "counts and bias are required");
    if (((uintptr_t)counts & 3u) || ((uintptr_t)bias & 3u))
        return fail(SLMOE_EINVAL, "counts and bias must be 4-byte aligned");
    return launch_signsgd_update(counts, E, step, bias, static_cast<cudaStream_t>(stream));
}

size_t slmoe_topk_workspace_size(int32_t T, int32_t E, int32_t k) {
    if (T < 0 || E < 1 || E > 4096 || k < 1 || k > E || k > 32 || (int64_t)T * k > (int64_t)INT32_MAX / 2) {
        fail(SLMOE_EINVAL, "T = %d, E = %d, k = %d outside the supported range", T, E, k);
        return 0;
    }
    const size_t nchunks = ((size_t)T + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    return align_up((nchunks ? nchunks : 1) * (size_t)E * 4, 256);
}

int slmoe_topk(const float *scores, const float *bias, int32_t T, int32_t E, int32_t k, int32_t *topk_idx,
               float *topk_w, int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos,
               int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    const size_t need = slmoe_topk_workspace_size(T, E, k);
    if (need == 0) return SLMOE_EINVAL;
    REQ(counts, "counts");
    REQ(offsets, "offsets");
    OPT(status, "status");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (T == 0) {
        if (cudaMemsetAsync(counts, 0, (size_t)E * 4, st) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, ((size_t)E + 1) * 4, st) != cudaSuccess)
            return check_launch("memset");
        return SLMOE_OK;
    }
    REQ(scores, "scores"); REQ(bias, "bias"); REQ(topk_idx, "topk_idx"); REQ(topk_w, "topk_w");
    REQ(perm, "perm"); REQ(slot_pos, "slot_pos"); REQ(workspace, "workspace");
    if (workspace_bytes < need)
        return fail(SLMOE_ENOSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    int32_t *chunk_counts = static_cast<int32_t *>(workspace);
    const int nchunks = (T + ROUTE_CHUNK - 1) / ROUTE_CHUNK;
    int rc;
    if ((rc = launch_topk(scores, bias, T, E, k, topk_idx, topk_w, chunk_counts, status, st))) return rc;
    if ((rc = launch_scan(chunk_counts, nchunks, E, counts, st))) return rc;
    return launch_scatter(topk_idx, chunk_counts, counts, T, E, k, offsets, perm, slot_pos, st);
}

int slmoe_mxfp4_quantize(const void *W, int64_t rows, int32_t K, uint8_t *packed, uint8_t *scales, void *stream) {
    g_err[0] = 0;
    if (rows < 0 || K <= 0 || K % 32) return fail(SLMOE_EINVAL, "rows >= 0 and K a positive multiple of 32 required");
    if (rows == 0) return SLMOE_OK;
    REQ(W, "W"); REQ(packed, "packed");
    if (!scales) return fail(SLMOE_EINVAL, "scales is NULL");
    return launch_mxfp4_quantize(W, rows, K, packed, scales, static_cast<cudaStream_t>(stream));
}

int slmoe_mxfp8_quantize(const float *X, int64_t rows, int32_t K, uint8_t *codes, uint8_t *scales, void *stream) {
    g_err[0] = 0;
    if (rows < 0 || K <= 0 || K % 32) return fail(SLMOE_EINVAL, "rows >= 0 and K a positive multiple of 32 required");
    if (rows == 0) return SLMOE_OK;
    REQ(X, "X"); REQ(codes, "codes");
    if (!scales) return fail(SLMOE_EINVAL, "scales is NULL");
    return launch_mxfp8_quantize(X, rows, K, codes, scales, static_cast<cudaStream_t>(stream));
}

int slmoe_wait_abort_check(int32_t *status, uint64_t wait_limit_ns, void *stream) {
    g_err[0] = 0;
    REQ(status, "status");
    if (wait_limit_ns == 0 || wait_limit_ns > 60000000000ull)
        return fail(SLMOE_EINVAL, "wait_limit_ns must be in (0, 60 s]");
    return tc_wait_abort_check(status, wait_limit_ns, static_cast<cudaStream_t>(stream));
}

size_t slmoe_backward_workspace_size(const slmoe_config *cfg) {
    Layout L;
    if (make_layout(cfg, &L)) return 0;
    if (cfg->dtype != SLMOE_BF16) {
        fail(SLMOE_EUNSUPPORTED, "the backward is built for the bf16 layer type");
        return 0;
    }
    return backward_workspace_bytes(cfg, nullptr);
}

int slmoe_backward_layout_get(const slmoe_config *cfg, slmoe_backward_layout *out) {
    if (!out) return fail(SLMOE_EINVAL, "out is NULL");
    if (slmoe_backward_workspace_size(cfg) == 0) return cfg && cfg->dtype != SLMOE_BF16 ? SLMOE_EUNSUPPORTED : SLMOE_EINVAL;
    BwdLayout L;
    backward_workspace_bytes(cfg, &L);
    out->dz = L.dz; out->dye = L.dye; out->dg = L.dg; out->gu = L.gu; out->dgu = L.dgu;
    out->dx_lat = L.dx_lat; out->gu_s = L.gu_s; out->dgu_s = L.dgu_s; out->total = L.total;
    return SLMOE_OK;
}

int slmoe_backward(const slmoe_config *cfg, const void *x, const slmoe_weights *w, const float *dy, float *dx,
                   const slmoe_grads *grads, int accumulate, const void *fwd_workspace, size_t fwd_workspace_bytes,
                   int32_t *status, void *workspace, size_t workspace_bytes, void *stream) {
    g_err[0] = 0;
    Layout L;
    int rc = make_layout(cfg, &L);
    if (rc) return rc;
    if (cfg->dtype != SLMOE_BF16) return fail(SLMOE_EUNSUPPORTED, "the backward is built for the bf16 layer type");
    if (cfg->T == 0) return SLMOE_OK;
    if (cfg->E > 4096) return fail(SLMOE_EUNSUPPORTED, "E > 4096");
    if (cfg->d_latent > 8192) return fail(SLMOE_EUNSUPPORTED, "d_latent > 8192 in the backward");
    if (!w || !grads) return fail(SLMOE_EINVAL, "weights and grads are required");
    REQ(x, "x"); REQ(dy, "dy"); REQ(dx, "dx");
    REQ(w->W_r, "W_r"); REQ(w->W_in, "W_in"); REQ(w->W13, "W13"); REQ(w->W2, "W2");
    REQ(w->gamma, "gamma"); REQ(w->W_out, "W_out");
    REQ(grads->dW_r, "dW_r"); REQ(grads->dW_in, "dW_in"); REQ(grads->dW13, "dW13"); REQ(grads->dW2, "dW2");
    REQ(grads->dgamma, "dgamma"); REQ(grads->dW_out, "dW_out");
    if (cfg->n_shared > 0) {
        REQ(w->W13_s, "W13_s"); REQ(w->W2_s, "W2_s"); REQ(grads->dW13_s, "dW13_s"); REQ(grads->dW2_s, "dW2_s");
    }
    OPT(status, "status");
    REQ(fwd_workspace, "fwd_workspace");
    if (fwd_workspace_bytes < L.pub.total)
        return fail(SLMOE_ENOSPACE, "forward workspace %zu bytes < %zu", fwd_workspace_bytes, L.pub.total);
    REQ(workspace, "workspace");
    const size_t need = backward_workspace_bytes(cfg, nullptr);
    if (workspace_bytes < need) return fail(SLMOE_ENOSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, need);
    if (accumulate != 0 && accumulate != 1) return fail(SLMOE_EINVAL, "accumulate must be 0 or 1");
    const char *fw = static_cast<const char *>(fwd_workspace);
    FwdSaved fs;
    fs.scores = reinterpret_cast<const float *>(fw + L.pub.scores);
    fs.topk_w = reinterpret_cast<const float *>(fw + L.pub.topk_w);
    fs.topk_idx = reinterpret_cast<const int32_t *>(fw + L.pub.topk_idx);
    fs.counts = reinterpret_cast<const int32_t *>(fw + L.pub.counts);
    fs.offsets = reinterpret_cast<const int32_t *>(fw + L.pub.offsets);
    fs.perm = reinterpret_cast<const int32_t *>(fw + L.pub.perm);
    fs.slot_pos = reinterpret_cast<const int32_t *>(fw + L.pub.slot_pos);
    fs.x_lat = reinterpret_cast<const __nv_bfloat16 *>(fw + L.pub.x_lat);
    fs.h = reinterpret_cast<const __nv_bfloat16 *>(fw + L.pub.h);
    fs.y_e = reinterpret_cast<const __nv_bfloat16 *>(fw + L.pub.y_e);
    fs.z = reinterpret_cast<const __nv_bfloat16 *>(fw + L.pub.z);
    fs.h_s = reinterpret_cast<const __nv_bfloat16 *>(fw + L.pub.h_s);
    fs.items1 = reinterpret_cast<const int4 *>(fw + L.items1);
    fs.n_items = reinterpret_cast<const int *>(fw + L.counters) + 8;
    return tc_backward(cfg, x, w, dy, dx, grads, accumulate, fs, static_cast<char *>(workspace), status,
                       static_cast<cudaStream_t>(stream));
}

int slmoe_forward(const slmoe_config *cfg, const void *x, const slmoe_weights *w,
                  const float *bias, const float *logit_offset, void *y, int32_t *topk_idx_out,
                  uint32_t *hist, int32_t *status, void *workspace, size_t workspace_bytes,
                  void *stream) {
    g_err[0] = 0;
    Layout L;
    int rc = make_layout(cfg, &L);
    if (rc) return rc;
    if (cfg->T == 0) return SLMOE_OK;
    REQ(workspace, "workspace");
    if (workspace_bytes < L.pub.total)
        return fail(SLMOE_ENOSPACE, "workspace %zu bytes < %zu needed", workspace_bytes, L.pub.total);
    if (!w) return fail(SLMOE_EINVAL, "weights is NULL");
    REQ(x, "x"); REQ(y, "y"); REQ(bias, "bias"); OPT(logit_offset, "logit_offset");
    REQ(w->W_r, "W_r"); REQ(w->W_in, "W_in"); REQ(w->W13, "W13"); REQ(w->W2, "W2");
    REQ(w->gamma, "gamma"); REQ(w->W_out, "W_out");
    if (cfg->n_shared > 0) { REQ(w->W13_s, "W13_s"); REQ(w->W2_s, "W2_s"); }
    if (cfg->dtype == SLMOE_MXFP4) {
        REQ(w->W13_scale, "W13_scale"); REQ(w->W2_scale, "W2_scale");
        // the packed weights are read by TMA with the FP4 expansion, which wants 32-byte alignment
        if (((uintptr_t)w->W13 | (uintptr_t)w->W2) & 31u)
            return fail(SLMOE_EINVAL, "W13 / W2 (MXFP4) are not 32-byte aligned");
    }
    OPT(topk_idx_out, "topk_idx_out"); OPT(hist, "hist"); OPT(status, "status");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    int32_t *stat = status ? status : reinterpret_cast<int32_t *>(ws + L.pub.status);
    if (!status && cudaMemsetAsync(stat, 0, 16, st) != cudaSuccess) return check_launch("memset");
    Routing R = {reinterpret_cast<float *>(ws + L.pub.scores),
                 reinterpret_cast<int32_t *>(ws + L.pub.topk_idx),
                 reinterpret_cast<float *>(ws + L.pub.topk_w),
                 reinterpret_cast<int32_t *>(ws + L.pub.counts),
                 reinterpret_cast<int32_t *>(ws + L.pub.offsets),
                 reinterpret_cast<int32_t *>(ws + L.pub.perm),
                 reinterpret_cast<int32_t *>(ws + L.pub.slot_pos),
                 reinterpret_cast<int32_t *>(ws + L.chunk_counts),
                 reinterpret_cast<int *>(ws + L.counters)};
    if (cudaMemsetAsync(R.counters, 0, 16 * sizeof(int), st) != cudaSuccess) return check_launch("memset");
    stage_event(0, st);
    if (cfg->dtype == SLMOE_F32) {
        if ((rc = route_impl(cfg, L, ws, x, w->W_r, bias, logit_offset, R, hist, stat, st))) return rc;
        if (topk_idx_out &&
            cudaMemcpyAsync(topk_idx_out, R.topk_idx, (size_t)cfg->T * cfg->k * 4, cudaMemcpyDeviceToDevice,
                            st) != cudaSuccess)
            return check_launch("copy topk_idx");
        return forward_f32(cfg, L, ws, x, w, R, y, st);
    }
    TcForward tf = {};
    tf.x_lat = ws + L.pub.x_lat;
    tf.h = ws + L.pub.h;
    tf.y_e = ws + L.pub.y_e;
    tf.z = ws + L.pub.z;
    tf.h_s = ws + L.pub.h_s;
    tf.topk_w = R.topk_w;
    tf.counts = R.counts;
    tf.offsets = R.offsets;
    tf.perm = R.perm;
    tf.slot_pos = R.slot_pos;
    tf.status = stat;
    tf.counters = R.counters;
    tf.items1 = reinterpret_cast<int4 *>(ws + L.items1);
    tf.items2 = reinterpret_cast<int4 *>(ws + L.items2);
    // the down-projection and the shared experts' gate|up need only x: fork them onto the
    // auxiliary stream, route on the caller's stream meanwhile, join before the routed experts
    // (the routing kernels are launched first so that they take the SMs first; the
    // persistent front kernels fill SMs as the router's tail wave frees them)
    AuxStreams *aux = nullptr;
    if ((rc = aux_streams(&aux))) return rc;
    if (cudaEventRecord(aux->fork, st) != cudaSuccess) return check_launch("fork");
    if ((rc = route_impl(cfg, L, ws, x, w->W_r, bias, logit_offset, R, hist, stat, st))) return rc;
    if (cudaStreamWaitEvent(aux->aux, aux->fork, 0) != cudaSuccess) return check_launch("fork wait");
    if ((rc = tc_forward_front(cfg, x, w, tf, aux->aux))) return rc;
    if (cudaEventRecord(aux->join, aux->aux) != cudaSuccess) return check_launch("join");
    if (topk_idx_out &&
        cudaMemcpyAsync(topk_idx_out, R.topk_idx, (size_t)cfg->T * cfg->k * 4, cudaMemcpyDeviceToDevice,
                        st) != cudaSuccess)
        return check_launch("copy topk_idx");
    if ((rc = tc_worklists(cfg, tf, st))) return rc;
    if (cudaStreamWaitEvent(st, aux->join, 0) != cudaSuccess) return check_launch("join wait");
    return tc_forward_back(cfg, w, tf, y, st);
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Routing with the library's own fixed scratch instead of a caller-supplied workspace.
// The scratch is one file-scope device array; its device address is looked up once per
// device (with that device current) and cached.  Same kernels and arithmetic as slmoe_route.

namespace slmoe {

static __device__ __align__(256) unsigned char g_route_scratch[SLMOE_ROUTE_NOALLOC_SCRATCH_BYTES];

// The scratch's device address belongs to the context that loaded this library's device
// code.  It is cached per device together with that context's id (cuCtxGetId: unique for the
// life of the process), so a call after cudaDeviceReset, or after the device's context was
// destroyed and made again, looks the address up anew instead of using a stale one.
struct ScratchAddr {
    unsigned long long ctx_id = 0;
    char *ptr = nullptr;
};
static ScratchAddr g_route_scratch_addr[MAX_DEVICES];
static std::mutex g_route_scratch_mu;
static PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
static PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;

static int driver_fn(const char *name, int version, void **fn) {
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, version, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !*fn) {
        cudaGetLastError();
        return fail(SLMOE_ECUDA, "driver entry point %s not available", name);
    }
    return SLMOE_OK;
}

// Id of the current context, or 0 when the thread has none yet (called with
// g_route_scratch_mu held).
static int current_ctx_id(unsigned long long *id) {
    int rc;
    if (!g_ctx_current && (rc = driver_fn("cuCtxGetCurrent", 4000, (void **)&g_ctx_current))) return rc;
    if (!g_ctx_id && (rc = driver_fn("cuCtxGetId", 12000, (void **)&g_ctx_id))) return rc;
    CUcontext ctx = nullptr;
    *id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS) return fail(SLMOE_ECUDA, "cuCtxGetCurrent failed");
    if (ctx && g_ctx_id(ctx, id) != CUDA_SUCCESS) return fail(SLMOE_ECUDA, "cuCtxGetId failed");
    return SLMOE_OK;
}

static int route_scratch(char **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES)
        return fail(SLMOE_ECUDA, "no current device");
    std::lock_guard<std::mutex> lock(g_route_scratch_mu);
    unsigned long long id = 0;
    int rc = current_ctx_id(&id);
    if (rc) return rc;
    ScratchAddr &s = g_route_scratch_addr[dev];
    if (!s.ptr || id == 0 || s.ctx_id != id) {
        // set-up: the lookup also makes the device's primary context current if it was not
        char *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress((void **)&ptr, g_route_scratch);
        if (e != cudaSuccess || !ptr) {
            cudaGetLastError();
            return fail(SLMOE_ECUDA, "device address of the routing scratch: %s", cudaGetErrorString(e));
        }
        if ((rc = current_ctx_id(&id))) return rc;
        if (id == 0) return fail(SLMOE_ECUDA, "no current CUDA context after set-up");
        s.ptr = ptr;
        s.ctx_id = id;
    }
    *out = s.ptr;
    return SLMOE_OK;
}

// Offsets of what a routing call keeps in the scratch: the zeroed tile counters, the
// per-chunk expert counts, the split router weights (bf16 type) and, when the caller passes
// no scores buffer, the scores.  Returns the bytes needed.
struct RouteScratch {
    size_t counters, chunk_counts, wr_split, scores, rt_split, total;
};

static RouteScratch route_scratch_layout(const slmoe_config *c, size_t nchunks, bool own_scores) {
    RouteScratch s = {};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off = align_up(off + (bytes ? bytes : 1), 256);
        return o;
    };
    s.counters = take(16 * sizeof(int));
    s.chunk_counts = take(nchunks * (size_t)c->E * 4);
    s.wr_split = c->dtype != SLMOE_F32 ? take((size_t)3 * c->E * c->d * 2) : 0;
    s.scores = own_scores ? take((size_t)c->T * c->E * 4) : 0;
    s.total = off;
    // the split-K router sums of a small bf16 batch, as in the workspace layout, when they fit
    // (else the router runs unsplit, its fp32 logit sums added in another order)
    if (c->dtype != SLMOE_F32 && c->T <= ROUTER_SPLITK_MAX_M) {
        const size_t at = take((size_t)ROUTER_SPLITK_MAX * c->T * c->E * 4);
        if (off <= (size_t)SLMOE_ROUTE_NOALLOC_SCRATCH_BYTES) {
            s.rt_split = at;
            s.total = off;
        }
    }
    return s;
}

}  // namespace slmoe

extern "C" int slmoe_route_noalloc(const slmoe_config *cfg, const void *x, const float *W_r,
                                   const float *bias, const float *logit_offset, int32_t *topk_idx,
                                   float *topk_w, float *scores, int32_t *counts, int32_t *offsets,
                                   int32_t *perm, int32_t *slot_pos, uint32_t *hist, int32_t *status,
                                   void *stream) {
    g_err[0] = 0;
    Layout L;
    int rc = make_layout(cfg, &L);
    if (rc) return rc;
    REQ(counts, "counts");
    REQ(offsets, "offsets");
    if (cfg->T > 0) {
        REQ(x, "x"); REQ(W_r, "W_r"); REQ(bias, "bias"); OPT(logit_offset, "logit_offset");
        REQ(topk_idx, "topk_idx"); REQ(topk_w, "topk_w"); REQ(perm, "perm"); REQ(slot_pos, "slot_pos");
        OPT(scores, "scores"); OPT(hist, "hist");
    }
    OPT(status, "status");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cfg->T == 0) {
        if (cudaMemsetAsync(counts, 0, cfg->E * 4, st) != cudaSuccess ||
            cudaMemsetAsync(offsets, 0, (cfg->E + 1) * 4, st) != cudaSuccess)
            return check_launch("memset");
        return SLMOE_OK;
    }
    const RouteScratch S = route_scratch_layout(cfg, L.nchunks, scores == nullptr);
    if (S.total > (size_t)SLMOE_ROUTE_NOALLOC_SCRATCH_BYTES)
        return fail(SLMOE_ENOSPACE,
                    "this routing call needs %zu bytes of scratch, more than the fixed %zu bytes "
                    "(pass a scores buffer, route fewer tokens per call, or use slmoe_route)",
                    S.total, (size_t)SLMOE_ROUTE_NOALLOC_SCRATCH_BYTES);
    char *scr = nullptr;
    if ((rc = route_scratch(&scr))) return rc;
    // route_impl reads the split router weights and the split-K router sums at these offsets
    L.wr_split = S.wr_split;
    L.rt_split = S.rt_split;
    Routing R = {scores ? scores : reinterpret_cast<float *>(scr + S.scores), topk_idx, topk_w,
                 counts, offsets, perm, slot_pos, reinterpret_cast<int32_t *>(scr + S.chunk_counts),
                 reinterpret_cast<int *>(scr + S.counters)};
    if (cudaMemsetAsync(R.counters, 0, 16 * sizeof(int), st) != cudaSuccess) return check_launch("memset");
    stage_event(0, st);
    return route_impl(cfg, L, scr, x, W_r, bias, logit_offset, R, hist, status, st);
}
