/*
 * slmoe.h - C ABI of the Stable LatentMoE forward path and its Quantile Balancing engine
 * on one NVIDIA GB300 (sm_103a).
 *
 * Sources, cited by page title and section:
 *   [K3-news] "苏神复盘 Kimi K3：896 个专家背后，藏着哪些关键技术取舍？"
 *             §01 LatentMoE 如何重新分配专家预算, §02 Stable LatentMoE 如何处理数值与负载风险
 *   [K3-arch] K3 architecture write-up (tahou.com): SiTU激活优化, 归一化策略调整, 负载均衡优化
 *   [SLMoE]   "Stable Latent MoE" concept note: 路由机制, Quantile Balancing,
 *             Latent-Space MoE, SiTU 激活, 训练基础设施 (static shapes, no host sync)
 *
 * Conventions shared by every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller.  Matrices are dense,
 *     row-major, with the nn.Linear convention W[out, in].
 *   - "stream" is a cudaStream_t passed as void* (NULL = the legacy default stream).  All
 *     work is enqueued on it; no call synchronises the host or copies device->host, so a
 *     call returns before its kernels finish ([SLMoE] 训练基础设施: no host sync on the
 *     critical path).  Calls that share output buffers must be ordered on one stream.
 *   - The library allocates no memory.  Scratch lives in a caller-provided workspace of at
 *     least slmoe_workspace_size() bytes, 256-byte aligned (slmoe_route_noalloc instead
 *     uses a fixed device array inside the library).  On the bf16 type,
 *     slmoe_forward creates, on its first call on a device, one auxiliary CUDA stream (lowest
 *     priority) and two events, kept until the process exits: it forks the down-projection
 *     and the shared experts' gate|up onto that stream, routes on the caller's stream
 *     meanwhile, and joins back through an event before the routed experts.  Consecutive
 *     calls on one device therefore share that stream; calls from several host threads on
 *     one device must be serialised by the caller.
 *   - Return value: SLMOE_OK (0) or a negative code.  Arguments are validated on the host
 *     before any launch; on error nothing is launched and slmoe_last_error() gives a
 *     thread-local message.  No C++ exception crosses the ABI.
 *   - Optional device status words (int32_t status[4], may be NULL) report anomalies
 *     without trapping: status[0] += number of NaN router scores met (a NaN score is never
 *     selected and is left out of histograms); status[1] is set to 1 when a histogram bin
 *     would pass 2^32-1; status[2] is set to 1 when a bounded device-side wait gave up (the
 *     outputs of that call are then invalid); status[3] is reserved.  The caller zeroes
 *     the words; calls only add or set.
 *   - Contraction work is the dense and grouped GEMMs on tcgen05 tensor cores (bf16 in,
 *     fp32 accumulate).  The fp32 layer type runs every step in fp32 on CUDA cores.
 */
#ifndef SLMOE_H
#define SLMOE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SLMOE_API __attribute__((visibility("default")))
#else
#define SLMOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define SLMOE_OK            0
#define SLMOE_EINVAL       (-1)  /* null pointer, misalignment, bad shape or k > E       */
#define SLMOE_EUNSUPPORTED (-2)  /* shape or type outside what the kernels are built for */
#define SLMOE_ECUDA        (-3)  /* a CUDA runtime or launch error                       */
#define SLMOE_ENOSPACE     (-4)  /* the workspace is smaller than slmoe_workspace_size() */

#define SLMOE_F32  0             /* x, projection weights and intermediates in fp32      */
#define SLMOE_BF16 1             /* the same in bf16 (fp32 accumulation, fp32 router)    */
/* The layer with MXFP4 weights and MXFP8 activations in the routed experts ([SLMoE]
 * 训练基础设施: MXFP4 weights, MXFP8 activations): W13 / W2 point to packed MXFP4 codes
 * [E, 2I, d_latent/2] / [E, d_latent, I/2] (bytes, 32-byte aligned; see slmoe_mxfp4_quantize)
 * with block scales W13_scale [E, 2I, d_latent/32] / W2_scale [E, d_latent, I/32].  The
 * routed experts' inputs x_lat and h are MXFP8 (see slmoe_mxfp8_quantize: blocks of 32 along
 * d_latent and I), produced by the epilogues of the down-projection and of the experts'
 * gate/up, and every routed-expert contraction runs on the block-scaled tensor cores (E2M1
 * x E4M3 products, exact, fp32 accumulation).  d_latent and I must be multiples of 128.
 * Everything else (router, shared experts, projections, y_e, z) is as SLMOE_BF16. */
#define SLMOE_MXFP4 2

/* Shape and constants of one layer.  beta1 / beta2 are the SiTU and soft-cap constants
 * ([K3-arch] SiTU激活优化: 4 and 25), eps the RMSNorm epsilon, nbins the QB histogram
 * width ([K3-arch] 负载均衡优化: 1000; at most 1024 here).
 * Limits: 1 <= k <= E <= 4096, k <= 32; d, d_latent, I, I_shared multiples of 8 (of 64 for
 * the bf16 type); n_shared <= 3; T >= 0 (T = 0 is a no-op). */
typedef struct slmoe_config {
    int32_t T;           /* tokens in the call                                   */
    int32_t d;           /* hidden width                                         */
    int32_t d_latent;    /* latent width of the routed experts                   */
    int32_t E;           /* routed experts                                       */
    int32_t k;           /* experts selected per token                           */
    int32_t I;           /* routed-expert intermediate width                     */
    int32_t n_shared;    /* always-on shared experts                             */
    int32_t I_shared;    /* shared-expert intermediate width                     */
    int32_t nbins;       /* QB histogram bins over [0, 1]                        */
    float   beta1;       /* SiTU gate bound                                      */
    float   beta2;       /* soft cap of the up branch                            */
    float   eps;         /* RMSNorm epsilon                                      */
    int32_t dtype;       /* SLMOE_F32 or SLMOE_BF16                              */
} slmoe_config;

/* Layer weights.  "act" = the layer type (fp32 for SLMOE_F32, bf16 for SLMOE_BF16).
 * Expert gate/up matrices hold the gate rows first ([SLMoE] SiTU 激活: the first half of
 * the last axis is the gate). */
typedef struct slmoe_weights {
    const float *W_r;    /* [E, d]                    fp32 router               */
    const void  *W_in;   /* [d_latent, d]             act  latent down-proj     */
    const void  *W13;    /* [E, 2I, d_latent]         act  expert gate|up       */
    const void  *W2;     /* [E, d_latent, I]          act  expert down          */
    const float *gamma;  /* [d_latent]                fp32 RMSNorm weight       */
    const void  *W_out;  /* [d, d_latent]             act  latent up-proj       */
    const void  *W13_s;  /* [n_shared, 2I_shared, d]  act  shared gate|up       */
    const void  *W2_s;   /* [n_shared, d, I_shared]   act  shared down          */
    const uint8_t *W13_scale;  /* SLMOE_MXFP4 only: [E, 2I, d_latent/32] E8M0    */
    const uint8_t *W2_scale;   /* SLMOE_MXFP4 only: [E, d_latent, I/32]   E8M0    */
} slmoe_weights;

/* Byte offsets of the intermediates inside the workspace, so that a caller can read a
 * stage's result after slmoe_forward (or slmoe_route) without a second code path.
 * Types: scores fp32 [T,E]; topk_idx int32 [T,k]; topk_w fp32 [T,k]; counts int32 [E];
 * offsets int32 [E+1]; perm int32 [T*k]; slot_pos int32 [T*k]; x_lat act [T,d_latent];
 * h act [T*k, I] (rows in perm order); y_e act [T*k, d_latent] (rows in perm order);
 * z act [T,d_latent]; h_s act [T, n_shared*I_shared]; status int32 [4].  act is fp32 for
 * SLMOE_F32 and bf16 otherwise, except that SLMOE_MXFP4 keeps x_lat and h as MXFP8: codes
 * [rows, K] bytes followed directly by their scales [rows, K/32] (K = d_latent, I). */
typedef struct slmoe_workspace_layout {
    size_t scores, topk_idx, topk_w, counts, offsets, perm, slot_pos;
    size_t x_lat, h, y_e, z, h_s, status;
    size_t total;
} slmoe_workspace_layout;

/* Bytes of workspace a slmoe_route or slmoe_forward call with this config needs
 * (0 on an invalid config; see slmoe_last_error). */
SLMOE_API size_t slmoe_workspace_size(const slmoe_config *cfg);

/* Fill *out with the workspace layout for cfg.  Returns SLMOE_OK or SLMOE_EINVAL. */
SLMOE_API int slmoe_workspace_layout_get(const slmoe_config *cfg, slmoe_workspace_layout *out);

/* Thread-local message of the last failed call on this thread ("" if none). */
SLMOE_API const char *slmoe_last_error(void);

/* Number of streaming multiprocessors of the current device (for sizing tests). */
SLMOE_API int slmoe_device_sm_count(void);

/* Stage profiling hook (thread-local).  When events is not NULL, slmoe_forward records
 * events[i] (a cudaEvent_t created by the caller, passed as void*) right after stage i, for
 * i < n:  0 start, 1 router scores, 2 top-k + permutation (+ histogram), 3 latent
 * down-projection, 4 expert gate|up + SiTU-GLU, 5 expert down, 6 combine + RMSNorm, 7 shared
 * gate|up + SiTU-GLU, 8 up-projection + shared down.  On the bf16 type, stages 3 and 7 run
 * on the library's auxiliary stream (recorded there), started at stage 0 and concurrent
 * with stages 1-2; stage 4 starts when 2 and 7 are both done.  NULL turns it off. */
SLMOE_API int slmoe_set_stage_events(void **events, int n);

/* Number of kernels this library has launched in this process (all threads). */
SLMOE_API long long slmoe_launch_count(void);

/*
 * slmoe_route - router scores, biased top-k and the expert-sorted permutation.
 *   [K3-news] §01-§02, [K3-arch] 负载均衡优化, [SLMoE] 路由机制.
 *   s[t,e]  = sigmoid(x_t . W_r[e] + logit_offset[e])      (fp32 logits)
 *   choose the k experts with the largest s[t,e] + bias[e]; ties go to the lower index;
 *   slots are ordered by biased score descending;
 *   topk_w[t,j] = s[t, topk_idx[t,j]] / sum_j s[t, topk_idx[t,j]]   (raw scores)
 *   counts[e] = tokens that chose e; offsets = exclusive scan of counts (offsets[E] = T*k);
 *   perm lists token ids by expert ascending, then token ascending;
 *   slot_pos[t*k+j] = position of (t, topk_idx[t,j]) in perm.
 * Arguments: x [T,d] act; W_r [E,d] fp32; bias [E] fp32; logit_offset [E] fp32 or NULL;
 *   outputs topk_idx [T,k] int32, topk_w [T,k] fp32, counts [E], offsets [E+1], perm [T*k],
 *   slot_pos [T*k] (all int32, all required); scores [T,E] fp32 or NULL (when NULL the
 *   scores stay in the workspace); hist [E,nbins] uint32 or NULL: when given, the scores'
 *   QB histogram is added into it (as slmoe_qb_histogram); status as above.
 * Errors: SLMOE_EINVAL on a null required pointer or a bad config, SLMOE_ENOSPACE on a
 *   short workspace, SLMOE_ECUDA on a launch failure.
 */
SLMOE_API int slmoe_route(const slmoe_config *cfg, const void *x, const float *W_r, const float *bias,
                const float *logit_offset, int32_t *topk_idx, float *topk_w, float *scores,
                int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos,
                uint32_t *hist, int32_t *status, void *workspace, size_t workspace_bytes,
                void *stream);

/*
 * slmoe_route_noalloc - slmoe_route without a workspace argument: the same kernels, the same
 * arithmetic and the same outputs, with the call's scratch taken from a fixed device array
 * inside this library instead of from the caller.  The pages describe no such call: it is
 * a convenience of this library for callers that cannot hand out device memory per call,
 * for instance a serving loop whose allocator has already given all of the device's memory
 * to weights and caches, or a latency-critical loop that must not call cudaMalloc or
 * cudaFree (cudaFree waits for the whole device).  The call makes no allocation call of any
 * kind (no cudaMalloc, cudaMallocAsync, cudaFree, nor a library routine that allocates); the
 * array itself is device memory that the CUDA runtime reserves together with this library's
 * device code on each device where that code is loaded.
 *
 * Scratch limit: SLMOE_ROUTE_NOALLOC_SCRATCH_BYTES (48 MiB) per device.  A call needs
 *   16 * 4 bytes of tile counters + ceil(T/16) * E * 4 bytes of per-chunk expert counts
 *   + 3 * E * d * 2 bytes of split router weights (bf16 type only)
 *   + T * E * 4 bytes of scores when scores is NULL,
 * each piece rounded up to 256 bytes.  With E = 896 and d = 7168 (bf16) that is 36.8 MiB
 * plus about 0.2 KiB per token with a caller scores buffer, 3.7 KiB per token without one.
 * A call that needs more returns SLMOE_ENOSPACE before anything is launched, and
 * slmoe_last_error() gives the bytes it needed.  A bf16 batch of at most 256 tokens also
 * takes 16 * T * E * 4 bytes for the split-K router sums that slmoe_route uses at that size,
 * when they fit under the limit; when they do not, the router runs unsplit here and its fp32
 * logits may differ from slmoe_route's in the last bits (the sums are added in another order).
 *
 * Zeroing: nothing in the scratch has to be zeroed by the caller.  The tile counters, the
 * only part that must start at zero, are cleared by each call on its own stream before its
 * first kernel; everything else in the scratch is written before it is read.  hist (when
 * given) accumulates as in slmoe_route, so the caller zeroes it.
 *
 * Set-up: the first call on each device looks up the scratch's device address with that
 * device current (cudaGetSymbolAddress) and keeps it, tied to the id of the device's CUDA
 * context; later calls in that context reuse the address, and a call made after the context
 * was destroyed and made again (cudaDeviceReset) looks it up anew.  Make the first call on a
 * device before capturing any stream into a CUDA graph.
 *
 * Overlap: there is one scratch per device, shared by every call on that device.  Two calls
 * that can run at the same time on one device (different streams not ordered by events, or
 * different host threads) race on it and give wrong results; order them on one stream or
 * with events.  When scores is NULL the scores are kept only in the scratch, and the next
 * call on the device overwrites them.
 *
 * Arguments and errors: as slmoe_route, without workspace and workspace_bytes; plus
 *   SLMOE_ENOSPACE when the call needs more scratch than the limit above.
 */
#define SLMOE_ROUTE_NOALLOC_SCRATCH_BYTES (48u * 1024u * 1024u)
SLMOE_API int slmoe_route_noalloc(const slmoe_config *cfg, const void *x, const float *W_r,
                const float *bias, const float *logit_offset, int32_t *topk_idx, float *topk_w,
                float *scores, int32_t *counts, int32_t *offsets, int32_t *perm, int32_t *slot_pos,
                uint32_t *hist, int32_t *status, void *stream);

/*
 * slmoe_topk - biased top-k selection, gate weights and the expert-sorted permutation from
 * router scores that are already computed (the scores a call of slmoe_route kept, or the
 * micro-batches of a Quantile Balancing engine that re-routes with updated biases).
 *   [K3-news] §02 (selection by score plus a per-expert bias that only steers selection);
 *   [K3-arch] 负载均衡优化 (QB re-centres the biases so that routing by biased score balances
 *   the loads).  The same kernels and rules as the selection and permutation of slmoe_route:
 *   choose the k experts with the largest scores[t,e] + bias[e] (fp32 add), ties to the lower
 *   index, slots by biased score descending; topk_w = chosen raw scores renormalised;
 *   counts, offsets, perm and slot_pos as in slmoe_route.
 * Arguments: scores [T,E] fp32; bias [E] fp32; outputs as slmoe_route (all required when
 *   T > 0; counts and offsets always); status as above (status[0] counts NaN scores);
 *   workspace of at least slmoe_topk_workspace_size(T, E, k) bytes (per-chunk expert
 *   counts), 256-byte aligned.  1 <= k <= min(E, 32), E <= 4096, T * k < 2^30.
 * Errors: SLMOE_EINVAL on a null or misaligned pointer or a bad shape, SLMOE_ENOSPACE on a
 *   short workspace, SLMOE_ECUDA on a launch failure.
 */
SLMOE_API size_t slmoe_topk_workspace_size(int32_t T, int32_t E, int32_t k);
SLMOE_API int slmoe_topk(const float *scores, const float *bias, int32_t T, int32_t E, int32_t k,
                int32_t *topk_idx, float *topk_w, int32_t *counts, int32_t *offsets, int32_t *perm,
                int32_t *slot_pos, int32_t *status, void *workspace, size_t workspace_bytes,
                void *stream);

/*
 * slmoe_wait_abort_check - exercises the failure path of the tensor-core kernels: every wait
 * of theirs on an mbarrier is bounded, and when one runs out the kernel stops all of its
 * roles, lets copies and MMAs already issued finish, frees its tensor memory, sets
 * status[2] = 1 and returns, leaving the context usable.  This call launches one tile of
 * the dense GEMM kernel whose copy-issuing thread is told to issue nothing, so the
 * MMA-issuing thread's first wait can only run out, after wait_limit_ns nanoseconds (every
 * wait of this launch has that limit; the layer calls use 4 s).  Nothing is read and
 * nothing but status is written.  The pages have no counterpart: this is for failure-
 * detection tests.  status: device int32[4], zeroed by the caller; wait_limit_ns in
 * (0, 6e10].  Errors: SLMOE_EINVAL on a null or misaligned status or a limit out of range,
 * SLMOE_ECUDA on a launch failure.
 */
SLMOE_API int slmoe_wait_abort_check(int32_t *status, uint64_t wait_limit_ns, void *stream);

/*
 * slmoe_mxfp4_quantize - bf16 weights to MXFP4 ([SLMoE] 训练基础设施: MXFP4 weights; the
 *   format is the OCP Microscaling one).  W [rows, K] bf16, K a multiple of 32.  Each block of
 *   32 consecutive values of a row shares the scale 2^e with e = floor(log2 max|v|) - 2,
 *   clamped to [-127, 127] (-127 for an all-zero block), stored as the byte e + 127 in
 *   scales [rows, K/32]; each value becomes the FP4 E2M1 code (sign, 2 exponent bits with
 *   bias 1, 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) nearest to v / 2^e, ties to
 *   the even mantissa, saturating at 6, sign bit for v < 0; two codes per byte in
 *   packed [rows, K/2], the lower-indexed value in the low nibble.  W 16-byte aligned.
 *   Errors: SLMOE_EINVAL on null or misaligned pointers, rows < 0, K not a positive multiple
 *   of 32.
 */
SLMOE_API int slmoe_mxfp4_quantize(const void *W, int64_t rows, int32_t K, uint8_t *packed, uint8_t *scales,
                                   void *stream);

/*
 * slmoe_mxfp8_quantize - fp32 values to MXFP8 ([SLMoE] 训练基础设施: MXFP8 activations; the
 *   format is the OCP Microscaling one with FP8 E4M3 elements).  X [rows, K] fp32, K a
 *   multiple of 32.  Each block of 32 consecutive values of a row shares the scale 2^e with
 *   e = floor(log2 max|v|) - 8, clamped to [-127, 127] (-127 for an all-zero block), stored
 *   as the byte e + 127 in scales [rows, K/32]; each value becomes the E4M3 code (sign, 4
 *   exponent bits with bias 7, 3 mantissa bits; largest value 448) nearest to v / 2^e, ties
 *   to the even mantissa, saturating at 448, sign bit for v < 0; codes [rows, K].  This is
 *   the conversion the SLMOE_MXFP4 layer applies to x_lat and h.  X and codes 16-byte
 *   aligned.  Errors: SLMOE_EINVAL on null or misaligned pointers, rows < 0, K not a positive
 *   multiple of 32.
 */
SLMOE_API int slmoe_mxfp8_quantize(const float *X, int64_t rows, int32_t K, uint8_t *codes, uint8_t *scales,
                                   void *stream);

/*
 * slmoe_qb_histogram - add per-expert score histograms of one micro-batch.
 *   [K3-arch] 负载均衡优化: scores in [0,1] are binned, 1000 bins; histograms of
 *   micro-batches and machines add.
 *   For every t < T, e < E with scores[t*E+e] not NaN:
 *     bin = min(nbins-1, max(0, floor(fl32(scores[t*E+e] * nbins))))  (one fp32 multiply)
 *     hist[e*nbins + bin] += 1
 *   scores [T,E] fp32, row-major; hist [E,nbins] uint32, accumulated in place (the caller
 *   zeroes it before the first micro-batch).  0 <= T < 2^31 (so that no count of one call
 *   can wrap); the running totals are checked against 2^32 - 1.  No workspace.
 * Errors: SLMOE_EINVAL on null pointers, E < 1, nbins < 1 or nbins > 1024.
 */
SLMOE_API int slmoe_qb_histogram(const float *scores, int64_t T, int32_t E, int32_t nbins,
                       uint32_t *hist, int32_t *status, void *stream);

/*
 * slmoe_qb_update - read each expert's (1 - k/E) quantile from its histogram and re-centre
 * the biases.  [K3-arch] 负载均衡优化 (quantile read from the binned distribution);
 * [K3-news] §02 (thresholds placed so that each expert gets its share).  The pages do not
 * print the update; this library fixes it as:
 *   N_e = sum_b hist[e,b];  r = (1 - k/E) * N_e;  j = first bin with C_j >= r
 *   q_e = (j + (r - C_{j-1}) / hist[e,j]) / nbins      (q_e = 0 when r = 0)
 *   bias[e] = mean_e(q) - q_e                           (overwrites bias)
 *   The rank search is exact integer arithmetic (ceil(r) = N_e - floor(N_e k / E)); q_e is
 *   interpolated in fp32 (absolute error below 3e-7) and the mean is an exact fixed-point sum
 *   (q_e * 2^31 rounded, added in int64), so the result does not depend on summation order;
 *   stored in fp32.  hist [E,nbins] uint32; q_out [E] fp32 or NULL;
 *   bias [E] fp32.  E <= 8192, nbins <= 1024.  One thread-block cluster; no workspace.
 */
SLMOE_API int slmoe_qb_update(const uint32_t *hist, int32_t E, int32_t nbins, int32_t k,
                    float *q_out, float *bias, void *stream);

/*
 * slmoe_signsgd_update - the fixed-step bias update that QB replaces, kept as the
 * comparison engine for it.  [K3-news] §02 (K2 balances without an auxiliary loss by moving
 * each expert's selection bias, SignSGD-like, a fixed step up or down); [K3-arch]
 * 负载均衡优化 (the SignSGD-style rule of K2, unstable at K3's expert count).  The pages
 * print no formula; this library fixes it as:
 *   N = sum_e counts[e];   bias[e] += step * sign(N - E * counts[e])
 *   i.e. an expert loaded below the mean load N / E is raised by step, one above it is
 *   lowered by step, one exactly at the mean is left as it is.  The sign is exact (int64);
 *   the update is one fp32 add (round to nearest) per expert.
 *   counts [E] int32: tokens routed to each expert since the last update (the counts of
 *   slmoe_route, summed over micro-batches by the caller if wanted); bias [E] fp32, updated in
 *   place; step > 0 and finite (the pages give no value).  E <= 65536.  One thread block; no
 *   workspace.
 * Errors: SLMOE_EINVAL on null or misaligned pointers, E outside [1, 65536], a step that is
 *   not finite and positive.
 */
SLMOE_API int slmoe_signsgd_update(const int32_t *counts, int32_t E, float step, float *bias, void *stream);

/*
 * slmoe_forward - one Stable LatentMoE layer (the FFN branch; the residual add is left to
 * the caller).  [K3-news] §01-§02, [K3-arch] SiTU激活优化 / 归一化策略调整,
 * [SLMoE] Latent-Space MoE.
 *   route as slmoe_route;  x_lat = x . W_in^T;
 *   for each chosen (t, e):  [g | u] = x_lat_t . W13[e]^T,
 *       h = beta1 tanh(g/beta1) sigmoid(g) * beta2 tanh(u/beta2),   y_e = h . W2[e]^T;
 *   c_t = sum_j topk_w[t,j] y_e(t,j)  (fp32, slot order);
 *   z_t = gamma * c_t / sqrt(mean(c_t^2) + eps);
 *   y_t = z_t . W_out^T + sum_s W2_s[s] . SiTU-GLU(W13_s[s] . x_t)
 * Arguments: x [T,d] act; w as slmoe_weights; bias [E] fp32; logit_offset [E] or NULL;
 *   y [T,d] fp32 for both layer types (written, not accumulated; the branch output is kept
 *   in fp32 because bf16 storage of a heavy-tailed output alone costs up to ~2% of its RMS); topk_idx_out [T,k] int32 or NULL: when given,
 *   the routing is exported there; hist [E,nbins] or NULL: QB histogram of the scores is
 *   added; status as above; workspace as slmoe_workspace_size().  The intermediates stay
 *   readable in the workspace (slmoe_workspace_layout_get).
 * Errors: as slmoe_route.
 */
SLMOE_API int slmoe_forward(const slmoe_config *cfg, const void *x, const slmoe_weights *w,
                  const float *bias, const float *logit_offset, void *y,
                  int32_t *topk_idx_out, uint32_t *hist, int32_t *status,
                  void *workspace, size_t workspace_bytes, void *stream);

/* Weight gradients of one layer, all fp32 and laid out as the weights (slmoe_weights). */
typedef struct slmoe_grads {
    float *dW_r;         /* [E, d]                   */
    float *dW_in;        /* [d_latent, d]            */
    float *dW13;         /* [E, 2I, d_latent]        */
    float *dW2;          /* [E, d_latent, I]         */
    float *dgamma;       /* [d_latent]               */
    float *dW_out;       /* [d, d_latent]            */
    float *dW13_s;       /* [n_shared, 2I_shared, d] */
    float *dW2_s;        /* [n_shared, d, I_shared]  */
} slmoe_grads;

/* Bytes of workspace a slmoe_backward call with this config needs (0 on an invalid config
 * or the fp32 layer type). */
SLMOE_API size_t slmoe_backward_workspace_size(const slmoe_config *cfg);

/* Byte offsets of the backward's intermediates inside its workspace (readable after the call):
 * dz fp32 [T,d_latent]; dy_e bf16 [T*k, d_latent] and dgu bf16 [T*k, 2I] (rows in the forward's
 * expert order); dg fp32 [T,k] (gate-weight gradients); gu fp32 [T*k, 2I] (recomputed
 * pre-activations of the routed experts); dx_lat bf16 [T,d_latent]; gu_s fp32 and dgu_s bf16
 * [T, 2I_shared] of the last shared expert.  Returns SLMOE_OK or an error code. */
typedef struct slmoe_backward_layout {
    size_t dz, dye, dg, gu, dgu, dx_lat, gu_s, dgu_s, total;
} slmoe_backward_layout;
SLMOE_API int slmoe_backward_layout_get(const slmoe_config *cfg, slmoe_backward_layout *out);

/*
 * slmoe_backward - gradients of one Stable LatentMoE layer call, for training it
 *   ([K3-arch] SiTU激活优化 / 归一化策略调整 / 负载均衡优化; [SLMoE] 训练基础设施: the pages
 *   train this layer, with histograms added across gradient-accumulation steps).
 *   Given dy = dL/dy for the layer output y of a slmoe_forward call, this computes the chain
 *   rule of that forward step by step:
 *     dW_out (+)= dy^T z;  dz = dy W_out;  RMSNorm:  dc = gamma dz / r - c (sum gamma dz c) / (n r^3),
 *       dgamma (+)= sum_t dz c / r  (c recomputed from y_e and the gate weights, r = sqrt(mean c^2 + eps));
 *     combine: dy_e(t,j) = g[t,j] dc_t,  dg[t,j] = dc_t . y_e(t,j);
 *     routed expert e:  dW2[e] (+)= dy_e^T h;  dh = dy_e W2[e];
 *       [dg | du] = [dh softcap(u) SiTU'(g) | dh SiTU(g) softcap'(u)]  ([g | u] recomputed);
 *       dW13[e] (+)= [dg | du]^T x_lat;  dx_lat += [dg | du] W13[e]  (summed over the k slots);
 *     dW_in (+)= dx_lat^T x;  dx = dx_lat W_in + (router) + (shared experts);
 *     router: ds_j = (dg_j - sum_i g_i dg_i) / sum_i s_i over the chosen experts,
 *       dlogit = ds s (1 - s) on the chosen experts (0 elsewhere), dW_r (+)= dlogit^T x,
 *       dx += dlogit W_r;  the selection itself and the bias pass no gradient;
 *     shared expert s: dW2_s (+)= dy^T h_s, [dg | du] as above from x W13_s^T (recomputed),
 *       dW13_s (+)= [dg | du]^T x, dx += [dg | du] W13_s.
 * Arguments: cfg, x, w as the forward call (bf16 layer type only); dy [T,d] fp32; dx [T,d]
 *   fp32 (written); grads: every pointer required, fp32, written (accumulate = 0) or added
 *   into (accumulate = 1, for gradient accumulation across micro-batches); fwd_workspace: the
 *   workspace of the slmoe_forward call on the same x, weights, bias and logit offset, not
 *   modified since (its routing, x_lat, h, y_e, z and h_s are read, nothing is written);
 *   status as above; workspace of slmoe_backward_workspace_size(cfg) bytes.
 *   Contractions run on the tensor cores (bf16 operands, fp32 accumulation); dz, dx and the
 *   weight gradients are fp32; the intermediates dy_e, [dg | du] and dx_lat are bf16.
 * Errors: SLMOE_EINVAL on a null or misaligned pointer or a bad config, SLMOE_EUNSUPPORTED for
 *   the fp32 layer type, SLMOE_ENOSPACE on a short workspace, SLMOE_ECUDA on a launch failure.
 */
SLMOE_API int slmoe_backward(const slmoe_config *cfg, const void *x, const slmoe_weights *w,
                   const float *dy, float *dx, const slmoe_grads *grads, int accumulate,
                   const void *fwd_workspace, size_t fwd_workspace_bytes, int32_t *status,
                   void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* SLMOE_H */
