// Internal launcher interface shared by the library's translation units (host side).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "slmoe.h"

namespace slmoe {

// Sets the thread-local error message and returns code.
int fail(int code, const char *fmt, ...);
// Maps a pending CUDA error (cudaGetLastError) to SLMOE_ECUDA with a message.
int check_launch(const char *what);

int sm_count();
// Records the caller's stage event i on st when stage events are set (profiling hook).
void stage_event(int i, cudaStream_t st);

// ---------------------------------------------------------------- full workspace layout
struct Layout {
    slmoe_workspace_layout pub;
    size_t chunk_counts;   // int32 [nchunks, E]: per-chunk expert counts, then bases
    size_t wr_split;       // bf16 [3, E, d]: router weight split hi / mid / lo
    size_t counters;       // int32 [16]: tile counters of the dynamically scheduled kernels
    size_t items1, items2; // int4 work lists of the routed-expert GEMMs (bf16 type)
    size_t rt_split;       // fp32 split-K logit sums of the router (bf16 type, small batches)
    size_t nchunks;
};
int make_layout(const slmoe_config *cfg, Layout *L);
int validate_config(const slmoe_config *cfg);

// ---------------------------------------------------------------- SIMT GEMM (CUDA cores)
// C[r, n] = epilogue( sum_s sum_k A_s[arow(r), k] * B_s[brow(n), k] ),  fp32 accumulate.
enum SimtEpi { SIMT_STORE = 0, SIMT_GLU = 1, SIMT_SIGMOID = 2 };
enum DType { DT_F32 = 0, DT_BF16 = 1 };

struct SimtSeg {
    const void *A;           // [rows, lda]
    const void *B;           // [N (or 2N for GLU), ldb] per group
    int64_t lda, ldb;
    int K;
    int64_t b_group_stride;  // elements between groups' B matrices
};

struct SimtGemm {
    SimtSeg seg[4];
    int nseg;
    const int32_t *a_index;        // nullable: A row of output row r is a_index[r]
    const int32_t *group_offsets;  // nullable: rows of group g are [off[g], off[g+1])
    int groups;                    // grid z (1 when not grouped)
    int M;                         // rows when not grouped; max rows per group when grouped
    int N;                         // output columns
    int glu_up_row;                // GLU: B row of the up half of column n is n + glu_up_row
    void *C;
    int64_t ldc;
    const float *mu;               // SIGMOID: logit offset per column (nullable)
    float beta1, beta2;
    int epi;
    int a_type, b_type, c_type;    // DType
};
int launch_simt_gemm(const SimtGemm &g, cudaStream_t st);

// ---------------------------------------------------------------- routing
int launch_topk(const float *scores, const float *bias, int T, int E, int k, int32_t *topk_idx,
                float *topk_w, int32_t *chunk_counts, int32_t *status, cudaStream_t st);
int launch_scan(int32_t *chunk_counts, int nchunks, int E, int32_t *counts, cudaStream_t st);
int launch_scatter(const int32_t *topk_idx, const int32_t *chunk_base, const int32_t *counts, int T,
                   int E, int k, int32_t *offsets, int32_t *perm, int32_t *slot_pos, cudaStream_t st);
constexpr int ROUTE_CHUNK = 16;  // tokens per top-k block / permutation chunk
// Tokens per pass of the routed-expert GEMMs: an expert with n tokens makes ceil(n / pass)
// work items per feature block, which also sizes the work lists in the workspace.
constexpr int GROUPED_PASS = 192;
// The MXFP4 layer's routed-expert GEMMs take short passes when the batch gives an expert few
// tokens on average (decode): their small token stages leave shared memory for more weight
// stages in flight.
constexpr int MX_SHORT_PASS = 32, MX_LONG_PASS = 192;
// The bf16 layer's expert down-projection takes one 128-row weight sub-tile per work item, in
// one of two accumulator sets, when the experts get many tokens (prefill); with at most 8
// tokens per expert on average (decode) the per-item cost dominates and items of two
// sub-tiles in one set are faster (0.60 against 0.455 ms at K3 decode).  The MXFP4
// layer always takes two.  down_block: output features per item.
constexpr int DOWN_NSUB = 1;
inline bool down_split(const slmoe_config *c) {
    return c->dtype != SLMOE_MXFP4 && (long long)c->T * c->k > 8LL * c->E;
}
inline int down_block(const slmoe_config *c) { return down_split(c) ? 128 * DOWN_NSUB : 256; }
inline int grouped_pass(const slmoe_config *c) {
    if (c->dtype != SLMOE_MXFP4) return GROUPED_PASS;
    return (long long)c->T * c->k <= 8LL * c->E ? MX_SHORT_PASS : MX_LONG_PASS;
}
// The router of a batch of at most ROUTER_SPLITK_MAX_M tokens splits its K blocks over up to
// ROUTER_SPLITK_MAX CTAs per tile (their fp32 partial logits live in the workspace).
constexpr int ROUTER_SPLITK_MAX_M = 256;
constexpr int ROUTER_SPLITK_MAX = 16;

// ---------------------------------------------------------------- QB
int launch_qb_histogram(const float *scores, int64_t T, int E, int nbins, uint32_t *hist,
                        int32_t *status, cudaStream_t st);
int launch_qb_update(const uint32_t *hist, int E, int nbins, int k, float *q_out, float *bias,
                     cudaStream_t st);
int launch_signsgd_update(const int32_t *counts, int E, float step, float *bias, cudaStream_t st);

// ---------------------------------------------------------------- combine + RMSNorm
int launch_combine_rmsnorm(int dtype, const void *y_e, const float *topk_w,
                           const int32_t *slot_pos, const float *gamma, int T, int d_latent,
                           int k, float eps, void *z, cudaStream_t st);

// ---------------------------------------------------------------- MXFP4 weights
int launch_mxfp4_quantize(const void *W, long long rows, int K, uint8_t *packed, uint8_t *scales, cudaStream_t st);
int launch_mxfp8_quantize(const float *X, long long rows, int K, uint8_t *codes, uint8_t *scales, cudaStream_t st);

// ---------------------------------------------------------------- backward (bf16 type)
// Intermediates of a forward call that the backward reads (views into its workspace).
struct FwdSaved {
    const float *scores, *topk_w;
    const int32_t *topk_idx, *counts, *offsets, *perm, *slot_pos;
    const __nv_bfloat16 *x_lat, *h, *y_e, *z, *h_s;
    const int4 *items1;            // the forward's gate|up work list and its count
    const int *n_items;
};
struct BwdLayout {
    size_t dy_b, dz, dye, dg, gu, dgu, dxe, dx_lat, gu_s, dgu_s, dl_perm, dgamma_part, counters;
    size_t nblk, total;
    size_t items_dglu, cap_dglu;   // 128-feature blocks of I
    size_t items_dxe, cap_dxe;     // 256-feature blocks of d_latent
};
size_t backward_workspace_bytes(const slmoe_config *c, BwdLayout *L);
int tc_backward(const slmoe_config *c, const void *x, const slmoe_weights *w, const float *dy, float *dx,
                const slmoe_grads *g, int accumulate, const FwdSaved &fs, char *ws, int32_t *status,
                cudaStream_t st);

}  // namespace slmoe
