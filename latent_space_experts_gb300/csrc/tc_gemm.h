// Tensor-core (tcgen05 / TMEM / TMA) path of the bf16 layer type.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"

namespace slmoe {

struct TcForward {
    void *x_lat, *h, *y_e, *z, *h_s;   // workspace buffers (bf16)
    const float *topk_w;
    const int32_t *counts, *offsets, *perm, *slot_pos;
    int32_t *status;
    int *counters;    // zeroed: tile counters [1] down, [2..4] shared, [5] up; item counters
                      // [6] expert gate|up, [7] expert down; item counts [8], [9]
    int4 *items1, *items2;              // work lists of the two routed-expert GEMMs
};

// Router scores s = sigmoid(x W_r^T + mu) with fp32-faithful logits: W_r is split into three
// bf16 pieces (hi + mid + lo == W_r exactly) whose products with the bf16 x are exact in
// fp32, accumulated on the tensor cores.  wsplit: workspace [3, E, d] bf16.
// counter: nullable zeroed tile counter for dynamic scheduling.  partial: nullable workspace
// for split-K logit sums of a small batch ([ROUTER_SPLITK_MAX, T, E] fp32).
int tc_router_scores(const slmoe_config *c, const void *x, const float *W_r, const float *mu,
                     __nv_bfloat16 *wsplit, float *scores, int32_t *status, int *counter, float *partial,
                     cudaStream_t st);

// The parts of the layer that need only x: latent down-projection and the shared experts'
// gate|up + SiTU-GLU (run concurrently with routing).
int tc_forward_front(const slmoe_config *c, const void *x, const slmoe_weights *w,
                     const TcForward &f, cudaStream_t st);

// The work lists of the two routed-expert GEMMs, built on the device from the expert counts
// and offsets of routing (launched on the routing stream, before it joins the front part).
int tc_worklists(const slmoe_config *c, const TcForward &f, cudaStream_t st);

// Everything after routing and the front part: the two grouped expert GEMMs, combine +
// RMSNorm, and the up-projection with the shared experts' down-projection.
int tc_forward_back(const slmoe_config *c, const slmoe_weights *w, const TcForward &f, void *y,
                    cudaStream_t st);

// ---------------------------------------------------------------- backward contractions
// A stored row-major matrix: p, its rows, columns and pitch (elements).  The dense GEMM reads A
// as [M rows, K cols] (K-major) or [K rows, M cols] (MN-major, maj & 1), B as [N rows, K cols]
// or [K rows, N cols] (maj & 2).
struct TcOperand {
    const void *p;
    long long pitch;
};
// SiTU-GLU derivative epilogue: the accumulator is dh [rows, F]; gu holds the fp32 gate and up
// pre-activations [rows, 2F]; [dg | du] goes to dgu (bf16, [rows, 2F]).
struct TcDglu {
    const float *gu;
    long long ld_gu;
    int F;
    __nv_bfloat16 *dgu;
    long long ld_dgu;
    float beta1, beta2;
};
// C[M, N] = (or +=) A . B^T in fp32 (dg == NULL), or the SiTU-GLU derivative of it.
int tc_dense_gemm(int maj, int M, int N, int K, TcOperand A, TcOperand B, void *C, long long ldc, int accumulate,
                  const TcDglu *dg, int32_t *status, int *counter, cudaStream_t st);
enum { TC_BWD_GU32 = 0, TC_BWD_DGLU = 1, TC_BWD_DXE = 2 };
// Grouped backward contractions on the routed experts' work lists (items of 192-token passes):
//   TC_BWD_GU32: gu[row] = W13[e] rows[index[row]] (fp32 gate|up pre-activations; the forward's
//                gate|up list, 128-feature blocks);
//   TC_BWD_DGLU: [dg | du][row] from dh = W2[e]^T rows[row] and gu (list of 128-feature blocks of I);
//   TC_BWD_DXE:  out[row] = W13[e]^T rows[row] (fp32; list of 256-feature blocks of d_latent).
int tc_grouped_bwd(int kind, const slmoe_config *c, const void *W, const void *rows, const int32_t *row_index,
                   const int4 *items, const int *n_items, int *counter, void *out, const float *gu,
                   __nv_bfloat16 *dgu, int32_t *status, cudaStream_t st);
// One work list of nfb feature blocks (192-token passes) from the expert counts and offsets.
int tc_worklist_single(const int32_t *counts, const int32_t *offsets, int E, int nfb, int4 *items, int *n_items,
                       int max_items, cudaStream_t st);

// Failure-path check: one launch of a tensor-core kernel whose bounded waits must run out
// (see slmoe_wait_abort_check).
int tc_wait_abort_check(int32_t *status, unsigned long long wait_limit_ns, cudaStream_t st);

}  // namespace slmoe
