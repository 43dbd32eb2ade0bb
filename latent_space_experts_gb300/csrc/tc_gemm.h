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

// Failure-path check: one launch of a tensor-core kernel whose bounded waits must run out
// (see slmoe_wait_abort_check).
int tc_wait_abort_check(int32_t *status, unsigned long long wait_limit_ns, cudaStream_t st);

}  // namespace slmoe
