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
};

// Router scores s = sigmoid(x W_r^T + mu) with fp32-faithful logits: W_r is split into three
// bf16 pieces (hi + mid + lo == W_r exactly) whose products with the bf16 x are exact in
// fp32, accumulated on the tensor cores.  wsplit: workspace [3, E, d] bf16.
int tc_router_scores(const slmoe_config *c, const void *x, const float *W_r, const float *mu,
                     __nv_bfloat16 *wsplit, float *scores, int32_t *status, cudaStream_t st);

// Everything after routing: down-projection, the two grouped expert GEMMs, combine +
// RMSNorm, shared experts and the up-projection.
int tc_forward_bf16(const slmoe_config *c, const void *x, const slmoe_weights *w,
                    const TcForward &f, void *y, cudaStream_t st);

}  // namespace slmoe
