"""GPU parity of the MXFP4 path: the quantiser bit-exact against the oracle's, and the
SLMOE_MXFP4 layer against the oracle's forward on the dequantised weights.

The routed experts' weights are quantised once (slmoe_mxfp4_quantize); the oracle takes the
GPU's codes and scales, dequantises them exactly (every MXFP4 value is a small integer times
a power of two) and runs its fp64 forward with the GPU's routing.  The layer's routed experts
compute in f16 on the GPU, which the oracle does not emulate: y is held to the bf16 bound,
max|err| <= 2e-2 RMS(ref).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import latent_space_experts_gb300 as lse
from gpu_util import BF16_TOL, assert_close_rms, need_gpu, to_dev

pytestmark = pytest.mark.gpu


def gpu_quantize(W):
    """packed, scales of a bf16 CUDA tensor [..., K] through slmoe_mxfp4_quantize."""
    K = W.shape[-1]
    rows = W.numel() // K
    packed = torch.empty(W.shape[:-1] + (K // 2,), dtype=torch.uint8, device="cuda")
    scales = torch.empty(W.shape[:-1] + (K // 32,), dtype=torch.uint8, device="cuda")
    lse.slmoe_mxfp4_quantize(W, rows, K, packed, scales)
    return packed, scales


def test_quantiser_matches_the_oracle_bit_for_bit():
    need_gpu()
    g = torch.Generator().manual_seed(0)
    rows, K = 300, 256
    w = torch.randn(rows, K, generator=g) * torch.exp(2 * torch.randn(rows, 1, generator=g))
    w[0] = 0.0                                                   # an all-zero row
    w[1, :32] = 0.0                                              # an all-zero block
    grid = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    mids = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0])
    w[2, :8], w[2, 8:16], w[2, 16] = grid, -mids, 4.0            # exact grid values and ties
    w[3, :32] = 1e-39                                            # subnormal block (bf16 keeps it)
    w[4, :32] = 3.0e38                                           # near the top of the range
    wb = w.to(torch.bfloat16)
    p, s = gpu_quantize(wb.cuda())
    p_ref, s_ref = oracle.mxfp4_quantize(wb.double().numpy())
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(p.cpu().numpy(), p_ref)


class LazyDequant:
    """Expert e's dequantised matrix on access (the oracle reads W13[e] / W2[e] only)."""

    def __init__(self, packed, scales):
        self.packed, self.scales = packed, scales
        self.shape = tuple(packed.shape[:-1]) + (2 * packed.shape[-1],)

    def __getitem__(self, e):
        return oracle.mxfp4_dequantize(self.packed[e].cpu().numpy(), self.scales[e].cpu().numpy())


def mxfp4_layer(inp):
    """The layer inputs with W13 / W2 quantised on the GPU; and the oracle's view of them."""
    q = dict(inp)
    q["W13"], q["W13_scale"] = gpu_quantize(inp["W13"])
    q["W2"], q["W2_scale"] = gpu_quantize(inp["W2"])
    ref = dict(inp)
    ref["W13"] = LazyDequant(q["W13"], q["W13_scale"])
    ref["W2"] = LazyDequant(q["W2"], q["W2_scale"])
    return q, ref


def run_mxfp4(shape, q):
    cfg = lse.config(shape, dtype=lse.MXFP4)
    ws = torch.zeros(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty(shape.T, shape.d, dtype=torch.float32, device="cuda")
    topk = torch.empty(shape.T, shape.k, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    lse.slmoe_forward(cfg, q["x"], lse.weights(q), q["bias"], q.get("logit_offset"), y, topk, None, status, ws)
    torch.cuda.synchronize()
    assert status.cpu().tolist()[1:3] == [0, 0], status
    return y, topk.cpu().numpy()


@pytest.mark.parametrize("over", [dict(T=300, d=512), dict(T=129, E=40, k=3, I=128, d=512),
                                  dict(T=600, E=2, k=1, I=384, d_latent=320, d=512), dict(T=1, d=512)])
def test_mxfp4_layer_matches_the_oracle(over):
    need_gpu()
    shp = synthetic.shape_with("mid", **over)
    inp = to_dev(synthetic.layer_inputs(shp, seed=12))
    q, ref_inp = mxfp4_layer(inp)
    y, topk = run_mxfp4(shp, q)
    ref = oracle.forward(ref_inp, shp.k, forced_topk_idx=topk)
    r = assert_close_rms(y, ref["y"], BF16_TOL, f"mxfp4 {over} y")
    print(f"mxfp4 {over}: max|err|/RMS {r:.2e}")


def test_mxfp4_k3_decode_and_prefill_sampled():
    """K3 widths: the decode batch on every token, the prefill batch on sampled tokens; the
    quantiser bit-exact on the routed experts those tokens reach."""
    need_gpu()
    shp = synthetic.LAYERS["k3_prefill"]
    inp = synthetic.layer_inputs(shp, seed=0, device="cuda")
    q, ref_inp = mxfp4_layer(inp)
    del inp["W13"], inp["W2"]
    torch.cuda.empty_cache()
    for T, n_tok in ((128, None), (8192, 24)):
        s = synthetic.shape_with("k3_prefill", T=T)
        qs = dict(q)
        qs["x"] = q["x"][:T].contiguous()
        y, topk = run_mxfp4(s, qs)
        tok = np.arange(T) if n_tok is None else np.unique(
            np.concatenate([[0, T - 1], np.random.default_rng(3).choice(T, n_tok, replace=False)]))
        rs = dict(ref_inp)
        rs["x"] = qs["x"]
        ref = oracle.forward(rs, s.k, forced_topk_idx=topk, tokens=tok)
        r = assert_close_rms(y[torch.as_tensor(tok, device="cuda")], ref["y"], BF16_TOL, f"mxfp4 K3 T={T} y")
        print(f"mxfp4 K3 T={T}: max|err|/RMS {r:.2e} on {len(tok)} tokens")
    W13 = synthetic.layer_inputs(synthetic.shape_with("k3_prefill", T=1, E=4), seed=0, device="cuda")["W13"]
    p, sc = gpu_quantize(W13)
    p_ref, s_ref = oracle.mxfp4_quantize(W13.double().cpu().numpy())
    assert np.array_equal(sc.cpu().numpy(), s_ref) and np.array_equal(p.cpu().numpy(), p_ref)
