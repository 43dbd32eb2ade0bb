"""GPU parity of the MXFP4 layer (MXFP4 weights, MXFP8 activations, block-scaled tensor cores).

The quantisers are bit-exact against the oracle's: slmoe_mxfp4_quantize (weights) and
slmoe_mxfp8_quantize (the conversion the layer's epilogues apply to x_lat and h).  The layer's
routed experts are checked stage by stage from the GPU's own inputs of each stage: x_lat's
MXFP8 codes against the oracle's conversion of x . W_in^T, h's codes against the oracle's
conversion of SiTU-GLU(W13[e] . x_lat) on the GPU's dequantised x_lat rows, y_e against W2[e]
applied to the GPU's dequantised h rows; and y end to end against the oracle's forward with
MXFP8 activations on the GPU's routing and the GPU's MXFP8 rounding decisions (``forced_mx``,
as the selection is forced: the stage checks show that each decision is a valid rounding).
Left to its own decisions the oracle rounds a few values near midpoints the other way, and at
K3 width one flipped x_lat value moves every h of that token by about 1e-3 relative, which
flips about 2 % of them in turn: y then differs by several per cent at single elements, the
quantisation noise of the format rather than an arithmetic error.

An MXFP8 code is an integer decided in floating point: the GPU converts its fp32 value, the
oracle its fp64 value, so the two may round differently where the value sits within the GPU's
own error of a rounding midpoint (or a block maximum within it of a power of two).  The stage
checks therefore bound the fraction of codes and of block scales that differ, and ask that
every GPU value in a block whose scale agrees is a correct rounding of a value within the
GPU's arithmetic error of the oracle's: |gpu - ref| <= half a grid step + rel |ref| + 1e-2 X
(X the block scale).  1e-2 X covers the tensor cores' fp32 accumulation: K / 16 steps (448 at
K3 width) that each round at about 2^-23 of a running sum up to the block maximum (256 X to
512 X) give about sqrt(448) 2^-23 512 X = 1.3e-3 X per standard deviation.  x_lat is a plain fp32
dot product: rel = 0, at most 1e-3 of the codes may differ.  h goes through three tanh.approx
evaluations (relative error up to about 2^-11 each): rel = 2e-3, and a 2e-3 relative error moves
a value across a midpoint of the E4M3 grid (steps of 6-12 %) for about 2 % of the codes, so at
most 3e-2 may differ.  y is held to the bf16 bound max|err| <= 2e-2 RMS(ref).
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import latent_space_experts_gb300 as lse
from gpu_util import BF16_STORE, BF16_TOL, assert_close_rms, need_gpu, to_dev

pytestmark = pytest.mark.gpu

MX_ABS = 1e-2           # fp32 accumulation error allowed, in units of the block scale X


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


def test_mxfp8_quantiser_matches_the_oracle_bit_for_bit():
    """Random values over a wide exponent range, every E4M3 value and every midpoint at a
    scale of 1, saturation, the subnormal grid, fp32 subnormals, zero blocks and -0."""
    need_gpu()
    rng = np.random.default_rng(1)
    rows, K = 512, 256
    x = (rng.normal(size=(rows, K)) * np.exp(4 * rng.normal(size=(rows, 1)))).astype(np.float32)
    vals = np.unique(np.abs(oracle.e4m3_decode(np.arange(127))))           # the 127 finite magnitudes
    x[0, :127], x[0, 127] = vals, 448.0                                    # every value, block max 448
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)
    x[1, :126], x[1, 126:] = mids, 300.0                                   # every midpoint: ties to even
    x[2, :128] = -mids[:128] if len(mids) >= 128 else np.resize(-mids, 128)
    x[3, :32] = np.linspace(449, 511, 32).astype(np.float32)               # past 448 after scaling
    x[3, 0] = 300.0
    x[4, :32] = np.float32(2.0 ** -130)                                    # fp32 subnormals
    x[4, 32:64] = 0.0
    x[5, 0], x[5, 1:32] = 256.0, np.linspace(0.0, 2.0 ** -5, 31)           # scale 1: the subnormal grid
    x[5, 32:64] = -1e-30
    x[5, 32] = 1.0                                                         # tiny negatives -> -0
    x[6, :32] = np.float32(3.0e38)
    X = torch.from_numpy(x).cuda()
    codes = torch.empty(rows, K, dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows, K // 32, dtype=torch.uint8, device="cuda")
    lse.slmoe_mxfp8_quantize(X, rows, K, codes, scales)
    c_ref, s_ref = oracle.mxfp8_quantize(x.astype(np.float64))
    assert np.array_equal(scales.cpu().numpy(), s_ref)
    c = codes.cpu().numpy()
    bad = np.argwhere(c != c_ref)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0]}: {c[tuple(bad[0])]:#x} vs {c_ref[tuple(bad[0])]:#x}"


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
    return y, topk.cpu().numpy(), lse.workspace_views(cfg, ws)


def check_mx8(codes, scales, ref, what, rel=0.0, mismatch=1e-3):
    """GPU MXFP8 codes / scales [rows, K] against the oracle's conversion of ref (fp64)."""
    c = codes.cpu().numpy()
    s = scales.cpu().numpy()
    c_ref, s_ref = oracle.mxfp8_quantize(ref)
    n_code, n_scale = int((c != c_ref).sum()), int((s != s_ref).sum())
    assert n_code <= mismatch * c.size and n_scale <= mismatch * s.size, (what, n_code, n_scale)
    got = oracle.mxfp8_dequantize(c, s)
    same = np.repeat(s == s_ref, 32, axis=-1)
    X = np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=-1)
    a = np.abs(ref) / X
    step = np.ldexp(1.0, (np.maximum(np.floor(np.log2(np.maximum(a, 2.0 ** -40))), -6) - 3).astype(np.int64)) * X
    sat = a > 448.0
    bound = np.where(sat, np.abs(ref) - 448.0 * X, 0.5 * step) + rel * np.abs(ref) + MX_ABS * X
    err = np.abs(got - ref)
    ok = (err <= bound) | ~same
    worst = np.unravel_index(int(np.argmax(np.where(same, err - bound, -np.inf))), err.shape)
    assert ok.all(), (what, worst, got[worst], ref[worst])
    print(f"{what}: {n_code} of {c.size} codes and {n_scale} of {s.size} scales differ from the oracle")
    return got


class LazyMx8:
    """Rows of an MXFP8 tensor (codes, scales on the device), dequantised on access."""

    def __init__(self, codes, scales):
        self.codes, self.scales = codes, scales

    def __getitem__(self, idx):
        i = torch.as_tensor(np.asarray(idx), device=self.codes.device)
        return oracle.mxfp8_dequantize(self.codes[i].cpu().numpy(), self.scales[i].cpu().numpy())


def forced_mx(views):
    return dict(x_lat=LazyMx8(views["x_lat"], views["x_lat_scales"]), h=LazyMx8(views["h"], views["h_scales"]),
                slot_pos=views["slot_pos"].cpu().numpy())


def check_stages(shp, ref_inp, views, topk, rows_per_expert=None):
    """x_lat, h and y_e of the GPU, each from the GPU's own previous stage (dequantised)."""
    x = ref_inp["x"].double().cpu().numpy()
    W_in = ref_inp["W_in"].double().cpu().numpy()
    xl = check_mx8(views["x_lat"], views["x_lat_scales"], x @ W_in.T, "x_lat")
    perm = views["perm"].cpu().numpy()
    offsets = views["offsets"].cpu().numpy()
    h_codes, h_scales = views["h"].cpu(), views["h_scales"].cpu()
    for e in np.nonzero(np.diff(offsets))[0][:12]:
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        rows = np.arange(lo, hi) if rows_per_expert is None else np.arange(lo, min(hi, lo + rows_per_expert))
        h_ref = oracle.expert_hidden(ref_inp, e, xl[perm[rows]])
        h = check_mx8(h_codes[rows], h_scales[rows], h_ref, f"h of expert {e}", rel=2e-3, mismatch=3e-2)
        y_ref = oracle.expert_output(ref_inp, e, h)
        assert_close_rms(views["y_e"][torch.as_tensor(rows, device="cuda")], y_ref, BF16_TOL, f"y_e of expert {e}",
                         BF16_STORE)


@pytest.mark.parametrize("over", [dict(T=300, d=512), dict(T=129, E=40, k=3, I=128, d=512),
                                  dict(T=600, E=2, k=1, I=384, d_latent=384, d=512), dict(T=1, d=512),
                                  dict(T=512, E=128, k=2, d=512, hot=True)])
def test_mxfp4_layer_matches_the_oracle(over):
    """Long (192-token) passes, and short (32-token) passes when the batch gives an expert at
    most 8 tokens on average (T = 1; the hot case, where every token also picks expert 5,
    so that it takes 16 short passes)."""
    need_gpu()
    over = dict(over)
    hot = over.pop("hot", False)
    shp = synthetic.shape_with("mid", **over)
    inp = to_dev(synthetic.layer_inputs(shp, seed=12))
    if hot:
        inp["bias"][5] += 10.0
    q, ref_inp = mxfp4_layer(inp)
    y, topk, views = run_mxfp4(shp, q)
    check_stages(shp, ref_inp, views, topk)
    ref = oracle.forward(ref_inp, shp.k, forced_topk_idx=topk, forced_mx=forced_mx(views))
    r = assert_close_rms(y, ref["y"], BF16_TOL, f"mxfp4 {over} y")
    print(f"mxfp4 {over}: max|err|/RMS {r:.2e}")


def test_mxfp4_k3_decode_and_prefill_sampled():
    """K3 widths: the decode batch on every token, the prefill batch on sampled tokens; the
    routed-expert stages on the first rows of 12 experts; the quantiser bit-exact on the
    routed experts those tokens reach."""
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
        y, topk, views = run_mxfp4(s, qs)
        rs = dict(ref_inp)
        rs["x"] = qs["x"]
        tok = np.arange(T) if n_tok is None else np.unique(
            np.concatenate([[0, T - 1], np.random.default_rng(3).choice(T, n_tok, replace=False)]))
        if n_tok is None:
            check_stages(s, rs, views, topk, rows_per_expert=64)
        ref = oracle.forward(rs, s.k, forced_topk_idx=topk, tokens=tok, forced_mx=forced_mx(views))
        r = assert_close_rms(y[torch.as_tensor(tok, device="cuda")], ref["y"], BF16_TOL, f"mxfp4 K3 T={T} y")
        print(f"mxfp4 K3 T={T}: max|err|/RMS {r:.2e} on {len(tok)} tokens")
        del views
    W13 = synthetic.layer_inputs(synthetic.shape_with("k3_prefill", T=1, E=4), seed=0, device="cuda")["W13"]
    p, sc = gpu_quantize(W13)
    p_ref, s_ref = oracle.mxfp4_quantize(W13.double().cpu().numpy())
    assert np.array_equal(sc.cpu().numpy(), s_ref) and np.array_equal(p.cpu().numpy(), p_ref)
