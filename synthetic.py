"""Seeded synthetic inputs for the Stable LatentMoE layer and the Quantile Balancing engine.

This module holds workload shapes and random draws only.  It contains no step of the
layer's arithmetic, so that the oracle (``oracle/``) and the CUDA library
(``latent_space_experts_gb300``) can both consume the very same tensors without sharing
any code that computes the method.

Shapes follow the write-ups on Kimi K3's MoE ("简单谈谈 K3 的 MoE 和 Attention" as summarised in
"苏神复盘 Kimi K3", section 01: hidden 7168, latent 3584, 896 routed experts, 16 active,
2 shared experts).  The routed intermediate width 512 and the smaller layer shapes are
the build's own choice; the pages state none of them.

Recipe (one torch generator per tensor, seed ``seed*1000 + tensor_id``):
  * x ~ N(0, 1); on the "mid" layer, 1 % of the entries (Bernoulli 0.01) are scaled by 50.
  * every weight matrix W[out, in] ~ N(0, 1/in).
  * router bias b: 0 ("tiny", K3 shapes), N(0, 0.05^2) ("mid").
  * router logit offset mu_e ~ N(0, 0.5^2) on the K3 shapes; "heavy skew" adds +2 on a
    seeded 10 % of the experts.
  * RMSNorm weight gamma = 1 + N(0, 0.1^2) (or exactly 1 with ``gamma_ones``).
  * bf16 layers store x and all projection weights rounded to bf16; W_r, b, mu and gamma
    stay fp32 (gamma is rounded to bf16 values but kept in an fp32 buffer).
  * QB engine: logits N(mu_e, 1) with mu_e ~ N(0, 0.5^2); micro-batch m uses seed 1 + m;
    the scores handed to the engine are fp32 sigmoids of those logits.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class LayerShape:
    name: str
    T: int
    d: int
    d_latent: int
    E: int
    k: int
    I: int
    n_shared: int
    I_shared: int
    dtype: str            # "f32" or "bf16": the type of x, the projections and the outputs
    nbins: int = 1000
    beta1: float = 4.0
    beta2: float = 25.0
    eps: float = 1e-6
    x_outliers: bool = False   # 1 % of x scaled by 50
    bias_std: float = 0.0
    mu_std: float = 0.0

    def as_dict(self):
        return asdict(self)


LAYERS = {
    "tiny": LayerShape("tiny", T=64, d=256, d_latent=128, E=16, k=2, I=64, n_shared=2,
                       I_shared=128, dtype="f32"),
    "mid": LayerShape("mid", T=4096, d=2048, d_latent=1024, E=64, k=4, I=256, n_shared=2,
                      I_shared=1024, dtype="bf16", x_outliers=True, bias_std=0.05),
    "k3_prefill": LayerShape("k3_prefill", T=8192, d=7168, d_latent=3584, E=896, k=16, I=512,
                             n_shared=2, I_shared=2048, dtype="bf16", mu_std=0.5),
    "k3_decode": LayerShape("k3_decode", T=128, d=7168, d_latent=3584, E=896, k=16, I=512,
                            n_shared=2, I_shared=2048, dtype="bf16", mu_std=0.5),
    # a 1/7 slice of the K3 prefill layer for profiler captures: the same per-expert shapes
    # and about the same tokens per expert (1170 * 16 / 128 = 146), 1.5 GB on the device
    "k3_slice": LayerShape("k3_slice", T=1170, d=7168, d_latent=3584, E=128, k=16, I=512,
                           n_shared=2, I_shared=2048, dtype="bf16", mu_std=0.5),
    # a 1/7 slice of the K3 decode batch for profiler captures: about 2.3 tokens per expert
    # (18 * 16 / 128), as in the 128-token batch over 896 experts
    "k3_decode_slice": LayerShape("k3_decode_slice", T=18, d=7168, d_latent=3584, E=128, k=16, I=512,
                                  n_shared=2, I_shared=2048, dtype="bf16", mu_std=0.5),
    # the K3 prefill batch and widths with 16 experts (top-2): the dense GEMMs (router,
    # down-projection, shared experts, up-projection) at full size, 1.6 GB on the device
    "k3_dense": LayerShape("k3_dense", T=8192, d=7168, d_latent=3584, E=16, k=2, I=512,
                           n_shared=2, I_shared=2048, dtype="bf16", mu_std=0.5),
}


@dataclass(frozen=True)
class QBShape:
    name: str = "qb_engine"
    T: int = 65536
    E: int = 896
    k: int = 16
    nbins: int = 1000
    micro_batches: int = 8
    mu_std: float = 0.5


QB = QBShape()

# tensor ids used to derive the per-tensor seeds
_TID = dict(x=1, W_r=2, bias=3, mu=4, W_in=5, W13=6, W2=7, gamma=8, W_out=9, W13_s=10,
            W2_s=11, skew=12, x_mask=13, qb_mu=20, qb_logits=21)


def shape_with(base: LayerShape | str, **over) -> LayerShape:
    """A copy of a named shape with some fields replaced (used for edge-case tests)."""
    if isinstance(base, str):
        base = LAYERS[base]
    d = base.as_dict()
    d.update(over)
    return LayerShape(**d)


def _gen(seed: int, tid: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + _TID[tid])
    return g


def _normal(shape, std, seed, tid, device, chunk_rows=None):
    """N(0, std^2) fp32, drawn in row chunks so that large tensors never need two fp32 copies."""
    g = _gen(seed, tid, device)
    out = torch.empty(shape, dtype=torch.float32, device=device)
    if out.numel() == 0:
        return out
    flat = out.view(shape[0], -1)
    step = chunk_rows or flat.shape[0]
    for r0 in range(0, flat.shape[0], step):
        r1 = min(flat.shape[0], r0 + step)
        flat[r0:r1] = torch.randn((r1 - r0, flat.shape[1]), generator=g, device=device,
                                  dtype=torch.float32)
    out.mul_(std)
    return out


def logit_offset(shape: LayerShape | str, seed: int = 0, device="cpu", heavy_skew=False):
    """The per-expert router logit offset mu of a layer (None when the shape has none):
    mu_e ~ N(0, mu_std^2); heavy skew adds +2 on a seeded 10 % of the experts."""
    if isinstance(shape, str):
        shape = LAYERS[shape]
    if shape.mu_std <= 0:
        return None
    E = shape.E
    mu = _normal((E,), shape.mu_std, seed, "mu", device)
    if heavy_skew:
        gs = _gen(seed, "skew", device)
        hot = torch.randperm(E, generator=gs, device=device)[: math.ceil(0.1 * E)]
        mu[hot] += 2.0
    return mu


def layer_inputs(shape: LayerShape | str, seed: int = 0, device="cpu", heavy_skew=False,
                 gamma_ones=False, T: int | None = None):
    """All inputs of one layer call as torch tensors on ``device``.

    Projection weights and x are returned in the layer's storage type (fp32 or bf16);
    W_r, bias, logit_offset and gamma are fp32.  ``logit_offset`` is None when the shape
    has no offset.
    """
    if isinstance(shape, str):
        shape = LAYERS[shape]
    Tn = shape.T if T is None else T
    wdt = torch.float32 if shape.dtype == "f32" else torch.bfloat16
    d, dl, E, I, ns, Is = shape.d, shape.d_latent, shape.E, shape.I, shape.n_shared, shape.I_shared

    def w(rows_shape, fan_in, tid):
        # generate per leading row in chunks of ~64 M elements, then cast
        per_row = math.prod(rows_shape[1:]) if len(rows_shape) > 1 else 1
        chunk = max(1, (1 << 26) // max(1, per_row))
        t = _normal(rows_shape, 1.0 / math.sqrt(fan_in), seed, tid, device, chunk_rows=chunk)
        return t.to(wdt) if wdt != torch.float32 else t

    x = _normal((Tn, d), 1.0, seed, "x", device)
    if shape.x_outliers:
        gm = _gen(seed, "x_mask", device)
        mask = torch.rand((Tn, d), generator=gm, device=device) < 0.01
        x = torch.where(mask, x * 50.0, x)
    x = x.to(wdt)

    W_r = _normal((E, d), 1.0 / math.sqrt(d), seed, "W_r", device)
    bias = _normal((E,), shape.bias_std, seed, "bias", device) if shape.bias_std > 0 else \
        torch.zeros(E, dtype=torch.float32, device=device)
    mu = logit_offset(shape, seed, device, heavy_skew)
    if gamma_ones:
        gamma = torch.ones(dl, dtype=torch.float32, device=device)
    else:
        gamma = 1.0 + _normal((dl,), 0.1, seed, "gamma", device)
        if wdt == torch.bfloat16:
            gamma = gamma.to(torch.bfloat16).to(torch.float32)

    return dict(
        x=x, W_r=W_r, bias=bias, logit_offset=mu, gamma=gamma,
        W_in=w((dl, d), d, "W_in"),
        W13=w((E, 2 * I, dl), dl, "W13"),
        W2=w((E, dl, I), I, "W2"),
        W_out=w((d, dl), dl, "W_out"),
        W13_s=w((ns, 2 * Is, d), d, "W13_s"),
        W2_s=w((ns, d, Is), Is, "W2_s"),
    )


def qb_logit_offsets(q: QBShape = QB, seed: int = 0, device="cpu"):
    return _normal((q.E,), q.mu_std, seed, "qb_mu", device)


def qb_scores(micro_batch: int, q: QBShape = QB, device="cpu", T: int | None = None, seed_base=1):
    """fp32 router scores of one QB micro-batch: sigmoid of logits N(mu_e, 1).

    Micro-batch m draws its logits from seed ``seed_base + m``; mu comes from seed 0.
    """
    Tn = q.T if T is None else T
    mu = qb_logit_offsets(q, 0, device)
    logits = _normal((Tn, q.E), 1.0, seed_base + micro_batch, "qb_logits", device,
                     chunk_rows=max(1, (1 << 24) // q.E))
    logits += mu
    return torch.sigmoid(logits)
