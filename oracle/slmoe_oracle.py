"""Oracle for the Stable LatentMoE forward path and its Quantile Balancing engine.

TEST INFRASTRUCTURE ONLY.  This module is a plain, slow, obviously correct fp64 CPU
statement of what the layer computes, forward and backward.  Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it; the product
library never does, and it shares no code with the CUDA path.

Sources (page title, then section):
  [K3-news]  "苏神复盘 Kimi K3：896 个专家背后，藏着哪些关键技术取舍？", §01 LatentMoE 如何重新分配
             专家预算 and §02 Stable LatentMoE 如何处理数值与负载风险.
  [K3-arch]  the K3 architecture write-up (tahou.com), sections 混合专家, SiTU激活优化,
             归一化策略调整, 负载均衡优化.
  [SLMoE]    "Stable Latent MoE" concept note, sections TL;DR, 路由机制, Quantile Balancing,
             Latent-Space MoE, SiTU 激活.

Readings where the pages are silent (all listed again in the design notes):
  * router score = sigmoid(x . W_r^T + mu_e); the selection uses score + b_e; the gate
    weights renormalise the raw scores of the chosen experts to sum 1 (the bias steers
    selection only, [K3-news] §02; no extra scale factor, [K3-arch] 归一化策略调整).
  * top-k ties go to the lower expert index; slot order is biased score descending.
  * an expert is gate/up -> SiTU-GLU -> expert down (I -> d_latent); the "four chained
    matmuls" of [K3-arch] 归一化策略调整 are down, expert up, expert down, up.
  * QB histograms bin the raw scores; the quantile is read by linear interpolation inside
    the bin that holds fractional rank r = (1 - k/E) * N; the update b_e <- mean(q) - q_e
    overwrites the bias.
  * the K2 rule that QB replaces (fixed-step, SignSGD-like) moves b_e by +step when the
    expert's load is below the mean load, by -step when above, not at all when equal.

Parity pins live in ``tests/test_oracle_pins.py``.  Three quantities stay "parity unpinned"
by the pages: the exact bias-update formula (the pages defer it to a technical report),
the fixed-step size of the SignSGD-like rule, and the balance that either rule reaches on
a given input.
"""
from __future__ import annotations

import numpy as np

# [K3-arch] SiTU激活优化: beta_1 = 4 on the gate branch, beta_2 = 25 on the linear branch.
BETA1 = 4.0
BETA2 = 25.0
# [K3-arch] 负载均衡优化: 1000 bins over [0, 1] were as good as 10000.
NBINS = 1000
EPS = 1e-6


def f64(a):
    """Widen an array-like (numpy array or torch tensor, any float type) to float64 numpy."""
    if hasattr(a, "detach"):
        return a.detach().cpu().double().numpy()
    return np.asarray(a, dtype=np.float64)


# ----------------------------------------------------------------------------------------
# Activations  ([K3-arch] SiTU激活优化; [SLMoE] SiTU 激活)
# ----------------------------------------------------------------------------------------

def sigmoid(v):
    v = np.asarray(v, dtype=np.float64)
    out = np.empty_like(v)
    pos = v >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-v[pos]))
    ev = np.exp(v[~pos])
    out[~pos] = ev / (1.0 + ev)
    return out


def situ(g, beta=BETA1):
    """Sigmoid Tanh Unit: beta * tanh(g / beta) * sigmoid(g); bounded in (-beta, beta)."""
    g = np.asarray(g, dtype=np.float64)
    return beta * np.tanh(g / beta) * sigmoid(g)


def softcap(u, beta=BETA2):
    """Soft cap of the linear (up) branch: beta * tanh(u / beta)."""
    u = np.asarray(u, dtype=np.float64)
    return beta * np.tanh(u / beta)


def situ_glu(gu, beta1=BETA1, beta2=BETA2):
    """SiTU-GLU on the last axis: the first half is the gate branch, the second the up branch."""
    half = gu.shape[-1] // 2
    return situ(gu[..., :half], beta1) * softcap(gu[..., half:], beta2)


# ----------------------------------------------------------------------------------------
# Router and biased top-k  ([K3-news] §01-§02; [SLMoE] 路由机制)
# ----------------------------------------------------------------------------------------

def router_scores(x, W_r, logit_offset=None):
    """s[t, e] = sigmoid(x_t . W_r[e] + mu_e) in fp64."""
    logits = f64(x) @ f64(W_r).T
    if logit_offset is not None:
        logits = logits + f64(logit_offset)[None, :]
    return sigmoid(logits)


def select_topk(scores, bias, k):
    """Top-k experts per token by biased score s + b.

    Returns (topk_idx [T,k] int32 in slot order, gates [T,k] fp64, gap [T] fp64) where the
    slot order is biased score descending with ties to the lower expert index, the gates
    are the chosen raw scores renormalised to sum 1, and gap is the distance between the
    k-th and (k+1)-th biased scores (inf when k == E).
    """
    s = f64(scores)
    T, E = s.shape
    biased = s + f64(bias)[None, :]
    idx = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((idx, -biased), axis=-1)          # primary -biased, then index
    sel = order[:, :k].astype(np.int32)
    rows = np.arange(T)[:, None]
    chosen = s[rows, sel]
    gates = chosen / chosen.sum(axis=1, keepdims=True)
    if k < E:
        gap = biased[rows[:, 0], order[:, k - 1]] - biased[rows[:, 0], order[:, k]]
    else:
        gap = np.full(T, np.inf)
    return sel, gates, gap


def permutation(topk_idx, E):
    """Expert-sorted token index: (counts[E], offsets[E+1], perm[T*k], slot_pos[T,k]).

    perm lists token ids grouped by expert (ascending) and, inside an expert, by token id
    (ascending); slot_pos[t, j] is the position in perm of the pair (t, topk_idx[t, j]).
    """
    ti = np.asarray(topk_idx, dtype=np.int64)
    T, k = ti.shape
    e_of = ti.reshape(-1)
    t_of = np.repeat(np.arange(T), k)
    j_of = np.tile(np.arange(k), T)
    order = np.lexsort((t_of, e_of))                      # expert ascending, then token
    perm = t_of[order]
    slot_pos = np.zeros((T, k), dtype=np.int64)
    slot_pos[t_of[order], j_of[order]] = np.arange(T * k)
    counts = np.bincount(e_of, minlength=E).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return counts, offsets, perm, slot_pos


def expert_loads(topk_idx, E):
    return np.bincount(np.asarray(topk_idx).reshape(-1), minlength=E)


# ----------------------------------------------------------------------------------------
# The layer  ([K3-news] §01-§02; [K3-arch] 归一化策略调整; [SLMoE] Latent-Space MoE)
# ----------------------------------------------------------------------------------------

def rmsnorm(c, gamma, eps=EPS):
    c = f64(c)
    return f64(gamma)[None, :] * c / np.sqrt(np.mean(c * c, axis=1, keepdims=True) + eps)


def forward(inp, k, beta1=BETA1, beta2=BETA2, eps=EPS, forced_topk_idx=None, tokens=None,
            mx_activations=False, forced_mx=None):
    """One Stable LatentMoE layer (the FFN branch, no residual add) in fp64.

    inp: dict of the layer inputs (see ``synthetic.layer_inputs``).  ``tokens`` restricts
    the computation to a subset of token rows (every step is per token);
    ``forced_topk_idx`` [T_all, k] replaces the oracle's own selection (the gates are
    still the oracle's renormalised fp64 scores of the forced experts).
    ``mx_activations`` takes the layer with MXFP4 weights and MXFP8 activations ([SLMoE]
    训练基础设施): x_lat and each routed expert's h pass through MXFP8 (``mxfp8_round_trip``,
    blocks of 32 along d_latent and I) before they meet the expert weights; inp["W13"] /
    inp["W2"] then hold the weights' dequantised values.  ``forced_mx`` replaces the MXFP8
    rounding decisions with given ones, as ``forced_topk_idx`` does the selection (a value
    within floating-point error of a rounding midpoint has two valid codes): a dict with the
    dequantised x_lat [T_all, d_latent], the dequantised h of every (token, slot) pair in
    permutation order [T_all * k, I] and slot_pos [T_all, k] (the pair's row in that order).

    Returns a dict with scores, topk_idx, gates, gap, x_lat, c (the gate-weighted combine),
    z (after RMSNorm), y_routed (z projected up), y_shared and y.
    """
    x_all = inp["x"]
    T_all = x_all.shape[0]
    tok = np.arange(T_all) if tokens is None else np.asarray(tokens)
    x = f64(x_all[tok] if tokens is not None else x_all)
    T = x.shape[0]

    # router: sigmoid scores, selection by biased score, renormalised raw-score gates
    s = router_scores(x, inp["W_r"], inp.get("logit_offset"))
    if forced_topk_idx is None:
        sel, gates, gap = select_topk(s, inp["bias"], k)
    else:
        sel = np.asarray(forced_topk_idx)[tok].astype(np.int32)
        chosen = s[np.arange(T)[:, None], sel]
        gates = chosen / chosen.sum(axis=1, keepdims=True)
        _, _, gap = select_topk(s, inp["bias"], k)

    # latent down-projection d -> d_latent
    x_lat = x @ f64(inp["W_in"]).T

    # routed experts in latent space, gate-weighted sum over the k chosen experts
    W13, W2 = inp["W13"], inp["W2"]
    d_lat = x_lat.shape[1]
    if forced_mx is not None:
        x_in = f64(forced_mx["x_lat"][tok])
    else:
        x_in = mxfp8_round_trip(x_lat) if mx_activations else x_lat
    c = np.zeros((T, d_lat))
    for e in np.unique(sel):
        tt, jj = np.nonzero(sel == e)
        gu = x_in[tt] @ f64(W13[int(e)]).T                 # [n, 2I]: gate rows first
        h = situ_glu(gu, beta1, beta2)
        if forced_mx is not None:
            h = f64(forced_mx["h"][np.asarray(forced_mx["slot_pos"])[tok[tt], jj]])
        elif mx_activations:
            h = mxfp8_round_trip(h)
        y_e = h @ f64(W2[int(e)]).T                        # [n, d_latent]
        np.add.at(c, tt, gates[tt, jj][:, None] * y_e)

    # RMSNorm after the combine, before the up-projection only
    z = rmsnorm(c, inp["gamma"], eps)
    y_routed = z @ f64(inp["W_out"]).T

    # two always-on shared experts on the full hidden width
    y_shared = np.zeros_like(y_routed)
    W13_s, W2_s = inp["W13_s"], inp["W2_s"]
    for si in range(W13_s.shape[0]):
        gu = x @ f64(W13_s[si]).T
        y_shared += situ_glu(gu, beta1, beta2) @ f64(W2_s[si]).T

    return dict(scores=s, topk_idx=sel, gates=gates, gap=gap, x_lat=x_lat, c=c, z=z,
                y_routed=y_routed, y_shared=y_shared, y=y_routed + y_shared, tokens=tok)


def expert_hidden(inp, e, rows_lat, beta1=BETA1, beta2=BETA2):
    """h = SiTU-GLU(W13[e] . x_lat) for given latent rows (used to check one stage)."""
    return situ_glu(f64(rows_lat) @ f64(inp["W13"][int(e)]).T, beta1, beta2)


# ----------------------------------------------------------------------------------------
# Quantile Balancing  ([K3-arch] 负载均衡优化; [K3-news] §02; [SLMoE] Quantile Balancing)
# ----------------------------------------------------------------------------------------

def qb_bins(scores_f32, nbins=NBINS):
    """Bin index of each fp32 score: floor(fl32(s * nbins)) clamped to [0, nbins-1].

    The product is one IEEE fp32 round-to-nearest multiply, exactly as the GPU does it.
    Returns (bins int64, valid mask); NaN scores are invalid and left out of the counts.
    """
    s = np.asarray(scores_f32, dtype=np.float32)
    valid = ~np.isnan(s)
    scaled = np.where(valid, s, np.float32(0)) * np.float32(nbins)   # fp32 * fp32 -> fp32
    b = np.floor(scaled.astype(np.float64)).astype(np.int64)
    return np.clip(b, 0, nbins - 1), valid


def qb_histogram(scores_f32, nbins=NBINS, hist=None):
    """Add the per-expert bin counts of a [T, E] fp32 score block into hist [E, nbins].

    Histograms of micro-batches add ([K3-arch] 负载均衡优化: the distribution is additive
    across machines and gradient-accumulation steps).
    """
    s = np.asarray(scores_f32, dtype=np.float32)
    T, E = s.shape
    b, valid = qb_bins(s, nbins)
    flat = (np.arange(E)[None, :] * nbins + b)[valid]
    add = np.bincount(flat, minlength=E * nbins).reshape(E, nbins).astype(np.uint64)
    if hist is None:
        return add
    return np.asarray(hist, dtype=np.uint64) + add


def qb_quantile(hist, k):
    """q_e: the (1 - k/E) quantile of expert e's scores, read from its histogram.

    With N_e counts and fractional rank r = (1 - k/E) * N_e, j is the first bin whose
    cumulative count C_j reaches r, and q_e = (j + (r - C_{j-1}) / hist[j]) / nbins
    (linear inside bin j).  An empty histogram (r = 0) gives q_e = 0.
    """
    h = np.asarray(hist, dtype=np.int64)
    E, nb = h.shape
    p = 1.0 - float(k) / float(E)
    q = np.zeros(E)
    for e in range(E):
        N = int(h[e].sum())
        r = p * float(N)
        if r == 0.0:
            q[e] = 0.0
            continue
        C = np.cumsum(h[e])
        j = int(np.searchsorted(C, r, side="left"))
        prev = float(C[j - 1]) if j > 0 else 0.0
        q[e] = (j + (r - prev) / float(h[e, j])) / nb
    return q


def qb_update(hist, k):
    """Bias update b_e <- mean_e(q) - q_e from the histograms (overwrites the bias)."""
    q = qb_quantile(hist, k)
    cbar = q.mean()
    return q, cbar - q


def signsgd_update(counts, bias, step):
    """The fixed-step bias update of K2 that QB replaces ([K3-news] §02: each expert's
    selection bias moves a fixed step up or down; [K3-arch] 负载均衡优化: the SignSGD-style
    rule).  With loads n_e and mean load N / E:  b_e + step if n_e < N / E, b_e - step if
    n_e > N / E, b_e if equal.  The comparison is made on the integers N and E * n_e; the
    sum is formed in fp64 (exact for fp32 operands within 29 binary orders of each other)
    and stored as fp32, the type of the bias."""
    n = np.asarray(counts, dtype=np.int64)
    E = n.shape[0]
    N = int(n.sum())
    b = np.asarray(bias, dtype=np.float32).copy()
    for e in range(E):
        diff = N - E * int(n[e])
        if diff > 0:
            b[e] = np.float32(float(b[e]) + float(np.float32(step)))
        elif diff < 0:
            b[e] = np.float32(float(b[e]) - float(np.float32(step)))
    return b


def expert_output(inp, e, h):
    """y_e = W2[e] . h for given hidden rows (used to check one stage)."""
    return f64(h) @ f64(inp["W2"][int(e)]).T


# ----------------------------------------------------------------------------------------
# Backward pass of the layer  ([K3-arch] SiTU激活优化 / 归一化策略调整 / 负载均衡优化;
# [SLMoE] 训练基础设施).  The pages train this layer; its gradient is the chain rule of the
# forward above, written out step by step in the same notation.  The selection (top-k of
# s + b) is piecewise constant and passes no gradient; the bias b is not trained by
# gradients (QB sets it), and the logit offset mu is an input of the synthetic workload.
# ----------------------------------------------------------------------------------------

def situ_grad(g, beta=BETA1):
    """d/dg [beta tanh(g/beta) sigmoid(g)] = sech^2(g/beta) sigmoid(g)
    + beta tanh(g/beta) sigmoid(g) (1 - sigmoid(g))."""
    g = np.asarray(g, dtype=np.float64)
    th = np.tanh(g / beta)
    sg = sigmoid(g)
    return (1.0 - th * th) * sg + beta * th * sg * (1.0 - sg)


def softcap_grad(u, beta=BETA2):
    """d/du [beta tanh(u/beta)] = 1 - tanh^2(u/beta)."""
    th = np.tanh(np.asarray(u, dtype=np.float64) / beta)
    return 1.0 - th * th


def situ_glu_backward(gu, dh, beta1=BETA1, beta2=BETA2):
    """Gradient of h = SiTU(g) * softcap(u) with respect to [g | u] (same layout as gu)."""
    half = gu.shape[-1] // 2
    g, u = gu[..., :half], gu[..., half:]
    dg = dh * softcap(u, beta2) * situ_grad(g, beta1)
    du = dh * situ(g, beta1) * softcap_grad(u, beta2)
    return np.concatenate([dg, du], axis=-1)


def rmsnorm_backward(c, gamma, dz, eps=EPS):
    """z = gamma * c / r with r = sqrt(mean(c^2) + eps):
    dc = gamma dz / r - c * sum(gamma dz c) / (n r^3);  dgamma = sum_t dz * c / r."""
    c, dz, gm = f64(c), f64(dz), f64(gamma)
    n = c.shape[1]
    r = np.sqrt(np.mean(c * c, axis=1, keepdims=True) + eps)
    gdz = gm[None, :] * dz
    dc = gdz / r - c * np.sum(gdz * c, axis=1, keepdims=True) / (n * r ** 3)
    dgamma = np.sum(dz * c / r, axis=0)
    return dc, dgamma


def backward(inp, k, dy, beta1=BETA1, beta2=BETA2, eps=EPS, forced_topk_idx=None, tokens=None):
    """Gradients of sum(dy * y) for one layer call, in fp64.

    dy [T, d] is the gradient arriving at the layer output y.  Returns dx [T, d] and the
    weight gradients dW_r [E, d], dW_in [d_l, d], dW13 [E, 2I, d_l], dW2 [E, d_l, I],
    dgamma [d_l], dW_out [d, d_l], dW13_s [n_s, 2I_s, d], dW2_s [n_s, d, I_s], plus the
    intermediates dz, dc, dg (gate weights), dx_lat and dlogit (router logits, [T, E]).
    The selection is the oracle's own unless forced_topk_idx gives it.  ``tokens`` restricts
    the call to a subset of token rows (dy rows of those tokens): every per-token result (dx,
    dz, dc, dg, dx_lat, dlogit) is then that of the full call for those tokens, while the
    weight gradients hold only those tokens' contributions.
    """
    x_all = inp["x"]
    if tokens is not None:
        tok = np.asarray(tokens)
        x = f64(x_all[tok])
        dy = f64(dy)[tok] if f64(dy).shape[0] == x_all.shape[0] else f64(dy)
        if forced_topk_idx is not None:
            forced_topk_idx = np.asarray(forced_topk_idx)[tok]
    else:
        x = f64(x_all)
        dy = f64(dy)
    T, d = x.shape
    W_r, W_in, W_out = f64(inp["W_r"]), f64(inp["W_in"]), f64(inp["W_out"])
    E = W_r.shape[0]

    # forward quantities the gradient needs (recomputed here, in fp64)
    s = router_scores(x, W_r, inp.get("logit_offset"))
    if forced_topk_idx is None:
        sel, gates, _ = select_topk(s, inp["bias"], k)
    else:
        sel = np.asarray(forced_topk_idx).astype(np.int64)
        chosen = s[np.arange(T)[:, None], sel]
        gates = chosen / chosen.sum(axis=1, keepdims=True)
    x_lat = x @ W_in.T
    d_lat = x_lat.shape[1]
    W13, W2 = inp["W13"], inp["W2"]
    c = np.zeros((T, d_lat))
    ye_of = {}
    for e in np.unique(sel):
        tt, jj = np.nonzero(sel == e)
        gu = x_lat[tt] @ f64(W13[int(e)]).T
        h = situ_glu(gu, beta1, beta2)
        ye = h @ f64(W2[int(e)]).T
        ye_of[int(e)] = (tt, jj, gu, h, ye)
        np.add.at(c, tt, gates[tt, jj][:, None] * ye)
    r = np.sqrt(np.mean(c * c, axis=1, keepdims=True) + eps)
    z = f64(inp["gamma"])[None, :] * c / r

    # up-projection y_routed = z W_out^T
    dW_out = dy.T @ z
    dz = dy @ W_out
    # RMSNorm after the combine
    dc, dgamma = rmsnorm_backward(c, inp["gamma"], dz, eps)

    # combine c_t = sum_j g[t,j] y_e(t,j), then the routed experts
    dg = np.zeros((T, k))
    dx_lat = np.zeros_like(x_lat)
    dW13 = np.zeros((E,) + tuple(W13.shape[1:]))
    dW2 = np.zeros((E,) + tuple(W2.shape[1:]))
    for e, (tt, jj, gu, h, ye) in ye_of.items():
        dg[tt, jj] = np.sum(dc[tt] * ye, axis=1)
        dye = gates[tt, jj][:, None] * dc[tt]
        dW2[e] = dye.T @ h
        dh = dye @ f64(W2[e])
        dgu = situ_glu_backward(gu, dh, beta1, beta2)
        dW13[e] = dgu.T @ x_lat[tt]
        np.add.at(dx_lat, tt, dgu @ f64(W13[e]))

    # latent down-projection x_lat = x W_in^T
    dW_in = dx_lat.T @ x
    dx = dx_lat @ W_in

    # router: g_j = s_j / S over the chosen experts, s = sigmoid(logit)
    rows = np.arange(T)[:, None]
    s_sel = s[rows, sel]
    S = s_sel.sum(axis=1, keepdims=True)
    ds_sel = (dg - np.sum(gates * dg, axis=1, keepdims=True)) / S
    dlogit = np.zeros((T, E))
    dlogit[rows, sel] = ds_sel * s_sel * (1.0 - s_sel)
    dW_r = dlogit.T @ x
    dx += dlogit @ W_r

    # shared experts on the full width
    W13_s, W2_s = inp["W13_s"], inp["W2_s"]
    dW13_s = np.zeros(W13_s.shape)
    dW2_s = np.zeros(W2_s.shape)
    for si in range(W13_s.shape[0]):
        gu = x @ f64(W13_s[si]).T
        h = situ_glu(gu, beta1, beta2)
        dW2_s[si] = dy.T @ h
        dh = dy @ f64(W2_s[si])
        dgu = situ_glu_backward(gu, dh, beta1, beta2)
        dW13_s[si] = dgu.T @ x
        dx += dgu @ f64(W13_s[si])

    return dict(dx=dx, dW_r=dW_r, dW_in=dW_in, dW13=dW13, dW2=dW2, dgamma=dgamma, dW_out=dW_out,
                dW13_s=dW13_s, dW2_s=dW2_s, dz=dz, dc=dc, dg=dg, dx_lat=dx_lat, dlogit=dlogit,
                topk_idx=sel, gates=gates, c=c, z=z)


# ----------------------------------------------------------------------------------------
# MXFP4 weights  ([SLMoE] 训练基础设施: MXFP4 weights, from quantisation-aware training on).
# The pages name the format only; this is the OCP Microscaling (MX) block format restated
# from its definition: blocks of 32 consecutive values along K share one power-of-two scale
# X = 2^e, stored as an E8M0 byte (e + 127); each value is an FP4 E2M1 number (sign bit,
# two exponent bits with bias 1, one mantissa bit), so magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
# Conversion of a block: e = floor(log2(max |v|)) - 2 (2 = the largest E2M1 exponent),
# clamped to [-127, 127] (-127 for an all-zero block); each v / X goes to the nearest E2M1
# magnitude, ties to the even mantissa, values past 6 to 6 (saturation); the sign bit is
# set for v < 0.  Packing: two codes per byte, the lower-indexed value in the low nibble.
# ----------------------------------------------------------------------------------------

MX_BLOCK = 32
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def mxfp4_quantize(W):
    """(packed uint8 [..., K/2], scales uint8 [..., K/32]) of W [..., K] (K a multiple of 32)."""
    w = f64(W)
    K = w.shape[-1]
    blocks = w.reshape(w.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    amax = np.max(np.abs(blocks), axis=-1)
    e = np.full(amax.shape, -127, dtype=np.int64)
    nz = amax > 0
    e[nz] = np.floor(np.log2(amax[nz])).astype(np.int64) - 2
    e = np.clip(e, -127, 127)
    scaled = blocks / np.ldexp(1.0, e)[..., None]
    mag = np.abs(scaled)
    # nearest magnitude; on a tie the even index (mantissa bit 0) wins
    dist = np.abs(mag[..., None] - E2M1_MAGNITUDES)
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    even = cand & (np.arange(8) % 2 == 0)
    idx = np.where(even.any(axis=-1), np.argmax(even, axis=-1), np.argmax(cand, axis=-1))
    codes = (idx | np.where(scaled < 0, 8, 0)).astype(np.uint8)
    codes = codes.reshape(w.shape)
    packed = (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


def mxfp4_dequantize(packed, scales):
    """The values [..., K] (fp64) that MXFP4 codes and their block scales stand for."""
    p = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    codes[..., 0::2] = p & 15
    codes[..., 1::2] = p >> 4
    mag = E2M1_MAGNITUDES[codes & 7]
    val = np.where(codes & 8, -mag, mag)
    X = np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    K = codes.shape[-1]
    return (val.reshape(codes.shape[:-1] + (K // MX_BLOCK, MX_BLOCK)) * X[..., None]).reshape(codes.shape)


# ----------------------------------------------------------------------------------------
# MXFP8 activations  ([SLMoE] 训练基础设施: MXFP8 activations beside the MXFP4 weights).  The
# same OCP Microscaling block format with FP8 E4M3 elements: sign bit, four exponent bits with
# bias 7 and three mantissa bits, so normal values 2^(E-7) (1 + m/8) for E = 1..15 (E = 15 with
# m = 7 is NaN, so the largest value is 448) and subnormal values m/8 * 2^-6.  A block of 32
# consecutive values along K shares X = 2^e, e = floor(log2(max |v|)) - 8 (8 = the largest E4M3
# exponent), clamped to [-127, 127] (-127 for an all-zero block), stored as the E8M0 byte
# e + 127.  Each v / X goes to the nearest E4M3 value, ties to the even mantissa, values past
# 448 to 448 (saturation); the sign bit is set for v < 0, so a negative value that rounds to
# zero is -0.  Which activations are MXFP8 is a reading: the pages name the formats only.
# Here they are the two operands that meet the MXFP4 weights, x_lat (before the experts'
# gate/up) and h (before the experts' down), blocked along the contraction dimension.
# ----------------------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_round(v):
    """Nearest E4M3 value to each v (fp64), ties to the even mantissa, saturating at 448."""
    v = f64(v)
    a = np.abs(v)
    _, ex = np.frexp(a)                      # a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1
    p = np.maximum(ex.astype(np.int64) - 1, -6)
    step = np.ldexp(1.0, p - 3)              # grid step of the binade (subnormals: 2^-9)
    r = np.minimum(np.rint(a / step) * step, E4M3_MAX)
    return np.where(v < 0, -r, r)


def e4m3_encode(r, negative):
    """E4M3 codes (uint8) of values r that are on the E4M3 grid; `negative` sets the sign bit."""
    a = np.abs(f64(r))
    _, ex = np.frexp(a)
    p = ex.astype(np.int64) - 1
    normal = a >= 2.0 ** -6
    E = np.where(normal, p + 7, 0)
    M = np.where(normal, np.ldexp(a, -p) * 8 - 8, a * 2.0 ** 9)
    code = (E << 3) | M.astype(np.int64)
    return (code | np.where(negative, 0x80, 0)).astype(np.uint8)


def e4m3_decode(codes):
    """Values (fp64) of E4M3 codes; the two NaN codes decode to NaN."""
    c = np.asarray(codes, dtype=np.int64)
    E = (c >> 3) & 15
    M = c & 7
    mag = np.where(E == 0, M / 8.0 * 2.0 ** -6, (1 + M / 8.0) * np.ldexp(1.0, E - 7))
    mag = np.where((E == 15) & (M == 7), np.nan, mag)
    return np.where(c & 0x80, -mag, mag)


def mxfp8_quantize(V):
    """(codes uint8 [..., K], scales uint8 [..., K/32]) of V [..., K] (K a multiple of 32)."""
    v = f64(V)
    K = v.shape[-1]
    blocks = v.reshape(v.shape[:-1] + (K // MX_BLOCK, MX_BLOCK))
    amax = np.max(np.abs(blocks), axis=-1)
    _, ex = np.frexp(amax)
    e = np.where(amax > 0, ex.astype(np.int64) - 1 - 8, -127)
    e = np.clip(e, -127, 127)
    scaled = blocks / np.ldexp(1.0, e)[..., None]
    codes = e4m3_encode(e4m3_round(scaled), scaled < 0).reshape(v.shape)
    return codes, (e + 127).astype(np.uint8)


def mxfp8_dequantize(codes, scales):
    """The values [..., K] (fp64) that MXFP8 codes and their block scales stand for."""
    val = e4m3_decode(codes)
    X = np.ldexp(1.0, np.asarray(scales, dtype=np.int64) - 127)
    K = val.shape[-1]
    return (val.reshape(val.shape[:-1] + (K // MX_BLOCK, MX_BLOCK)) * X[..., None]).reshape(val.shape)


def mxfp8_round_trip(V):
    """V quantised to MXFP8 and back (fp64): the value an MXFP8 activation carries."""
    return mxfp8_dequantize(*mxfp8_quantize(V))
