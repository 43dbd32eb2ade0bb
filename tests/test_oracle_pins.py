"""Pins for the oracle: facts the K3 pages and plain mathematics fix, none of them a
re-statement of the oracle's own formulas.  CPU only.

Sources are cited by page title and section:
  [K3-news] "苏神复盘 Kimi K3：896 个专家背后，藏着哪些关键技术取舍？" §01, §02
  [K3-arch] K3 architecture write-up (tahou.com): SiTU激活优化, 归一化策略调整, 负载均衡优化
  [SLMoE]   "Stable Latent MoE" concept note: TL;DR, Quantile Balancing, SiTU 激活
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_constants_match_the_pages():
    """[K3-arch] SiTU激活优化 / 负载均衡优化, [K3-news] §01: constants printed on the pages."""
    g = json.load(open(os.path.join(GOLDEN, "k3_constants.json")))
    assert oracle.BETA1 == g["beta1"]["value"]
    assert oracle.BETA2 == g["beta2"]["value"]
    assert oracle.NBINS == g["nbins"]["value"]
    k3 = synthetic.LAYERS["k3_prefill"]
    assert (k3.d, k3.d_latent, k3.E, k3.k, k3.n_shared) == (
        g["d_model"]["value"], g["d_latent"]["value"], g["routed_experts"]["value"],
        g["active_routed"]["value"], g["shared_experts"]["value"])
    assert synthetic.LAYERS["k3_decode"].d == k3.d
    E0, k0 = g["pre_latent_config"]["value"]
    assert k0 / E0 == k3.k / k3.E          # same sparsity before and after LatentMoE


# ---------------------------------------------------------------- SiTU and the soft cap

def test_situ_special_values():
    """[K3-arch] SiTU激活优化: gate output confined to (-beta, beta), beta = 4."""
    assert oracle.situ(0.0) == 0.0
    assert abs(oracle.situ(60.0) - 4.0) < 1e-9            # saturates at +beta
    assert abs(oracle.situ(-60.0)) < 1e-20                 # and at 0 for g -> -inf
    h = 1e-5
    slope = (oracle.situ(h) - oracle.situ(-h)) / (2 * h)
    assert abs(slope - 0.5) < 1e-8                         # SiTU'(0) = SiLU'(0) = 1/2


@pytest.mark.parametrize("g", [1e-3, -1e-3, 0.1, -0.1, 1.0, -1.0, 2.5])
def test_situ_close_to_silu_for_small_inputs(g):
    """[K3-news] §02: the soft cap keeps the original function for small activations.

    With y = g/beta, SiTU/SiLU = tanh(y)/y and the Taylor series of tanh gives
    1 - y^2/3 <= tanh(y)/y <= 1 - y^2/3 + 2y^4/15.
    """
    silu = g / (1.0 + math.exp(-g))
    y = g / 4.0
    ratio = float(oracle.situ(g)) / silu
    assert 1 - y * y / 3 - 1e-15 <= ratio <= 1 - y * y / 3 + 2 * y ** 4 / 15 + 1e-15


def test_situ_bounds_and_monotone():
    g = np.linspace(-1e3, 1e3, 200001)
    s = oracle.situ(g)
    assert np.all(s <= 4.0) and np.all(s > -4.0)           # fp64 rounds the far tail to 4
    assert np.all(s[np.abs(g) < 60] < 4.0)
    silu_min = -0.2784645427610738                         # min of g*sigmoid(g)
    assert s.min() >= silu_min - 1e-12                     # |tanh(y)/y| <= 1
    pos = g > 0
    assert np.all(np.diff(s[pos]) >= 0)


def test_softcap():
    """[K3-arch] SiTU激活优化: soft cap beta_2 = 25 on the linear branch."""
    assert oracle.softcap(0.0) == 0.0
    assert abs(oracle.softcap(1e-3) - 1e-3) < 1e-12
    assert abs(oracle.softcap(1e4) - 25.0) < 1e-12
    assert abs(oracle.softcap(-1e4) + 25.0) < 1e-12
    u = np.linspace(-1e4, 1e4, 100001)
    assert np.all(np.abs(oracle.softcap(u)) <= 25.0)
    assert np.allclose(oracle.softcap(-u), -oracle.softcap(u))


def test_situ_glu_gate_is_first_half():
    """[SLMoE] SiTU 激活: gate = first half of the last axis, up = second half.

    gate >> beta1 saturates SiTU at 4; a tiny up value passes the cap unchanged, so the
    product is 4e-3.  Swapping the halves would give SiTU(1e-3) * cap(40) ~ 1.15e-2.
    """
    h = oracle.situ_glu(np.array([40.0, 1e-3]))
    assert abs(h[0] - 4e-3) < 1e-10
    big = oracle.situ_glu(np.array([1e3, 1e3]))
    assert abs(big[0] - 100.0) < 1e-9                      # |h| < beta1 * beta2
    rng = np.random.default_rng(0)
    gu = rng.normal(scale=50.0, size=(1000, 64))
    assert np.all(np.abs(oracle.situ_glu(gu)) < 100.0)


# ---------------------------------------------------------------- router and top-k

def test_router_scores_closed_forms():
    x = np.zeros((3, 8))
    W = np.ones((5, 8))
    assert np.all(oracle.router_scores(x, W) == 0.5)       # sigmoid(0) = 1/2
    mu = np.array([50.0, -50.0, 0.0, 0.0, 0.0])
    s = oracle.router_scores(x, W, mu)
    assert abs(s[0, 0] - 1.0) < 1e-20 and s[0, 1] < 1e-20
    x1 = np.zeros((1, 8)); x1[0, 2] = 3.0
    W1 = np.zeros((5, 8)); W1[4, 2] = 1.0                  # W_r is [E, d]: row e is expert e
    s1 = oracle.router_scores(x1, W1)
    assert abs(s1[0, 4] - 1 / (1 + math.exp(-3.0))) < 1e-15 and np.all(s1[0, :4] == 0.5)


def _brute_topk_set(v, k):
    """The unique k-subset whose members all beat all non-members under (value desc, index asc)."""
    E = len(v)
    found = []
    for S in itertools.combinations(range(E), k):
        rest = [j for j in range(E) if j not in S]
        if all((v[i] > v[j]) or (v[i] == v[j] and i < j) for i in S for j in rest):
            found.append(set(S))
    assert len(found) == 1
    return found[0]


@pytest.mark.parametrize("E,k", [(6, 1), (7, 2), (10, 3), (12, 3)])
def test_topk_matches_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    T = 200
    s = np.round(rng.uniform(size=(T, E)) * 8) / 8         # coarse grid: many exact ties
    b = np.round(rng.normal(scale=0.2, size=E) * 8) / 8
    sel, gates, gap = oracle.select_topk(s, b, k)
    for t in range(T):
        v = s[t] + b
        assert set(sel[t].tolist()) == _brute_topk_set(v, k)
        vs = v[sel[t]]
        for j in range(k - 1):                              # slot order: desc, ties by index
            assert vs[j] > vs[j + 1] or (vs[j] == vs[j + 1] and sel[t, j] < sel[t, j + 1])
        srt = np.sort(v)[::-1]
        assert gap[t] == srt[k - 1] - srt[k]
        assert abs(gates[t].sum() - 1.0) < 1e-12
        # gates are the raw scores (not the biased ones) renormalised
        raw = s[t, sel[t]]
        assert np.allclose(gates[t] * raw.sum(), raw, rtol=0, atol=1e-12)


def test_bias_steers_selection_only():
    """[K3-news] §02: the bias moves the selection threshold, the weights stay the raw scores."""
    s = np.array([[0.9, 0.8, 0.1]])
    sel0, g0, _ = oracle.select_topk(s, np.zeros(3), 1)
    sel1, g1, _ = oracle.select_topk(s, np.array([0.0, 0.0, 0.85]), 1)
    assert sel0[0, 0] == 0 and sel1[0, 0] == 2
    assert g0[0, 0] == 1.0 and g1[0, 0] == 1.0
    sel2, g2, _ = oracle.select_topk(s, np.array([0.0, 0.0, 0.85]), 2)
    assert set(sel2[0]) == {0, 2}
    assert abs(g2[0, list(sel2[0]).index(0)] - 0.9 / 1.0) < 1e-12


# ---------------------------------------------------------------- permutation

def _random_routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (37, 16, 2), (200, 9, 9), (64, 64, 4)])
def test_permutation_invariants_and_brute_force(T, E, k):
    ti = _random_routing(T, E, k, T + E)
    counts, offsets, perm, slot_pos = oracle.permutation(ti, E)
    assert counts.sum() == T * k and offsets[0] == 0 and offsets[-1] == T * k
    assert np.all(np.diff(offsets) == counts)
    # brute force: walk experts, then tokens in order
    exp_perm = [t for e in range(E) for t in range(T) if e in ti[t]]
    assert perm.tolist() == exp_perm
    for t in range(T):
        for j in range(k):
            p = slot_pos[t, j]
            e = ti[t, j]
            assert perm[p] == t and offsets[e] <= p < offsets[e + 1]
    assert sorted(slot_pos.reshape(-1).tolist()) == list(range(T * k))


# ---------------------------------------------------------------- the layer

def _tiny(seed=0, **over):
    shp = synthetic.shape_with("tiny", **over)
    return shp, synthetic.layer_inputs(shp, seed=seed)


def _dense_ffn(x_lat, W13, W2):
    return oracle.situ_glu(x_lat @ oracle.f64(W13).T) @ oracle.f64(W2).T


def test_rmsnorm_unit_rms():
    """[K3-arch] 归一化策略调整: one RMSNorm before the up-projection; gamma = 1 gives RMS 1."""
    rng = np.random.default_rng(1)
    c = rng.normal(scale=3.0, size=(50, 128))
    z = oracle.rmsnorm(c, np.ones(128))
    rms = np.sqrt((z * z).mean(axis=1))
    ms = (c * c).mean(axis=1)
    assert np.all(np.abs(rms - 1.0) <= 1e-6 / ms)           # 1 - O(eps / mean(c^2))
    assert np.allclose(oracle.rmsnorm(7.0 * c, np.ones(128)), z, atol=1e-7)


def test_identical_experts_reduce_to_one_dense_ffn():
    """If all routed experts are equal, the renormalised gates sum to 1 and the routed branch
    is up(RMSNorm(FFN(down(x)))) whatever the routing ([K3-news] §01-§02)."""
    shp, inp = _tiny(seed=3)
    inp["W13"][:] = inp["W13"][0]
    inp["W2"][:] = inp["W2"][0]
    out = oracle.forward(inp, shp.k)
    x = oracle.f64(inp["x"])
    x_lat = x @ oracle.f64(inp["W_in"]).T
    c = _dense_ffn(x_lat, inp["W13"][0], inp["W2"][0])
    assert np.allclose(out["c"], c, rtol=1e-12, atol=1e-12)
    z = oracle.rmsnorm(c, inp["gamma"])
    y = z @ oracle.f64(inp["W_out"]).T
    for s in range(shp.n_shared):
        y += _dense_ffn(x, inp["W13_s"][s], inp["W2_s"][s])
    assert np.allclose(out["y"], y, rtol=1e-11, atol=1e-11)


def test_k_equals_E_is_a_dense_mixture():
    shp, inp = _tiny(seed=4, E=5, k=5)
    out = oracle.forward(inp, 5)
    x = oracle.f64(inp["x"])
    s = 1.0 / (1.0 + np.exp(-(x @ oracle.f64(inp["W_r"]).T)))
    w = s / s.sum(axis=1, keepdims=True)
    x_lat = x @ oracle.f64(inp["W_in"]).T
    c = sum(w[:, [e]] * _dense_ffn(x_lat, inp["W13"][e], inp["W2"][e]) for e in range(5))
    assert np.allclose(out["c"], c, rtol=1e-12, atol=1e-12)


def test_projection_orientation_and_norm_position():
    """Weights are [out, in]; expert row 0 is a gate row and row I an up row; the norm sits
    between the combine and the up-projection.  Built so that a transposed W13 (square on
    this shape: 2I = d_latent) or a swapped gate/up pair gives a visibly different output."""
    shp, inp = _tiny(seed=5)
    I, dl, d = shp.I, shp.d_latent, shp.d
    inp["gamma"] = torch.ones(dl)
    inp["W_in"].zero_()
    for l in range(dl):
        inp["W_in"][l, l] = 1.0                            # x_lat = x[:d_latent]
    inp["W13"].zero_(); inp["W2"].zero_(); inp["W13_s"].zero_()
    inp["W13"][:, 0, 5] = 1.0                              # gate_0 reads latent 5
    inp["W13"][:, I, 7] = 1.0                              # up_0 reads latent 7
    inp["W2"][:, 3, 0] = 100.0                             # latent out 3 reads h_0
    inp["x"].zero_()
    inp["x"][:, 5] = 40.0
    inp["x"][:, 7] = 1e-3
    out = oracle.forward(inp, shp.k)
    c = out["c"]
    assert np.allclose(c[:, 3], 0.4, rtol=1e-6)            # 100 * SiTU(40) * cap(1e-3) ~ 0.4
    assert np.all(np.delete(c, 3, axis=1) == 0)
    z = out["z"]
    assert np.all(z[:, 3] > 0) and np.all(np.delete(z, 3, axis=1) == 0)
    ms = (c * c).mean(axis=1)
    assert np.all(np.abs(np.sqrt((z * z).mean(axis=1)) - 1.0) <= 1e-6 / ms)
    y = out["y"]
    col = oracle.f64(inp["W_out"])[:, 3]                   # y = W_out z: column 3 of W_out
    assert np.allclose(y, z[:, [3]] * col[None, :], rtol=1e-12, atol=1e-12)


def test_forced_routing_and_token_subsets_agree():
    shp, inp = _tiny(seed=6)
    full = oracle.forward(inp, shp.k)
    sub = oracle.forward(inp, shp.k, tokens=np.array([3, 17, 40]))
    assert np.allclose(sub["y"], full["y"][[3, 17, 40]], rtol=1e-12, atol=1e-12)
    forced = oracle.forward(inp, shp.k, forced_topk_idx=full["topk_idx"])
    assert np.allclose(forced["y"], full["y"], rtol=0, atol=0)


# ---------------------------------------------------------------- Quantile Balancing

def test_histogram_counts_and_additivity():
    """[K3-arch] 负载均衡优化: per-expert histograms over [0, 1]; counts add across
    micro-batches and machines."""
    a = synthetic.qb_scores(0, T=3000).numpy()
    b = synthetic.qb_scores(1, T=2000).numpy()
    ha = oracle.qb_histogram(a)
    hb = oracle.qb_histogram(b)
    assert ha.shape == (896, 1000)
    assert np.all(ha.sum(axis=1) == 3000)
    assert np.array_equal(ha + hb, oracle.qb_histogram(np.concatenate([a, b])))
    assert np.array_equal(oracle.qb_histogram(b, hist=ha), ha + hb)


def test_bins_against_per_value_binning():
    """Binning a value = floor of its single-rounded fp32 product with 1000; checked value by
    value through fp64 (exact product, then one rounding to fp32) and against the exact
    rational floor, which may differ only within one fp32 ulp of a bin edge."""
    rng = np.random.default_rng(2)
    s = rng.uniform(size=20000).astype(np.float32)
    edge = (np.arange(0, 1001) / 1000.0).astype(np.float32)
    s = np.concatenate([s, edge, np.nextafter(edge, np.float32(0)), np.nextafter(edge, np.float32(2))])
    s = s[(s >= 0) & (s <= 1)]
    b, valid = oracle.qb_bins(s)
    assert valid.all()
    for v, bv in zip(s.tolist(), b.tolist()):
        p = float(np.float32(v * 1000.0))                  # exact product, one fp32 rounding
        assert bv == min(999, math.floor(p))
        exact = min(999, math.floor(v * 1000.0)) if v * 1000.0 != 1000.0 else 999
        if bv != exact:
            assert abs(v * 1000.0 - round(v * 1000.0)) <= np.spacing(np.float32(v * 1000.0))
    bb, _ = oracle.qb_bins(np.array([0.0, 1.0, 0.5, 0.0005, 0.9995], np.float32))
    assert bb.tolist() == [0, 999, 500, 0, 999]
    bn, vn = oracle.qb_bins(np.array([np.nan, 0.25], np.float32))
    assert vn.tolist() == [False, True]
    h = oracle.qb_histogram(np.array([[np.nan], [0.25]], np.float32))
    assert h.sum() == 1 and h[0, 250] == 1


def test_quantile_closed_forms():
    E, k = 8, 2
    p = 1 - k / E
    uniform = np.ones((E, 1000), dtype=np.uint64)           # one count per bin
    q = oracle.qb_quantile(uniform, k)
    assert np.allclose(q, p, rtol=0, atol=1e-15)            # linear inside bins: q = p
    point = np.zeros((E, 1000), dtype=np.uint64)
    point[:, 123] = 10
    q = oracle.qb_quantile(point, k)
    assert np.allclose(q, (123 + p) / 1000, rtol=0, atol=1e-15)
    empty = np.zeros((E, 1000), dtype=np.uint64)
    assert np.all(oracle.qb_quantile(empty, k) == 0.0)


def test_quantile_within_one_bin_of_exact():
    """The histogram quantile lies within one bin width (1e-3, plus fp32 edge rounding) of the
    ceil(r)-th smallest score, r = (1 - k/E) N."""
    s = synthetic.qb_scores(2, T=4000).numpy()
    E, k = s.shape[1], 16
    q = oracle.qb_quantile(oracle.qb_histogram(s), k)
    r = (1 - k / E) * s.shape[0]
    exact = np.sort(s, axis=0)[math.ceil(r) - 1]
    assert np.max(np.abs(q - exact)) <= 1e-3 + 1e-6


def test_bias_update_properties():
    s = synthetic.qb_scores(3, T=4000).numpy()
    h = oracle.qb_histogram(s)
    q, b = oracle.qb_update(h, 16)
    assert abs(b.sum()) < 1e-12
    assert np.allclose(q + b, q.mean(), rtol=0, atol=1e-15)
    same = np.repeat(h[:1], h.shape[0], axis=0)
    _, b0 = oracle.qb_update(same, 16)
    assert np.all(np.abs(b0) <= 1e-15)                      # mean of equal values, fp64


def test_qb_rebalances_loads():
    """[K3-news] §02: QB places each expert's selection threshold so that it receives its
    share of tokens.  Loads always sum to T*k; the skewed max/mean load shrinks."""
    E, k = 64, 4
    rng = np.random.default_rng(7)
    mu = rng.normal(scale=0.5, size=E)
    logits = rng.normal(size=(20000, E)) + mu
    s = (1 / (1 + np.exp(-logits))).astype(np.float32)
    sel0, _, _ = oracle.select_topk(s, np.zeros(E), k)
    L0 = oracle.expert_loads(sel0, E)
    _, b = oracle.qb_update(oracle.qb_histogram(s), k)
    sel1, _, _ = oracle.select_topk(s, b, k)
    L1 = oracle.expert_loads(sel1, E)
    assert L0.sum() == L1.sum() == 20000 * k
    assert L1.max() / L1.mean() < 0.5 * (L0.max() / L0.mean())


# ---------------------------------------------------------------- fixed-step (SignSGD) rule
def test_signsgd_hand_cases():
    """[K3-news] §02: K2 raises or lowers each expert's selection bias by a fixed step."""
    step = np.float32(1e-3)
    b = oracle.signsgd_update([3, 1, 2], np.zeros(3, np.float32), step)    # mean 2
    assert b.tolist() == [-step, step, 0.0]
    b = oracle.signsgd_update([1, 2], np.array([0.5, 0.5], np.float32), 0.25)   # mean 1.5
    assert b.tolist() == [0.75, 0.25]
    b = oracle.signsgd_update([0, 0, 0, 9], np.array([0, 0, 0, 0], np.float32), 0.5)
    assert b.tolist() == [0.5, 0.5, 0.5, -0.5]
    neg0 = np.array([-0.0, 1.0], np.float32)
    b = oracle.signsgd_update([5, 5], neg0, 0.5)                           # every load at the mean
    assert np.array_equal(b.view(np.uint32), neg0.view(np.uint32))


def test_signsgd_sign_rule_and_step_against_exact_arithmetic():
    """The direction is decided by exact rational comparison with the mean load, and each
    moved bias equals the fp32 round-to-nearest sum of the old bias and +-step."""
    from fractions import Fraction
    rng = np.random.default_rng(11)
    for E in (1, 2, 7, 64, 897):
        n = rng.integers(0, 40, size=E)
        if E > 2:
            n[: E // 3] = int(round(n.mean()))                   # many loads near the mean
        b0 = rng.normal(scale=0.05, size=E).astype(np.float32)
        step = np.float32(rng.uniform(1e-4, 1e-2))
        b1 = oracle.signsgd_update(n, b0, step)
        mean = Fraction(int(n.sum()), E)
        for e in range(E):
            if Fraction(int(n[e])) < mean:
                want = np.float32(b0[e]) + step                   # numpy fp32 add (IEEE RN)
            elif Fraction(int(n[e])) > mean:
                want = np.float32(b0[e]) - step
            else:
                want = b0[e]
            assert b1[e].view(np.uint32) == np.float32(want).view(np.uint32), e


def test_signsgd_needs_many_steps_where_qb_needs_one():
    """[K3-news] §02 / [K3-arch] 负载均衡优化: the fixed-step rule probes its way to balance,
    QB reads the thresholds from the score distribution in one update.  On a skewed router
    one fixed step of 1e-3 leaves the imbalance almost unchanged, QB halves it at once, and
    repeated fixed steps keep shrinking it (the step size itself is the caller's: the pages
    give none)."""
    E, k = 64, 4
    rng = np.random.default_rng(7)
    mu = rng.normal(scale=0.5, size=E)
    s = (1 / (1 + np.exp(-(rng.normal(size=(20000, E)) + mu)))).astype(np.float32)

    def imbalance(bias):
        sel, _, _ = oracle.select_topk(s, bias, k)
        L = oracle.expert_loads(sel, E)
        assert L.sum() == 20000 * k
        return L.max() / L.mean(), L

    r0, L0 = imbalance(np.zeros(E))
    b = oracle.signsgd_update(L0, np.zeros(E, np.float32), 1e-3)
    r1, _ = imbalance(b)
    _, bq = oracle.qb_update(oracle.qb_histogram(s), k)
    rq, _ = imbalance(bq)
    assert r1 > 0.9 * r0 and rq < 0.5 * r0
    b = np.zeros(E, np.float32)
    for _ in range(60):
        _, L = imbalance(b)
        b = oracle.signsgd_update(L, b, 1e-2)
    r60, _ = imbalance(b)
    assert r60 < 0.75 * r0

