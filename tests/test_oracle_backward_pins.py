"""Pins of the oracle's backward pass, on CPU: every gradient against central finite
differences of the oracle's own forward (fp64, selection held fixed), the activation
derivatives against closed forms and special values, and the norm's gradient against finite
differences of the norm alone.  A dropped term, a wrong sign or a transposed operand in any
step of the chain rule moves at least one of these far outside the bound."""
import numpy as np
import pytest

import oracle
import synthetic


def test_situ_and_softcap_derivatives():
    g = np.concatenate([np.linspace(-30, 30, 601), [0.0, 1e-6, -1e-6]])
    h = 1e-6
    fd = (oracle.situ(g + h) - oracle.situ(g - h)) / (2 * h)
    assert np.max(np.abs(fd - oracle.situ_grad(g))) < 1e-8
    assert oracle.situ_grad(0.0) == 0.5                      # sech^2(0) sigmoid(0) + 0
    assert abs(oracle.situ_grad(60.0)) < 1e-10               # flat at +beta
    assert abs(oracle.situ_grad(-60.0)) < 1e-10              # flat at 0
    u = np.linspace(-200, 200, 801)
    fdu = (oracle.softcap(u + h) - oracle.softcap(u - h)) / (2 * h)
    assert np.max(np.abs(fdu - oracle.softcap_grad(u))) < 1e-8
    assert oracle.softcap_grad(0.0) == 1.0
    assert np.allclose(oracle.softcap_grad(u), oracle.softcap_grad(-u))


def test_situ_glu_backward_layout():
    """The gate half of the gradient sits in the first half, the up half in the second."""
    rng = np.random.default_rng(0)
    gu = rng.normal(scale=3.0, size=(7, 10))
    dh = rng.normal(size=(7, 5))
    got = oracle.situ_glu_backward(gu, dh)
    h = 1e-6
    for i in range(10):
        e = np.zeros(10)
        e[i] = h
        fd = np.sum(dh * (oracle.situ_glu(gu + e) - oracle.situ_glu(gu - e)), axis=1) / (2 * h)
        assert np.max(np.abs(fd - got[:, i])) < 1e-7


def test_rmsnorm_backward_matches_finite_differences():
    rng = np.random.default_rng(1)
    c = rng.normal(size=(4, 9))
    gamma = 1 + 0.1 * rng.normal(size=9)
    dz = rng.normal(size=(4, 9))
    dc, dgamma = oracle.rmsnorm_backward(c, gamma, dz, 1e-6)
    h = 1e-6
    for t in range(4):
        for i in range(9):
            e = np.zeros_like(c)
            e[t, i] = h
            fd = np.sum(dz * (oracle.rmsnorm(c + e, gamma) - oracle.rmsnorm(c - e, gamma))) / (2 * h)
            assert abs(fd - dc[t, i]) < 1e-7
    for i in range(9):
        e = np.zeros(9)
        e[i] = h
        fd = np.sum(dz * (oracle.rmsnorm(c, gamma + e) - oracle.rmsnorm(c, gamma - e))) / (2 * h)
        assert abs(fd - dgamma[i]) < 1e-7


def tiny_layer(seed):
    shp = synthetic.shape_with("tiny", T=5, d=12, d_latent=8, E=6, k=2, I=4, n_shared=2, I_shared=6,
                               mu_std=0.5, bias_std=0.1)
    inp = synthetic.layer_inputs(shp, seed=seed)
    out = {k: (None if v is None else np.asarray(v.double().numpy())) for k, v in inp.items()}
    # larger weights so that the soft caps and the saturating gate are in play
    out["W13"] = out["W13"] * 6.0
    out["W13_s"] = out["W13_s"] * 6.0
    return shp, out


@pytest.mark.parametrize("seed", [0, 1])
def test_backward_matches_finite_differences_of_the_forward(seed):
    shp, inp = tiny_layer(seed)
    k = shp.k
    rng = np.random.default_rng(10 + seed)
    dy = rng.normal(size=(shp.T, shp.d))
    sel = oracle.forward(inp, k)["topk_idx"]

    def loss(p):
        return float(np.sum(dy * oracle.forward(p, k, forced_topk_idx=sel)["y"]))

    g = oracle.backward(inp, k, dy, forced_topk_idx=sel)
    h = 1e-6
    names = {"x": "dx", "W_r": "dW_r", "W_in": "dW_in", "W13": "dW13", "W2": "dW2", "gamma": "dgamma",
             "W_out": "dW_out", "W13_s": "dW13_s", "W2_s": "dW2_s"}
    for name, gname in names.items():
        base = inp[name]
        flat_idx = rng.choice(base.size, min(base.size, 40), replace=False)
        scale = max(1.0, np.max(np.abs(g[gname])))
        for fi in flat_idx:
            idx = np.unravel_index(fi, base.shape)
            p_plus = dict(inp)
            p_minus = dict(inp)
            p_plus[name] = base.copy()
            p_minus[name] = base.copy()
            p_plus[name][idx] += h
            p_minus[name][idx] -= h
            fd = (loss(p_plus) - loss(p_minus)) / (2 * h)
            assert abs(fd - g[gname][idx]) <= 1e-6 * scale, (name, idx, fd, g[gname][idx])
    assert g["dW13"].shape == inp["W13"].shape and g["dW2_s"].shape == inp["W2_s"].shape


def test_backward_router_gradient_only_on_chosen_experts():
    shp, inp = tiny_layer(2)
    dy = np.random.default_rng(3).normal(size=(shp.T, shp.d))
    g = oracle.backward(inp, shp.k, dy)
    chosen = np.zeros((shp.T, shp.E), bool)
    chosen[np.arange(shp.T)[:, None], g["topk_idx"]] = True
    assert np.all(g["dlogit"][~chosen] == 0.0)
    # the gate weights sum to 1, so the gradient of the scores sums to zero after weighting
    rows = np.arange(shp.T)[:, None]
    s = oracle.router_scores(inp["x"], inp["W_r"], inp["logit_offset"])[rows, g["topk_idx"]]
    ds = g["dlogit"][rows, g["topk_idx"]] / (s * (1 - s))
    assert np.allclose(np.sum(ds * s, axis=1), 0.0, atol=1e-12)


def test_backward_with_identical_experts_has_no_router_gradient():
    """All routed experts equal: the combine is the same FFN whatever the gate weights (they
    sum to 1), so the router receives no gradient and every expert's weight gradient is the
    gate-weighted share of one dense FFN's."""
    shp, inp = tiny_layer(4)
    inp["W13"][:] = inp["W13"][0]
    inp["W2"][:] = inp["W2"][0]
    dy = np.random.default_rng(5).normal(size=(shp.T, shp.d))
    g = oracle.backward(inp, shp.k, dy)
    assert np.max(np.abs(g["dW_r"])) < 1e-12 and np.max(np.abs(g["dg"] - g["dg"][:, :1])) < 1e-12
    # summed over experts, the routed weight gradients are those of one dense FFN driven by dc
    x_lat = inp["x"] @ inp["W_in"].T
    gu = x_lat @ inp["W13"][0].T
    h = oracle.situ_glu(gu)
    dgu = oracle.situ_glu_backward(gu, g["dc"] @ inp["W2"][0])
    assert np.allclose(g["dW13"].sum(axis=0), dgu.T @ x_lat, atol=1e-12)
    assert np.allclose(g["dW2"].sum(axis=0), g["dc"].T @ h, atol=1e-12)


def test_backward_token_subsets_match_the_full_call():
    """Per-token results of a token subset equal the full call's rows for those tokens."""
    shp, inp = tiny_layer(7)
    dy = np.random.default_rng(8).normal(size=(shp.T, shp.d))
    full = oracle.backward(inp, shp.k, dy)
    tok = [0, 3, 4]
    sub = oracle.backward(inp, shp.k, dy, forced_topk_idx=full["topk_idx"], tokens=tok)
    for name in ("dx", "dz", "dc", "dg", "dx_lat", "dlogit"):
        assert np.allclose(sub[name], full[name][tok], atol=1e-12, rtol=0), name
