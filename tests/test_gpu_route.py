"""GPU parity of slmoe_route against the oracle: router scores, biased top-k selection
(bit-exact outside near ties), gate weights, and the expert-sorted permutation (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import latent_space_experts_gb300 as lse
from gpu_util import (NEAR_TIE, check_selection_and_permutation, need_gpu, route_buffers, run_route,
                      to_dev)

# Router scores must stay within half the near-tie gap of the oracle: then every token whose
# k-th/(k+1)-th biased gap is >= 1e-5 is decided the same way on both sides.
SCORE_TOL = NEAR_TIE / 2

pytestmark = pytest.mark.gpu


def check_route(shape, inp_cpu, score_tol):
    cfg = lse.config(shape)
    inp = to_dev(inp_cpu)
    out = run_route(cfg, inp)
    T, E, k = shape.T, shape.E, shape.k
    s_ref = oracle.router_scores(inp_cpu["x"], inp_cpu["W_r"], inp_cpu.get("logit_offset"))
    s_gpu = out["scores"].double().numpy()
    serr = np.max(np.abs(s_gpu - s_ref)) if T else 0.0
    assert serr <= score_tol, f"score error {serr:.2e}"

    sel_ref, gates_ref, gap = oracle.select_topk(s_ref, inp_cpu["bias"], k)
    sel = out["topk_idx"].numpy()
    w = out["topk_w"].double().numpy()
    keep = gap >= NEAR_TIE
    for t in np.nonzero(keep)[0]:
        assert set(sel[t].tolist()) == set(sel_ref[t].tolist()), f"token {t}"
        ref_w = dict(zip(sel_ref[t].tolist(), gates_ref[t].tolist()))
        for j in range(k):
            assert abs(w[t, j] - ref_w[int(sel[t, j])]) <= 1e-5
    # every token (excluded ones too): k distinct experts, slot order valid under the GPU's
    # own fp32 biased scores, weights sum to 1
    b = inp_cpu["bias"].numpy()
    for t in range(T):
        assert len(set(sel[t].tolist())) == k and sel[t].min() >= 0 and sel[t].max() < E
        v = (out["scores"][t].numpy() + b)[sel[t]]
        for j in range(k - 1):
            assert v[j] > v[j + 1] or (v[j] == v[j + 1] and sel[t, j] < sel[t, j + 1])
        rest = np.setdiff1d(np.arange(E), sel[t])
        if rest.size:
            vb = out["scores"][t].numpy() + b
            worst = v.min()
            assert np.all((vb[rest] < worst) | ((vb[rest] == worst) & (rest > sel[t][v == worst].max())))
        assert abs(w[t].sum() - 1.0) < 1e-5

    counts, offsets, perm, slot_pos = oracle.permutation(sel, E)
    assert np.array_equal(out["counts"].numpy(), counts)
    assert np.array_equal(out["offsets"].numpy(), offsets)
    assert np.array_equal(out["perm"].numpy()[:T * k], perm)
    assert np.array_equal(out["slot_pos"].numpy()[:T * k].reshape(T, k), slot_pos)
    return int((~keep).sum()), serr


@pytest.mark.parametrize("name", ["tiny", "mid"])
def test_route_configs(name):
    need_gpu()
    shp = synthetic.LAYERS[name]
    inp = synthetic.layer_inputs(shp, seed=0)
    excluded, serr = check_route(shp, inp, score_tol=SCORE_TOL)
    print(f"{name}: near-tie tokens excluded {excluded}/{shp.T}, max score err {serr:.2e}")


@pytest.mark.parametrize("over", [dict(T=1), dict(T=65, E=33, k=5), dict(T=130, E=4, k=4),
                                  dict(T=200, E=96, k=8), dict(T=3, E=1, k=1)])
def test_route_edge_shapes_f32(over):
    need_gpu()
    shp = synthetic.shape_with("tiny", **over)
    inp = synthetic.layer_inputs(shp, seed=1)
    check_route(shp, inp, score_tol=SCORE_TOL)


@pytest.mark.parametrize("over", [dict(T=1), dict(T=77, E=40, k=3), dict(T=300, E=256, k=16, d=512)])
def test_route_edge_shapes_bf16(over):
    need_gpu()
    shp = synthetic.shape_with("mid", **over)
    inp = synthetic.layer_inputs(shp, seed=2)
    check_route(shp, inp, score_tol=SCORE_TOL)


def test_route_exact_ties_and_saturated_scores():
    """All-equal scores pick the lowest indices; s = 1.0 exactly (saturated sigmoid) ties too."""
    need_gpu()
    shp = synthetic.shape_with("tiny", T=64, E=16, k=4)
    inp = synthetic.layer_inputs(shp, seed=3)
    inp["W_r"].zero_()
    out = run_route(lse.config(shp), to_dev(inp))
    assert np.all(out["scores"].numpy() == 0.5)
    assert np.array_equal(out["topk_idx"].numpy(), np.tile(np.arange(4), (64, 1)))
    assert np.allclose(out["topk_w"].numpy(), 0.25)
    mu = torch.zeros(16)
    mu[[3, 9, 12]] = 100.0                       # sigmoid saturates to exactly 1.0 in fp32
    inp["logit_offset"] = mu
    out = run_route(lse.config(shp), to_dev(inp))
    assert np.all(out["scores"].numpy()[:, [3, 9, 12]] == 1.0)
    assert np.array_equal(out["topk_idx"].numpy()[:, :3], np.tile([3, 9, 12], (64, 1)))
    assert np.all(out["topk_idx"].numpy()[:, 3] == 0)


def test_route_zero_token_experts_and_bias():
    """A large negative bias empties experts; counts are 0 and offsets stay monotone."""
    need_gpu()
    shp = synthetic.shape_with("tiny", T=64, E=16, k=2)
    inp = synthetic.layer_inputs(shp, seed=4)
    inp["bias"] = torch.zeros(16)
    inp["bias"][8:] = -10.0
    out = run_route(lse.config(shp), to_dev(inp))
    assert np.all(out["counts"].numpy()[8:] == 0)
    assert np.all(out["topk_idx"].numpy() < 8)
    check_route(shp, inp, score_tol=SCORE_TOL)


def test_route_nan_scores_are_counted():
    need_gpu()
    shp = synthetic.shape_with("tiny", T=8, E=16, k=2)
    inp = synthetic.layer_inputs(shp, seed=5)
    inp["x"][5, 0] = float("nan")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = run_route(lse.config(shp), to_dev(inp), status=status)
    assert int(status[0]) == 16
    assert np.array_equal(out["topk_idx"].numpy()[5], [0, 1])   # nothing but NaN: lowest index
    ref = oracle.router_scores(inp["x"][[0, 1, 2]], inp["W_r"])
    sel_ref, _, _ = oracle.select_topk(ref, inp["bias"][:], 2)
    assert np.array_equal(np.sort(out["topk_idx"].numpy()[[0, 1, 2]], 1), np.sort(sel_ref, 1))


def test_route_empty_batch():
    need_gpu()
    shp = synthetic.shape_with("tiny", T=0)
    cfg = lse.config(shp)
    counts = torch.full((16,), 7, dtype=torch.int32, device="cuda")
    offsets = torch.full((17,), 7, dtype=torch.int32, device="cuda")
    ws = torch.empty(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    lse.slmoe_route(cfg, None, None, None, None, None, None, None, counts, offsets, None, None, None,
                    None, ws)
    torch.cuda.synchronize()
    assert counts.sum().item() == 0 and offsets.sum().item() == 0


def gpu_topk(scores, bias, k, status=None):
    """slmoe_topk through the C ABI on a [T, E] fp32 score matrix already on the device."""
    T, E = scores.shape
    b = route_buffers(T, E, k)
    del b["scores"]
    ws = torch.empty(lse.slmoe_topk_workspace_size(T, E, k), dtype=torch.uint8, device="cuda")
    lse.slmoe_topk(scores, bias, T, E, k, b["topk_idx"], b["topk_w"], b["counts"], b["offsets"],
                   b["perm"], b["slot_pos"], status, ws)
    torch.cuda.synchronize()
    return {n: v.cpu().numpy() for n, v in b.items()}


def check_topk_call(scores, bias, k, near_tie_bound):
    out = gpu_topk(scores, bias, k)
    s_ref = scores.double().cpu().numpy()          # the very fp32 scores, widened exactly
    return check_selection_and_permutation(
        s_ref, scores, bias, out["topk_idx"], out["topk_w"], out["counts"], out["offsets"],
        out["perm"], out["slot_pos"], 0.0, near_tie_bound), out


@pytest.mark.parametrize("micro_batch,bias_std", [(0, 0.0), (1, 0.05)])
def test_topk_from_scores_at_the_qb_engine_size(micro_batch, bias_std):
    """65536 tokens x 896 experts, top-16, from the QB engine's fp32 scores."""
    need_gpu()
    q = synthetic.QB
    sc = synthetic.qb_scores(micro_batch, q, device="cuda")
    g = torch.Generator(device="cpu").manual_seed(77 + micro_batch)
    bias = (torch.randn(q.E, generator=g) * bias_std).cuda()
    (n_tie, _), out = check_topk_call(sc, bias, q.k, int(0.05 * q.T))
    assert out["counts"].sum() == q.T * q.k
    print(f"QB-engine top-k: near-tie tokens {n_tie}/{q.T}")


@pytest.mark.parametrize("T,E,k", [(1, 896, 16), (333, 7, 3), (100, 64, 32), (5, 4096, 32),
                                   (1000, 1, 1), (4097, 300, 10)])
def test_topk_from_scores_edge_shapes(T, E, k):
    need_gpu()
    g = torch.Generator(device="cpu").manual_seed(T * 31 + E)
    sc = torch.sigmoid(torch.randn(T, E, generator=g)).cuda()
    bias = (torch.randn(E, generator=g) * 0.1).cuda()
    check_topk_call(sc, bias, k, T)


def test_topk_exact_ties_nan_and_empty():
    need_gpu()
    T, E, k = 40, 16, 4
    sc = torch.full((T, E), 0.5, device="cuda")
    sc[3, 5] = float("nan")
    bias = torch.zeros(E, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = gpu_topk(sc, bias, k, status)
    assert int(status[0]) == 1
    exp = np.tile(np.arange(4), (T, 1))
    assert np.array_equal(out["topk_idx"], exp)
    assert np.allclose(out["topk_w"], 0.25)
    ws = torch.empty(lse.slmoe_topk_workspace_size(0, E, k), dtype=torch.uint8, device="cuda")
    counts = torch.full((E,), 3, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), 3, dtype=torch.int32, device="cuda")
    lse.slmoe_topk(None, None, 0, E, k, None, None, counts, offsets, None, None, None, ws)
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0


def test_route_k3_router_shape():
    """slmoe_route at the K3 router's widths (d = 7168, E = 896, k = 16) with a ragged
    number of tokens: the top-k kernel's looping path for large E and several scan chunks."""
    need_gpu()
    shp = synthetic.shape_with("k3_decode", T=1000, d_latent=64, I=64, n_shared=0)
    inp = synthetic.layer_inputs(shp, seed=9)
    excluded, serr = check_route(shp, inp, score_tol=SCORE_TOL)
    assert excluded <= 0.05 * shp.T
    print(f"K3 router shape: near-tie tokens excluded {excluded}/{shp.T}, max score err {serr:.2e}")
