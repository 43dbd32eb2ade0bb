"""GPU parity of slmoe_backward against the oracle's fp64 backward.

The forward runs first (slmoe_forward); the oracle takes the GPU's selection (forced routing)
and computes every gradient in fp64 from the exact inputs, without emulating the bf16
roundings of the GPU's intermediates.  End to end, each gradient must be within a relative
Frobenius error of 1e-2 and a max error of 0.1 RMS(ref) (gpu_util.BWD_FRO / BWD_MAX: four bf16
roundings lie between the inputs and a gradient).  Each stage is also checked on its own, from
the GPU's own inputs of that stage, at 2e-3 RMS (exact bf16 products, fp32 sums), with the
mid workload's x outliers (1 % of x scaled by 50) that push the gates into saturation.
Gradient accumulation across micro-batches (accumulate = 1) must add the micro-batches'
gradients, while the forward's QB histograms add in the same way.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import latent_space_experts_gb300 as lse
from gpu_util import BF16_STORE, assert_close_grad, assert_close_rms, need_gpu, to_dev

pytestmark = pytest.mark.gpu

GRADS = ("dW_r", "dW_in", "dW13", "dW2", "dgamma", "dW_out", "dW13_s", "dW2_s")
WEIGHT_OF = dict(dW_r="W_r", dW_in="W_in", dW13="W13", dW2="W2", dgamma="gamma", dW_out="W_out",
                 dW13_s="W13_s", dW2_s="W2_s")


def zero_grads(inp):
    return {g: torch.zeros(inp[w].shape, dtype=torch.float32, device="cuda") for g, w in WEIGHT_OF.items()}


def forward_backward(shape, inp, dy, grads, accumulate, hist=None):
    cfg = lse.config(shape)
    ws = torch.zeros(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty(shape.T, shape.d, dtype=torch.float32, device="cuda")
    topk = torch.empty(shape.T, shape.k, dtype=torch.int32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    W = lse.weights(inp)
    lse.slmoe_forward(cfg, inp["x"], W, inp["bias"], inp.get("logit_offset"), y, topk, hist, status, ws)
    bws = torch.zeros(lse.slmoe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    dx = torch.full((shape.T, shape.d), float("nan"), dtype=torch.float32, device="cuda")
    lse.slmoe_backward(cfg, inp["x"], W, dy, dx, lse.grads(grads), accumulate, ws, status, bws)
    torch.cuda.synchronize()
    assert status.cpu().tolist()[1:3] == [0, 0], status
    return y, topk.cpu().numpy(), dx


def layer(over, seed):
    over = dict(over)
    over.setdefault("x_outliers", False)
    shp = synthetic.shape_with("mid", **over)
    inp_cpu = synthetic.layer_inputs(shp, seed=seed)
    g = torch.Generator().manual_seed(100 + seed)
    dy = torch.randn(shp.T, shp.d, generator=g)
    return shp, inp_cpu, dy


def err_stats(got, ref):
    got = got.detach().double().cpu().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    err = np.abs(got - ref)
    r = float(np.sqrt(np.mean(ref * ref)))
    if r == 0.0:
        return float(err.max()), float(err.max())
    return float(err.max()) / r, float(np.max(err / (np.abs(ref) + r)))


def check_grads(shp, inp_cpu, dy_cpu, dx, grads, topk, scale=1.0, what="", skip=()):
    ref = oracle.backward(inp_cpu, shp.k, dy_cpu.double().numpy(), forced_topk_idx=topk)
    pairs = [("dx", dx, ref["dx"])] + [(n, grads[n], scale * ref[n]) for n in GRADS
                                       if n not in skip and not (n in ("dW13_s", "dW2_s") and shp.n_shared == 0)]
    print(what, {n: "max/RMS %.2e, max/(|ref|+RMS) %.2e" % err_stats(g, r) for n, g, r in pairs})
    for n, g, r in pairs:
        assert_close_grad(g, r, f"{what} {n}")
    return ref


@pytest.mark.parametrize("over,seed", [
    (dict(T=300, d=512), 0),                                     # several tiles, ragged T
    (dict(T=130, d=256, d_latent=384, E=8, k=8, I=128), 1),      # k = E, ragged latent tiles
    (dict(T=77, d=512, E=40, k=3, I=192, n_shared=0), 2),        # experts without tokens, no shared
    (dict(T=600, d=512, E=2, k=1, I=384, n_shared=3, I_shared=320), 3),   # > 256 rows per expert
])
def test_backward_matches_the_oracle(over, seed):
    need_gpu()
    shp, inp_cpu, dy = layer(over, seed)
    inp = to_dev(inp_cpu)
    grads = zero_grads(inp)
    for g in grads.values():
        g.fill_(float("nan"))              # accumulate = 0 must overwrite every element
    _, topk, dx = forward_backward(shp, inp, dy.cuda(), grads, 0)
    check_grads(shp, inp_cpu, dy, dx, grads, topk, what=str(over))


def test_backward_accumulates_across_micro_batches_with_the_qb_histogram():
    """Two micro-batches: weight gradients added in place (accumulate = 1 after a first call
    with 0), and the forward's QB histograms of the two batches added in place, as gradient
    accumulation does ([K3-arch] 负载均衡优化: the distribution adds across accumulation steps)."""
    need_gpu()
    shp = synthetic.shape_with("mid", T=200, d=512, x_outliers=False)
    inps = [synthetic.layer_inputs(shp, seed=s) for s in (5, 5)]
    # the same weights, different tokens and output gradients for the second micro-batch
    g = torch.Generator().manual_seed(9)
    inps[1]["x"] = torch.randn(shp.T, shp.d, generator=g).to(torch.bfloat16)
    dys = [torch.randn(shp.T, shp.d, generator=g) for _ in range(2)]
    grads = zero_grads(to_dev(inps[0]))
    hist = torch.zeros(shp.E, shp.nbins, dtype=torch.int32, device="cuda")
    refs = []
    for m in range(2):
        inp = to_dev(inps[m])
        _, topk, dx = forward_backward(shp, inp, dys[m].cuda(), grads, 1 if m else 0, hist=hist)
        ref = oracle.backward(inps[m], shp.k, dys[m].double().numpy(), forced_topk_idx=topk)
        assert_close_grad(dx, ref["dx"], f"dx micro-batch {m}")
        refs.append(ref)
    for name in GRADS:
        assert_close_grad(grads[name], refs[0][name] + refs[1][name], f"accumulated {name}")
    h = hist.cpu().numpy().view(np.uint32).astype(np.int64)
    assert np.all(h.sum(axis=1) == 2 * shp.T)


def test_backward_of_identical_experts_gives_no_router_gradient():
    """All routed experts equal: the gate weights sum to 1, so the router gradient vanishes
    (up to bf16 rounding) while the expert gradients do not."""
    need_gpu()
    shp, inp_cpu, dy = layer(dict(T=256, d=512), 6)
    inp_cpu["W13"][:] = inp_cpu["W13"][0]
    inp_cpu["W2"][:] = inp_cpu["W2"][0]
    inp = to_dev(inp_cpu)
    grads = zero_grads(inp)
    _, topk, dx = forward_backward(shp, inp, dy.cuda(), grads, 0)
    ref = check_grads(shp, inp_cpu, dy, dx, grads, topk, what="identical experts", skip=("dW_r",))
    assert np.max(np.abs(ref["dW_r"])) < 1e-12
    assert float(grads["dW_r"].abs().max()) <= 1e-3 * float(grads["dW_in"].abs().max())


SAME = 2e-3     # stage checks from the GPU's own operands: exact bf16 products, fp32 sums


def f64(t):
    return t.detach().double().cpu().numpy()


def bf16_round(a):
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16).double().numpy()


def check_backward_stages(shp, inp, fw, bw, grads, dy, experts):
    """Each backward stage against the oracle's formula applied to the GPU's own inputs of
    that stage (so a stage is judged on its own arithmetic, not on the roundings before it)."""
    T, k, I = shp.T, shp.k, shp.I
    perm, offsets = f64(fw["perm"]).astype(np.int64), f64(fw["offsets"]).astype(np.int64)
    slot_pos = f64(fw["slot_pos"]).astype(np.int64).reshape(T, k)
    dy_b = bf16_round(f64(dy))
    W_out = oracle.f64(inp["W_out"])
    assert_close_rms(bw["dz"], dy_b @ W_out, SAME, "stage dz")
    assert_close_rms(grads["dW_out"], dy_b.T @ f64(fw["z"]), SAME, "stage dW_out")
    # norm + combine backward from the GPU's y_e and gates
    ye = f64(fw["y_e"])
    gw = f64(fw["topk_w"])
    c = np.einsum("tj,tjd->td", gw, ye[slot_pos])
    dc, dgamma = oracle.rmsnorm_backward(c, inp["gamma"], f64(bw["dz"]), shp.eps)
    assert_close_rms(grads["dgamma"], dgamma, SAME, "stage dgamma")
    dye_ref = np.zeros_like(ye)
    dye_ref[slot_pos.reshape(-1)] = (gw[:, :, None] * dc[:, None, :]).reshape(T * k, -1)
    assert_close_rms(bw["dye"], dye_ref, SAME, "stage dy_e", BF16_STORE)
    # dg = dc . y_e: judged against the scale of such a dot product (it vanishes for k = 1,
    # where the norm makes the output independent of the scale of c = y_e)
    dg_ref = np.einsum("td,tjd->tj", dc, ye[slot_pos])
    scale = float(np.sqrt(np.mean(dc * dc) * np.mean(ye * ye) * dc.shape[1]))
    assert np.max(np.abs(f64(bw["dg"]) - dg_ref)) <= SAME * scale, "stage dg"
    xl = f64(fw["x_lat"])
    h = f64(fw["h"])
    dye = f64(bw["dye"])
    gu = f64(bw["gu"])
    dgu = f64(bw["dgu"])
    for e in experts:
        p = np.arange(offsets[e], offsets[e + 1])
        if p.size == 0:
            continue
        W13, W2 = oracle.f64(inp["W13"][int(e)]), oracle.f64(inp["W2"][int(e)])
        assert_close_rms(gu[p], xl[perm[p]] @ W13.T, SAME, f"stage gu expert {e}")
        dgu_ref = oracle.situ_glu_backward(gu[p], dye[p] @ W2)
        assert_close_rms(dgu[p], dgu_ref, SAME, f"stage dgu expert {e}", BF16_STORE)
        assert_close_rms(grads["dW2"][int(e)], dye[p].T @ h[p], SAME, f"stage dW2 expert {e}")
        assert_close_rms(grads["dW13"][int(e)], dgu[p].T @ xl[perm[p]], SAME, f"stage dW13 expert {e}")
    # x_lat gradient: each row's W13[e]^T dgu summed over the token's slots
    dxe = np.zeros((T * k, xl.shape[1]))
    for e in np.unique(np.searchsorted(offsets, np.arange(T * k), side="right") - 1):
        p = np.arange(offsets[e], offsets[e + 1])
        dxe[p] = dgu[p] @ oracle.f64(inp["W13"][int(e)])
    dx_lat_ref = dxe[slot_pos].sum(axis=1)
    assert_close_rms(bw["dx_lat"], dx_lat_ref, SAME, "stage dx_lat", BF16_STORE)
    x = oracle.f64(inp["x"])
    assert_close_rms(grads["dW_in"], f64(bw["dx_lat"]).T @ x, SAME, "stage dW_in")
    if shp.n_shared:
        s = shp.n_shared - 1
        W13s, W2s = oracle.f64(inp["W13_s"][s]), oracle.f64(inp["W2_s"][s])
        gus = f64(bw["gu_s"])
        assert_close_rms(gus, x @ W13s.T, SAME, "stage gu_s")
        assert_close_rms(bw["dgu_s"], oracle.situ_glu_backward(gus, dy_b @ W2s), SAME, "stage dgu_s", BF16_STORE)
        assert_close_rms(grads["dW13_s"][s], f64(bw["dgu_s"]).T @ x, SAME, "stage dW13_s")
        hs = f64(fw["h_s"])[:, s * shp.I_shared:(s + 1) * shp.I_shared]
        assert_close_rms(grads["dW2_s"][s], dy_b.T @ hs, SAME, "stage dW2_s")


@pytest.mark.parametrize("over,seed", [(dict(T=300, d=512, x_outliers=True), 0),
                                       (dict(T=77, d=512, E=40, k=3, I=192, x_outliers=True), 2),
                                       (dict(T=600, d=512, E=2, k=1, I=384, n_shared=3, I_shared=320), 3)])
def test_backward_stages(over, seed):
    need_gpu()
    shp, inp_cpu, dy = layer(over, seed)
    inp = to_dev(inp_cpu)
    grads = zero_grads(inp)
    cfg = lse.config(shp)
    ws = torch.zeros(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty(shp.T, shp.d, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    W = lse.weights(inp)
    lse.slmoe_forward(cfg, inp["x"], W, inp["bias"], inp["logit_offset"], y, None, None, status, ws)
    bws = torch.zeros(lse.slmoe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    dx = torch.empty(shp.T, shp.d, dtype=torch.float32, device="cuda")
    dyd = dy.cuda()
    lse.slmoe_backward(cfg, inp["x"], W, dyd, dx, lse.grads(grads), 0, ws, status, bws)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    check_backward_stages(shp, inp_cpu, lse.workspace_views(cfg, ws), lse.backward_views(cfg, bws), grads, dyd,
                          range(shp.E))


def test_backward_k3_prefill_sampled():
    """The K3 prefill layer (T = 8192, E = 896, k = 16): dx of sampled tokens against the
    oracle's backward of those tokens (end to end, forced routing), and the stages of the
    hottest, coldest and some random experts, of sampled tokens and of sampled weight rows,
    from the GPU's own inputs of each stage."""
    need_gpu()
    shp = synthetic.LAYERS["k3_prefill"]
    inp = synthetic.layer_inputs(shp, seed=0, device="cuda")
    T, k, d, dl = shp.T, shp.k, shp.d, shp.d_latent
    g = torch.Generator(device="cuda").manual_seed(3)
    dy = torch.randn(T, d, generator=g, device="cuda")
    grads = zero_grads(inp)
    cfg = lse.config(shp)
    ws = torch.zeros(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty(T, d, dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    W = lse.weights(inp)
    lse.slmoe_forward(cfg, inp["x"], W, inp["bias"], inp["logit_offset"], y, None, None, status, ws)
    bws = torch.zeros(lse.slmoe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    dx = torch.empty(T, d, dtype=torch.float32, device="cuda")
    lse.slmoe_backward(cfg, inp["x"], W, dy, dx, lse.grads(grads), 0, ws, status, bws)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    fw, bw = lse.workspace_views(cfg, ws), lse.backward_views(cfg, bws)
    rng = np.random.default_rng(4)
    tok = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 30, replace=False)]))
    topk = fw["topk_idx"].cpu().numpy()
    ref = oracle.backward(inp, k, dy, forced_topk_idx=topk, tokens=tok)
    fro, mx = assert_close_grad(dx[torch.as_tensor(tok, device="cuda")], ref["dx"], "K3 dx")
    print(f"K3 prefill dx on {len(tok)} tokens: Frobenius {fro:.2e}, max/RMS {mx:.2e}")
    # stages from the GPU's own inputs
    perm = fw["perm"].cpu().numpy().astype(np.int64)
    offsets = fw["offsets"].cpu().numpy().astype(np.int64)
    counts = np.diff(offsets)
    used = np.nonzero(counts > 0)[0]
    experts = np.unique(np.concatenate([np.argsort(-counts, kind="stable")[:3],
                                        [e for e in used if counts[e] <= 3][:3], rng.choice(used, 4, replace=False)]))
    slot_pos = fw["slot_pos"].cpu().numpy().astype(np.int64).reshape(T, k)
    tok_d = torch.as_tensor(tok, device="cuda")
    dy_b = bf16_round(f64(dy[tok_d]))
    assert_close_rms(bw["dz"][tok_d], dy_b @ oracle.f64(inp["W_out"]), SAME, "K3 stage dz")
    rows = rng.choice(d, 16, replace=False)
    dyb_all = dy.to(torch.bfloat16).double()
    assert_close_rms(grads["dW_out"][torch.as_tensor(rows, device="cuda")],
                     f64(dyb_all[:, torch.as_tensor(rows, device="cuda")].T @ fw["z"].double()), SAME, "K3 stage dW_out")
    ye_tok = f64(fw["y_e"][torch.as_tensor(slot_pos[tok].reshape(-1), device="cuda")]).reshape(len(tok), k, dl)
    gw = f64(fw["topk_w"][tok_d])
    c = np.einsum("tj,tjd->td", gw, ye_tok)
    dc, _ = oracle.rmsnorm_backward(c, inp["gamma"], f64(bw["dz"][tok_d]), shp.eps)
    dye_tok = f64(bw["dye"][torch.as_tensor(slot_pos[tok].reshape(-1), device="cuda")]).reshape(len(tok), k, dl)
    assert_close_rms(dye_tok, gw[:, :, None] * dc[:, None, :], SAME, "K3 stage dy_e", BF16_STORE)
    for e in experts:
        p = np.arange(offsets[e], offsets[e + 1])
        pd = torch.as_tensor(p, device="cuda")
        xl = f64(fw["x_lat"][torch.as_tensor(perm[p], device="cuda")])
        W13, W2 = oracle.f64(inp["W13"][int(e)]), oracle.f64(inp["W2"][int(e)])
        gu, dye, dgu = f64(bw["gu"][pd]), f64(bw["dye"][pd]), f64(bw["dgu"][pd])
        assert_close_rms(gu, xl @ W13.T, SAME, f"K3 stage gu expert {e}")
        assert_close_rms(dgu, oracle.situ_glu_backward(gu, dye @ W2), SAME, f"K3 stage dgu expert {e}", BF16_STORE)
        assert_close_rms(grads["dW2"][int(e)], dye.T @ f64(fw["h"][pd]), SAME, f"K3 stage dW2 expert {e}")
        assert_close_rms(grads["dW13"][int(e)], dgu.T @ xl, SAME, f"K3 stage dW13 expert {e}")
    print(f"K3 prefill backward stages checked on experts {experts.tolist()} (loads {counts[experts].tolist()})")
