"""GPU parity of the Quantile Balancing engine: histogram counts bit-exact against the oracle
on the same fp32 scores, quantiles and biases within 1e-6 (both in fp64 from identical counts)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
import latent_space_experts_gb300 as lse
from gpu_util import need_gpu, run_route, to_dev
from test_gpu_route import check_topk_call

pytestmark = pytest.mark.gpu


def gpu_hist(scores, nbins=1000, hist=None, status=None):
    T, E = scores.shape
    if hist is None:
        hist = torch.zeros(E, nbins, dtype=torch.int32, device="cuda")
    lse.slmoe_qb_histogram(scores, T, E, nbins, hist, status)
    return hist


def test_qb_engine_full_size_eight_micro_batches():
    """65536 tokens x 896 experts per micro-batch, 8 micro-batches added in place, then the
    (1 - 16/896) quantile and the bias update."""
    need_gpu()
    q = synthetic.QB
    hist = torch.zeros(q.E, q.nbins, dtype=torch.int32, device="cuda")
    ref = np.zeros((q.E, q.nbins), dtype=np.uint64)
    for m in range(q.micro_batches):
        s = synthetic.qb_scores(m, q, device="cuda")
        gpu_hist(s, q.nbins, hist)
        ref = oracle.qb_histogram(s.cpu().numpy(), q.nbins, ref)
    torch.cuda.synchronize()
    h = hist.cpu().numpy().view(np.uint32).astype(np.uint64)
    assert np.array_equal(h, ref)
    assert np.all(h.sum(axis=1) == q.T * q.micro_batches)
    q_out = torch.empty(q.E, device="cuda")
    bias = torch.empty(q.E, device="cuda")
    lse.slmoe_qb_update(hist, q.E, q.nbins, q.k, q_out, bias)
    q_ref, b_ref = oracle.qb_update(ref, q.k)
    assert np.max(np.abs(q_out.cpu().numpy() - q_ref)) <= 1e-6
    assert np.max(np.abs(bias.cpu().numpy() - b_ref)) <= 1e-6


@pytest.mark.parametrize("T,E,nbins", [(1, 1, 1000), (1000, 33, 1000), (5000, 64, 999), (777, 100, 10),
                                       (200000, 40, 1000), (3, 2048, 1000), (2000, 70, 1024),
                                       (3000, 600, 1000), (5, 4096, 1000), (4000, 300, 7)])
def test_histogram_shapes(T, E, nbins):
    """Bit-exact bins against the oracle over expert counts that give the launch different
    cluster sizes (1 to 32 expert slabs and more: the cluster size follows from how many
    clusters fit at once), ragged last slabs, few and many tokens per CTA, and bin counts
    whose rows split unevenly over a cluster's CTAs."""
    need_gpu()
    g = torch.Generator(device="cpu").manual_seed(T + E)
    s = torch.rand(T, E, generator=g, dtype=torch.float32)
    s[0, 0] = 0.0
    s[-1, -1] = 1.0
    hist = gpu_hist(s.cuda(), nbins)
    torch.cuda.synchronize()
    assert np.array_equal(hist.cpu().numpy().view(np.uint32), oracle.qb_histogram(s.numpy(), nbins))


def test_histogram_edges_and_nan():
    need_gpu()
    edges = (np.arange(0, 1001) / 1000.0).astype(np.float32)
    vals = np.concatenate([edges, np.nextafter(edges, np.float32(0)), np.nextafter(edges, np.float32(2)),
                           [np.nan, np.nan]]).astype(np.float32)
    vals = np.clip(np.nan_to_num(vals, nan=-1.0), 0, 1).astype(np.float32)
    vals[-2:] = np.nan
    s = np.stack([vals, vals[::-1]], axis=1).copy()
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    hist = gpu_hist(torch.from_numpy(s).cuda(), 1000, status=status)
    torch.cuda.synchronize()
    assert np.array_equal(hist.cpu().numpy().view(np.uint32), oracle.qb_histogram(s, 1000))
    assert int(status[0]) == 4


@pytest.mark.parametrize("T,E", [(4099, 96), (1000, 896)])
def test_histogram_edges_nan_and_alignment_match_the_oracle(T, E):
    """Bin edges, out-of-range values and NaN spread over rows and experts, at a shape whose
    rows do not divide evenly among a cluster's CTAs, from a 16-byte aligned matrix and from
    the same values one float further on (4-byte aligned)."""
    need_gpu()
    g = torch.Generator(device="cpu").manual_seed(T * 7 + E)
    s = torch.rand(T, E, generator=g, dtype=torch.float32)
    edges = torch.arange(0, 1001, dtype=torch.float32) / 1000
    s.view(-1)[:edges.numel()] = edges
    s.view(-1)[edges.numel():2 * edges.numel()] = torch.nextafter(edges, torch.zeros(()))
    s[5, :] = float("nan")
    s[T - 1, 3] = float("nan")
    s[:, 7] = 1.0
    s[9, 3], s[10, 4] = -0.5, 2.0
    ref = oracle.qb_histogram(s.numpy(), 1000)
    n_nan = int(torch.isnan(s).sum())
    aligned = s.cuda()
    buf = torch.empty(T * E + 1, dtype=torch.float32, device="cuda")
    buf[1:] = aligned.view(-1)
    shifted = buf[1:].view(T, E)
    assert aligned.data_ptr() % 16 == 0 and shifted.data_ptr() % 16 == 4
    for x in (aligned, shifted):
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
        hist = gpu_hist(x, 1000, status=status)
        torch.cuda.synchronize()
        assert np.array_equal(hist.cpu().numpy().view(np.uint32), ref)
        assert int(status[0]) == n_nan and int(status[1]) == 0


def test_update_closed_forms_on_gpu():
    need_gpu()
    E, k = 8, 2
    uni = torch.ones(E, 1000, dtype=torch.int32, device="cuda")
    q_out = torch.empty(E, device="cuda")
    bias = torch.empty(E, device="cuda")
    lse.slmoe_qb_update(uni, E, 1000, k, q_out, bias)
    assert np.allclose(q_out.cpu().numpy(), 1 - k / E, atol=1e-7)
    assert np.allclose(bias.cpu().numpy(), 0.0, atol=1e-7)
    empty = torch.zeros(E, 1000, dtype=torch.int32, device="cuda")
    lse.slmoe_qb_update(empty, E, 1000, k, q_out, bias)
    assert np.all(q_out.cpu().numpy() == 0.0)


def test_fused_route_histogram_matches_standalone():
    """slmoe_route(hist=...) bins the GPU's own fp32 scores: identical to binning them on the host."""
    need_gpu()
    shp = synthetic.LAYERS["mid"]
    inp = to_dev(synthetic.layer_inputs(shp, seed=0))
    hist = torch.zeros(shp.E, shp.nbins, dtype=torch.int32, device="cuda")
    out = run_route(lse.config(shp), inp, hist=hist)
    ref = oracle.qb_histogram(out["scores"].numpy(), shp.nbins)
    assert np.array_equal(hist.cpu().numpy().view(np.uint32), ref)


def test_qb_rebalances_k3_routing():
    """Route 8 micro-batches of K3-shaped scores, update the bias by QB, route a held-out
    micro-batch on the GPU (slmoe_topk) with no bias and with the QB bias: each routing is
    checked against the oracle's selection, and max/mean load is reported before and after
    (the pages fix no target value)."""
    need_gpu()
    q = synthetic.QB
    T = 8192
    hist = torch.zeros(q.E, q.nbins, dtype=torch.int32, device="cuda")
    for m in range(q.micro_batches):
        gpu_hist(synthetic.qb_scores(m, q, device="cuda", T=T), q.nbins, hist)
    bias = torch.empty(q.E, device="cuda")
    lse.slmoe_qb_update(hist, q.E, q.nbins, q.k, None, bias)
    held = synthetic.qb_scores(q.micro_batches, q, device="cuda", T=T)
    ratios = []
    for b in (torch.zeros(q.E, device="cuda"), bias):
        (_, _), out = check_topk_call(held, b, q.k, int(0.05 * T))
        L = out["counts"]
        assert L.sum() == T * q.k
        ratios.append(L.max() / L.mean())
    print(f"max/mean load before QB {ratios[0]:.2f}, after {ratios[1]:.2f}")
    assert ratios[1] < ratios[0]


def signsgd_case(E, seed, big=False):
    """Counts with an exact integer mean m that many experts hit exactly (zero-sum
    deviations around m), so all three branches of the rule are taken; biases with -0.0."""
    rng = np.random.default_rng(seed)
    m = (1 << 28) if big else 3000
    dev = np.zeros(E, np.int64)
    half = rng.integers(-2000, 2001, size=E // 2)
    half[rng.random(E // 2) < 0.3] = 0
    dev[0:2 * (E // 2):2], dev[1:2 * (E // 2):2] = half, -half      # pairs +d, -d: sum 0
    dev = rng.permutation(dev)
    n = m + dev
    assert n.min() >= 0 and n.max() < 2**31
    b = rng.normal(scale=0.05, size=E).astype(np.float32)
    b[::5] = -0.0
    return n.astype(np.int32), b


@pytest.mark.parametrize("E,big", [(1, False), (7, False), (896, False), (1000, False),
                                   (8, True), (65536, False)])
def test_signsgd_update_matches_the_oracle_bit_for_bit(E, big):
    need_gpu()
    n, b0 = signsgd_case(E, seed=E, big=big)
    step = np.float32(1e-3)
    counts = torch.from_numpy(n).cuda()
    bias = torch.from_numpy(b0.copy()).cuda()
    lse.slmoe_signsgd_update(counts, E, float(step), bias)
    ref = oracle.signsgd_update(n, b0, step)
    assert np.array_equal(bias.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    moved = (bias.cpu().numpy().view(np.uint32) != b0.view(np.uint32)).sum()
    assert moved == int((n.astype(np.int64) * E != int(n.astype(np.int64).sum())).sum())


def test_signsgd_loop_on_k3_micro_batches_follows_the_oracle():
    """Eight micro-batches of K3-shaped scores (E = 896, k = 16): each is routed with the
    current bias (top-k on the host, test infrastructure), its loads feed one fixed-step
    update on the GPU, and the GPU bias follows the oracle's bit for bit.  On a held-out
    micro-batch the max/mean load is reported for no balancing, the fixed-step rule and QB
    (one update from the same eight histograms); the pages fix no target value."""
    need_gpu()
    q = synthetic.QB
    T, step = 8192, np.float32(1e-3)
    bias_g = torch.zeros(q.E, device="cuda")
    bias_o = np.zeros(q.E, np.float32)
    hist = torch.zeros(q.E, q.nbins, dtype=torch.int32, device="cuda")
    for m in range(q.micro_batches):
        sc = synthetic.qb_scores(m, q, device="cuda", T=T)
        gpu_hist(sc, q.nbins, hist)
        sel, _, _ = oracle.select_topk(sc.cpu().numpy(), bias_o, q.k)
        L = oracle.expert_loads(sel, q.E).astype(np.int32)
        assert L.sum() == T * q.k
        # the GPU routes the same micro-batch with its own (bit-identical) bias: its selection
        # matches the oracle's outside near ties
        check_topk_call(sc, bias_g, q.k, int(0.05 * T))
        lse.slmoe_signsgd_update(torch.from_numpy(L).cuda(), q.E, float(step), bias_g)
        bias_o = oracle.signsgd_update(L, bias_o, step)
        assert np.array_equal(bias_g.cpu().numpy().view(np.uint32), bias_o.view(np.uint32)), m
    qbias = torch.empty(q.E, device="cuda")
    lse.slmoe_qb_update(hist, q.E, q.nbins, q.k, None, qbias)
    held = synthetic.qb_scores(q.micro_batches, q, device="cuda", T=T).cpu().numpy()
    ratios = {}
    for name, b in (("none", np.zeros(q.E)), ("fixed step", bias_o), ("QB", qbias.cpu().numpy())):
        sel, _, _ = oracle.select_topk(held, b, q.k)
        L = oracle.expert_loads(sel, q.E)
        assert L.sum() == T * q.k
        ratios[name] = L.max() / L.mean()
    print("max/mean load on a held-out micro-batch:", {k: round(v, 2) for k, v in ratios.items()})
    assert ratios["QB"] < ratios["none"]
