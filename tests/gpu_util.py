"""Helpers shared by the GPU parity tests (no arithmetic of the method lives here)."""
import numpy as np
import pytest
import torch

import latent_space_experts_gb300 as lse

NEAR_TIE = 1e-5          # tokens whose oracle k-th/(k+1)-th biased gap is below this are excluded
BF16_TOL = 2e-2          # max|err| <= 2e-2 * RMS(ref) on bf16 paths
F32_TOL = 1e-4           # max|err| <= 1e-4 * RMS(ref) on fp32 paths
BF16_STORE = 2.0 ** -7   # extra elementwise allowance for intermediates stored in bf16
# Backward gradients pass through up to four bf16 roundings (dy, dy_e, [dg | du], dx_lat; and
# the forward's stored x_lat, h, y_e, z): relative RMS error about 2^-9 * sqrt(4) / sqrt(3) =
# 2.3e-3 per product.  Held to a relative Frobenius error of 1e-2 and a max error of 0.1 RMS.
BWD_FRO = 1e-2
BWD_MAX = 0.1


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    lse.build()
    lse.load()


def to_dev(inp, device="cuda"):
    return {k: (v.to(device) if v is not None else None) for k, v in inp.items()}


def rms(a):
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a)))


def assert_close_rms(got, ref, tol, what="", rel=0.0):
    """max|got - ref| <= tol * RMS(ref), elementwise widened by rel * |ref| when rel > 0.

    rel > 0 is used only for intermediates that the bf16 layer stores in bf16 (x_lat, h,
    y_e, z): their storage alone rounds by up to 2^-9 |value|.  The layer output y is held to
    the plain bound.
    """
    got = got.detach().float().cpu().double().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    if not got.size:
        return 0.0
    err = np.abs(got - ref)
    bound = tol * rms(ref) + rel * np.abs(ref)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (f"{what}: |err| {err.flat[worst]:.3e} > bound {bound.flat[worst]:.3e} "
                                  f"at {np.unravel_index(worst, err.shape)} (ref {ref.flat[worst]:.4e}, "
                                  f"RMS {rms(ref):.3e})")
    return float(err.max()) / max(rms(ref), 1e-300)


def route_buffers(T, E, k, device="cuda"):
    return dict(topk_idx=torch.empty(T, k, dtype=torch.int32, device=device),
                topk_w=torch.empty(T, k, dtype=torch.float32, device=device),
                scores=torch.empty(T, E, dtype=torch.float32, device=device),
                counts=torch.empty(E, dtype=torch.int32, device=device),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=device),
                perm=torch.empty(max(T * k, 1), dtype=torch.int32, device=device),
                slot_pos=torch.empty(max(T * k, 1), dtype=torch.int32, device=device))


def run_route(cfg, inp, hist=None, status=None):
    T, E, k = cfg.T, cfg.E, cfg.k
    b = route_buffers(T, E, k)
    ws = torch.empty(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    lse.slmoe_route(cfg, inp["x"], inp["W_r"], inp["bias"], inp.get("logit_offset"), b["topk_idx"],
                    b["topk_w"], b["scores"], b["counts"], b["offsets"], b["perm"], b["slot_pos"],
                    hist, status, ws)
    torch.cuda.synchronize()
    return {n: v.cpu() for n, v in b.items()}


def host(a):
    """A numpy copy of a torch tensor (any device) or an array-like."""
    if hasattr(a, "detach"):
        return a.detach().cpu().numpy()
    return np.asarray(a)


def check_topk_valid(scores_f32, bias_f32, sel, w):
    """Every token's selection is a valid biased top-k under the GPU's own fp32 scores, with
    the stated rules (vectorised over tokens): k distinct experts, slots ordered by fp32
    biased score descending with ties to the lower index, every unchosen expert below the
    weakest chosen one (or equal to it with a higher index), gate weights summing to 1."""
    s = host(scores_f32).astype(np.float32)
    T, E = s.shape
    k = sel.shape[1]
    if T == 0:
        return
    assert sel.min() >= 0 and sel.max() < E
    vb = s + host(bias_f32).astype(np.float32)[None, :]          # the fp32 add of the kernel
    srt = np.sort(sel, axis=1)
    assert np.all(srt[:, 1:] != srt[:, :-1]), "repeated expert in a token's selection"
    rows = np.arange(T)[:, None]
    v = vb[rows, sel]
    nxt_ok = (v[:, :-1] > v[:, 1:]) | ((v[:, :-1] == v[:, 1:]) & (sel[:, :-1] < sel[:, 1:]))
    assert np.all(nxt_ok), "slot order"
    worst = v[:, -1]
    worst_idx = sel[:, -1]
    chosen = np.zeros((T, E), bool)
    chosen[rows, sel] = True
    idx = np.arange(E)[None, :]
    ok = chosen | (vb < worst[:, None]) | ((vb == worst[:, None]) & (idx > worst_idx[:, None]))
    bad = np.nonzero(~ok.all(axis=1))[0]
    assert bad.size == 0, f"tokens {bad[:5]} leave out an expert that beats a chosen one"
    assert np.all(np.abs(np.asarray(w, np.float64).sum(axis=1) - 1.0) < 1e-5)


def check_selection_and_permutation(scores_ref, scores_gpu, bias, sel, w, counts, offsets, perm,
                                    slot_pos, score_tol, near_tie_bound):
    """Bit-exact selection on every token whose oracle k-th/(k+1)-th biased gap is at least
    NEAR_TIE, gate weights within 1e-5, validity of every token's selection, and the
    permutation outputs equal to the oracle's permutation of the GPU's selection.  Returns
    (near-tie tokens, max score error); asserts the near-tie count <= near_tie_bound."""
    import oracle
    T, k = sel.shape
    E = scores_gpu.shape[1]
    s_gpu = host(scores_gpu).astype(np.float32)
    serr = float(np.max(np.abs(s_gpu.astype(np.float64) - scores_ref))) if T else 0.0
    assert serr <= score_tol, f"score error {serr:.2e}"
    sel_ref, gates_ref, gap = oracle.select_topk(scores_ref, bias, k)
    keep = gap >= NEAR_TIE
    n_tie = int((~keep).sum())
    assert n_tie <= near_tie_bound, f"{n_tie} near-tie tokens > bound {near_tie_bound}"
    o_gpu, o_ref = np.argsort(sel, axis=1), np.argsort(sel_ref, axis=1)
    rows = np.arange(T)[:, None]
    e_gpu, e_ref = sel[rows, o_gpu], sel_ref[rows, o_ref]
    diff = np.nonzero(keep & np.any(e_gpu != e_ref, axis=1))[0]
    assert diff.size == 0, f"selection differs on tokens {diff[:5]}"
    werr = np.abs(np.asarray(w, np.float64)[rows, o_gpu] - gates_ref[rows, o_ref])[keep]
    assert werr.size == 0 or werr.max() <= 1e-5, f"gate weight error {werr.max():.2e}"
    check_topk_valid(s_gpu, bias, sel, w)
    c_ref, off_ref, perm_ref, sp_ref = oracle.permutation(sel, E)
    assert np.array_equal(np.asarray(counts), c_ref)
    assert np.array_equal(np.asarray(offsets), off_ref)
    assert np.array_equal(np.asarray(perm)[:T * k], perm_ref)
    assert np.array_equal(np.asarray(slot_pos).reshape(-1)[:T * k].reshape(T, k), sp_ref)
    return n_tie, serr


def assert_close_grad(got, ref, what=""):
    """Backward gradients: ||got - ref||_F <= BWD_FRO ||ref||_F and max|got - ref| <= BWD_MAX RMS(ref).
    Returns (Frobenius ratio, max / RMS)."""
    got = got.detach().double().cpu().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = got - ref
    if not np.any(ref):                       # a gradient that vanishes exactly (e.g. dW_r at k = 1)
        assert not np.any(got), f"{what}: expected exact zeros, max |got| {np.max(np.abs(got)):.3e}"
        return 0.0, 0.0
    fro = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    mx = float(np.max(np.abs(err)) / max(rms(ref), 1e-300))
    assert fro <= BWD_FRO, f"{what}: relative Frobenius error {fro:.3e} > {BWD_FRO}"
    assert mx <= BWD_MAX, f"{what}: max error {mx:.3e} RMS > {BWD_MAX}"
    return fro, mx
