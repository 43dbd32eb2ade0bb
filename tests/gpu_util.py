"""Helpers shared by the GPU parity tests (no arithmetic of the method lives here)."""
import numpy as np
import pytest
import torch

import latent_space_experts_gb300 as lse

NEAR_TIE = 1e-5          # tokens whose oracle k-th/(k+1)-th biased gap is below this are excluded
BF16_TOL = 2e-2          # max|err| <= 2e-2 * RMS(ref) on bf16 paths
F32_TOL = 1e-4           # max|err| <= 1e-4 * RMS(ref) on fp32 paths
BF16_STORE = 2.0 ** -7   # extra elementwise allowance for intermediates stored in bf16


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
