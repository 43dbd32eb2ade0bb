"""Helpers shared by the GPU parity tests (no arithmetic of the method lives here)."""
import numpy as np
import pytest
import torch

import latent_space_experts_gb300 as lse

NEAR_TIE = 1e-5          # tokens whose oracle k-th/(k+1)-th biased gap is below this are excluded
BF16_TOL = 2e-2          # max|err| <= 2e-2 * RMS(ref) on bf16 paths
F32_TOL = 1e-4           # max|err| <= 1e-4 * RMS(ref) on fp32 paths


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


def assert_close_rms(got, ref, tol, what=""):
    got = got.detach().float().cpu().double().numpy() if hasattr(got, "detach") else np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    bound = tol * rms(ref)
    assert err <= bound, f"{what}: max|err| {err:.3e} > {tol} * RMS(ref) = {bound:.3e}"
    return err / max(rms(ref), 1e-300)


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
