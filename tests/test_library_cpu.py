"""The C ABI library builds, loads without a GPU, exports every symbol the header declares,
and rejects bad arguments on the host before any launch.  CPU only."""
import ctypes
import os
import re

import pytest

import synthetic
import latent_space_experts_gb300 as lse

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "slmoe.h")


@pytest.fixture(scope="module")
def lib():
    lse.build()
    return lse.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(slmoe_\w+)\s*\(", text)))


def test_header_declares_the_four_calls():
    syms = declared_symbols()
    for s in ("slmoe_route", "slmoe_qb_histogram", "slmoe_qb_update", "slmoe_forward",
              "slmoe_workspace_size", "slmoe_last_error"):
        assert s in syms


def test_every_declared_symbol_is_exported(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), s
        assert s in lse.__all__, f"binding does not expose {s}"


def test_workspace_size_and_layout(lib):
    for name, shp in synthetic.LAYERS.items():
        cfg = lse.config(shp)
        n = lse.slmoe_workspace_size(cfg)
        L = lse.slmoe_workspace_layout_get(cfg)
        assert L["total"] == n > 0
        offs = [L[k] for k in ("scores", "topk_idx", "topk_w", "counts", "offsets", "perm",
                               "slot_pos", "x_lat", "h", "y_e", "z", "h_s", "status")]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
        es = 2 if shp.dtype == "bf16" else 4
        assert L["h"] - L["x_lat"] >= shp.T * shp.d_latent * es
        assert L["z"] - L["y_e"] >= shp.T * shp.k * shp.d_latent * es


@pytest.mark.parametrize("field,value", [("k", 0), ("k", 33), ("E", 0), ("E", 5000), ("d", 100),
                                         ("dtype", 7), ("nbins", 0), ("n_shared", 4), ("T", -1)])
def test_bad_configs_are_rejected(lib, field, value):
    cfg = lse.config(synthetic.LAYERS["mid"])
    setattr(cfg, field, value)
    assert lib.slmoe_workspace_size(ctypes.byref(cfg)) == 0
    assert lib.slmoe_last_error().decode() != ""
    with pytest.raises(lse.SlmoeError):
        lse.slmoe_workspace_size(cfg)


def test_k_above_E_is_rejected(lib):
    cfg = lse.config(synthetic.LAYERS["tiny"])
    cfg.k = cfg.E + 1
    assert lib.slmoe_workspace_size(ctypes.byref(cfg)) == 0
    assert "k" in lib.slmoe_last_error().decode()


def test_null_and_misaligned_arguments_fail_before_launch(lib):
    cfg = lse.config(synthetic.LAYERS["tiny"])
    n = lse.slmoe_workspace_size(cfg)
    fake = ctypes.c_void_p(1 << 20)                 # never dereferenced: validation fails first
    args = [ctypes.byref(cfg)] + [None] * 13 + [fake, n, None]
    rc = lib.slmoe_route(*args)
    assert rc == -1 and "NULL" in lib.slmoe_last_error().decode()
    mis = ctypes.c_void_p((1 << 20) + 4)
    rc = lib.slmoe_route(ctypes.byref(cfg), *([fake] * 11), None, None, mis, n, None)
    assert rc == -1 and "aligned" in lib.slmoe_last_error().decode()
    rc = lib.slmoe_route(ctypes.byref(cfg), *([fake] * 11), None, None, fake, n - 256, None)
    assert rc == -4
    rc = lib.slmoe_qb_histogram(None, 10, 4, 1000, fake, None, None)
    assert rc == -1
    rc = lib.slmoe_qb_histogram(fake, 10, 4, 1025, fake, None, None)
    assert rc == -1
    rc = lib.slmoe_qb_update(fake, 4, 1000, 5, None, fake, None)
    assert rc == -1
    w = lse.Weights()
    rc = lib.slmoe_forward(ctypes.byref(cfg), fake, ctypes.byref(w), fake, None, fake, None, None,
                           None, fake, n, None)
    assert rc == -1 and "W_r" in lib.slmoe_last_error().decode()


@pytest.mark.parametrize("E,step", [(0, 1e-3), (65537, 1e-3), (4, 0.0), (4, -1e-3),
                                    (4, float("inf")), (4, float("nan"))])
def test_signsgd_update_rejects_bad_arguments(lib, E, step):
    fake = ctypes.c_void_p(1 << 20)                 # never dereferenced: validation fails first
    assert lib.slmoe_signsgd_update(fake, E, step, fake, None) == -1
    assert lib.slmoe_last_error().decode() != ""


def test_signsgd_update_rejects_null_and_misaligned_pointers(lib):
    fake = ctypes.c_void_p(1 << 20)
    mis = ctypes.c_void_p((1 << 20) + 2)
    assert lib.slmoe_signsgd_update(None, 4, 1e-3, fake, None) == -1
    assert lib.slmoe_signsgd_update(fake, 4, 1e-3, None, None) == -1
    assert lib.slmoe_signsgd_update(mis, 4, 1e-3, fake, None) == -1
    assert "aligned" in lib.slmoe_last_error().decode()


def test_empty_batch_forward_returns_before_any_cuda_call(lib):
    """T = 0: nothing to compute, so slmoe_forward succeeds without touching its pointers."""
    cfg = lse.config(synthetic.shape_with("mid", T=0))
    w = lse.Weights()
    rc = lib.slmoe_forward(ctypes.byref(cfg), None, ctypes.byref(w), None, None, None, None, None,
                           None, None, 0, None)
    assert rc == 0


def test_small_batches_get_room_for_the_split_router():
    """A bf16 batch of at most 256 tokens reserves [16, T, E] fp32 for the router's split-K
    logit sums in the workspace; a larger batch does not split and needs no such room."""
    E = 896
    def total(T):
        return lse.slmoe_workspace_size(lse.config(synthetic.shape_with("k3_decode", T=T)))
    # growth from 256 to 257 tokens loses the split region (16 * 256 * E * 4 bytes) but adds
    # one token's worth of everything else
    per_token = total(300) - total(299)
    assert total(257) < total(256) + per_token
    assert total(256) - total(255) >= 16 * E * 4


def test_router_weight_split_is_exact_in_three_bf16_pieces():
    """The router's fp32 weights go to the tensor cores as three bf16 pieces, hi = bf16(w),
    mid = bf16(w - hi), lo = bf16(w - hi - mid) (round to nearest, differences in fp32):
    hi + mid + lo == w exactly for normal fp32 values, and each piece times a bf16 activation
    is exact in fp32, so the logits are the fp32 weights' logits up to the order of the adds.
    Checked here with torch's round-to-nearest bf16 conversion, the same rounding the GPU
    split uses."""
    import numpy as np
    import torch
    rng = np.random.default_rng(3)
    mant = rng.uniform(1.0, 2.0, 200000)
    expo = rng.integers(-60, 61, 200000)
    sign = rng.choice([-1.0, 1.0], 200000)
    w = torch.from_numpy((sign * mant * 2.0 ** expo).astype(np.float32))
    w = torch.cat([w, torch.randn(100000) / 84.7])                 # the K3 router's N(0, 1/d)
    hi = w.to(torch.bfloat16)
    r1 = w - hi.float()
    mid = r1.to(torch.bfloat16)
    r2 = r1 - mid.float()
    lo = r2.to(torch.bfloat16)
    assert torch.equal(lo.float(), r2)                             # the remainder fits bf16
    total = hi.double() + mid.double() + lo.double()
    assert torch.equal(total, w.double())
    x = torch.randn(300000).to(torch.bfloat16)
    for piece in (hi, mid, lo):                                     # products exact in fp32
        assert torch.equal((x.float() * piece.float()).double(), x.double() * piece.double())


@pytest.mark.parametrize("T,E,k", [(-1, 8, 2), (10, 0, 1), (10, 8, 9), (10, 64, 33), (10, 5000, 4),
                                   (1 << 30, 64, 2)])
def test_topk_workspace_rejects_bad_shapes(lib, T, E, k):
    assert lib.slmoe_topk_workspace_size(T, E, k) == 0
    assert lib.slmoe_last_error().decode() != ""


def test_topk_workspace_size(lib):
    # one int32 count per (16-token chunk, expert), rounded up to 256 bytes
    assert lib.slmoe_topk_workspace_size(65536, 896, 16) == 4096 * 896 * 4
    assert lib.slmoe_topk_workspace_size(17, 3, 1) == 256
    assert lib.slmoe_topk_workspace_size(0, 8, 2) > 0


def test_topk_and_abort_check_validate_on_the_host(lib):
    """Null or misaligned pointers and bad limits are refused before any CUDA call."""
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    ws = lib.slmoe_topk_workspace_size(64, 16, 2)
    args = lambda counts: (fake, fake, 64, 16, 2, fake, fake, counts, fake, fake, fake, None, fake, ws, None)
    assert lib.slmoe_topk(*args(None)) == -1
    assert lib.slmoe_topk(*args(odd)) == -1
    assert lib.slmoe_topk(fake, fake, 64, 16, 2, fake, fake, fake, fake, fake, fake, None, fake, ws - 256,
                          None) == -4
    assert lib.slmoe_wait_abort_check(None, 1000, None) == -1
    assert lib.slmoe_wait_abort_check(fake, 0, None) == -1
    assert lib.slmoe_wait_abort_check(fake, 10 ** 12, None) == -1


@pytest.mark.parametrize("field,value,ok", [("d_latent", 320, False), ("I", 192, False), ("d_latent", 384, True),
                                            ("I", 384, True)])
def test_mxfp4_layer_needs_128_multiples(lib, field, value, ok):
    """The MXFP4 layer reads K blocks of 128 (d_latent and I) on the block-scaled tensor cores."""
    cfg = lse.config(synthetic.LAYERS["mid"], dtype=lse.MXFP4)
    setattr(cfg, field, value)
    assert (lib.slmoe_workspace_size(ctypes.byref(cfg)) > 0) == ok


def test_mxfp8_quantize_validates_on_the_host(lib):
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    assert lib.slmoe_mxfp8_quantize(fake, 4, 48, fake, fake, None) == -1      # K not a multiple of 32
    assert lib.slmoe_mxfp8_quantize(fake, -1, 32, fake, fake, None) == -1
    assert lib.slmoe_mxfp8_quantize(None, 4, 32, fake, fake, None) == -1
    assert lib.slmoe_mxfp8_quantize(odd, 4, 32, fake, fake, None) == -1
    assert lib.slmoe_mxfp8_quantize(fake, 4, 32, fake, None, None) == -1
    assert lib.slmoe_mxfp8_quantize(fake, 0, 32, fake, fake, None) == 0       # nothing to do
