"""slmoe_route_noalloc (routing with the library's fixed per-device scratch, no workspace
argument) against slmoe_route (the same routing with a caller workspace), through the C ABI.

The GPU tests make two no-allocation calls in a row on one stream, with different inputs and
with the scores kept by the caller and in the scratch, and compare each call's outputs with
slmoe_route on the same input.  The second call only comes out right if each call clears the
scratch's tile counters itself.  The file name makes pytest collect it last, so the tests run
both after the whole suite and, run alone, in a fresh process where the first call sets the
scratch up.  The size limit is checked on the host, without a GPU.
"""
import ctypes

import pytest
import torch

import synthetic
import latent_space_experts_gb300 as lse
from gpu_util import F32_TOL, assert_close_rms, need_gpu, route_buffers, run_route, to_dev

SCRATCH_LIMIT = 48 * 1024 * 1024
ENOSPACE = -4


def k3_router_shape(T):
    """The K3 router (d = 7168, E = 896, k = 16, bf16) with the expert widths cut down: only
    x, W_r, the bias and the logit offsets take part in routing."""
    return synthetic.shape_with("k3_decode", T=T, d_latent=64, I=64, n_shared=0)


def route_noalloc(cfg, inp, keep_scores, hist=None):
    b = route_buffers(cfg.T, cfg.E, cfg.k)
    lse.slmoe_route_noalloc(cfg, inp["x"], inp["W_r"], inp["bias"], inp.get("logit_offset"),
                            b["topk_idx"], b["topk_w"], b["scores"] if keep_scores else None,
                            b["counts"], b["offsets"], b["perm"], b["slot_pos"], hist, None)
    return b


def compare(got, ref, T, k, keep_scores):
    for n in ("topk_idx", "counts", "offsets"):
        assert torch.equal(got[n].cpu(), ref[n]), n
    for n in ("perm", "slot_pos"):
        assert torch.equal(got[n].cpu()[:T * k], ref[n][:T * k]), n
    assert_close_rms(got["topk_w"], ref["topk_w"].double().numpy(), F32_TOL, "topk_w")
    if keep_scores:
        assert_close_rms(got["scores"], ref["scores"].double().numpy(), F32_TOL, "scores")


@pytest.mark.gpu
@pytest.mark.parametrize("family", ["k3_router_bf16", "tiny_f32"])
def test_noalloc_matches_route_on_two_calls_in_a_row(family):
    need_gpu()
    if family == "k3_router_bf16":
        shapes = [k3_router_shape(128), k3_router_shape(1000)]
    else:
        shapes = [synthetic.shape_with("tiny", T=200), synthetic.shape_with("tiny", T=77, E=33, k=5)]
    inps = [to_dev(synthetic.layer_inputs(s, seed=40 + i)) for i, s in enumerate(shapes)]
    cfgs = [lse.config(s) for s in shapes]
    hists = [torch.zeros(s.E, s.nbins, dtype=torch.int32, device="cuda") for s in shapes]

    # two no-allocation calls back to back on the current stream: the first keeps the scores
    # in the caller's buffer, the second leaves them in the scratch and adds a histogram
    got = [route_noalloc(cfgs[0], inps[0], keep_scores=True),
           route_noalloc(cfgs[1], inps[1], keep_scores=False, hist=hists[1])]
    torch.cuda.synchronize()

    for i, (s, cfg, inp) in enumerate(zip(shapes, cfgs, inps)):
        ref_hist = torch.zeros_like(hists[i]) if i == 1 else None
        ref = run_route(cfg, inp, hist=ref_hist)
        compare(got[i], ref, s.T, s.k, keep_scores=(i == 0))
        if i == 1:
            assert torch.equal(hists[1].cpu(), ref_hist.cpu())
            assert int(hists[1].sum()) == s.T * s.E


@pytest.mark.gpu
def test_noalloc_empty_batch():
    need_gpu()
    cfg = lse.config(synthetic.shape_with("tiny", T=0))
    counts = torch.full((16,), 7, dtype=torch.int32, device="cuda")
    offsets = torch.full((17,), 7, dtype=torch.int32, device="cuda")
    lse.slmoe_route_noalloc(cfg, None, None, None, None, None, None, None, counts, offsets, None,
                            None, None, None)
    torch.cuda.synchronize()
    assert int(counts.abs().sum()) == 0 and int(offsets.abs().sum()) == 0


def test_noalloc_rejects_calls_beyond_the_scratch_on_the_host():
    """A call that needs more than the fixed scratch returns SLMOE_ENOSPACE before any CUDA
    call, and its message gives the bytes it needed and the limit."""
    lse.build()
    lib = lse.load()
    fake = ctypes.c_void_p(1 << 20)           # aligned, never dereferenced on this path
    cfg = lse.config(k3_router_shape(8192))
    split = 3 * 896 * 7168 * 2
    need = split + 8192 * 896 * 4            # dominated by the split weights and the scores
    assert need > SCRATCH_LIMIT
    args = [fake] * 12
    rc = lib.slmoe_route_noalloc(ctypes.byref(cfg), *args[:6], None, *args[6:10], None, None, None)
    assert rc == ENOSPACE
    msg = lse.slmoe_last_error()
    assert "scratch" in msg and str(SCRATCH_LIMIT) in msg
    needed = int(msg.split("needs ")[1].split(" bytes")[0])
    assert needed >= need
