"""The bounded-wait failure path of the tensor-core kernels, made to run out on purpose.

slmoe_wait_abort_check launches one tile of the dense GEMM kernel whose copy-issuing thread
issues nothing, so the MMA thread's wait on its first operand stage can only give up.  With a
1 ms limit the launch must come back promptly with status[2] = 1 (and no other status word
set), leave the context usable, and a normal layer call on the same stream right after it must
still match the oracle.  Nothing faults, traps or hangs: every wait in the kernel is bounded
and nothing is in flight when it stops.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import synthetic
import latent_space_experts_gb300 as lse
from gpu_util import BF16_TOL, assert_close_rms, need_gpu, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    need_gpu()
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    lse.slmoe_wait_abort_check(status, 1_000_000)      # 1 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert status.cpu().tolist() == [0, 0, 1, 0], status
    assert dt < 1.0, f"the aborted launch took {dt:.3f} s"

    # a second abort on the same stream, then a normal layer call: both behave
    status.zero_()
    lse.slmoe_wait_abort_check(status, 2_000_000)
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 1, 0]

    shp = synthetic.shape_with("mid", T=300, d=512)
    inp_cpu = synthetic.layer_inputs(shp, seed=11)
    inp = to_dev(inp_cpu)
    cfg = lse.config(shp)
    ws = torch.zeros(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty(shp.T, shp.d, dtype=torch.float32, device="cuda")
    topk = torch.empty(shp.T, shp.k, dtype=torch.int32, device="cuda")
    st2 = torch.zeros(4, dtype=torch.int32, device="cuda")
    lse.slmoe_forward(cfg, inp["x"], lse.weights(inp), inp["bias"], inp.get("logit_offset"), y, topk,
                      None, st2, ws)
    torch.cuda.synchronize()
    assert st2.cpu().tolist() == [0, 0, 0, 0]
    ref = oracle.forward(inp_cpu, shp.k, forced_topk_idx=topk.cpu().numpy())
    assert_close_rms(y, ref["y"], BF16_TOL, "y after an aborted launch")


def test_wait_abort_check_rejects_bad_arguments():
    need_gpu()
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    for limit in (0, 10**12):
        with pytest.raises(lse.SlmoeError):
            lse.slmoe_wait_abort_check(status, limit)
    with pytest.raises(lse.SlmoeError):
        lse.slmoe_wait_abort_check(None, 1000)
    torch.cuda.synchronize()
    assert int(status.abs().sum()) == 0
