"""The host side of a multi-GPU bench run, on CPU: two gloo ranks.

One process per GPU runs an independent replica of the layer; the job's time per step is
the slowest rank's, and the job's throughput counts the tokens of every rank.  These tests
run bench.py's helpers for that in two processes joined by a gloo process group (no GPU).
"""
import multiprocessing as mp
import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        ms = bench.max_over_ranks(3.5 + rank, world, device="cpu")    # rank 1 is the slow one
        bench.barrier(world)
        q.put((rank, ms, bench.job_throughput(8192, world, ms)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_count_every_ranks_tokens():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    assert [g[1] for g in got] == [4.5, 4.5]
    assert all(g[2] == pytest.approx(2 * 8192 / 4.5e-3) for g in got)


def test_one_rank_is_the_plain_time():
    import bench
    assert bench.max_over_ranks(2.0, 1) == 2.0
    assert bench.job_throughput(8192, 1, 4.0) == pytest.approx(8192 / 4e-3)


def test_oracle_inputs_widened_once_give_the_same_layer():
    """bench.py hands the oracle its dense inputs already in fp64 (as the GPU keeps its weights
    resident): the oracle's results are the same as from the stored inputs."""
    import numpy as np
    import bench
    import oracle
    import synthetic
    shp = synthetic.shape_with("mid", T=48, d=256, d_latent=128, E=16, k=2, I=64, I_shared=128)
    inp = synthetic.layer_inputs(shp, seed=9)
    tok = np.arange(0, 48, 3)
    a = oracle.forward({k: (v.cpu() if v is not None else None) for k, v in inp.items()}, shp.k, tokens=tok)
    b = oracle.forward(bench.oracle_inputs(inp), shp.k, tokens=tok)
    assert np.array_equal(a["topk_idx"], b["topk_idx"])
    assert np.array_equal(a["y"], b["y"])
