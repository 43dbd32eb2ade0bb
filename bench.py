"""Benchmark of the Stable LatentMoE forward hot path on GB300.

One step = one slmoe_forward over one batch of the workload (router scores, biased top-k,
permutation, QB histogram of the step's scores, latent down-projection, both routed-expert
GEMMs with the fused SiTU-GLU, combine + RMSNorm, shared experts, up-projection) followed by
the QB bias update (slmoe_qb_update).  Inputs and weights are resident in HBM when timing
starts; weights (10.2 GB at the K3 shape) exceed the L2 (about 129 MB), so no flush is
needed.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload k3_prefill|k3_decode|mid]
                  [--impl ours|reference] [--skew] [--qb-only]

Prints one JSON line (rank 0).  N > 1 runs one independent replica per GPU (weak scaling):
the layer has no data-path exchange on one node in this design.  --impl reference times the
fp64 oracle on the host cores on a bounded sample of the same workload.  --qb-only runs just
the QB engine measurement (histogram of 65536 x 896 scores + bias update), a small process
for profiling that kernel.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "LatentMoE fwd tokens/s at K3 shape (1xGB300)"
UNIT = "tokens/s"
PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STAGES = ["start", "router", "topk+permute+hist", "down", "expert gate|up", "expert down",
          "combine+rmsnorm", "shared gate|up", "up+shared down"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return PEAKS_FALLBACK, "fallback"


def work_model(shp, counts=None):
    """Algorithmic FLOPs and bytes per stage for one step (weights touched + kernel I/O)."""
    T, d, dl, E, k, I, ns, Is = shp.T, shp.d, shp.d_latent, shp.E, shp.k, shp.I, shp.n_shared, shp.I_shared
    touched = E if counts is None else int((counts > 0).sum())
    st = {
        "router": dict(flops=2 * T * d * E, bytes=T * d * 2 + E * d * 4 + T * E * 4, bound="tensor"),
        "topk+permute+hist": dict(flops=0, bytes=2 * T * E * 4 + T * k * 16, bound="hbm"),
        "down": dict(flops=2 * T * d * dl, bytes=T * d * 2 + dl * d * 2 + T * dl * 2, bound="tensor"),
        "expert gate|up": dict(flops=2 * T * k * dl * 2 * I,
                               bytes=touched * 2 * I * dl * 2 + T * dl * 2 + T * k * I * 2, bound="hbm"),
        "expert down": dict(flops=2 * T * k * I * dl,
                            bytes=touched * dl * I * 2 + T * k * I * 2 + T * k * dl * 2, bound="hbm"),
        "combine+rmsnorm": dict(flops=0, bytes=T * k * dl * 2 + T * dl * 2, bound="hbm"),
        "shared gate|up": dict(flops=2 * T * d * 2 * Is * ns, bytes=T * d * 2 + ns * 2 * Is * d * 2 + T * ns * Is * 2,
                               bound="tensor"),
        "up+shared down": dict(flops=2 * T * (dl + ns * Is) * d,
                               bytes=T * dl * 2 + T * ns * Is * 2 + d * (dl + ns * Is) * 2 + T * d * 2,
                               bound="tensor"),
    }
    layer_flops = sum(v["flops"] for v in st.values())
    layer_bytes = (E * d * 4 + dl * d * 2 + touched * 3 * I * dl * 2 + d * dl * 2 + ns * 3 * Is * d * 2
                   + T * d * 2 * 2)
    return st, layer_flops, layer_bytes


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms during a region."""
    Q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def start(self):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        self.f.seek(0)
        rows = [r.split(", ") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        samples = []
        for r in rows:
            try:
                ts = time.mktime(time.strptime(r[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + float("0." + r[0].split(".")[1])
                samples.append((ts, float(r[2]), float(r[3]), r[5:]))
            except (ValueError, IndexError):
                continue
        inside = [s for s in samples if t0 - 0.2 <= s[0] <= t1 + 0.2] or samples
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i, v in enumerate(s[3][1:5]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(s[1] for s in inside) if inside else None,
                "sm_max_mhz": max(s[2] for s in inside) if inside else None,
                "reasons": reasons, "samples": len(inside)}


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    return world, rank, local


def max_over_ranks(v, world, device="cuda"):
    """The largest of the ranks' values (the slowest rank's time), on every rank."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, ms_per_step):
    """Whole-job throughput: the units every rank processed in one step, over the step time
    of the slowest rank (replicas: each rank runs the full batch)."""
    return units_per_rank * world / (ms_per_step * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def oracle_inputs(inp):
    """The layer inputs on the host for the oracle: the dense tensors (x, router, latent
    projections, shared experts, norm) widened to the oracle's fp64 once, as the GPU keeps
    its weights resident; the routed experts' weights (40 GB in fp64 at K3) stay in their
    storage type and the oracle widens each chosen expert's matrices per call."""
    import numpy as np
    out = {}
    for k, v in inp.items():
        if v is None or k in ("W13", "W2"):
            out[k] = v.cpu() if v is not None else None
        else:
            out[k] = np.ascontiguousarray(v.detach().cpu().double().numpy())
    return out


def oracle_sample(shp, inp_cpu, n_tok):
    """Time the fp64 oracle on n_tok tokens of the workload (routing included)."""
    import numpy as np
    import oracle
    tok = np.arange(n_tok)
    t0 = time.perf_counter()
    oracle.forward(inp_cpu, shp.k, tokens=tok)
    dt = time.perf_counter() - t0
    return n_tok / dt, dt


def oracle_tokens(shp, inp_cpu, target_s):
    """Tokens per oracle sample so that one sample takes at most about target_s seconds.
    Trials double the token count until one takes a quarter of the target; the count is then
    scaled by target / trial time.  A sample's cost grows more slowly than its token count
    (tokens share experts, whose weights are widened once per sample), so the scaled sample
    does not overshoot."""
    cap = 4096
    n = min(4, shp.T)
    while True:
        _, dt = oracle_sample(shp, inp_cpu, n)
        if dt >= target_s / 4 or n >= min(shp.T, cap):
            break
        n = min(2 * n, shp.T, cap)
    return max(1, min(shp.T, cap, int(n * target_s / max(dt, 1e-6))))


def profiled_traffic(stage):
    """DRAM bytes per launch of a stage's kernel at the bench workload, as recorded in the
    committed ncu summaries under profiles/ ("bench-traffic:" lines), used only while the
    kernel's source file still has the SHA-256 recorded with the capture; else None."""
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None
    pat = re.compile(r"bench-traffic: (.+?) = (\d+) bytes per launch; source (\S+) sha256 ([0-9a-f]{64})")
    for name in sorted(os.listdir(pdir)):
        with open(os.path.join(pdir, name), errors="replace") as f:
            for line in f:
                m = pat.search(line)
                if not m or m.group(1) != stage:
                    continue
                src = os.path.join(ROOT, m.group(3))
                if not os.path.exists(src):
                    continue
                if hashlib.sha256(open(src, "rb").read()).hexdigest() == m.group(4):
                    return int(m.group(2))
    return None


def cpu_cores():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max((i.get("num_threads", 1) for i in info), default=1)
        return int(n)
    except Exception:
        return os.cpu_count() or 1


def run_reference(args):
    """The oracle as the reference arm: fp64 CPU forward on a bounded token sample per step."""
    import torch
    import synthetic
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shp = synthetic.LAYERS[args.workload]
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = synthetic.layer_inputs(shp, seed=0, device=dev)
    inp_cpu = oracle_inputs(inp)
    del inp
    # each step is a bounded sample: the whole run (warm-up + timed) takes about ref_seconds
    n_tok = args.ref_tokens or oracle_tokens(shp, inp_cpu, args.ref_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_sample(shp, inp_cpu, n_tok)
    t = []
    for _ in range(args.steps):
        _, dt = oracle_sample(shp, inp_cpu, n_tok)
        t.append(dt)
    total = sum(t)
    value = n_tok * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "T": shp.T, "d": shp.d, "d_latent": shp.d_latent,
                       "E": shp.E, "k": shp.k, "I": shp.I, "n_shared": shp.n_shared,
                       "I_shared": shp.I_shared, "sample_tokens_per_step": n_tok},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{n_tok} tokens of the {args.workload} batch per step (routing, "
                                       f"experts, norm, shared experts), fp64 numpy"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def qb_engine(hbm):
    """QB engine on one GPU: histogram bandwidth over one 65536 x 896 fp32 micro-batch of
    scores (235 MB, larger than L2) and the time of one bias update, CUDA events on the
    launching stream after warm-up."""
    import torch
    import latent_space_experts_gb300 as lse
    import synthetic
    stream = torch.cuda.current_stream()
    q = synthetic.QB
    sc = synthetic.qb_scores(0, q, device="cuda")
    qh = torch.zeros(q.E, q.nbins, dtype=torch.int32, device="cuda")
    for _ in range(3):
        lse.slmoe_qb_histogram(sc, q.T, q.E, q.nbins, qh)
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 50
    g0.record(stream)
    for _ in range(reps):
        lse.slmoe_qb_histogram(sc, q.T, q.E, q.nbins, qh)
    g1.record(stream)
    torch.cuda.synchronize()
    tq = g0.elapsed_time(g1) / reps * 1e-3
    qbias = torch.empty(q.E, device="cuda")
    for _ in range(3):
        lse.slmoe_qb_update(qh, q.E, q.nbins, q.k, None, qbias)
    g0.record(stream)
    for _ in range(reps):
        lse.slmoe_qb_update(qh, q.E, q.nbins, q.k, None, qbias)
    g1.record(stream)
    torch.cuda.synchronize()
    tu = g0.elapsed_time(g1) / reps * 1e-3
    # the fixed-step rule QB replaces, on the loads of one micro-batch
    counts = torch.full((q.E,), q.T * q.k // q.E, dtype=torch.int32, device="cuda")
    counts[: q.E // 2] += 1
    counts[q.E // 2:] -= 1
    sbias = torch.zeros(q.E, device="cuda")
    for _ in range(3):
        lse.slmoe_signsgd_update(counts, q.E, 1e-3, sbias)
    g0.record(stream)
    for _ in range(reps):
        lse.slmoe_signsgd_update(counts, q.E, 1e-3, sbias)
    g1.record(stream)
    torch.cuda.synchronize()
    ts = g0.elapsed_time(g1) / reps * 1e-3
    qbytes = q.T * q.E * 4 + 2 * q.E * q.nbins * 4
    return {"GB/s": round(qbytes / tq / 1e9, 1), "frac_of_hbm": round(qbytes / tq / 1e9 / hbm, 4),
            "us_per_micro_batch": round(tq * 1e6, 2), "bytes": qbytes,
            "update_us": round(tu * 1e6, 2), "signsgd_update_us": round(ts * 1e6, 2),
            "engine_ms": round((q.micro_batches * tq + tu) * 1e3, 4),
            "note": "65536 x 896 fp32 scores per micro-batch (235 MB > L2); engine = 8 histograms + 1 update"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="k3_prefill", choices=["k3_prefill", "k3_decode", "mid", "k3_slice", "k3_dense"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=None,
                    help="oracle tokens per reference step (default: sized from --ref-seconds)")
    ap.add_argument("--ref-seconds", type=float, default=120.0,
                    help="about how long the whole reference run (warm-up + timed steps) takes")
    ap.add_argument("--cpu-baseline-tokens", type=int, default=None,
                    help="oracle tokens of the cpu_baseline sample (default: sized from --cpu-seconds)")
    ap.add_argument("--cpu-seconds", type=float, default=25.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--qb-only", action="store_true", help="only the QB engine measurement")
    ap.add_argument("--no-graph", action="store_true", help="time the step without a CUDA graph")
    ap.add_argument("--skew", action="store_true", help="heavy skew (10%% hot experts)")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)

    import numpy as np
    import torch
    import latent_space_experts_gb300 as lse
    import synthetic

    world, rank, local = dist_setup(args)
    lse.build()
    lse.load()
    if args.qb_only:
        if rank == 0:
            pk, pk_kind = peaks()
            print(json.dumps({"qb_histogram": qb_engine(pk["hbm_gbs"]), "peak_source": pk_kind}))
        return
    shp = synthetic.LAYERS[args.workload]
    cfg = lse.config(shp)
    inp = synthetic.layer_inputs(shp, seed=rank, device="cuda", heavy_skew=args.skew)
    ws = torch.zeros(lse.slmoe_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    y = torch.empty(shp.T, shp.d, dtype=torch.float32, device="cuda")
    hist = torch.zeros(shp.E, shp.nbins, dtype=torch.int32, device="cuda")
    bias = inp["bias"].clone()
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    W = lse.weights(inp)
    stream = torch.cuda.current_stream()

    def step(x, out=None):
        lse.slmoe_forward(cfg, x, W, bias, inp["logit_offset"], y if out is None else out, None, hist,
                          status, ws)
        lse.slmoe_qb_update(hist, shp.E, shp.nbins, shp.k, None, bias)

    for _ in range(max(3, args.warmup)):
        step(inp["x"])
    torch.cuda.synchronize()
    assert status.cpu().tolist()[1:3] == [0, 0], f"device status {status.cpu().tolist()}"

    # the timed step is replayed from a CUDA graph of the same calls (the library's launches are
    # stream-ordered, its auxiliary stream joins the capture through the fork/join events);
    # the graph only removes host launch gaps between the step's ~15 kernels
    graph = None
    launches_per_step = None
    if not args.no_graph:
        l_cap = lse.slmoe_launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step(inp["x"])
        launches_per_step = lse.slmoe_launch_count() - l_cap
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
        assert status.cpu().tolist()[1:3] == [0, 0], f"device status {status.cpu().tolist()}"

    # ---------------- device-resident timing
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    l0 = lse.slmoe_launch_count()
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    e0.record(stream)
    for _ in range(args.steps):
        if graph is not None:
            graph.replay()
        else:
            step(inp["x"])
    e1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier(world)
    launches = (launches_per_step * args.steps if graph is not None
                else lse.slmoe_launch_count() - l0)
    ms = max_over_ranks(e0.elapsed_time(e1), world) / args.steps
    clocks = sampler.stop(w0, w1) if sampler else None

    # ---------------- per-stage timing (events recorded by the library on this stream)
    nst = len(STAGES)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(min(args.steps, 50))]
    for row in ev:
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    stage_ms = [0.0] * nst
    for row in ev:
        lse.slmoe_set_stage_events(row)
        step(inp["x"])
    lse.slmoe_set_stage_events(None)
    torch.cuda.synchronize()
    # stage i ends at event i.  On the bf16 type the down-projection (3) and the shared
    # gate|up (7) run on the library's auxiliary stream from the start (0), concurrently with
    # routing (1, 2); the routed experts (4) start when both branches are done.
    start_of = {3: 0, 7: 3, 4: None}
    for row in ev:
        t = [row[0].elapsed_time(e) for e in row]
        for i in range(1, nst):
            if i == 4:
                t_start = max(t[2], t[7])
            elif i == 8:
                t_start = t[6]
            else:
                t_start = t[start_of.get(i, i - 1)]
            stage_ms[i] += (t[i] - t_start) / len(ev)
    counts = lse.workspace_views(cfg, ws)["counts"].cpu().numpy()
    st_model, layer_flops, layer_bytes = work_model(shp, counts)
    pk, pk_kind = peaks()
    hbm = pk["hbm_gbs"]
    tc = pk["bf16_tflops_sustained"]
    stages = {}
    for i in range(1, nst):
        m = st_model[STAGES[i]]
        t = stage_ms[i] * 1e-3
        stages[STAGES[i]] = {"ms": round(stage_ms[i], 4),
                             "GB/s": round(m["bytes"] / t / 1e9, 1) if t > 0 else None,
                             "TFLOP/s": round(m["flops"] / t / 1e12, 1) if t > 0 else None,
                             "bound": m["bound"]}
    # the dominant kernel on the critical path (the concurrent front part excluded)
    dom = max((1, 2, 4, 5, 6, 8), key=lambda i: stage_ms[i])
    dm = st_model[STAGES[dom]]
    t_dom = stage_ms[dom] * 1e-3
    if dm["bound"] == "hbm":
        roof = {"bound": "hbm", "achieved": round(dm["bytes"] / t_dom / 1e9, 1), "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": round(dm["flops"] / t_dom / 1e12, 1), "peak": tc,
                "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = profiled_traffic(STAGES[dom]) if args.workload == "k3_prefill" else None
    roof["kernel"] = STAGES[dom]
    roof["peak_source"] = f"{pk_kind} ({'sustained bf16' if roof['bound'] == 'tensor' else 'hbm copy'})"
    t_layer = max(layer_flops / (tc * 1e12), layer_bytes / (hbm * 1e9))

    # ---------------- end to end through the public API, host buffers
    # Every step uploads its input from pinned host memory and reads its result back.  As a
    # serving loop would, the copies run on their own streams with two device buffers each, so
    # that step i+1's upload and step i's read-back overlap the compute of the steps beside them;
    # the timed region runs from before the first upload to the end of the last read-back.
    x_host = inp["x"].cpu().pin_memory()
    y_host = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    x_dev = [torch.empty_like(inp["x"]) for _ in range(2)]
    y_dev = [y, torch.empty_like(y)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_steps(n, start):
        done, out = [None, None], [None, None]
        ready = [None, None]
        s_in.wait_event(start)
        with torch.cuda.stream(s_in):
            x_dev[0].copy_(x_host, non_blocking=True)
            ready[0] = s_in.record_event()
        for i in range(n):
            b = i % 2
            if i + 1 < n:                       # upload step i+1 once step i-1 has read its buffer
                nb = 1 - b
                if done[nb] is not None:
                    s_in.wait_event(done[nb])
                with torch.cuda.stream(s_in):
                    x_dev[nb].copy_(x_host, non_blocking=True)
                    ready[nb] = s_in.record_event()
            stream.wait_event(ready[b])
            if out[b] is not None:              # y buffer b: step i-2's read-back is done
                stream.wait_event(out[b])
            step(x_dev[b], y_dev[b])
            done[b] = stream.record_event()
            s_out.wait_event(done[b])
            with torch.cuda.stream(s_out):
                y_host[b].copy_(y_dev[b], non_blocking=True)
                out[b] = s_out.record_event()
        for ev in out:
            if ev is not None:
                stream.wait_event(ev)

    w0e = torch.cuda.Event()
    w0e.record(stream)
    e2e_steps(3, w0e)
    torch.cuda.synchronize()
    barrier(world)
    n_e2e = max(3, min(args.steps, 100))
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    e2e_steps(n_e2e, f0)
    f1.record(stream)
    torch.cuda.synchronize()
    assert status.cpu().tolist()[1:3] == [0, 0], f"device status {status.cpu().tolist()}"
    assert torch.equal(y_host[(n_e2e - 1) % 2], y_dev[(n_e2e - 1) % 2].cpu())
    ms_e2e = max_over_ranks(f0.elapsed_time(f1), world) / n_e2e

    # ---------------- QB engine histogram bandwidth (65536 x 896 fp32 per micro-batch)
    qb = qb_engine(hbm) if rank == 0 else None

    # ---------------- oracle on the host cores (bounded sample)
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_cpu = oracle_inputs(inp)
        n_tok = args.cpu_baseline_tokens or oracle_tokens(shp, inp_cpu, args.cpu_seconds)
        v, dt = oracle_sample(shp, inp_cpu, n_tok)
        cpu_base = {"value": round(v, 3), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                    "sample": f"{n_tok} tokens of the {args.workload} batch, fp64 numpy ({dt:.1f} s)"}

    if rank == 0:
        tokens = shp.T
        line = {
            "metric": METRIC, "value": round(job_throughput(tokens, world, ms), 1), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": shp.dtype,
            "data": "synthetic",
            "config": {"workload": args.workload, "T": shp.T, "d": shp.d, "d_latent": shp.d_latent,
                       "E": shp.E, "k": shp.k, "I": shp.I, "n_shared": shp.n_shared, "I_shared": shp.I_shared,
                       "router": "fp32 logits (3-piece bf16 split)", "skew": bool(args.skew),
                       "parallelism": f"replicas x{world}",
                       "l2": "no flush: weights (10.2 GB at K3) exceed L2 every step",
                       "cuda_graph": graph is not None},
            "roofline": roof,
            "layer_roofline": {"ms": round(t_layer * 1e3, 4), "frac": round(t_layer * 1e3 / ms, 4),
                               "flops": layer_flops, "bytes": layer_bytes,
                               "peaks": f"{pk_kind}: {tc} TFLOP/s sustained bf16, {hbm} GB/s"},
            "stages": stages,
            "qb_histogram": qb,
            "cpu_baseline": cpu_base,
            "e2e": {"value": round(job_throughput(tokens, world, ms_e2e), 1), "unit": UNIT,
                    "h2d_bytes_per_step": x_host.numel() * x_host.element_size(),
                    "d2h_bytes_per_step": y_host[0].numel() * y_host[0].element_size(),
                    "copies": "own streams, double-buffered, overlapping the neighbouring steps"},
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
