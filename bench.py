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


# The block-scaled MMA of the MXFP4 layer (E2M1 x E4M3) runs at the FP8 tensor rate: the
# measured bf16 peak times the nominal ratio 4.5 / 2.25 PFLOP/s.
MX_TENSOR_RATIO = 2.0


def work_model(shp, counts=None, mx=False):
    """FLOPs and bytes per stage of one step.  "bytes" are the layer's algorithmic bytes
    (weights touched, the layer's input x and its fp32 output y); "inter" are the
    intermediates a stage reads or writes (scores, x_lat, h, y_e, z, h_s), which a fused
    design could avoid and which are reported separately.  mx: the MXFP4 layer type, whose
    routed-expert weights take 17/32 bytes each (half a byte per code plus one scale byte per
    32) and whose x_lat and h are MXFP8 (33/32 bytes per value)."""
    wb = 17 / 32 if mx else 2.0
    ab = 33 / 32 if mx else 2.0          # bytes per x_lat / h value
    T, d, dl, E, k, I, ns, Is = shp.T, shp.d, shp.d_latent, shp.E, shp.k, shp.I, shp.n_shared, shp.I_shared
    touched = E if counts is None else int((counts > 0).sum())
    st = {
        "router": dict(flops=2 * T * d * E, bytes=T * d * 2 + E * d * 4, inter=T * E * 4, bound="tensor"),
        "topk+permute+hist": dict(flops=0, bytes=0, inter=2 * T * E * 4 + T * k * 16, bound="hbm"),
        "down": dict(flops=2 * T * d * dl, bytes=T * d * 2 + dl * d * 2, inter=int(T * dl * ab), bound="tensor"),
        "expert gate|up": dict(flops=2 * T * k * dl * 2 * I, bytes=int(touched * 2 * I * dl * wb),
                               inter=int(T * dl * ab + T * k * I * ab), bound="hbm"),
        "expert down": dict(flops=2 * T * k * I * dl, bytes=int(touched * dl * I * wb),
                            inter=int(T * k * I * ab) + T * k * dl * 2, bound="hbm"),
        "combine+rmsnorm": dict(flops=0, bytes=0, inter=T * k * dl * 2 + T * dl * 2 + T * k * 8, bound="hbm"),
        "shared gate|up": dict(flops=2 * T * d * 2 * Is * ns, bytes=T * d * 2 + ns * 2 * Is * d * 2,
                               inter=T * ns * Is * 2, bound="tensor"),
        "up+shared down": dict(flops=2 * T * (dl + ns * Is) * d, bytes=d * (dl + ns * Is) * 2 + T * d * 4,
                               inter=T * dl * 2 + T * ns * Is * 2, bound="tensor"),
    }
    layer_flops = sum(v["flops"] for v in st.values())
    layer_bytes = int(E * d * 4 + dl * d * 2 + touched * 3 * I * dl * wb + d * dl * 2 + ns * 3 * Is * d * 2
                      + T * d * 2 + T * d * 4)
    return st, layer_flops, layer_bytes


def tensor_peak(pk, timed_s, reasons):
    """The bf16 tensor peak a tensor-bound figure is judged against: the burst figure for a
    timed region shorter than two seconds or one that saw no power capping, the sustained
    figure (a seconds-long loop under the power cap) otherwise."""
    if timed_s >= 2.0 and "sw_power_cap" in (reasons or []):
        return pk["bf16_tflops_sustained"], "sustained bf16"
    return pk["bf16_tflops"], "burst bf16"


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


# Tokens of the workload's batch that one oracle sample runs (both the cpu_baseline leg and
# each step of --impl reference time this same sample, so the two figures agree).
CPU_SAMPLE_TOKENS = 512


def oracle_sample(shp, inp_cpu, n_tok):
    """Time the fp64 oracle on the first n_tok tokens of the batch (routing included)."""
    import numpy as np
    import oracle
    tok = np.arange(n_tok)
    t0 = time.perf_counter()
    oracle.forward(inp_cpu, shp.k, tokens=tok)
    dt = time.perf_counter() - t0
    return n_tok / dt, dt


def _blas_threads_fns():
    """(get, set) of the BLAS thread count of the OpenBLAS that numpy loaded, looked up in the
    process's own mapped libraries (no extra package needed); (None, None) if not found."""
    import ctypes
    import numpy  # noqa: F401  (loads the BLAS)
    try:
        paths = {l.split()[-1] for l in open("/proc/self/maps") if "blas" in l.lower() and ".so" in l}
    except OSError:
        return None, None
    for path in sorted(paths):
        try:
            lib = ctypes.CDLL(path)
        except OSError:
            continue
        for get, set_ in (("scipy_openblas_get_num_threads64_", "scipy_openblas_set_num_threads64_"),
                          ("openblas_get_num_threads64_", "openblas_set_num_threads64_"),
                          ("openblas_get_num_threads", "openblas_set_num_threads")):
            if hasattr(lib, get) and hasattr(lib, set_):
                g, s = getattr(lib, get), getattr(lib, set_)
                g.restype = ctypes.c_int
                s.argtypes = [ctypes.c_int]
                return g, s
    return None, None


def oracle_sample_threads(shp, inp_cpu, n_tok, threads):
    """oracle_sample with the BLAS limited to `threads` threads (None: as configured).
    Returns (tokens/s, seconds) or (None, None) when the BLAS thread count cannot be set."""
    if threads is None:
        return oracle_sample(shp, inp_cpu, n_tok)
    get, set_ = _blas_threads_fns()
    if get is None:
        return None, None
    before = get()
    set_(threads)
    try:
        return oracle_sample(shp, inp_cpu, n_tok)
    finally:
        set_(before)


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
    """Threads the oracle's BLAS runs on (the host's core count if it cannot be read)."""
    get, _ = _blas_threads_fns()
    if get is not None:
        return int(get())
    return os.cpu_count() or 1


def reference_tokens(shp, inp_cpu, args):
    """Oracle tokens per reference step: the cpu_baseline sample (CPU_SAMPLE_TOKENS), unless
    --steps + --warmup samples of it would take much longer than --ref-seconds; then the
    sample shrinks so that the run stays within a few minutes (said in the line)."""
    n = min(shp.T, args.ref_tokens or CPU_SAMPLE_TOKENS)
    _, dt = oracle_sample(shp, inp_cpu, n)
    runs = args.steps + args.warmup
    if args.ref_tokens is None and runs * dt > args.ref_seconds:
        n = max(8, int(n * args.ref_seconds / (runs * dt)))
    return n


def run_reference(args):
    """The oracle as the reference arm: fp64 CPU forward on a bounded token sample per step
    (the same sample the cpu_baseline leg of the default run times)."""
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
    n_tok = reference_tokens(shp, inp_cpu, args)
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
                             "sample": f"the first {n_tok} tokens of the {args.workload} batch per step "
                                       f"(routing, experts, norm, shared experts), fp64 numpy, all cores"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def qb_engine(hbm):
    """QB engine on one GPU: histogram bandwidth over one 65536 x 896 fp32 micro-batch of
    scores (235 MB, larger than L2) and the time of one bias update, CUDA events on the
    launching stream.  The histogram is warmed up for about 0.1 s (the clocks settle after
    whatever ran before) and timed over about 0.2 s, with the SM clocks sampled meanwhile."""
    import torch
    import latent_space_experts_gb300 as lse
    import synthetic
    stream = torch.cuda.current_stream()
    q = synthetic.QB
    sc = synthetic.qb_scores(0, q, device="cuda")
    qh = torch.zeros(q.E, q.nbins, dtype=torch.int32, device="cuda")
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    for _ in range(2000):
        lse.slmoe_qb_histogram(sc, q.T, q.E, q.nbins, qh)
    torch.cuda.synchronize()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 4000
    w0 = time.time()
    g0.record(stream)
    for _ in range(reps):
        lse.slmoe_qb_histogram(sc, q.T, q.E, q.nbins, qh)
    g1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    clocks = sampler.stop(w0, w1)
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
            "engine_ms": round((q.micro_batches * tq + tu) * 1e3, 4), "clocks": clocks,
            "note": "65536 x 896 fp32 scores per micro-batch (235 MB > L2); engine = 8 histograms + 1 update"}


def mxfp4_inputs(inp):
    """The layer inputs with the routed experts' W13 / W2 quantised to MXFP4 on the device."""
    import torch
    import latent_space_experts_gb300 as lse
    mx = dict(inp)
    for name in ("W13", "W2"):
        W = inp[name]
        K = W.shape[-1]
        mx[name] = torch.empty(W.shape[:-1] + (K // 2,), dtype=torch.uint8, device="cuda")
        mx[name + "_scale"] = torch.empty(W.shape[:-1] + (K // 32,), dtype=torch.uint8, device="cuda")
        lse.slmoe_mxfp4_quantize(W, W.numel() // K, K, mx[name], mx[name + "_scale"])
    return mx


def qb_balance(step=1e-3):
    """QB-engine balance on the GPU: eight 65536 x 896 micro-batches of scores are binned into
    one histogram and routed (slmoe_topk) with a bias that the fixed-step rule updates after
    each micro-batch; one QB update then reads the histogram.  A held-out micro-batch (seed 9)
    is routed with no bias, with the fixed-step bias and with the QB bias, and max/mean
    expert load is reported for each (the pages fix no target)."""
    import torch
    import latent_space_experts_gb300 as lse
    import synthetic
    q = synthetic.QB
    E, k, T = q.E, q.k, q.T
    hist = torch.zeros(E, q.nbins, dtype=torch.int32, device="cuda")
    ws = torch.empty(lse.slmoe_topk_workspace_size(T, E, k), dtype=torch.uint8, device="cuda")
    buf = dict(topk_idx=torch.empty(T, k, dtype=torch.int32, device="cuda"),
               topk_w=torch.empty(T, k, dtype=torch.float32, device="cuda"),
               counts=torch.empty(E, dtype=torch.int32, device="cuda"),
               offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
               perm=torch.empty(T * k, dtype=torch.int32, device="cuda"),
               slot_pos=torch.empty(T * k, dtype=torch.int32, device="cuda"))

    def route(scores, bias):
        lse.slmoe_topk(scores, bias, T, E, k, buf["topk_idx"], buf["topk_w"], buf["counts"], buf["offsets"],
                       buf["perm"], buf["slot_pos"], None, ws)
        return buf["counts"]

    fixed = torch.zeros(E, device="cuda")
    for m in range(q.micro_batches):
        sc = synthetic.qb_scores(m, q, device="cuda")
        lse.slmoe_qb_histogram(sc, T, E, q.nbins, hist)
        lse.slmoe_signsgd_update(route(sc, fixed), E, step, fixed)
        del sc
    qbias = torch.empty(E, device="cuda")
    lse.slmoe_qb_update(hist, E, q.nbins, k, None, qbias)
    held = synthetic.qb_scores(q.micro_batches, q, device="cuda")
    out = {}
    for name, b in (("no bias", torch.zeros(E, device="cuda")), (f"{q.micro_batches} fixed steps of {step:g}", fixed),
                    ("QB", qbias)):
        c = route(held, b).double()
        out[name] = round(float(c.max() / c.mean()), 3)
    torch.cuda.synchronize()
    return {"max_over_mean_load": out,
            "held_out": f"micro-batch {q.micro_batches + 1} (seed {q.micro_batches + 1}), {T} tokens x {E} experts, top-{k}",
            "routing": "slmoe_topk on the GPU; histograms and both bias updates on the GPU"}


class LayerRun:
    """One layer configuration on the device: workspace, outputs, the step (slmoe_forward +
    slmoe_qb_update) and, unless disabled, a CUDA graph of that step."""

    def __init__(self, shp, inp, x, mu, use_graph=True, warmup=3, dtype=None):
        import torch
        import latent_space_experts_gb300 as lse
        self.lse, self.shp, self.inp, self.x, self.mu = lse, shp, inp, x, mu
        self.cfg = lse.config(shp, dtype=dtype)
        self.mx = dtype == lse.MXFP4
        self.ws = torch.zeros(lse.slmoe_workspace_size(self.cfg), dtype=torch.uint8, device="cuda")
        self.y = torch.empty(shp.T, shp.d, dtype=torch.float32, device="cuda")
        self.hist = torch.zeros(shp.E, shp.nbins, dtype=torch.int32, device="cuda")
        self.bias = inp["bias"].clone()
        self.status = torch.zeros(4, dtype=torch.int32, device="cuda")
        self.W = lse.weights(inp)
        self.stream = torch.cuda.current_stream()
        for _ in range(max(3, warmup)):
            self.step(self.x)
        torch.cuda.synchronize()
        self.check_status()
        self.graph, self.launches_per_step = None, None
        if use_graph:
            l_cap = lse.slmoe_launch_count()
            self.graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self.graph):
                self.step(self.x)
            self.launches_per_step = lse.slmoe_launch_count() - l_cap
            for _ in range(3):
                self.graph.replay()
            torch.cuda.synchronize()
            self.check_status()

    def step(self, x, out=None):
        shp = self.shp
        self.lse.slmoe_forward(self.cfg, x, self.W, self.bias, self.mu, self.y if out is None else out, None,
                               self.hist, self.status, self.ws)
        self.lse.slmoe_qb_update(self.hist, shp.E, shp.nbins, shp.k, None, self.bias)

    def check_status(self):
        st = self.status.cpu().tolist()
        assert st[1:3] == [0, 0], f"device status {st}"

    def timed(self, steps):
        """ms per step over `steps` steps, CUDA events on the launching stream; and the number
        of this library's kernels launched in that region."""
        import torch
        l0 = self.lse.slmoe_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(self.stream)
        for _ in range(steps):
            if self.graph is not None:
                self.graph.replay()
            else:
                self.step(self.x)
        e1.record(self.stream)
        torch.cuda.synchronize()
        launches = (self.launches_per_step * steps if self.graph is not None
                    else self.lse.slmoe_launch_count() - l0)
        return e0.elapsed_time(e1) / steps, launches

    def counts(self):
        return self.lse.workspace_views(self.cfg, self.ws)["counts"].cpu().numpy()


def backward_work(shp):
    """FLOPs and algorithmic bytes of one slmoe_backward call: every contraction of the
    backward (dgrad and wgrad of the up-projection, shared experts, routed experts and
    down-projection, plus the recomputed pre-activations of both kinds of experts and the
    router's two thin products), and the bytes of the weights read, the fp32 gradients
    written, x and dy read and dx written."""
    T, d, dl, E, k, I, ns, Is = shp.T, shp.d, shp.d_latent, shp.E, shp.k, shp.I, shp.n_shared, shp.I_shared
    Tk = T * k
    flops = (2 * 2 * T * d * dl            # dz, dW_out
             + ns * 2 * T * d * 8 * Is     # gu_s recompute (2 Is), dh_s (Is), dW2_s (Is), dx (2 Is), dW13_s (2 Is)
             + 2 * Tk * dl * 8 * I         # gu recompute (2I), dh (I), dx_lat rows (2I), dW2 (I), dW13 (2I)
             + 2 * 2 * T * dl * d          # dx from dx_lat, dW_in
             + 2 * 2 * Tk * d)             # router: dx and dW_r
    weights = E * d * 4 + dl * d * 2 + E * 3 * I * dl * 2 + d * dl * 2 + ns * 3 * Is * d * 2
    grads = (E * d + dl * d + E * 3 * I * dl + dl + d * dl + ns * 3 * Is * d) * 4
    nbytes = weights + grads + T * d * 2 + T * d * 4 + T * d * 4
    return flops, nbytes


def backward_bench(run, pk, reps=5):
    """slmoe_backward of the bench batch (after one forward that leaves its intermediates in
    the workspace): ms per call, CUDA events on the launching stream, and its roofline."""
    import torch
    lse, shp, cfg = run.lse, run.shp, run.cfg
    g = {n: torch.zeros(run.inp[w].shape, dtype=torch.float32, device="cuda") for n, w in
         (("dW_r", "W_r"), ("dW_in", "W_in"), ("dW13", "W13"), ("dW2", "W2"), ("dgamma", "gamma"),
          ("dW_out", "W_out"), ("dW13_s", "W13_s"), ("dW2_s", "W2_s"))}
    G = lse.grads(g)
    bws = torch.zeros(lse.slmoe_backward_workspace_size(cfg), dtype=torch.uint8, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(5)
    dy = torch.randn(shp.T, shp.d, generator=gen, device="cuda")
    dx = torch.empty(shp.T, shp.d, dtype=torch.float32, device="cuda")
    run.step(run.x)
    st = torch.zeros(4, dtype=torch.int32, device="cuda")
    for _ in range(2):
        lse.slmoe_backward(cfg, run.x, run.W, dy, dx, G, 0, run.ws, st, bws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(run.stream)
    for _ in range(reps):
        lse.slmoe_backward(cfg, run.x, run.W, dy, dx, G, 0, run.ws, st, bws)
    e1.record(run.stream)
    torch.cuda.synchronize()
    assert st.cpu().tolist()[1:3] == [0, 0], st
    ms = e0.elapsed_time(e1) / reps
    flops, nbytes = backward_work(shp)
    tc = pk["bf16_tflops"]
    t_roof = max(flops / (tc * 1e12), nbytes / (pk["hbm_gbs"] * 1e9))
    del g, G, bws
    return {"ms_per_call": round(ms, 3), "tokens_per_s": round(shp.T / (ms * 1e-3), 1),
            "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1),
            "roofline": {"ms": round(t_roof * 1e3, 4), "frac": round(t_roof * 1e3 / ms, 4), "flops": flops,
                         "bytes": nbytes, "tensor_peak_tflops": tc, "hbm_gbs": pk["hbm_gbs"]},
            "note": "weight gradients fp32 (overwritten); contractions on tcgen05 (bf16 operands)"}


def tensor_seconds(st_model, flops, tc, mx):
    """Time of the layer's FLOPs at the tensor peak tc (TFLOP/s); on the MXFP4 layer type the
    routed experts' FLOPs run at MX_TENSOR_RATIO times that rate."""
    routed = st_model["expert gate|up"]["flops"] + st_model["expert down"]["flops"] if mx else 0
    return (flops - routed) / (tc * 1e12) + routed / (MX_TENSOR_RATIO * tc * 1e12)


def layer_summary(run, ms, pk, timed_s, reasons):
    """Tokens/s and the whole-layer roofline of one timed layer configuration."""
    st_model, flops, nbytes = work_model(run.shp, run.counts(), run.mx)
    tc, tc_kind = tensor_peak(pk, timed_s, reasons)
    t_flops, t_bytes = tensor_seconds(st_model, flops, tc, run.mx), nbytes / (pk["hbm_gbs"] * 1e9)
    t_layer = max(t_flops, t_bytes)
    lr = {"ms": round(t_layer * 1e3, 4), "frac": round(t_layer * 1e3 / ms, 4),
          "bound": "tensor" if t_flops >= t_bytes else "hbm", "flops": flops,
          "bytes": nbytes, "tensor_peak_tflops": tc, "tensor_peak": tc_kind, "hbm_gbs": pk["hbm_gbs"]}
    if run.mx:
        lr["routed_expert_tensor_peak"] = f"{MX_TENSOR_RATIO:g} x {tc_kind} (block-scaled FP8 rate, nominal ratio)"
    return {"ms_per_step": round(ms, 4), "tokens_per_s": round(run.shp.T / (ms * 1e-3), 1),
            "layer_roofline": lr, "experts_touched": int((run.counts() > 0).sum())}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="k3_prefill", choices=["k3_prefill", "k3_decode", "mid", "k3_slice", "k3_decode_slice",
                                                                     "k3_dense"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-tokens", type=int, default=None,
                    help="oracle tokens per reference step (default: the cpu_baseline sample)")
    ap.add_argument("--ref-seconds", type=float, default=240.0,
                    help="the reference run shrinks its sample if it would take much longer than this")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the decode / mid sub-results, the QB engine and the QB balance in the line")
    ap.add_argument("--qb-only", action="store_true", help="only the QB engine measurement")
    ap.add_argument("--bwd-only", action="store_true",
                    help="only the backward measurement of the workload (one forward first)")
    ap.add_argument("--no-graph", action="store_true", help="time the step without a CUDA graph")
    ap.add_argument("--skew", action="store_true", help="heavy skew (10%% hot experts)")
    ap.add_argument("--mxfp4", action="store_true",
                    help="run the workload as the MXFP4 layer type (routed-expert weights quantised once)")
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
    pk, pk_kind = peaks()
    hbm = pk["hbm_gbs"]
    if args.qb_only:
        if rank == 0:
            print(json.dumps({"qb_histogram": qb_engine(hbm), "peak_source": pk_kind}))
        return
    shp = synthetic.LAYERS[args.workload]
    inp = synthetic.layer_inputs(shp, seed=rank, device="cuda", heavy_skew=args.skew)
    if args.bwd_only:
        if rank == 0:
            brun = LayerRun(shp, inp, inp["x"], inp["logit_offset"], use_graph=False)
            print(json.dumps({"workload": args.workload, "backward": backward_bench(brun, pk, reps=args.steps)}))
        return
    run_inp = mxfp4_inputs(inp) if args.mxfp4 else inp
    run = LayerRun(shp, run_inp, inp["x"], inp["logit_offset"], use_graph=not args.no_graph, warmup=args.warmup,
                   dtype=lse.MXFP4 if args.mxfp4 else None)
    for _ in range(max(0, args.warmup - 3)):
        run.timed(1)

    # ---------------- device-resident timing
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    if sampler:
        sampler.start()
    barrier(world)
    torch.cuda.synchronize()
    w0 = time.time()
    ms_rank, launches = run.timed(args.steps)
    w1 = time.time()
    barrier(world)
    ms = max_over_ranks(ms_rank, world)
    clocks = sampler.stop(w0, w1) if sampler else None
    timed_s = ms * args.steps * 1e-3
    reasons = clocks["reasons"] if clocks else []
    run.check_status()

    # ---------------- per-stage timing (events recorded by the library on this stream)
    nst = len(STAGES)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nst)] for _ in range(min(args.steps, 50))]
    for row in ev:
        for e in row:
            e.record(run.stream)
    torch.cuda.synchronize()
    stage_ms = [0.0] * nst
    for row in ev:
        lse.slmoe_set_stage_events(row)
        run.step(run.x)
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
    counts = run.counts()
    st_model, layer_flops, layer_bytes = work_model(shp, counts, run.mx)
    tc, tc_kind = tensor_peak(pk, timed_s, reasons)
    stages = {}
    for i in range(1, nst):
        m = st_model[STAGES[i]]
        t = stage_ms[i] * 1e-3
        stages[STAGES[i]] = {"ms": round(stage_ms[i], 4),
                             "GB/s": round(m["bytes"] / t / 1e9, 1) if t > 0 else None,
                             "GB/s_with_intermediates": round((m["bytes"] + m["inter"]) / t / 1e9, 1) if t > 0 else None,
                             "TFLOP/s": round(m["flops"] / t / 1e12, 1) if t > 0 else None,
                             "bound": m["bound"]}
    # the dominant kernel on the critical path (the concurrent front part excluded)
    dom = max((1, 2, 4, 5, 6, 8), key=lambda i: stage_ms[i])
    dm = st_model[STAGES[dom]]
    t_dom = stage_ms[dom] * 1e-3
    if dm["bound"] == "hbm":
        roof = {"bound": "hbm", "achieved": round(dm["bytes"] / t_dom / 1e9, 1), "peak": hbm, "unit": "GB/s"}
        roof["achieved_with_intermediates"] = round((dm["bytes"] + dm["inter"]) / t_dom / 1e9, 1)
        roof["peak_source"] = f"{pk_kind} hbm copy"
    else:
        roof = {"bound": "tensor", "achieved": round(dm["flops"] / t_dom / 1e12, 1), "peak": tc,
                "unit": "TFLOP/s", "peak_source": f"{pk_kind} {tc_kind}"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = profiled_traffic(STAGES[dom]) if args.workload == "k3_prefill" else None
    roof["kernel"] = STAGES[dom]
    roof["algorithmic_bytes"] = dm["bytes"]
    summary = layer_summary(run, ms, pk, timed_s, reasons)
    lr = summary["layer_roofline"]
    t_sus = max(tensor_seconds(st_model, layer_flops, pk["bf16_tflops_sustained"], run.mx), layer_bytes / (hbm * 1e9))
    lr["frac_vs_sustained_peak"] = round(t_sus * 1e3 / ms, 4)

    # ---------------- end to end through the public API, host buffers
    # Every step uploads its input from pinned host memory and reads its result back.  As a
    # serving loop would, the copies run on their own streams with two device buffers each, so
    # that step i+1's upload and step i's read-back overlap the compute of the steps beside them;
    # the timed region runs from before the first upload to the end of the last read-back.
    stream, y = run.stream, run.y
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
            run.step(x_dev[b], y_dev[b])
            done[b] = stream.record_event()
            s_out.wait_event(done[b])
            with torch.cuda.stream(s_out):
                y_host[b].copy_(y_dev[b], non_blocking=True)
                out[b] = s_out.record_event()
        for ev_ in out:
            if ev_ is not None:
                stream.wait_event(ev_)

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
    run.check_status()
    assert torch.equal(y_host[(n_e2e - 1) % 2], y_dev[(n_e2e - 1) % 2].cpu())
    ms_e2e = max_over_ranks(f0.elapsed_time(f1), world) / n_e2e
    del x_host, y_host, x_dev, y_dev

    # ---------------- the other layer workloads and the QB engine (rank 0, reported only)
    extra = {}
    qb = qb_engine(hbm) if rank == 0 and not args.no_extra else None
    if rank == 0 and not args.no_extra:
        if args.workload == "k3_prefill":
            # K3 decode: the same weights, the first 128 tokens of the batch; uniform and with
            # heavy skew (10 % of the experts get +2 on their logit offset)
            dshp = synthetic.LAYERS["k3_decode"]
            for name, skew in (("k3_decode", False), ("k3_decode_heavy_skew", True)):
                mu = synthetic.logit_offset(dshp, seed=rank, device="cuda", heavy_skew=skew)
                drun = LayerRun(dshp, inp, inp["x"][: dshp.T].contiguous(), mu)
                dms, _ = drun.timed(200)
                extra[name] = layer_summary(drun, dms, pk, dms * 0.2, reasons)
                del drun
        if args.workload == "k3_prefill":
            # the MXFP4 layer type: the same weights with the routed experts quantised once
            mx = mxfp4_inputs(inp)
            for name, T in (("k3_decode_mxfp4", 128), ("k3_prefill_mxfp4", shp.T)):
                s_mx = synthetic.shape_with(shp, T=T)
                mrun = LayerRun(s_mx, mx, inp["x"][:T].contiguous(), inp["logit_offset"], dtype=lse.MXFP4)
                mms, _ = mrun.timed(100)
                extra[name] = layer_summary(mrun, mms, pk, mms * 0.1, reasons)
                extra[name]["note"] = ("routed experts on the block-scaled tensor cores: weights MXFP4 (E2M1 + "
                                       "E8M0 per 32), x_lat and h MXFP8 (E4M3 + E8M0 per 32); the rest as the "
                                       "bf16 layer")
                del mrun
            del mx
        mshp = synthetic.LAYERS["mid"]
        minp = synthetic.layer_inputs(mshp, seed=0, device="cuda")
        mrun = LayerRun(mshp, minp, minp["x"], minp["logit_offset"])
        mms, _ = mrun.timed(200)
        extra["mid"] = layer_summary(mrun, mms, pk, mms * 0.2, reasons)
        del mrun, minp
        extra["qb_balance"] = qb_balance()
        if args.workload == "k3_prefill":
            extra["k3_prefill_backward"] = backward_bench(run, pk)

    # ---------------- oracle on the host cores (the same sample the reference arm times)
    cpu_base = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        inp_cpu = oracle_inputs(inp)
        n_tok = min(shp.T, CPU_SAMPLE_TOKENS)
        oracle_sample(shp, inp_cpu, min(n_tok, 16))          # page in the widened inputs
        v_all, dt_all = oracle_sample_threads(shp, inp_cpu, n_tok, None)
        v_one, dt_one = oracle_sample_threads(shp, inp_cpu, n_tok, 1)
        cpu_base = {"value": round(v_all, 3), "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                    "sample": f"the first {n_tok} tokens of the {args.workload} batch, fp64 numpy "
                              f"({dt_all:.1f} s on all cores)",
                    "one_thread": ({"value": round(v_one, 3), "seconds": round(dt_one, 1)} if v_one
                                   else "BLAS thread count not settable here")}

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
                       "routed_expert_weights": "mxfp4" if args.mxfp4 else "bf16",
                       "parallelism": f"replicas x{world}",
                       "l2": "no flush: weights (10.2 GB at K3) exceed L2 every step",
                       "cuda_graph": run.graph is not None},
            "roofline": roof,
            "layer_roofline": lr,
            "stages": stages,
            "qb_histogram": qb,
            "workloads": extra,
            "cpu_baseline": cpu_base,
            "e2e": {"value": round(job_throughput(tokens, world, ms_e2e), 1), "unit": UNIT,
                    "h2d_bytes_per_step": inp["x"].numel() * inp["x"].element_size(),
                    "d2h_bytes_per_step": y.numel() * y.element_size(),
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
