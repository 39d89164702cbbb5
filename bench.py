"""Benchmark of one Muon/NorMuon optimizer step on the GPT-2-124M body.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

Prints ONE JSON line (rank 0).  The step is the whole hot path -- momentum,
Nesterov, normalisation, five Newton-Schulz iterations, NorMuon, write-back --
on seeded synthetic gradients (a bank of 4 gradient sets cycled through,
inputs larger than L2).  ``value`` is device time per step (CUDA graph of
``muon_step``, CUDA events, max over ranks); ``e2e`` is the same step through
the public Python API with the step's gradients copied in from pinned host
memory and the updated parameters copied back, inside the timed region, the
copies of neighbouring steps overlapping the step on two copy streams
(``e2e.serial_ms``: the same with every copy on the step's stream).
Per-kernel times come from a second pass of K steps with per-stage CUDA
events.  ``--impl reference`` times the fp64 CPU oracle on a bounded sample of
the same workload instead.  With torchrun (N > 1) every rank runs an
independent replica of the workload on its own GPU (no data-path collective).
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Muon/NorMuon step ms on GPT-2-124M body; NS TFLOP/s & % of bf16 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ---------------------------------------------------------------------------- work model

def work_model(wl, grad_bytes):
    """Algorithmic flops / bytes of one step of workload ``wl``."""
    ns = wl.ns_steps
    gram = poly = upd = 0
    gram_b = poly_b = upd_first_b = upd_b = 0
    elems = 0
    for (r, c) in wl.sub_shapes():
        m, n = min(r, c), max(r, c)
        gram += m * (m + 1) * n          # upper triangle of X X^T (incl. diagonal)
        poly += m * m * (m + 1)          # upper triangle of A A
        upd += 2 * m * m * n             # P X
        elems += r * c
        # HBM bytes per launch (2-byte elements): the first iteration works on u
        # (bf16 hi + lo), later ones on the fp16 iterate
        gram_b += 2 * m * n + 2 * m * m            # read X (u hi), write A
        poly_b += 2 * m * m + 2 * m * m            # read A, write P
        upd_first_b += 2 * m * m + 3 * 2 * m * n   # read P, u hi, u lo; write X1
        upd_b += 2 * m * m + 2 * 2 * m * n         # read P, X; write X' 
    return {
        "elems": elems,
        "gram_flops": gram, "poly_flops": poly, "update_flops": upd,
        "gram_bytes": gram_b, "poly_bytes": poly_b,
        "update_bytes": (upd_first_b + (ns - 1) * upd_b) / ns,   # mean per launch
        "ns_flops": ns * (gram + poly + upd),
        "ns_flops_dense": ns * sum(4 * min(r, c) ** 2 * max(r, c) + 2 * min(r, c) ** 3 for r, c in wl.sub_shapes()),
        "momentum_bytes": elems * (grad_bytes + 4 + 4 + 2 + 2),   # g, buf r/w, u as bf16 hi + lo
        "apply_bytes": elems * (2 + 4 + 4),                        # O bf16, p r/w
    }


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        power = [num(r[3]) for r in rows if num(r[3]) is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ---------------------------------------------------------------------------- oracle timing

_ORACLE_INPUTS = {}


def oracle_sample_time(wl, layers=1, repeats=1, seed_step=0):
    """fp64 oracle on the first ``layers`` layers' matrices.

    Returns a dict: ``sample_ms`` (the fastest of ``repeats`` timings of one
    step of the sample), ``scale`` (parameters of the workload / parameters
    sampled; every layer holds the same shapes), ``ms`` = sample_ms * scale,
    and a description of the sample.
    """
    import numpy as np

    import oracle
    from workloads import grads_for, params_for

    per_layer = 3
    nl = max(1, len(wl.matrices) // per_layer)
    layers = max(1, min(layers, nl))
    idx = list(range(min(len(wl.matrices), layers * per_layer)))
    shapes = [(wl.matrices[i].rows, wl.matrices[i].cols, wl.matrices[i].split, wl.matrices[i].lr_mul,
               wl.matrices[i].wd_mul) for i in idx]
    key = (wl.name, layers, seed_step)
    if key not in _ORACLE_INPUTS:  # drawing the inputs is not part of the timed oracle step
        _ORACLE_INPUTS[key] = ([p.double().numpy() for p in params_for(wl, idx)],
                               [g.double().numpy() for g in grads_for(wl, seed_step, indices=idx)])
    params, grads = _ORACLE_INPUTS[key]
    cfg = oracle.OracleConfig(lr=wl.lr, momentum=wl.momentum, beta2=wl.beta2, ns_steps=wl.ns_steps,
                              normuon=wl.normuon)
    times = []
    for _ in range(repeats):
        orc = oracle.MuonOracle(shapes, cfg)
        t0 = time.perf_counter()
        orc.step(params, grads)
        times.append(time.perf_counter() - t0)
    scale = len(wl.matrices) / len(idx)
    sample_ms = min(times) * 1e3
    desc = (f"{layers} of {nl} layers ({len(idx)} of {len(wl.matrices)} parameters), one step, fp64 numpy, "
            f"fastest of {repeats}" + ("" if scale == 1 else f", scaled x{scale:g} to the whole workload"))
    return {"ms": sample_ms * scale, "sample_ms": sample_ms, "scale": scale, "layers": layers, "repeats": repeats,
            "sample": desc}


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count()


# ---------------------------------------------------------------------------- ranks
def rank_barrier(world):
    """Barrier over the ranks of a multi-GPU run (replicas: each rank steps its own copy)."""
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def rank_max(x, world, device):
    """Max of a per-rank time over all ranks (the slowest replica sets the step time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------- reference arm

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from workloads import workload

    wl = workload(args.workload)
    # size the per-step sample so that warm-up + timed steps take about --ref-budget seconds:
    # the whole workload when that fits, else the largest number of layers that does
    probe = oracle_sample_time(wl, layers=1)
    nl = max(1, len(wl.matrices) // 3)
    per_step_s = args.ref_budget / (args.steps + args.warmup)
    layers = int(max(1, min(nl, per_step_s // max(probe["sample_ms"] * 1e-3, 1e-9))))
    for k in range(args.warmup):
        oracle_sample_time(wl, layers=layers, seed_step=k % 4)
    runs = [oracle_sample_time(wl, layers=layers, seed_step=k % 4) for k in range(args.steps)]
    v = statistics.mean(r["ms"] for r in runs)
    sample_ms = statistics.mean(r["sample_ms"] for r in runs)
    scale = runs[0]["scale"]
    sample = runs[0]["sample"]
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "ms", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": v, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "description": wl.description},
        "sample_ms_per_step": sample_ms, "scale": scale,
        "cpu_baseline": {"value": v, "unit": "ms", "cores": cores(), "kind": "oracle", "sample": sample,
                         "sample_ms": sample_ms, "scale": scale},
        "e2e": {"value": v, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- our arm

def adam_measure(args, dev, hbm):
    """Graph-replayed fused Adam step on the GPT-2 embedding / head / scalar groups."""
    import torch

    from optimizer_nesterov_momentum_gb300 import AdamGroup, AdamTensorSpec
    from workloads import adam_grads_for, adam_params_for, adam_workload

    wl = adam_workload("gpt2-124m-adam")
    grp = AdamGroup([AdamTensorSpec(t.numel, t.lr, t.weight_decay) for t in wl.tensors], grad_dtype=wl.grad_dtype)
    params = [p.reshape(-1).to(dev) for p in adam_params_for(wl)]
    bank = [[g.reshape(-1).to(dev) for g in adam_grads_for(wl, k)] for k in range(2)]
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for k in range(3):
            grp.step(params, bank[k % 2])
    torch.cuda.current_stream().wait_stream(stream)
    graphs = []
    for k in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            grp.step(params, bank[k])
        graphs.append(g)
    for k in range(3):
        graphs[k % 2].replay()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for k in range(args.steps):
        graphs[k % 2].replay()
    end.record()
    torch.cuda.synchronize()
    ms = start.elapsed_time(end) / args.steps
    nbytes = wl.numel * (2 + 3 * 4 + 3 * 4)   # g bf16; p, m, v read and written
    gbs = nbytes / (ms * 1e-3) / 1e9
    launches = grp.launch_count()
    grp.close()
    return {"workload": wl.name, "description": wl.description, "elements": wl.numel, "ms": ms,
            "bound": "hbm", "achieved": gbs, "unit": "GB/s", "peak": hbm, "frac": gbs / hbm,
            "algorithmic_per_step": nbytes, "gpu_launches": launches * args.steps,
            "launch": "cuda graph of muon_adam_step", "l2": "inputs larger than L2 (2.0 GB per step)"}


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__

    __graft_entry__.build()
    from optimizer_nesterov_momentum_gb300 import MatrixSpec, Muon
    from workloads import grads_for, params_for, workload

    wl = workload(args.workload)
    nbank = 4
    specs = [MatrixSpec(m.rows, m.cols, m.split, m.lr_mul, m.wd_mul) for m in wl.matrices]
    params = [p.to(dev) for p in params_for(wl)]
    bank = [[g.to(dev) for g in grads_for(wl, k, device=str(dev))] for k in range(nbank)]
    grad_bytes = 2 if wl.grad_dtype == "bf16" else 4
    opt = Muon(specs, lr=wl.lr, momentum=wl.momentum, beta2=wl.beta2, weight_decay=wl.weight_decay,
               ns_steps=wl.ns_steps, normuon=wl.normuon, grad_dtype=wl.grad_dtype, ns_form=args.ns_form)
    launches = opt.launch_count()
    model = work_model(wl, grad_bytes)

    # warm-up (eager), then capture one graph per gradient set, then reset state
    stream = torch.cuda.Stream(device=dev)
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        for k in range(max(args.warmup, 3)):
            opt.step(params, bank[k % nbank])
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    graphs = []
    for k in range(nbank):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            opt.step(params, bank[k])
        graphs.append(g)
    opt.reset()
    for k in range(max(args.warmup, 3)):
        graphs[k % nbank].replay()
    opt.sync_status()

    def barrier():
        rank_barrier(world)

    def max_over_ranks(x):
        return rank_max(x, world, dev)

    # ---- timed region: graph replays
    barrier()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        start.record()
        for k in range(args.steps):
            graphs[k % nbank].replay()
        end.record()
        torch.cuda.synchronize()
    barrier()
    ms = max_over_ranks(start.elapsed_time(end) / args.steps)
    clocks = clk.summary()

    # ---- spread of single steps: a second pass with an event after every replay
    # (the events add about 1 % to a step, so ``value`` comes from the pass above)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    torch.cuda.synchronize()
    marks[0].record()
    for k in range(args.steps):
        graphs[k % nbank].replay()
        marks[k + 1].record()
    torch.cuda.synchronize()
    per_step = [marks[k].elapsed_time(marks[k + 1]) for k in range(args.steps)]
    step_stats = {"mean": statistics.fmean(per_step), "median": statistics.median(per_step),
                  "std": statistics.pstdev(per_step), "min": min(per_step), "max": max(per_step),
                  "pass": "second pass, one event per replay"}
    opt.sync_status()

    # ---- eager step timing (same work, launched through the API each step)
    torch.cuda.synchronize()
    start.record()
    for k in range(args.steps):
        opt.step(params, bank[k % nbank])
    end.record()
    torch.cuda.synchronize()
    eager_ms = max_over_ranks(start.elapsed_time(end) / args.steps)

    # ---- per-stage times: second pass with CUDA events around every launch
    opt.set_profiling(True)
    acc = None
    for k in range(args.steps):
        opt.step(params, bank[k % nbank])
        st = opt.stage_times()
        acc = st if acc is None else {kk: acc[kk] + st[kk] for kk in acc}
    opt.set_profiling(False)
    stage_ms = {kk: v / args.steps for kk, v in acc.items()}

    # ---- end to end through the public API with host buffers: every step copies its
    # gradients in from pinned host memory and reads the updated parameters back.  Each
    # step's gradients, the parameters and their snapshots live in single flat buffers
    # (the matrices are views into them), so a step enqueues three copies instead of one
    # per matrix and direction: the host's enqueue rate cannot set the pace.
    def flat_views(flat, like):
        out, o = [], 0
        for t in like:
            out.append(flat[o:o + t.numel()].view(t.shape))
            o += t.numel()
        return out

    n_grad = sum(g.numel() for g in bank[0])
    n_param = sum(p.numel() for p in params)
    gdt = bank[0][0].dtype
    host_grads = []
    for gs in bank:
        hf = torch.empty(n_grad, dtype=gdt).pin_memory()
        for dst, src in zip(flat_views(hf, gs), gs):
            dst.copy_(src.cpu())
        host_grads.append(hf)
    host_params = torch.empty(n_param, dtype=torch.float32).pin_memory()
    pflat = torch.empty(n_param, dtype=torch.float32, device=dev)
    e2e_params = flat_views(pflat, params)
    for dst, src in zip(e2e_params, params):
        dst.copy_(src)
    h2d = n_grad * host_grads[0].element_size()
    d2h = n_param * 4
    main = torch.cuda.current_stream()

    # serial: copy in, step, copy out, all on one stream
    gflat = torch.empty(n_grad, dtype=gdt, device=dev)
    dev_grads = flat_views(gflat, bank[0])
    torch.cuda.synchronize()
    barrier()
    start.record()
    for k in range(args.steps):
        gflat.copy_(host_grads[k % nbank], non_blocking=True)
        opt.step(e2e_params, dev_grads)
        host_params.copy_(pflat, non_blocking=True)
    end.record()
    torch.cuda.synchronize()
    barrier()
    e2e_serial_ms = max_over_ranks(start.elapsed_time(end) / args.steps)

    # pipelined: step k+1's gradients are copied in on one stream while step k runs
    # (device gradients double-buffered), and step k's parameters are snapshotted on
    # the device and copied out on another stream while step k+1 runs
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    dgr_flat = [torch.empty(n_grad, dtype=gdt, device=dev) for _ in range(2)]
    dgr = [flat_views(f, bank[0]) for f in dgr_flat]
    snap = [torch.empty(n_param, dtype=torch.float32, device=dev) for _ in range(2)]
    in_done = [torch.cuda.Event() for _ in range(2)]
    step_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def copy_in(k):
        slot = k % 2
        with torch.cuda.stream(s_in):
            if k >= 2:
                s_in.wait_event(step_done[slot])  # step k - 2 is done with this buffer
            dgr_flat[slot].copy_(host_grads[k % nbank], non_blocking=True)
            in_done[slot].record(s_in)

    def pipelined_pass():
        torch.cuda.synchronize()
        barrier()
        start.record(main)
        copy_in(0)
        for k in range(args.steps):
            slot = k % 2
            if k + 1 < args.steps:
                copy_in(k + 1)
            main.wait_event(in_done[slot])
            opt.step(e2e_params, dgr[slot], stream=main)
            if k >= 2:
                main.wait_event(out_done[slot])  # the copy-out of step k - 2 is done with this snapshot
            snap[slot].copy_(pflat, non_blocking=True)
            step_done[slot].record(main)
            with torch.cuda.stream(s_out):
                s_out.wait_event(step_done[slot])
                host_params.copy_(snap[slot], non_blocking=True)
                out_done[slot].record(s_out)
        main.wait_stream(s_in)
        main.wait_stream(s_out)
        end.record(main)
        torch.cuda.synchronize()
        barrier()
        return max_over_ranks(start.elapsed_time(end) / args.steps)

    # the host link's rate varies from run to run (other tenants of the machine share it):
    # three passes, the median reported, all three listed
    e2e_passes = [pipelined_pass() for _ in range(3)]
    e2e_ms = statistics.median(e2e_passes)
    opt.sync_status()

    # ---- roofline of each stage.  The tensor peak is the burst figure when the clock record
    # shows the SMs at (or near) their maximum with no power cap -- a short timed region, as
    # here -- and the sustained (power-capped) figure otherwise; both fractions are reported.
    peaks, peak_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    tc_burst = float(peaks["bf16_tflops"])
    tc_sustained = float(peaks.get("bf16_tflops_sustained", tc_burst))
    at_max = (clocks.get("sm_mhz") is not None and clocks.get("sm_max_mhz")
              and clocks["sm_mhz"] >= 0.95 * clocks["sm_max_mhz"] and "sw_power_cap" not in clocks["reasons"])
    tc_peak = tc_burst if at_max else tc_sustained
    tc_key = "bf16_tflops" if at_max else "bf16_tflops_sustained"
    nsi = wl.ns_steps
    kern = {}
    kern["momentum"] = {"ms": stage_ms["momentum"], "bound": "hbm",
                        "achieved": model["momentum_bytes"] / (stage_ms["momentum"] * 1e-3) / 1e9, "unit": "GB/s",
                        "algorithmic_per_launch": model["momentum_bytes"]}
    kern["apply"] = {"ms": stage_ms["apply"], "bound": "hbm",
                     "achieved": model["apply_bytes"] / (stage_ms["apply"] * 1e-3) / 1e9, "unit": "GB/s",
                     "algorithmic_per_launch": model["apply_bytes"]}
    # the Newton-Schulz stages' work as the library planned it (the Gram-pair order moves
    # m x m products into the Gram and update launches and adds a product stage)
    planned = opt.stage_work()
    for name in ("gram", "poly", "update", "product"):
        # a product is bound by whichever of its flops (at the tensor peak) and its
        # HBM bytes (at the copy peak) takes longer; both fractions are reported
        fl_step, by_step, n_launch = planned[name]
        if n_launch == 0:
            continue
        per_launch_ms = stage_ms[name] / n_launch
        flops, nbytes = fl_step / n_launch, by_step / n_launch
        tflops = flops / (per_launch_ms * 1e-3) / 1e12
        gbs = nbytes / (per_launch_ms * 1e-3) / 1e9
        hbm_bound = nbytes / hbm > flops / 1e3 / tc_peak
        kern[name] = {"ms": stage_ms[name], "ms_per_launch": per_launch_ms, "launches": n_launch,
                      "bound": "hbm" if hbm_bound else "tensor",
                      "achieved": gbs if hbm_bound else tflops, "unit": "GB/s" if hbm_bound else "TFLOP/s",
                      "algorithmic_per_launch": nbytes if hbm_bound else flops,
                      "tflops": tflops, "frac_tensor": tflops / tc_peak,
                      "frac_tensor_burst": tflops / tc_burst, "frac_tensor_sustained": tflops / tc_sustained,
                      "gbs": gbs, "frac_hbm": gbs / hbm, "bytes_per_launch": nbytes, "flops_per_launch": flops}
    for name in ("norm_scale", "lane_stats"):
        kern[name] = {"ms": stage_ms[name]}
    for k, v in kern.items():
        if "achieved" in v:
            v["peak"] = hbm if v["unit"] == "GB/s" else tc_peak
            v["frac"] = v["achieved"] / v["peak"]
    ns_ms = stage_ms["gram"] + stage_ms["poly"] + stage_ms["update"] + stage_ms.get("product", 0.0)
    ns_flops_exec = sum(planned[k][0] for k in ("gram", "poly", "update", "product"))
    ns_tflops = ns_flops_exec / (ns_ms * 1e-3) / 1e12
    total_stage = sum(stage_ms.values())
    dom = max((k for k in ("momentum", "apply", "gram", "poly", "update", "product") if k in kern),
              key=lambda k: kern[k]["ms"])
    # DRAM traffic per launch of the dominant kernel, from the single-pass ncu capture summarised in
    # profiles/dram_traffic_<workload>.md (a line "traffic_bytes_per_launch <stage> <bytes>")
    traffic = None
    tr_path = os.path.join(ROOT, "profiles", f"dram_traffic_{wl.name}.md")
    # the capture was taken in the default (Gram-pair) order; another order's launches differ
    if os.path.exists(tr_path) and args.ns_form == "gram_pairs":
        with open(tr_path) as f:
            for line in f:
                parts = line.split()
                if len(parts) == 3 and parts[0] == "traffic_bytes_per_launch" and parts[1] == dom:
                    traffic = float(parts[2])
    d = kern[dom]
    roofline = {"bound": d["bound"], "achieved": d["achieved"], "peak": d["peak"], "unit": d["unit"],
                "frac": d["frac"], "traffic": traffic, "kernel": dom,
                "algorithmic_bytes_per_launch": d.get("bytes_per_launch", d.get("algorithmic_per_launch")),
                "peak_source": f"{peak_src} ({'hbm_gbs' if d['unit'] == 'GB/s' else tc_key})",
                "share_of_step": d["ms"] / total_stage}
    if d["unit"] == "TFLOP/s":
        roofline["frac_burst"] = d["achieved"] / tc_burst
        roofline["frac_sustained"] = d["achieved"] / tc_sustained
        roofline["peak_choice"] = ("burst: SM clock at maximum, no power cap during the timed region" if at_max
                                   else "sustained: SM clock below maximum or power-capped during the timed region")

    adam = None if args.no_adam else adam_measure(args, dev, hbm)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        r = oracle_sample_time(wl, layers=args.cpu_layers, repeats=3)
        cpu = {"value": r["ms"], "unit": "ms", "cores": cores(), "kind": "oracle", "sample": r["sample"],
               "sample_ms": r["sample_ms"], "scale": r["scale"]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": ms, "unit": "ms", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16+fp16", "data": "synthetic",
            "config": {"workload": wl.name, "description": wl.description, "matrices": len(wl.sub_shapes()),
                       "elements": model["elems"], "ns_steps": nsi, "grad_dtype": wl.grad_dtype,
                       "launch": "cuda graph of muon_step",
                       "tensor_core_operands": "bf16 (first Newton-Schulz iteration), fp16 (later ones); fp32 state",
                       "l2": "inputs larger than L2 (grads+params+momentum "
                       f"{(model['elems'] * (grad_bytes + 8)) / 1e6:.0f} MB > 129 MB)",
                       "parallelism": "replicas" if world > 1 else "single"},
            "ns": {"order": args.ns_form,
                   "tflops_algorithmic": ns_tflops, "flops_algorithmic": ns_flops_exec,
                   "frac_of_bf16_peak": ns_tflops / tc_peak,
                   "frac_of_burst": ns_tflops / tc_burst, "frac_of_sustained": ns_tflops / tc_sustained,
                   "flops_standard_order": model["ns_flops"],
                   "tflops_standard_order_equivalent": model["ns_flops"] / (ns_ms * 1e-3) / 1e12,
                   "tflops_dense_equivalent": model["ns_flops_dense"] / (ns_ms * 1e-3) / 1e12,
                   "ms": ns_ms, "peak_tflops": tc_peak, "peak_source": f"{peak_src} ({tc_key})",
                   "note": "tflops_algorithmic: the products the step runs (symmetric ones counted once per "
                           "upper-triangle element); the *_equivalent rates divide the standard order's work "
                           "by the same time"},
            "eager_ms_per_step": eager_ms,
            "kernels": kern,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "step_ms_stats": step_stats,
            "e2e": {"value": e2e_ms, "unit": "ms", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelined": True, "passes_ms": e2e_passes, "serial_ms": e2e_serial_ms,
                    "note": "gradients copied in from pinned host memory and parameters read back every step; "
                            "copies of neighbouring steps overlap the step on two copy streams; one flat "
                            "buffer per direction (three copies per step); median of three timed passes"},
            "gpu_launches": launches * args.steps,
            "clocks": clocks,
            "next_rows": {"adam": adam},
        }
        print(json.dumps(line), flush=True)
    opt.close()
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="gpt2-124m")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-layers", type=int, default=2)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-adam", action="store_true", help="skip the Adam-group measurement")
    ap.add_argument("--ns-form", default="gram_pairs", choices=["gram_pairs", "standard"],
                    help="order of the Newton-Schulz products (muon_config.ns_form)")
    ap.add_argument("--ref-budget", type=float, default=150.0,
                    help="seconds the reference arm (the fp64 oracle) may spend on warm-up + timed steps")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
