"""Runs a few eager optimizer steps of a named synthetic workload and exits.

A minimal driver for profilers (one muon_step per iteration, no CUDA graphs,
no timing, no oracle), e.g.

    python run_steps.py --workload gpt2-124m --steps 2
    python run_steps.py --adam gpt2-124m-adam --steps 3
"""

from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="gpt2-124m")
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--engine", default="tcgen05", choices=["tcgen05", "simt"])
    ap.add_argument("--adam", default=None, help="run the Adam group of this workload instead")
    a = ap.parse_args()
    if a.adam:
        return run_adam(a)

    import torch

    from optimizer_nesterov_momentum_gb300 import MatrixSpec, Muon, build
    from workloads import grads_for, params_for, workload

    build.build()
    wl = workload(a.workload)
    specs = [MatrixSpec(m.rows, m.cols, m.split, m.lr_mul, m.wd_mul) for m in wl.matrices]
    params = [p.cuda() for p in params_for(wl)]
    grads = [g.cuda() for g in grads_for(wl, 0, device="cuda")]
    opt = Muon(specs, lr=wl.lr, momentum=wl.momentum, beta2=wl.beta2, ns_steps=wl.ns_steps, normuon=wl.normuon,
               grad_dtype=wl.grad_dtype, gemm_engine=a.engine)
    for _ in range(a.steps):
        opt.step(params, grads)
    opt.sync_status()
    torch.cuda.synchronize()
    print(f"ran {a.steps} steps of {wl.name} ({opt.launch_count()} launches per step)")
    opt.close()


def run_adam(a):
    import torch

    from optimizer_nesterov_momentum_gb300 import AdamGroup, AdamTensorSpec, build
    from workloads import adam_grads_for, adam_params_for, adam_workload

    build.build()
    wl = adam_workload(a.adam)
    grp = AdamGroup([AdamTensorSpec(t.numel, t.lr, t.weight_decay) for t in wl.tensors], grad_dtype=wl.grad_dtype)
    params = [p.reshape(-1).cuda() for p in adam_params_for(wl)]
    grads = [g.reshape(-1).cuda() for g in adam_grads_for(wl, 0)]
    for _ in range(a.steps):
        grp.step(params, grads)
    torch.cuda.synchronize()
    print(f"ran {a.steps} Adam steps of {wl.name} ({grp.launch_count()} launches per step)")
    grp.close()


if __name__ == "__main__":
    main()
