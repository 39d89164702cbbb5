"""Runs a few eager optimizer steps of a named synthetic workload and exits.

A minimal driver for profilers (one muon_step per iteration, no CUDA graphs,
no timing, no oracle), e.g.

    python -m optimizer_nesterov_momentum_gb300.run_steps --workload gpt2-124m --steps 2
"""

from __future__ import annotations

import argparse
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="gpt2-124m")
    ap.add_argument("--steps", type=int, default=2)
    ap.add_argument("--engine", default="tcgen05", choices=["tcgen05", "simt"])
    a = ap.parse_args()

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


if __name__ == "__main__":
    main()
