"""Worst parity errors of the CUDA path against the fp64 oracle, per named workload.

Runs the same comparison as the GPU parity tests (tests/parity_util.py) and
prints one JSON line per workload with the largest relative Frobenius error of
each checked quantity and the NS-dependent errors divided by their bound
(<= 1 passes).  Needs a GPU.  Usage:

    python -m tests.parity_report [workload ...]
"""

import json
import sys

from tests.parity_util import Shape, run_parity
from workloads import grads_for, params_for, workload

# (workload, steps, sampled parents or None for all, oracle NS implementation)
CASES = {
    "tiny": (1, None, "iterate"),
    "gpt2-124m": (1, None, "iterate"),
    "gpt2-124m-normuon-200": (5, None, "iterate"),
    "gpt2-medium": (1, [0, 1, 2, 70, 71], "iterate"),
    "stress": (1, [0, 20], "closed_form"),
}


def report(name):
    steps, sample, impl = CASES[name]
    wl = workload(name)
    shapes = [Shape(m.rows, m.cols, m.split, m.lr_mul, m.wd_mul) for m in wl.matrices]
    big = name in ("gpt2-medium", "stress")
    grads = [[g.cpu() for g in grads_for(wl, k, device="cuda" if big else None)] for k in range(steps)]
    errs, _, _ = run_parity(shapes, params_for(wl), grads, lr=wl.lr, momentum=wl.momentum, beta2=wl.beta2,
                            ns_steps=wl.ns_steps, normuon=wl.normuon, grad_dtype=wl.grad_dtype,
                            check_parents=sample, ns_impl=impl)
    keys = ["momentum", "ortho", "v_stage", "v_e2e", "delta_stage", "delta_e2e", "ortho_ratio", "v_e2e_ratio",
            "delta_e2e_ratio"]
    return {"workload": name, "steps": steps, "parents_checked": "all" if sample is None else sample,
            "oracle_ns": impl, **{k: getattr(errs, k) for k in keys}}


def main():
    names = sys.argv[1:] or list(CASES)
    for n in names:
        print(json.dumps(report(n)), flush=True)


if __name__ == "__main__":
    main()
