"""Seeded synthetic workloads shared by the oracle-side tests and the GPU path.

This package only *describes* shapes and *draws* inputs (parameters and
gradients).  It holds none of the optimizer's arithmetic: no momentum, no
normalisation, no Newton-Schulz, no second moment.  Both the fp64 oracle and
the CUDA path consume exactly the bits produced here.
"""

from .shapes import MatrixShape, WORKLOADS, workload
from .adam import ADAM_WORKLOADS, AdamTensor, AdamWorkload, adam_grads_for, adam_params_for, adam_workload
from .generators import (
    lowrank_plus_noise,
    power_law_spectrum,
    log_uniform_spectrum,
    gaussian_params,
    grads_for,
    params_for,
    seed_for,
)

__all__ = [
    "ADAM_WORKLOADS",
    "AdamTensor",
    "AdamWorkload",
    "adam_grads_for",
    "adam_params_for",
    "adam_workload",
    "MatrixShape",
    "WORKLOADS",
    "workload",
    "lowrank_plus_noise",
    "power_law_spectrum",
    "log_uniform_spectrum",
    "gaussian_params",
    "grads_for",
    "params_for",
    "seed_for",
]
