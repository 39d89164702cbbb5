"""fp64 CPU oracle of the Muon / NorMuon optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may use it.  It
shares no code with the CUDA path; the two meet only through the seeded
inputs of the ``workloads`` package.

Pinned by ``tests/test_oracle_pins.py`` against closed forms (the SVD form of
an odd matrix polynomial, the classic Newton-Schulz limit U V^T), invariants
(the singular-value band, norm preservation), hand-derived recurrences and a
second pure-Python brute-force implementation on an 8 x 16 matrix.
"""

from .muon_oracle import (
    NS_COEFFS,
    NORM_EPS,
    V_FLOOR,
    FP32_MAX,
    OracleConfig,
    MuonOracle,
    bf16_round,
    fp16_round,
    momentum_update,
    nesterov_direction,
    split_matrix,
    merge_matrix,
    orient_wide,
    frobenius_normalise,
    newton_schulz,
    newton_schulz_closed_form,
    zeropower_via_newtonschulz5,
    normuon_scale,
    shape_scale,
    write_back,
)
from .schedules import lr_multiplier, scheduled_lr, scheduled_momentum
from .adam_oracle import ADAM_BETAS, ADAM_EPS, AdamConfig, AdamOracle, adam_moments, adam_param_update

__all__ = [
    "ADAM_BETAS",
    "ADAM_EPS",
    "AdamConfig",
    "AdamOracle",
    "adam_moments",
    "adam_param_update",
    "lr_multiplier",
    "scheduled_lr",
    "scheduled_momentum",
    "NS_COEFFS",
    "NORM_EPS",
    "V_FLOOR",
    "FP32_MAX",
    "OracleConfig",
    "MuonOracle",
    "bf16_round",
    "fp16_round",
    "momentum_update",
    "nesterov_direction",
    "split_matrix",
    "merge_matrix",
    "orient_wide",
    "frobenius_normalise",
    "newton_schulz",
    "newton_schulz_closed_form",
    "zeropower_via_newtonschulz5",
    "normuon_scale",
    "shape_scale",
    "write_back",
]
