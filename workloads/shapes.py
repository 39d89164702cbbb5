"""Matrix shape lists of the workloads the optimizer step is tested and timed on.

Shapes follow the GPT-2 bodies the modded-nanogpt write-ups train:

* GPT-2-124M: 12 layers, d = 768.  Per layer one attention bank of shape
  [768, 3072] that is viewed as four [768, 768] matrices (Q, K, V, O) before
  the optimizer touches it (FixMuonLR record write-up, change 2, "attention
  reshape moved earlier"), one MLP up-projection ``c_fc`` [768, 3072] whose
  lr multiplier is 2.0 = sqrt(4) (same write-up, change 1, "MLP
  up-projection lr_mul"), and one down-projection ``c_proj`` [3072, 768].
* GPT-2-medium: 24 layers, d = 1024, same structure.
* A stress set of 4096-wide matrices, including tall and wide ones, so that
  the transpose-to-the-short-side path is exercised at size.
* A tiny set of four 64x256 matrices (plain Muon, fp32 gradients).
"""

from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Tuple


@dataclass(frozen=True)
class MatrixShape:
    """One parameter matrix handed to the optimizer.

    ``split`` > 1 marks a bank that the optimizer views as ``split`` separate
    matrices of shape rows x (cols / split) laid out one after the other in
    memory (the ``view`` of a contiguous [rows, cols] tensor).
    """

    name: str
    rows: int
    cols: int
    split: int = 1
    lr_mul: float = 1.0
    wd_mul: float = 1.0

    @property
    def sub_shape(self) -> Tuple[int, int]:
        return self.rows, self.cols // self.split

    @property
    def numel(self) -> int:
        return self.rows * self.cols


@dataclass(frozen=True)
class Workload:
    name: str
    matrices: Tuple[MatrixShape, ...]
    grad_kind: str  # "lowrank", "powerlaw", "loguniform"
    grad_dtype: str  # "f32" or "bf16"
    normuon: bool
    lr: float
    momentum: float = 0.95
    beta2: float = 0.95
    weight_decay: float = 0.0
    ns_steps: int = 5
    steps: int = 1
    base_seed: int = 0
    description: str = ""

    @property
    def numel(self) -> int:
        return sum(m.numel for m in self.matrices)

    def sub_shapes(self) -> List[Tuple[int, int]]:
        out = []
        for m in self.matrices:
            out.extend([m.sub_shape] * m.split)
        return out


def _gpt2_body(layers: int, d: int) -> Tuple[MatrixShape, ...]:
    mats = []
    for layer in range(layers):
        mats.append(MatrixShape(f"h{layer}.attn.qkvo", d, 4 * d, split=4))
        mats.append(MatrixShape(f"h{layer}.mlp.c_fc", d, 4 * d, lr_mul=2.0))
        mats.append(MatrixShape(f"h{layer}.mlp.c_proj", 4 * d, d))
    return tuple(mats)


def _stress() -> Tuple[MatrixShape, ...]:
    mats = [MatrixShape(f"sq{i}", 4096, 4096) for i in range(16)]
    mats += [MatrixShape(f"wide{i}", 4096, 16384) for i in range(4)]
    mats += [MatrixShape(f"tall{i}", 16384, 4096) for i in range(4)]
    return tuple(mats)


WORKLOADS = {
    "tiny": Workload(
        name="tiny",
        matrices=tuple(MatrixShape(f"w{i}", 64, 256) for i in range(4)),
        grad_kind="lowrank",
        grad_dtype="f32",
        normuon=False,
        lr=0.02,
        base_seed=0,
        description="4 fp32 matrices 64x256, plain Muon, one step",
    ),
    "gpt2-124m": Workload(
        name="gpt2-124m",
        matrices=_gpt2_body(12, 768),
        grad_kind="lowrank",
        grad_dtype="bf16",
        normuon=True,
        lr=0.03,
        base_seed=2000,
        description="GPT-2-124M body: 48x768^2 (qkvo banks split), 12 c_fc 768x3072 (lr_mul 2), "
        "12 c_proj 3072x768; NorMuon, one step",
    ),
    "gpt2-124m-plain": Workload(
        name="gpt2-124m-plain",
        matrices=_gpt2_body(12, 768),
        grad_kind="lowrank",
        grad_dtype="bf16",
        normuon=False,
        lr=0.02,
        base_seed=2000,
        description="GPT-2-124M body, plain Muon (shape scale max(1,R/C)^0.5), one step",
    ),
    "gpt2-124m-normuon-200": Workload(
        name="gpt2-124m-normuon-200",
        matrices=_gpt2_body(12, 768),
        grad_kind="lowrank",
        grad_dtype="bf16",
        normuon=True,
        lr=0.03,
        steps=200,
        base_seed=3000,
        description="GPT-2-124M body, NorMuon, 200 consecutive steps on fresh grads",
    ),
    "gpt2-medium": Workload(
        name="gpt2-medium",
        matrices=_gpt2_body(24, 1024),
        grad_kind="powerlaw",
        grad_dtype="bf16",
        normuon=True,
        lr=0.03,
        base_seed=4000,
        description="GPT-2-medium body: 96x1024^2, 24x1024x4096, 24x4096x1024; s_i = i^-0.5",
    ),
    "stress": Workload(
        name="stress",
        matrices=_stress(),
        grad_kind="loguniform",
        grad_dtype="bf16",
        normuon=True,
        lr=0.03,
        base_seed=5000,
        description="16x4096^2, 4x4096x16384, 4x16384x4096; singular values log-uniform on [1e-4, 1]",
    ),
}


def workload(name: str) -> Workload:
    try:
        return WORKLOADS[name]
    except KeyError:
        raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}") from None
