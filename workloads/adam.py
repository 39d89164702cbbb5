"""Seeded inputs for the Adam groups (token embedding, output head, scalars).

Shapes and learning rates follow "modded-nanogpt 的 FlexAttention 记录解析",
section "优化器分工" (embedding lr 0.6, head lr 0.008, scalar parameters lr
0.04) on the GPT-2 (124M) body (vocabulary 50304, width 768).  The pages name
the scalar group but not its members; the stand-in is two 12-element vectors
(one entry per layer) and two single numbers.

Gradients, drawn with ``numpy.random.Generator(PCG64([seed, index]))``:

* embedding: only rows of tokens present in the step's batch are non-zero.
  The batch is 8 sequences of 64 Ki tokens (the same page's hyper-parameter
  table); token ranks follow a Zipf law (frequency of rank k proportional to
  1/k), so a row is present with probability 1 - (1 - f_k)^T.  Present rows
  are N(0, 1e-3).
* head and scalars: dense N(0, 1e-3).

Parameters are N(0, 0.02) in fp32.  Nothing here computes any part of Adam.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch


@dataclass(frozen=True)
class AdamTensor:
    name: str
    shape: Tuple[int, ...]
    lr: float
    weight_decay: float = 0.0
    grad: str = "dense"  # or "token_rows"

    @property
    def numel(self) -> int:
        n = 1
        for d in self.shape:
            n *= d
        return n


@dataclass(frozen=True)
class AdamWorkload:
    name: str
    tensors: Tuple[AdamTensor, ...]
    grad_dtype: str
    base_seed: int
    tokens_per_step: int
    description: str

    @property
    def numel(self) -> int:
        return sum(t.numel for t in self.tensors)


VOCAB, N_EMBD, N_LAYER = 50304, 768, 12

ADAM_WORKLOADS: Dict[str, AdamWorkload] = {
    w.name: w
    for w in [
        AdamWorkload(
            "gpt2-124m-adam",
            (
                AdamTensor("wte", (VOCAB, N_EMBD), 0.6, grad="token_rows"),
                AdamTensor("lm_head", (VOCAB, N_EMBD), 0.008),
                AdamTensor("skip_weights", (N_LAYER,), 0.04),
                AdamTensor("lambdas", (N_LAYER,), 0.04),
                AdamTensor("scalar_a", (1,), 0.04),
                AdamTensor("scalar_b", (1,), 0.04),
            ),
            "bf16",
            5000,
            8 * 64 * 1024,
            "GPT-2-124M embedding and head (50304 x 768 each) and a scalar group; Adam lr 0.6 / 0.008 / 0.04",
        ),
        AdamWorkload(
            "adam-ragged",
            (
                AdamTensor("a", (1,), 0.04),
                AdamTensor("b", (3,), 0.3, weight_decay=0.01),
                AdamTensor("c", (4,), 0.002),
                AdamTensor("d", (4095,), 0.6),
                AdamTensor("e", (64, 65), 0.008, weight_decay=0.1),
                AdamTensor("f", (12345,), 0.04, grad="token_rows"),
                AdamTensor("g", (4096, 3), 0.3),
            ),
            "bf16",
            6000,
            4096,
            "ragged sizes (1 .. 12345 elements), mixed lrs and L2 terms",
        ),
    ]
}


def adam_workload(name: str) -> AdamWorkload:
    return ADAM_WORKLOADS[name]


def _rng(seed: int, index: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([int(seed), int(index)]))


def _token_rows_present(rng: np.random.Generator, rows: int, tokens: int) -> np.ndarray:
    ranks = np.arange(1, rows + 1, dtype=np.float64)
    freq = (1.0 / ranks) / np.sum(1.0 / ranks)
    p_present = -np.expm1(tokens * np.log1p(-freq))
    return rng.random(rows) < p_present


def adam_params_for(wl: AdamWorkload) -> List[torch.Tensor]:
    out = []
    for i, t in enumerate(wl.tensors):
        rng = _rng(wl.base_seed + 1_000_000, i)
        out.append(torch.from_numpy((rng.standard_normal(t.numel) * 0.02).astype(np.float32)).reshape(t.shape))
    return out


def adam_grads_for(wl: AdamWorkload, step: int, device: Optional[str] = None, dtype: Optional[str] = None) -> List[torch.Tensor]:
    """Gradients of ``step`` (0-based), cast to the workload's dtype (or ``dtype``)."""
    dt = torch.bfloat16 if (dtype or wl.grad_dtype) == "bf16" else torch.float32
    out = []
    for i, t in enumerate(wl.tensors):
        rng = _rng(wl.base_seed + step, i)
        g = (rng.standard_normal(t.numel) * 1e-3).astype(np.float32)
        if t.grad == "token_rows":
            rows = t.shape[0]
            present = _token_rows_present(rng, rows, wl.tokens_per_step)
            g = g.reshape(rows, -1) * present[:, None].astype(np.float32)
        g = torch.from_numpy(np.ascontiguousarray(g)).reshape(t.shape).to(dt)
        out.append(g.to(device) if device else g)
    return out
