"""Seeded synthetic tensor lists for the optimizer step.

This module only describes and draws inputs: tensor shapes, flags, group
hyperparameters and the random values of weights and gradients.  It holds
none of the step's arithmetic, so the CUDA path and the fp64 oracle can both
take their inputs from here without sharing any of the method.

The five full-size workloads follow the SomaSpeed page's first optimizer
paragraph (what a step does to each gradient) and the
RLinf mixed-precision section ("Retaining Low-Precision Gradients": bf16
gradients on fp32 state).  Unstated hyperparameters take the PPO settings of
the veRL write-up ("Training Configuration": lr 5e-6, grad_clip 1) and
PyTorch's AdamW defaults (betas 0.9/0.999, eps 1e-8).

A normal N(0, s) below means standard deviation s.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Callable, Optional, Sequence

import numpy as np

F32 = "f32"
BF16 = "bf16"
F16 = "f16"


@dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    grad_dtype: str = F32
    group: int = 0
    trainable: bool = True
    owned: bool = True
    zero_grad: bool = False  # every gradient element of this tensor is 0
    param_lowp: Optional[str] = None  # BF16 / F16: a model copy of the fp32 master weights

    @property
    def numel(self) -> int:
        n = 1
        for s in self.shape:
            n *= int(s)
        return n


@dataclass(frozen=True)
class GroupSpec:
    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    divisor: float = 0.0  # the group's own gradient divisor; 0 = the list's


@dataclass(frozen=True)
class Workload:
    name: str
    tensors: tuple
    groups: tuple
    grad_divisor: float
    max_norm: float
    steps: int
    grad_std: float
    param_std: float = 0.02
    seed: int = 1234
    # lr of every group at step t (1-based); None keeps each group's lr.
    lr_at: Optional[Callable[[int], Sequence[float]]] = field(default=None, compare=False)

    @property
    def trainable_numel(self) -> int:
        return sum(t.numel for t in self.tensors if t.trainable)

    @property
    def owned_numel(self) -> int:
        return sum(t.numel for t in self.tensors if t.trainable and t.owned)

    def group_lrs(self, step: int) -> list:
        if self.lr_at is None:
            return [g.lr for g in self.groups]
        return list(self.lr_at(step))

    def effective_bytes_per_step(self) -> int:
        """Bytes per step under the stated accounting: 32 B per trainable
        element with fp32 gradients, 28 B with 16-bit gradients (plus 2 B for
        a 16-bit model copy)."""
        total = 0
        for t in self.tensors:
            if t.trainable:
                total += t.numel * ((32 if t.grad_dtype == F32 else 28) + (2 if t.param_lowp else 0))
        return total

    def algorithmic_bytes_per_step(self) -> int:
        """Exact bytes the step must move: the norm reads owned gradients
        once; the update reads g, p, m, v and writes p, m, v."""
        total = 0
        for t in self.tensors:
            if not t.trainable:
                continue
            gb = 4 if t.grad_dtype == F32 else 2
            total += t.numel * (gb + 24 + (2 if t.param_lowp else 0))
            if t.owned:
                total += t.numel * gb
        return total


# ---------------------------------------------------------------------------
# Workload definitions
# ---------------------------------------------------------------------------

def tiny() -> Workload:
    """12 fp32 tensors, last two frozen, one group, divisor 4; clipping fires."""
    shapes = [(64, 32), (32,), (128, 64), (64,), (64, 64), (64,), (256, 64),
              (256,), (64, 256), (64,), (16, 64), (16,)]
    tensors = tuple(
        TensorSpec(name=f"t{i}", shape=s, grad_dtype=F32, group=0,
                   trainable=(i < 10), owned=True)
        for i, s in enumerate(shapes))
    return Workload(name="tiny-12", tensors=tensors,
                    groups=(GroupSpec(lr=1e-3, weight_decay=0.01),),
                    grad_divisor=4.0, max_norm=1.0, steps=3, grad_std=1.0,
                    seed=1235)


def _transformer_blocks(n_blocks: int, width: int, mlp: int, grad_dtype: str,
                        replicated_every: int = 0) -> tuple:
    """q/k/v/o [w,w], up/gate [mlp,w], down [w,mlp], RMSNorm [w] per block.
    Matrices are group 0 (decayed), norm weights group 1 (no decay).  With
    replicated_every=k, list index i with i % k == k-1 is replicated
    (updated, not in the norm)."""
    out = []
    idx = 0
    for b in range(n_blocks):
        for nm, shp, grp in (("q", (width, width), 0), ("k", (width, width), 0),
                             ("v", (width, width), 0), ("o", (width, width), 0),
                             ("up", (mlp, width), 0), ("gate", (mlp, width), 0),
                             ("down", (width, mlp), 0), ("norm", (width,), 1)):
            owned = True
            if replicated_every and idx % replicated_every == replicated_every - 1:
                owned = False
            out.append(TensorSpec(name=f"b{b}.{nm}", shape=shp, grad_dtype=grad_dtype,
                                  group=grp, trainable=True, owned=owned))
            idx += 1
    return tuple(out)


def action_expert(n_blocks: int = 18, width: int = 1024, mlp: int = 4096,
                  steps: int = 10, master: bool = False) -> Workload:
    """~300M-parameter action-expert-like head, bf16 grads, two groups.  With
    master=True the fp32 weights are master copies of bf16 model weights."""
    tensors = _transformer_blocks(n_blocks, width, mlp, BF16)
    if master:
        tensors = tuple(replace(t, param_lowp=BF16) for t in tensors)
    return Workload(
        name=f"action-expert-{n_blocks}x{width}x{mlp}" + ("-master" if master else ""),
        tensors=tensors,
        groups=(GroupSpec(lr=5e-6, weight_decay=0.01), GroupSpec(lr=5e-6, weight_decay=0.0)),
        grad_divisor=64.0, max_norm=1.0, steps=steps, grad_std=1e-3, seed=1236)


def many_small(count: int = 20000, max_numel: int = 65536, steps: int = 10) -> Workload:
    """`count` 1-D fp32 tensors with log-uniform sizes in [1, max_numel];
    10% frozen, 1% of the trainable ones with all-zero gradients."""
    rng = np.random.Generator(np.random.PCG64(1237))
    u = rng.random(count)
    sizes = np.clip(np.rint(np.exp(u * math.log(max_numel))), 1, max_numel).astype(np.int64)
    frozen = set(rng.choice(count, size=count // 10, replace=False).tolist())
    trainable_idx = [i for i in range(count) if i not in frozen]
    n_zero = max(1, len(trainable_idx) // 100)
    zero = set(rng.choice(np.array(trainable_idx), size=n_zero, replace=False).tolist())
    tensors = tuple(
        TensorSpec(name=f"s{i}", shape=(int(sizes[i]),), grad_dtype=F32, group=0,
                   trainable=(i not in frozen), owned=True, zero_grad=(i in zero))
        for i in range(count))
    return Workload(name=f"many-small-{count}", tensors=tensors,
                    groups=(GroupSpec(lr=5e-6, weight_decay=0.0),),
                    grad_divisor=8.0, max_norm=1.0, steps=steps, grad_std=1e-2, seed=1238)


def hsdp_shard_view(n_blocks: int = 32, width: int = 4096, mlp: int = 11008,
                    steps: int = 10) -> Workload:
    """7B-parameter list seen as one HSDP shard: 25% of the tensors are
    replicated (updated but excluded from the norm)."""
    return Workload(
        name=f"hsdp-shard-{n_blocks}x{width}x{mlp}",
        tensors=_transformer_blocks(n_blocks, width, mlp, BF16, replicated_every=4),
        groups=(GroupSpec(lr=5e-6, weight_decay=0.01), GroupSpec(lr=5e-6, weight_decay=0.0)),
        grad_divisor=128.0, max_norm=1.0, steps=steps, grad_std=1e-4, seed=1239)


def cosine_lr(peak: float, steps: int) -> Callable[[int], Sequence[float]]:
    def lr_at(t: int):
        return (peak * 0.5 * (1.0 + math.cos(math.pi * (t - 1) / steps)),)
    return lr_at


def flat(numel: int = 1_500_000_000, steps: int = 10) -> Workload:
    """One flat fp32 tensor plus four 64-element biases; gradients small
    enough that clipping does not fire; lr follows a cosine each step."""
    tensors = (TensorSpec(name="flat", shape=(numel,), grad_dtype=F32),) + tuple(
        TensorSpec(name=f"bias{i}", shape=(64,), grad_dtype=F32) for i in range(4))
    return Workload(name=f"flat-{numel}", tensors=tensors,
                    groups=(GroupSpec(lr=1e-4, weight_decay=0.1),),
                    grad_divisor=1.0, max_norm=1.0, steps=steps, grad_std=1e-5,
                    seed=1240, lr_at=cosine_lr(1e-4, steps))


FULL = {
    "tiny": tiny,
    "action_expert": action_expert,
    "many_small": many_small,
    "hsdp_shard": hsdp_shard_view,
    "flat": flat,
}

# Reduced sizes that the oracle finishes in well under a second but that
# still span many chunks and leave ragged tails (odd widths, odd lengths).
SMALL = {
    "tiny": tiny,
    "action_expert": lambda: action_expert(n_blocks=3, width=96, mlp=380),
    "many_small": lambda: many_small(count=2000),
    "hsdp_shard": lambda: hsdp_shard_view(n_blocks=4, width=128, mlp=344),
    "flat": lambda: flat(numel=1_500_007),
}


def with_steps(w: Workload, steps: int) -> Workload:
    lr_at = w.lr_at
    if lr_at is not None and w.name.startswith("flat"):
        lr_at = cosine_lr(w.groups[0].lr, steps)
    return replace(w, steps=steps, lr_at=lr_at)
