"""Draw the seeded weights and gradients of a `Workload` with torch.

Each tensor gets its own generator, seeded from (workload seed, kind, step,
tensor index), so a tensor's values do not depend on which other tensors are
drawn or in which order.  Values drawn on the CPU and on a CUDA device differ
(different generators), so a consumer never takes a CPU draw for values that
were drawn on a device: it copies them from the tensors actually used, or
draws them again on the same kind of device, where the same seed gives the
same values.
"""
from __future__ import annotations

import hashlib

import torch

from .configs import BF16, F16, F32, Workload

_DTYPES = {F32: torch.float32, BF16: torch.bfloat16, F16: torch.float16}


def torch_dtype(tag: str) -> torch.dtype:
    return _DTYPES[tag]


def tensor_seed(seed: int, kind: str, step: int, index: int) -> int:
    h = hashlib.sha256(f"{seed}/{kind}/{step}/{index}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _normal(shape, std: float, seed: int, device, dtype) -> torch.Tensor:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    x.mul_(std)
    return x if dtype == torch.float32 else x.to(dtype)


def _kind(w: Workload, k: int, kind: str, shard_rank: int) -> str:
    """Seed kind of tensor k.  With shard_rank r > 0, a sharded tensor (one
    the list flags as owned; a replicated one is the same on every rank) is
    rank r's own shard and gets its own values; rank 0 draws what a single
    GPU draws."""
    if shard_rank and w.tensors[k].owned:
        return f"{kind}/rank{shard_rank}"
    return kind


def draw_param(w: Workload, k: int, device="cpu", shard_rank: int = 0) -> torch.Tensor:
    """fp32 weight k of the workload, N(0, param_std)."""
    return _normal(w.tensors[k].shape, w.param_std, tensor_seed(w.seed, _kind(w, k, "param", shard_rank), 0, k),
                   device, torch.float32)


def draw_grad(w: Workload, k: int, step: int, device="cpu", shard_rank: int = 0) -> torch.Tensor:
    """Gradient k of step `step` in its grad dtype (zeros if zero_grad)."""
    t = w.tensors[k]
    dt = _DTYPES[t.grad_dtype]
    if t.zero_grad:
        return torch.zeros(t.shape, device=device, dtype=dt)
    return _normal(t.shape, w.grad_std, tensor_seed(w.seed, _kind(w, k, "grad", shard_rank), step, k), device, dt)


def draw_params(w: Workload, device="cpu") -> list:
    """fp32 weights N(0, param_std) for every tensor, frozen ones included."""
    return [_normal(t.shape, w.param_std, tensor_seed(w.seed, "param", 0, i), device, torch.float32)
            for i, t in enumerate(w.tensors)]


def draw_grads(w: Workload, step: int, device="cpu", out=None) -> list:
    """Gradients of step `step` (1-based) in each tensor's grad dtype,
    N(0, grad_std), zeros for tensors flagged zero_grad.  Frozen tensors get
    gradients too, so that a test can check nobody reads or writes them.
    With `out`, values are written into those tensors instead."""
    res = []
    for i in range(len(w.tensors)):
        g = draw_grad(w, i, step, device)
        if out is not None:
            out[i].copy_(g)
            del g
            res.append(out[i])
        else:
            res.append(g)
    return res


def zero_moments(w: Workload, device="cpu"):
    m = [torch.zeros(t.shape, device=device, dtype=torch.float32) for t in w.tensors]
    v = [torch.zeros(t.shape, device=device, dtype=torch.float32) for t in w.tensors]
    return m, v
