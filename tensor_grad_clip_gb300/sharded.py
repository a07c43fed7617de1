"""The optimizer step over a shard group (FSDP/HSDP ranks).

Every rank owns some shards; the SomaSpeed page takes one global clipping
decision in which each gradient shard counts once (its second optimizer
paragraph, on batching the work over the tensor list).  The ranks exchange one
float64 each: their owned square-sum.

    step = ShardedStep(opt, group)           # after torch.distributed init
    step(tensor_list, grad_divisor, max_norm)

runs soma_opt_sumsq, an all-gather of the per-rank sums over `group`, and
soma_opt_step_from_sumsq, which adds them in rank order on the device, so
every rank applies the same clip coefficient.
"""
from __future__ import annotations

import contextlib
from typing import Sequence

import torch
import torch.distributed as dist


def owned_flags(num_tensors: int, rank: int, world: int, sharded: Sequence[bool]) -> list:
    """Ownership of a list present on every rank of a group: a sharded entry
    (a different shard on each rank) is owned by its holder; a replicated
    entry (the same tensor on every rank) is owned by one rank only, chosen
    round-robin by list index, so that it enters the norm once."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    return [bool(sharded[k]) or (k % world == rank) for k in range(num_tensors)]


def gather_rank_sums(local: torch.Tensor, group=None) -> torch.Tensor:
    """All ranks' one-element float64 tensors, rank r at index r, on the
    device of `local`.  A gloo group exchanges host copies (gloo moves host
    memory; the copy to the host waits for the square-sum kernel)."""
    world = dist.get_world_size(group)
    staged = local.is_cuda and dist.get_backend(group) == "gloo"
    src = local.cpu() if staged else local
    parts = [torch.empty_like(src) for _ in range(world)]
    dist.all_gather(parts, src, group=group)
    out = torch.cat(parts)
    return out.to(local.device, non_blocking=False) if staged else out


class ShardedStep:
    def __init__(self, opt, group=None, device=None):
        self.opt = opt
        self.group = group
        dev = torch.device("cuda", opt.device) if device is None else device
        self.local = torch.zeros(1, dtype=torch.float64, device=dev)

    def __call__(self, tensors, grad_divisor: float, max_norm: float, stream=None):
        """One step; the all-gather runs on the same stream as both kernels."""
        ctx = torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()
        with ctx:
            self.opt.sumsq(tensors, grad_divisor, self.local)
            sums = gather_rank_sums(self.local, self.group)
            self.opt.step_from_sumsq(tensors, grad_divisor, max_norm, sums)
        return sums
