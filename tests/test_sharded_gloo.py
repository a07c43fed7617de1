"""The shard-group exchange on CPU: two gloo ranks, each holding its own
shards of the sharded tensors plus the replicated ones.  Every entry must be
owned exactly once, and the norm from the gathered per-rank sums (added in
rank order) must equal the oracle's norm over the whole model."""
import math
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _shard_grad(w, k, rank):
    import workloads as W
    t = w.tensors[k]
    seed = W.tensor_seed(w.seed, f"shard{rank}", 1, k)
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(t.shape, generator=g) * w.grad_std).to(W.torch_dtype(t.grad_dtype))


def _worker(rank, port, out_path):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import oracle
    import workloads as W
    from tensor_grad_clip_gb300.sharded import gather_rank_sums, owned_flags
    dist.init_process_group("gloo", rank=rank, world_size=WORLD, init_method=f"tcp://127.0.0.1:{port}")
    w = W.SMALL["hsdp_shard"]()
    sharded = [t.owned for t in w.tensors]          # the list's replicated entries are not sharded
    flags = owned_flags(len(w.tensors), rank, WORLD, sharded)
    local = 0.0
    for k, t in enumerate(w.tensors):
        if not flags[k]:
            continue
        g = _shard_grad(w, k, rank) if sharded[k] else W.draw_grad(w, k, 1, "cpu")
        local += oracle.tensor_sqsum(g, w.grad_divisor)
    sums = gather_rank_sums(torch.tensor([local], dtype=torch.float64))
    all_flags = [None] * WORLD
    dist.all_gather_object(all_flags, flags)
    with open(out_path + f".{rank}", "w") as f:
        f.write(f"{sums.tolist()}\n{all_flags}\n")
    dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_norm_matches_the_whole_model(tmp_path):
    sys.path.insert(0, ROOT)
    import ast
    import oracle
    import workloads as W
    port = _free_port()
    out = str(tmp_path / "rank")
    mp.start_processes(_worker, args=(port, out), nprocs=WORLD, start_method="spawn", join=True)
    res = [open(out + f".{r}").read().splitlines() for r in range(WORLD)]
    sums = [ast.literal_eval(r[0]) for r in res]
    flags = ast.literal_eval(res[0][1])
    assert sums[0] == sums[1] and len(sums[0]) == WORLD  # every rank sees the same values
    w = W.SMALL["hsdp_shard"]()
    sharded = [t.owned for t in w.tensors]
    for k in range(len(w.tensors)):
        owners = [r for r in range(WORLD) if flags[r][k]]
        assert owners == (list(range(WORLD)) if sharded[k] else [k % WORLD])
    # the whole model once: every rank's shard of each sharded tensor, each replicated tensor once
    total = 0.0
    for k, t in enumerate(w.tensors):
        if sharded[k]:
            for r in range(WORLD):
                total += oracle.tensor_sqsum(_shard_grad(w, k, r), w.grad_divisor)
        else:
            total += oracle.tensor_sqsum(W.draw_grad(w, k, 1, "cpu"), w.grad_divisor)
    norm_ranks = math.sqrt(sum(sums[0]))
    assert math.isclose(norm_ranks, math.sqrt(total), rel_tol=1e-12)
    assert oracle.clip_coef(norm_ranks, w.max_norm) < 1.0 or norm_ranks < 1.0
