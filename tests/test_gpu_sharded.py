"""ShardedStep, the multi-rank step that bench.py runs under torchrun, end to
end through torch.distributed.

The SomaSpeed page takes one global clipping decision in which each gradient
shard counts once (second optimizer paragraph; its HSDP paragraph has the
matching shards synchronise their gradients).  Here:

* one rank in an NCCL group of one: the all-gather runs on the step's stream;
* two ranks in a gloo group, two processes sharing the one GPU: each holds
  its own shards of the sharded tensors (own seeds) and a copy of every
  replicated tensor, which only its round-robin owner counts in the norm.

After each of 3 chained steps, every rank's tensors are compared with the
fp64 oracle run over the whole model (every rank's shard of each sharded
tensor as its own entry, each replicated tensor once), and the ranks' norms
must be equal bit for bit.  The ranks' kernels never wait on one another:
each rank's square-sum finishes before its host joins the all-gather.
"""
import math
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
STEPS = 3

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    import workloads as W
    return W.with_steps(W.SMALL["hsdp_shard"](), STEPS)


def _worker(rank, world, backend, port, out_path):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist

    import workloads as W
    from parity_harness import DeviceList, make_opt
    from tensor_grad_clip_gb300 import TensorList
    from tensor_grad_clip_gb300.sharded import ShardedStep, owned_flags
    torch.cuda.set_device(0)
    dist.init_process_group(backend, rank=rank, world_size=world, init_method=f"tcp://127.0.0.1:{port}")
    w = _workload()
    sharded = [t.owned for t in w.tensors]
    flags = owned_flags(len(w.tensors), rank, world, sharded)
    params = [W.draw_param(w, k, "cpu", shard_rank=rank) for k in range(len(w.tensors))]
    dl = DeviceList(w, params)
    tl = TensorList(dl.p, dl.g, dl.m, dl.v, groups=[t.group for t in w.tensors],
                    trainable=[t.trainable for t in w.tensors], owned=flags)
    opt = make_opt(w)
    step = ShardedStep(opt)
    stream = torch.cuda.Stream()
    res = {}
    for s in range(1, STEPS + 1):
        grads = [W.draw_grad(w, k, s, "cpu", shard_rank=rank) for k in range(len(w.tensors))]
        dl.load_grads(grads)
        snap = dl.snapshot()
        stream.wait_stream(torch.cuda.current_stream())
        sums = step(tl, w.grad_divisor, w.max_norm, stream=stream)
        norm, coef, nonfinite = opt.get_norm(stream)
        torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        dl.check_snapshot(snap)
        dl.check_guards()
        res[f"norm{s}"] = np.array([norm, coef, nonfinite], dtype=np.float64)
        res[f"sums{s}"] = sums.cpu().numpy()
        for k in range(len(w.tensors)):
            res[f"p{s}_{k}"] = dl.p[k].cpu().numpy()
            res[f"m{s}_{k}"] = dl.m[k].cpu().numpy()
            res[f"v{s}_{k}"] = dl.v[k].cpu().numpy()
    res["steps"] = np.array([opt.get_group_step(q) for q in range(len(w.groups))])
    res["flags"] = np.array(flags)
    np.savez(out_path + f".{rank}.npz", **res)
    opt.close()
    dist.destroy_process_group()


def _run(world, backend, tmp_path):
    port = _free_port()
    out = str(tmp_path / "rank")
    mp.start_processes(_worker, args=(world, backend, port, out), nprocs=world, start_method="spawn", join=True)
    return [np.load(out + f".{r}.npz") for r in range(world)]


def _check_against_whole_model(res, world):
    import workloads as W
    from parity_harness import NORM_RTOL, assert_close
    from oracle import GroupState, OracleOptimizer
    w = _workload()
    sharded = [t.owned for t in w.tensors]
    # every entry owned exactly once across the ranks
    for k in range(len(w.tensors)):
        owners = [r for r in range(world) if res[r]["flags"][k]]
        assert owners == (list(range(world)) if sharded[k] else [k % world]), (k, owners)
    # the whole model: (tensor, rank) for each rank's shard, (tensor, owner) once per replicated tensor
    entries = [(k, r) for k in range(len(w.tensors)) for r in (range(world) if sharded[k] else [k % world])]
    orc = OracleOptimizer([W.draw_param(w, k, "cpu", shard_rank=r) for k, r in entries],
                          [(w.tensors[k].group, w.tensors[k].trainable, True) for k, r in entries],
                          [GroupState(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                                      weight_decay=g.weight_decay) for g in w.groups])
    for s in range(1, STEPS + 1):
        rn, rc = orc.step([W.draw_grad(w, k, s, "cpu", shard_rank=r) for k, r in entries], w.grad_divisor,
                          w.max_norm)
        norms = [res[r][f"norm{s}"] for r in range(world)]
        for r in range(world):
            assert norms[r].tobytes() == norms[0].tobytes(), "ranks derived different norms"
            assert np.array_equal(res[r][f"sums{s}"], res[0][f"sums{s}"])
        norm, coef, nonfinite = norms[0]
        assert nonfinite == 0
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s, norm, rn)
        assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s, coef, rc)
        for e, (k, owner) in enumerate(entries):
            ranks = [owner] if sharded[k] else list(range(world))  # every rank's replicated copy
            for r in ranks:
                nm = f"step {s} rank {r} {w.tensors[k].name}"
                assert_close(nm + " p", res[r][f"p{s}_{k}"], orc.params[e])
                assert_close(nm + " m", res[r][f"m{s}_{k}"], orc.exp_avg[e])
                assert_close(nm + " v", res[r][f"v{s}_{k}"], orc.exp_avg_sq[e])
    for r in range(world):
        assert list(res[r]["steps"]) == [STEPS] * len(w.groups)


@pytest.mark.timeout(600)
def test_sharded_step_one_rank_nccl(tmp_path):
    res = _run(1, "nccl", tmp_path)
    _check_against_whole_model(res, 1)


@pytest.mark.timeout(600)
def test_sharded_step_two_ranks_gloo_one_gpu(tmp_path):
    res = _run(2, "gloo", tmp_path)
    _check_against_whole_model(res, 2)
