"""bench.py's multi-rank path, launched the way a multi-GPU benchmark is
launched (torchrun, one process per rank), here with two ranks sharing the
one GPU over a gloo group.

Each rank holds its own shards of the sharded tensors and a copy of every
replicated tensor, owning a replicated one only if it is its round-robin
owner, so the norm that rank 0 prints must be the whole model's: every rank's
shard of each sharded tensor once, each replicated tensor once (the SomaSpeed
page's "each gradient shard contributes once", second optimizer paragraph).
The ranks' kernels never wait on one another: each rank's square-sum finishes
before its host joins the all-gather.
"""
import json
import math
import os
import socket
import subprocess
import sys

import pytest
import torch

import oracle
import workloads as W
from parity_harness import NORM_RTOL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.timeout(900)
def test_bench_two_ranks_print_the_whole_model_norm():
    world = 2
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={world}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--gpus", str(world),
           "--workload", "hsdp_shard", "--blocks", "1", "--steps", "3", "--warmup", "1", "--no-e2e",
           "--no-cpu-baseline", "--per-config", "none"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=800)
    assert out.returncode == 0, out.stdout[-2000:] + out.stderr[-4000:]
    lines = [x for x in out.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1, out.stdout  # rank 0 alone prints
    line = json.loads(lines[0])
    assert line["n_gpus"] == world and line["value"] > 0 and line["scaling"] == "weak"
    assert "gloo" in line["config"]["parallelism"]
    assert line["gpu_launches"] == 3 * 3  # square-sum, finish and update kernels per step

    # The whole model at the printed step: the bench draws every rank's
    # step-1 gradients on the device once and does not reload them.  The same
    # seeds on the same device give the same values here.
    oracle.lib()
    w = W.hsdp_shard_view(n_blocks=1)
    total = 0.0
    for k, t in enumerate(w.tensors):
        ranks = range(world) if t.owned else [k % world]  # replicated: counted once
        for r in ranks:
            g = W.draw_grad(w, k, 1, torch.device("cuda", 0), shard_rank=r if t.owned else 0).cpu()
            total += oracle.tensor_sqsum(g, w.grad_divisor)
    expected = math.sqrt(total)
    assert math.isclose(line["last_norm"], expected, rel_tol=NORM_RTOL), (line["last_norm"], expected)
    assert math.isclose(line["last_clip_coef"], oracle.clip_coef(expected, w.max_norm), rel_tol=NORM_RTOL)
