"""Parity at full size, in the layout and launch configuration bench.py times.

The 20 000-tensor list (104 M) is compared element by element after each of
3 chained steps.  For the action-expert (302 M), 7B shard-view (6.48 G) and
flat (1.5 G) lists, over 10 chained steps:

* the norm is the oracle's own fp64 sum over every owned gradient, taken
  in pieces of at most 2^26 elements on a thread pool and added in list
  order;
* the update is checked on a seeded sample of elements per tensor: the first
  and last 32 and 128 random ones.  The oracle carries their fp64 state
  across steps, each element depending only on its own p, m, v, g, the
  oracle's c and the group constants;
* gradients are bit-unchanged, and the sentinel gaps between tensors are
  intact.

A single tensor of more than 2^31 elements covers 64-bit offsets.
"""
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_harness import NORM_RTOL, assert_close
from tensor_grad_clip_gb300 import SomaOpt, TensorList, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.lib()


def oracle_norm(w, fb, divisor, pool):
    """sqrt of the oracle's sum of (g/d)^2 over owned tensors; large tensors
    are summed in pieces of 2^26 elements, pieces added in list order."""
    piece = 1 << 26
    tasks = [(k, a) for k, t in enumerate(w.tensors) if t.trainable and t.owned
             for a in range(0, t.numel, piece)]

    def one(task):
        k, a = task
        return oracle.tensor_sqsum(fb.g[k][a:a + piece].cpu(), divisor)

    total = 0.0
    for x in pool.map(one, tasks):
        total += x
    return math.sqrt(total)


def sample_indices(numel, seed, k):
    rng = np.random.default_rng(seed * 1000 + k)
    head = np.arange(min(32, numel))
    tail = np.arange(max(0, numel - 32), numel)
    rand = rng.integers(0, numel, size=min(128, numel))
    return np.unique(np.concatenate([head, tail, rand]))


def run_full(w, steps, extra_idx=None, graph=False):
    dev = torch.device("cuda", 0)
    fb = W.FlatBuffers(w, dev, grad_step=1)
    opt = SomaOpt(0)
    for q in w.groups:
        opt.add_group(lr=q.lr, betas=(q.beta1, q.beta2), eps=q.eps, weight_decay=q.weight_decay)
    tl = TensorList(fb.p, fb.g, fb.m, fb.v, groups=[t.group for t in w.tensors],
                    trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors])
    idx, state = [], []
    for k, t in enumerate(w.tensors):
        ix = sample_indices(t.numel, w.seed, k)
        if extra_idx is not None:
            ix = np.unique(np.concatenate([ix, extra_idx]))
        ix_t = torch.from_numpy(ix).to(dev)
        idx.append(ix_t)
        p0 = fb.p[k][ix_t].double().cpu().numpy()
        state.append([p0.copy(), np.zeros_like(p0), np.zeros_like(p0)])
    pool = ThreadPoolExecutor(16)
    stream = torch.cuda.Stream() if graph else None
    cuda_graph = torch.cuda.CUDAGraph() if graph else None
    for s in range(1, steps + 1):
        if s > 1:
            fb.load_grads(s)
        lrs = w.group_lrs(s)
        for q, lr in enumerate(lrs):
            opt.set_lr(q, lr)
        gbits = torch.int16 if fb.grad_dtype == torch.bfloat16 else torch.int32
        g_before = fb.G.view(gbits).clone()
        if graph:  # captured once, replayed with the lr pushed each step
            stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                opt.push_groups(stream)
                if s == 1:
                    opt.step_graph(tl, w.grad_divisor, w.max_norm, stream)
                    with torch.cuda.graph(cuda_graph, stream=stream):
                        opt.step_graph(tl, w.grad_divisor, w.max_norm, stream)
                else:
                    cuda_graph.replay()
            norm, coef, nonfinite = opt.get_norm(stream)
            torch.cuda.current_stream().wait_stream(stream)
        else:
            opt.step(tl, w.grad_divisor, w.max_norm)
            norm, coef, nonfinite = opt.get_norm()
        rn = oracle_norm(w, fb, w.grad_divisor, pool)
        rc = oracle.clip_coef(rn, w.max_norm)
        assert not nonfinite
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s, norm, rn)
        assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s, coef, rc)
        if rc == 1.0:
            assert coef == 1.0
        assert torch.equal(fb.G.view(gbits), g_before), "gradients changed"
        del g_before
        for k, t in enumerate(w.tensors):
            q = w.groups[t.group]
            p_s, m_s, v_s = state[k]
            oracle.adamw_update(p_s, fb.g[k][idx[k]].cpu(), m_s, v_s, lr=lrs[t.group], beta1=q.beta1,
                                beta2=q.beta2, eps=q.eps, weight_decay=q.weight_decay, step=s, c=rc,
                                divisor=w.grad_divisor)
            assert_close(f"step {s} {t.name} p", fb.p[k][idx[k]].cpu().numpy(), p_s)
            assert_close(f"step {s} {t.name} m", fb.m[k][idx[k]].cpu().numpy(), m_s)
            assert_close(f"step {s} {t.name} v", fb.v[k][idx[k]].cpu().numpy(), v_s)
    if graph:
        opt.pull_groups(stream)
        del cuda_graph
    for q in range(len(w.groups)):
        assert opt.get_group_step(q) == steps
    torch.cuda.synchronize()
    assert fb.gaps_intact(), "a write landed outside a tensor"
    plan = opt.plan()
    opt.close()
    pool.shutdown()
    del fb
    torch.cuda.empty_cache()
    return plan


@pytest.mark.parametrize("name", ["action_expert", "flat", "hsdp_shard"])
def test_full_size_parity(name):
    w = W.FULL[name]()
    plan = run_full(w, steps=10)
    assert plan["trainable_numel"] == w.trainable_numel
    assert plan["owned_numel"] == w.owned_numel


def test_full_size_graph_replays():
    # The graph-capturable step at full size: one capture, replays with the
    # lr pushed each step (the flat list's cosine schedule), sampled against
    # the oracle like the regular step.
    w = W.with_steps(W.FULL["flat"](), 4)
    run_full(w, steps=4, graph=True)
    w = W.with_steps(W.FULL["action_expert"](), 3)
    run_full(w, steps=3, graph=True)


def test_tensor_beyond_2_pow_31_elements():
    n = (1 << 31) + 13
    w = W.Workload(name="huge", tensors=(W.TensorSpec("huge", (n,), W.BF16),),
                   groups=(W.GroupSpec(lr=1e-4, weight_decay=0.01),), grad_divisor=4.0, max_norm=1.0,
                   steps=2, grad_std=1e-3, seed=77)
    around = np.arange((1 << 31) - 20, (1 << 31) + 13)
    run_full(w, steps=2, extra_idx=around)


def test_full_size_many_small_every_element():
    # The 20 000-tensor list at full size (104 M trainable elements), every
    # element against the oracle after each of 3 chained steps.  The flat
    # buffers come back to the host once per step and are sliced per tensor.
    from parity_harness import make_oracle
    w = W.with_steps(W.FULL["many_small"](), 3)
    dev = torch.device("cuda", 0)
    fb = W.FlatBuffers(w, dev, grad_step=1)
    P0 = fb.P.cpu()
    sl = [slice(fb.offsets[k], fb.offsets[k] + t.numel) for k, t in enumerate(w.tensors)]
    orc = make_oracle(w, [P0[s_] for s_ in sl])
    opt = SomaOpt(0)
    for q in w.groups:
        opt.add_group(lr=q.lr, betas=(q.beta1, q.beta2), eps=q.eps, weight_decay=q.weight_decay)
    tl = TensorList(fb.p, fb.g, fb.m, fb.v, groups=[t.group for t in w.tensors],
                    trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors])
    for s in range(1, w.steps + 1):
        if s > 1:
            fb.load_grads(s)
        G = fb.G.cpu()
        opt.step(tl, w.grad_divisor, w.max_norm)
        norm, coef, nonfinite = opt.get_norm()
        rn, rc = orc.step([G[s_] for s_ in sl], w.grad_divisor, w.max_norm)
        assert not nonfinite
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s, norm, rn)
        assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s, coef, rc)
        assert torch.equal(fb.G.cpu().view(torch.int32), G.view(torch.int32)), "gradients changed"
        P, M, V = fb.P.cpu().numpy(), fb.M.cpu().numpy(), fb.V.cpu().numpy()
        for k, t in enumerate(w.tensors):
            if t.trainable:
                assert_close(f"step {s} {t.name} p", P[sl[k]], orc.params[k])
                assert_close(f"step {s} {t.name} m", M[sl[k]], orc.exp_avg[k])
                assert_close(f"step {s} {t.name} v", V[sl[k]], orc.exp_avg_sq[k])
            elif t.numel:
                assert np.array_equal(P[sl[k]].view(np.int32), P0[sl[k]].numpy().view(np.int32))
    torch.cuda.synchronize()
    assert fb.gaps_intact(), "a write landed outside a tensor"
    opt.close()
    del fb
    torch.cuda.empty_cache()
