"""The shard-group step on one GPU: R ranks emulated as R handles with their
own tensor lists, launched one after another (nothing waits on anything).
Rank r holds its own shard of every sharded tensor plus a copy of every
replicated tensor; ownership follows sharded.owned_flags.  The per-rank sums
are gathered into one device array, as an all-gather would, and every rank
then steps with the global norm.  Checked against the fp64 oracle run over
the whole model (every shard, every replicated tensor once)."""
import math
from dataclasses import replace

import numpy as np
import pytest
import torch

import workloads as W
from oracle import GroupState, OracleOptimizer
from parity_harness import NORM_RTOL, DeviceList, assert_close, make_opt
from tensor_grad_clip_gb300 import build
from tensor_grad_clip_gb300.sharded import owned_flags

pytestmark = pytest.mark.gpu
R = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _param(w, k, r, sharded):
    if not sharded[k]:
        return W.draw_param(w, k, "cpu")
    g = torch.Generator().manual_seed(W.tensor_seed(w.seed, f"param-shard{r}", 0, k))
    return torch.randn(w.tensors[k].shape, generator=g) * w.param_std


def _grad(w, k, r, s, sharded):
    if not sharded[k]:
        return W.draw_grad(w, k, s, "cpu")
    g = torch.Generator().manual_seed(W.tensor_seed(w.seed, f"grad-shard{r}", s, k))
    return (torch.randn(w.tensors[k].shape, generator=g) * w.grad_std).to(W.torch_dtype(w.tensors[k].grad_dtype))


@pytest.mark.parametrize("name", ["hsdp_shard", "tiny"])
def test_emulated_ranks_match_the_whole_model(name):
    w = W.with_steps(W.SMALL[name](), 3)
    n = len(w.tensors)
    sharded = [t.owned for t in w.tensors]
    if name == "tiny":  # no replicated entries in the tiny list: make every third one replicated
        sharded = [k % 3 != 2 for k in range(n)]
    ranks = []
    for r in range(R):
        flags = owned_flags(n, r, R, sharded)
        wr = replace(w, tensors=tuple(replace(t, owned=flags[k]) for k, t in enumerate(w.tensors)))
        params = [_param(w, k, r, sharded) for k in range(n)]
        ranks.append((wr, DeviceList(wr, params), make_opt(wr), params))
    # oracle over the whole model: shard (k, r) for sharded k, one copy of replicated k
    keys = [(k, r) for k in range(n) for r in (range(R) if sharded[k] else [0])]
    orc = OracleOptimizer([ranks[r][3][k].double().numpy().reshape(-1) for k, r in keys],
                          [(w.tensors[k].group, w.tensors[k].trainable, True) for k, r in keys],
                          [GroupState(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps, weight_decay=g.weight_decay)
                           for g in w.groups])
    sums = torch.zeros(R, dtype=torch.float64, device="cuda")
    for s in range(1, w.steps + 1):
        for r, (wr, dl, opt, _) in enumerate(ranks):
            dl.load_grads([_grad(w, k, r, s, sharded) for k in range(n)])
            opt.sumsq(dl.tl, w.grad_divisor, sums[r:r + 1])
        for wr, dl, opt, _ in ranks:
            opt.step_from_sumsq(dl.tl, w.grad_divisor, w.max_norm, sums)
        norms = [opt.get_norm() for _, _, opt, _ in ranks]
        rn, rc = orc.step([_grad(w, k, r, s, sharded) for k, r in keys], w.grad_divisor, w.max_norm)
        assert all(x == norms[0] for x in norms)  # every rank derives the same bits
        assert math.isclose(norms[0][0], rn, rel_tol=NORM_RTOL) and math.isclose(norms[0][1], rc, rel_tol=NORM_RTOL)
        for i, (k, r) in enumerate(keys):
            if not w.tensors[k].trainable:
                continue
            for rr in (range(R) if not sharded[k] else [r]):
                dl = ranks[rr][1]
                assert_close(f"step {s} {k}/{rr} p", dl.p[k].cpu().numpy(), orc.params[i])
                assert_close(f"step {s} {k}/{rr} m", dl.m[k].cpu().numpy(), orc.exp_avg[i])
                assert_close(f"step {s} {k}/{rr} v", dl.v[k].cpu().numpy(), orc.exp_avg_sq[i])
        for k in range(n):
            if not sharded[k]:  # replicated copies stay bit-identical across ranks
                for rr in range(1, R):
                    assert torch.equal(ranks[rr][1].p[k], ranks[0][1].p[k])
        for _, dl, _, _ in ranks:
            dl.check_guards()
    for _, _, opt, _ in ranks:
        assert [opt.get_group_step(q) for q in range(len(w.groups))] == [g.step for g in orc.groups]
        opt.close()


def test_local_sum_is_the_owned_square_sum():
    import oracle
    w = W.with_steps(W.SMALL["hsdp_shard"](), 1)
    params = W.draw_params(w, "cpu")
    grads = W.draw_grads(w, 1, "cpu")
    dl = DeviceList(w, params)
    dl.load_grads(grads)
    opt = make_opt(w)
    out = torch.zeros(2, dtype=torch.float64, device="cuda")
    opt.sumsq(dl.tl, w.grad_divisor, out[1:])
    ref = sum(oracle.tensor_sqsum(g, w.grad_divisor) for g, t in zip(grads, w.tensors) if t.trainable and t.owned)
    assert out[0].item() == 0.0
    assert math.isclose(out[1].item(), ref, rel_tol=NORM_RTOL)
    for q in range(len(w.groups)):
        assert opt.get_group_step(q) == 0  # the local sum alone is not a step
    opt.close()


def test_rank_sums_up_to_the_limit_are_added_in_rank_order():
    # soma_opt_step_from_sumsq with SOMA_MAX_RANKS per-rank sums (this rank's
    # own square-sum at one index, the others drawn): the norm is the square
    # root of their fp64 sum taken in index order, bit for bit (one add chain
    # and a correctly rounded square root on both sides), c is the oracle's
    # coefficient of that norm, and every tensor is updated with that c.
    import oracle
    from tensor_grad_clip_gb300 import _abi
    w = W.with_steps(W.SMALL["tiny"](), 1)
    params = W.draw_params(w, "cpu")
    grads = W.draw_grads(w, 1, "cpu")
    dl = DeviceList(w, params)
    dl.load_grads(grads)
    opt = make_opt(w)
    n = _abi.SOMA_MAX_RANKS
    parts = torch.rand(n, generator=torch.Generator().manual_seed(11), dtype=torch.float64) * 0.5
    local = torch.zeros(1, dtype=torch.float64, device="cuda")
    opt.sumsq(dl.tl, w.grad_divisor, local)
    parts[n // 3] = local.item()
    opt.step_from_sumsq(dl.tl, w.grad_divisor, w.max_norm, parts.cuda())
    norm, coef, nonfinite = opt.get_norm()
    total = 0.0
    for x in parts.tolist():
        total += x
    assert not nonfinite
    assert norm == math.sqrt(total)
    assert coef == oracle.clip_coef(math.sqrt(total), w.max_norm) < 1.0
    q = w.groups[0]
    for k, t in enumerate(w.tensors):
        if not t.trainable:
            continue
        p = params[k].double().numpy().reshape(-1).copy()
        m, v = np.zeros_like(p), np.zeros_like(p)
        oracle.adamw_update(p, grads[k], m, v, lr=q.lr, beta1=q.beta1, beta2=q.beta2, eps=q.eps,
                            weight_decay=q.weight_decay, step=1, c=coef, divisor=w.grad_divisor)
        assert_close(f"{t.name} p", dl.p[k].cpu().numpy(), p)
        assert_close(f"{t.name} m", dl.m[k].cpu().numpy(), m)
        assert_close(f"{t.name} v", dl.v[k].cpu().numpy(), v)
    opt.close()
