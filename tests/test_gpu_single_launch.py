"""The single-launch step for small lists (one thread-block cluster does the
square-sum, the norm and the update): it is taken when it should be, gives
the same bits as the two-kernel step on the same tables, and follows the
fp64 oracle at its size limit and on either side of it."""
import pytest
import torch

import workloads as W
from parity_harness import DeviceList, make_opt, run_parity
from tensor_grad_clip_gb300 import SomaError, _abi, build

pytestmark = pytest.mark.gpu

T = W.TensorSpec


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _custom(tensors, groups=None, divisor=4.0, steps=3):
    groups = groups or (W.GroupSpec(lr=1e-3, weight_decay=0.01), W.GroupSpec(lr=2e-3, beta1=0.8, eps=1e-6))
    return W.Workload(name="custom", tensors=tuple(tensors), groups=tuple(groups), grad_divisor=divisor,
                      max_norm=1.0, steps=steps, grad_std=1.0)


def _copies_list(big=30001):
    # mixed gradient dtypes, model copies, a replicated and a frozen entry
    return _custom([T("a", (96, 80), W.BF16, param_lowp=W.BF16), T("b", (80,), W.F16, group=1, param_lowp=W.F16),
                    T("c", (5003,), W.F32, owned=False), T("d", (7,), W.BF16),
                    T("e", (big,), W.F32, group=1, param_lowp=W.BF16), T("frozen", (33,), trainable=False)])


def _run(w, timing_at=(), single=None, tuning=None):
    """Chained steps; timing is on (two kernels) at the steps in timing_at."""
    dl = DeviceList(w, W.draw_params(w, "cpu"))
    opt = make_opt(w)
    if tuning:
        opt.set_tuning(**tuning)
    if single is not None:
        opt.set_single_launch(single)
    norms, plans = [], []
    for s in range(1, w.steps + 1):
        dl.load_grads(W.draw_grads(w, s, "cpu"))
        opt.set_timing(s in timing_at)
        for q, lr in enumerate(w.group_lrs(s)):
            opt.set_lr(q, lr)
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
        norms.append(opt.get_norm())
        plans.append(opt.plan())
    torch.cuda.synchronize()
    state = [x.cpu().clone() for x in dl.p + dl.m + dl.v] + [x.cpu().clone() for x in dl.plow if x is not None]
    opt.close()
    return norms, plans, state


def _bits(x):
    return x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32)


def _assert_same(a, b):
    assert a[0] == b[0]  # norm, c and the non-finite count of every step
    for x, y in zip(a[2], b[2]):
        assert torch.equal(_bits(x), _bits(y))


@pytest.mark.parametrize("which", ["tiny", "copies", "copies_large", "many_chunks"])
def test_same_bits_as_the_two_kernel_step(which):
    # copies_large: 82 771 elements under a raised limit, more than one vector
    # per thread in each CTA's share, so no update vector is loaded early
    w = {"copies": _copies_list(), "copies_large": _copies_list(70001)}.get(which) or W.with_steps(W.SMALL["tiny"](), 3)
    tuning = dict(update_chunk=64, norm_chunk=64) if which == "many_chunks" else None
    single = 1 << 20 if which == "copies_large" else None
    one = _run(w, tuning=tuning, single=single)
    two = _run(w, timing_at=range(1, w.steps + 1), tuning=tuning, single=single)
    for p in one[1]:
        assert p["launches_per_step"] == 1 and p["single_launch_ctas"] >= 2, p
    for p in two[1]:
        assert p["launches_per_step"] == 2 and p["single_launch_ctas"] == 0, p
    _assert_same(one, two)
    if which == "many_chunks":  # each CTA of the cluster walks many chunks
        assert one[1][0]["norm_chunks"] > 8 * one[1][0]["single_launch_ctas"]


def test_single_and_two_kernel_steps_interleaved():
    # steps 2 and 4 run as two kernels (timing on), the others as one launch,
    # each launched right behind the other kind on the same stream
    w = W.with_steps(W.SMALL["tiny"](), 5)
    _assert_same(_run(w), _run(w, timing_at=(2, 4)))


@pytest.mark.parametrize("which", ["tiny", "copies"])
def test_oracle_parity(which):
    w = W.SMALL["tiny"]() if which == "tiny" else _copies_list()
    run_parity(w, expect_launches=1)


def test_size_limit():
    # the automatic limit is 4096 trainable elements per CTA of the cluster;
    # a list at the limit runs as one launch, one element more as two kernels
    probe = _run(_custom([T("x", (100,))], steps=1))
    k = probe[1][0]["single_launch_ctas"]
    assert k in (2, 4, 8, 16)
    limit = 4096 * k
    for extra, launches in ((0, 1), (1, 2)):
        w = _custom([T("big", (limit - 1000 + extra,), W.BF16), T("norm", (1000,), group=1),
                     T("frozen", (64,), trainable=False)], steps=2)
        run_parity(w, expect_launches=launches)
    # an explicit limit; 0 turns the single launch off
    w = _custom([T("a", (12345,)), T("b", (7655,), W.BF16, group=1)], steps=2)
    run_parity(w, single_launch=20000, expect_launches=1)
    run_parity(w, single_launch=19999, expect_launches=2)
    run_parity(w, single_launch=0, expect_launches=2)


def test_group_divisors():
    # each chunk's partial scaled by its group's 1/d^2, c/d per group: the
    # oracle's results, and the two-kernel step's bits
    groups = (W.GroupSpec(lr=1e-3, weight_decay=0.01), W.GroupSpec(lr=2e-3, divisor=16.0),
              W.GroupSpec(lr=5e-4, divisor=0.5))
    w = _custom([T("a", (3000,)), T("b", (500,), W.BF16, group=1), T("c", (20011,), group=2, param_lowp=W.BF16),
                 T("d", (9,), W.F16, group=1, owned=False)], groups=groups)
    run_parity(w, expect_launches=1)
    one = _run(w)
    two = _run(w, timing_at=range(1, w.steps + 1))
    assert all(p["launches_per_step"] == 1 for p in one[1]) and all(p["launches_per_step"] == 2 for p in two[1])
    _assert_same(one, two)


def test_graph_steps_run_as_one_launch():
    # the graph-capturable step takes the single launch too, its CTAs deriving
    # the group constants from the device table: the same bits as regular steps
    w = W.with_steps(W.SMALL["tiny"](), 3)
    reg = _run(w)
    dl = DeviceList(w, W.draw_params(w, "cpu"))
    opt = make_opt(w)
    stream = torch.cuda.current_stream()
    opt.push_groups(stream)
    norms, plans = [], []
    for s in range(1, w.steps + 1):
        dl.load_grads(W.draw_grads(w, s, "cpu"))
        opt.step_graph(dl.tl, w.grad_divisor, w.max_norm, stream)
        norms.append(opt.get_norm())
        plans.append(opt.plan())
    opt.pull_groups(stream)
    assert all(p["launches_per_step"] == 1 and p["single_launch_ctas"] >= 2 for p in plans), plans
    assert [opt.get_group_step(q) for q in range(len(w.groups))] == [w.steps] * len(w.groups)
    torch.cuda.synchronize()
    state = [x.cpu().clone() for x in dl.p + dl.m + dl.v]
    opt.close()
    _assert_same(reg, (norms, plans, state))


def test_limit_changes_drop_prepared_lists_and_graph_handles_refuse_them():
    w = W.with_steps(W.SMALL["tiny"](), 1)
    dl = DeviceList(w, W.draw_params(w, "cpu"))
    dl.load_grads(W.draw_grads(w, 1, "cpu"))
    opt = make_opt(w)
    opt.step(dl.tl, w.grad_divisor, w.max_norm)
    assert opt.cache_stats()["entries"] == 1 and opt.plan()["launches_per_step"] == 1
    opt.set_single_launch(0)  # the tables are cut differently now: rebuilt at the next step
    assert opt.cache_stats()["entries"] == 0
    opt.step(dl.tl, w.grad_divisor, w.max_norm)
    assert opt.plan()["launches_per_step"] == 2 and opt.cache_stats()["builds"] == 2
    opt.close()
    g = make_opt(w)
    stream = torch.cuda.current_stream()
    g.push_groups(stream)
    g.step_graph(dl.tl, w.grad_divisor, w.max_norm, stream)
    with pytest.raises(SomaError) as e:
        g.set_single_launch(0)  # a captured graph may hold these tables
    assert e.value.status == _abi.SOMA_ERR_STATE
    torch.cuda.synchronize()
    g.close()
