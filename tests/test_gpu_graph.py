"""The graph-capturable step: captured once with torch.cuda.graph, replayed
with fresh gradients and a changing learning rate, checked against the fp64
oracle after every replay; plus the rules that keep a captured graph valid."""
import math
from dataclasses import replace

import pytest
import torch

import workloads as W
from parity_harness import NORM_RTOL, DeviceList, assert_close, make_opt, make_oracle, sixty_four_groups
from tensor_grad_clip_gb300 import SomaError, _abi, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


class _DevArray:
    """A torch view of library-owned device memory."""

    def __init__(self, ptr, n, typestr="<f8"):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr, "data": (ptr, False),
                                         "version": 3}


def _check_state(w, dl, orc, step):
    for k, t in enumerate(w.tensors):
        if t.trainable:
            assert_close(f"replay {step} {t.name} p", dl.p[k].cpu().numpy(), orc.params[k])
            assert_close(f"replay {step} {t.name} m", dl.m[k].cpu().numpy(), orc.exp_avg[k])
            assert_close(f"replay {step} {t.name} v", dl.v[k].cpu().numpy(), orc.exp_avg_sq[k])


@pytest.mark.parametrize("lr_route", ["push_groups", "device_table"])
def test_captured_step_replays_match_the_oracle(lr_route):
    w = W.SMALL["flat"]()              # cosine lr, wd 0.1, no clipping
    w2 = W.with_steps(W.SMALL["hsdp_shard"](), 6)  # two groups, replicated tensors, bf16
    for wl in (w, w2):
        params = W.draw_params(wl, "cpu")
        dl = DeviceList(wl, params)
        opt = make_opt(wl)
        orc = make_oracle(wl, params)
        stream = torch.cuda.Stream()
        table = torch.as_tensor(_DevArray(opt.device_groups(), 8 * _abi.SOMA_MAX_GROUPS), device="cuda")
        graph = torch.cuda.CUDAGraph()
        for s in range(1, wl.steps + 1):
            grads = W.draw_grads(wl, s, "cpu")
            dl.load_grads(grads)
            lrs = wl.group_lrs(s)
            for q, lr in enumerate(lrs):
                orc.set_lr(q, lr)
                opt.set_lr(q, lr)
            stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                if s == 1 or lr_route == "push_groups":
                    opt.push_groups(stream)
                else:
                    for q, lr in enumerate(lrs):
                        table[8 * q].fill_(lr)  # lr is the first field of a 64-byte entry
                if s == 1:
                    opt.step_graph(dl.tl, wl.grad_divisor, wl.max_norm, stream)  # outside capture
                    with torch.cuda.graph(graph, stream=stream):
                        opt.step_graph(dl.tl, wl.grad_divisor, wl.max_norm, stream)
                else:
                    graph.replay()
            norm, coef, nonfinite = opt.get_norm(stream)
            rn, rc = orc.step(grads, wl.grad_divisor, wl.max_norm)
            assert not nonfinite
            assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s, norm, rn)
            assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s, coef, rc)
            torch.cuda.current_stream().wait_stream(stream)
            _check_state(wl, dl, orc, s)
        opt.pull_groups(stream)
        for q in range(len(wl.groups)):
            assert opt.get_group_step(q) == wl.steps == orc.groups[q].step
        del graph
        opt.close()


@pytest.mark.parametrize("group_div", [False, True])
def test_graph_replays_equal_regular_steps_bit_for_bit(group_div):
    # Regular steps derive each group's constants on the host, graph replays
    # on the device, with the same fp64 operations rounded one at a time: the
    # weights and moments agree bit for bit, also after a resume at a large
    # step count and with a learning rate that changes every step.
    w = W.with_steps(W.SMALL["hsdp_shard"](), 4)  # two groups, bf16 grads, replicated tensors
    if group_div:
        w = replace(w, groups=(replace(w.groups[0], divisor=3.0), w.groups[1]))
    _regular_vs_graph(w, (123457, 7))


@pytest.mark.parametrize("single", [False, True], ids=["two_kernels", "single_launch"])
def test_sixty_four_groups_graph_replays_equal_regular_steps(single):
    # The device group table at the group limit: every group's constants and
    # step count, derived on the device, match the host's for regular steps.
    _regular_vs_graph(sixty_four_groups(), tuple(1000 * q + 1 for q in range(64)),
                      single_launch=None if single else 0)


def _regular_vs_graph(w, resume, single_launch=None):
    finals, norms = [], []
    for graph_mode in (False, True):
        params = W.draw_params(w, "cpu")
        dl = DeviceList(w, params)
        opt = make_opt(w)
        if single_launch is not None:
            opt.set_single_launch(single_launch)
        for q, t in enumerate(resume):
            opt.set_group_step(q, t)
        stream = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        got = []
        for s in range(1, w.steps + 1):
            dl.load_grads(W.draw_grads(w, s, "cpu"))
            for q in range(len(w.groups)):
                opt.set_lr(q, w.groups[q].lr * (1.0 + 0.37 * s + 0.11 * q))
            stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                if not graph_mode:
                    opt.step(dl.tl, w.grad_divisor, w.max_norm, stream)
                else:
                    opt.push_groups(stream)
                    if s == 1:
                        opt.step_graph(dl.tl, w.grad_divisor, w.max_norm, stream)
                        with torch.cuda.graph(graph, stream=stream):
                            opt.step_graph(dl.tl, w.grad_divisor, w.max_norm, stream)
                    else:
                        graph.replay()
            got.append(opt.get_norm(stream))
            torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        if graph_mode:
            opt.pull_groups(stream)
        stepped = [any(t.trainable and t.group == q for t in w.tensors) for q in range(len(w.groups))]
        assert ([opt.get_group_step(q) for q in range(len(w.groups))] ==
                [t + (w.steps if stepped[q] else 0) for q, t in enumerate(resume)])
        finals.append([x.cpu().view(torch.int32) for x in dl.p + dl.m + dl.v])
        norms.append(got)
        del graph
        opt.close()
    assert norms[0] == norms[1]
    for k, (a, b) in enumerate(zip(*finals)):
        assert torch.equal(a, b), k


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # the refused steps capture nothing
def test_rules_that_keep_a_captured_graph_valid():
    w = W.with_steps(W.SMALL["tiny"](), 1)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    other = DeviceList(w, params)
    opt = make_opt(w)
    with pytest.raises(SomaError) as e:  # groups not on the device yet
        opt.step_graph(dl.tl, w.grad_divisor, w.max_norm)
    assert e.value.status == _abi.SOMA_ERR_STATE
    opt.push_groups()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        with pytest.raises(SomaError):  # first call for a list inside capture
            with torch.cuda.graph(graph, stream=stream):
                opt.step_graph(dl.tl, w.grad_divisor, w.max_norm, stream)
    torch.cuda.synchronize()
    opt.step_graph(dl.tl, w.grad_divisor, w.max_norm)
    for call in (lambda: opt.step_graph(other.tl, w.grad_divisor, w.max_norm),
                 lambda: opt.step(other.tl, w.grad_divisor, w.max_norm),
                 lambda: opt.set_tuning(update_chunk=1024)):
        with pytest.raises(SomaError) as e:
            call()
        assert e.value.status == _abi.SOMA_ERR_STATE
    opt.step(dl.tl, w.grad_divisor, w.max_norm)  # the same list still works on the regular path
    torch.cuda.synchronize()
    opt.close()


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")  # the refused steps capture nothing
def test_regular_and_multirank_steps_refuse_stream_capture():
    # Their constants are fixed at enqueue time, so a captured launch would
    # replay stale step counts: capture is refused, and nothing changes.
    w = W.with_steps(W.SMALL["tiny"](), 2)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    opt = make_opt(w)
    dl.load_grads(W.draw_grads(w, 1, "cpu"))
    opt.step(dl.tl, w.grad_divisor, w.max_norm)  # the list is prepared
    torch.cuda.synchronize()
    p_before = [x.clone() for x in dl.p]
    sums = torch.zeros(1, dtype=torch.float64, device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    calls = (lambda s: opt.step(dl.tl, w.grad_divisor, w.max_norm, s),
             lambda s: opt.sumsq(dl.tl, w.grad_divisor, sums, s),
             lambda s: opt.step_from_sumsq(dl.tl, w.grad_divisor, w.max_norm, sums, s))
    for call in calls:
        graph = torch.cuda.CUDAGraph()
        with pytest.raises(SomaError) as e:
            with torch.cuda.stream(stream):
                with torch.cuda.graph(graph, stream=stream):
                    call(stream)
        assert e.value.status == _abi.SOMA_ERR_STATE
        assert "soma_opt_step_graph" in str(e.value)
        del graph
    torch.cuda.synchronize()
    assert opt.get_group_step(0) == 1
    for a, b in zip(p_before, dl.p):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    opt.step(dl.tl, w.grad_divisor, w.max_norm)  # still usable outside capture
    assert opt.get_group_step(0) == 2
    opt.close()


def test_regular_and_graph_steps_mixed_on_one_handle():
    # The documented rule: push_groups before graph steps that follow regular
    # ones, pull_groups before regular steps that follow graph steps.  Every
    # step is compared with the oracle.
    w = W.with_steps(W.SMALL["hsdp_shard"](), 6)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    opt = make_opt(w)
    orc = make_oracle(w, params)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    for s in range(1, w.steps + 1):
        grads = W.draw_grads(w, s, "cpu")
        dl.load_grads(grads)
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            if s in (1, 2, 5, 6):  # regular steps
                if s == 5:
                    opt.pull_groups(stream)
                opt.step(dl.tl, w.grad_divisor, w.max_norm, stream)
            else:  # graph steps 3 and 4
                if s == 3:
                    opt.push_groups(stream)
                    opt.step_graph(dl.tl, w.grad_divisor, w.max_norm, stream)  # step 3, outside capture
                    with torch.cuda.graph(graph, stream=stream):
                        opt.step_graph(dl.tl, w.grad_divisor, w.max_norm, stream)
                else:
                    graph.replay()  # step 4
        norm, coef, _ = opt.get_norm(stream)
        torch.cuda.current_stream().wait_stream(stream)
        rn, rc = orc.step(grads, w.grad_divisor, w.max_norm)
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s, norm, rn)
        _check_state(w, dl, orc, s)
    assert [opt.get_group_step(q) for q in range(len(w.groups))] == [6] * len(w.groups)
    del graph
    opt.close()
