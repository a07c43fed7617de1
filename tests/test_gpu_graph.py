"""The graph-capturable step: captured once with torch.cuda.graph, replayed
with fresh gradients and a changing learning rate, checked against the fp64
oracle after every replay; plus the rules that keep a captured graph valid."""
import math

import numpy as np
import pytest
import torch

import workloads as W
from parity_harness import NORM_RTOL, DeviceList, assert_close, make_opt, make_oracle
from tensor_grad_clip_gb300 import SomaError, TensorList, _abi, build

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


def test_graph_step_equals_regular_step():
    w = W.with_steps(W.SMALL["action_expert"](), 4)
    finals = []
    for graph_mode in (False, True):
        params = W.draw_params(w, "cpu")
        dl = DeviceList(w, params)
        opt = make_opt(w)
        if graph_mode:
            opt.push_groups()
        for s in range(1, w.steps + 1):
            dl.load_grads(W.draw_grads(w, s, "cpu"))
            (opt.step_graph if graph_mode else opt.step)(dl.tl, w.grad_divisor, w.max_norm)
        torch.cuda.synchronize()
        finals.append([x.cpu().double().numpy() for x in dl.p + dl.m + dl.v])
        opt.close()
    for a, b in zip(*finals):
        assert_close("graph vs regular", b, a, rtol=1e-6, atol=1e-12)


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
