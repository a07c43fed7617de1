"""Seeded random lists against the fp64 oracle: sizes from 0 to tens of
thousands of elements, all gradient dtypes, bf16/fp16 model copies, several
groups (some with their own divisor), frozen and replicated entries, buffers
shifted off the 16-byte grid, and chunk sizes from the smallest allowed up to
the automatic ones.  Each case runs two chained steps through the C ABI and
is compared element by element after each."""
import numpy as np
import pytest

import workloads as W
from parity_harness import run_parity
from tensor_grad_clip_gb300 import build

pytestmark = pytest.mark.gpu

CASES = 24


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _random_case(seed):
    rng = np.random.Generator(np.random.PCG64(9000 + seed))
    ngroups = int(rng.integers(1, 5))
    groups = []
    for q in range(ngroups):
        groups.append(W.GroupSpec(lr=float(10 ** rng.uniform(-4, -2)), beta1=float(rng.choice([0.0, 0.8, 0.9])),
                                  beta2=float(rng.choice([0.99, 0.999])), eps=float(rng.choice([1e-8, 1e-6])),
                                  weight_decay=float(rng.choice([0.0, 0.01, 0.1])),
                                  divisor=float(rng.choice([0.0, 0.0, 3.0, 16.0]))))
    ntensors = int(rng.integers(1, 40))
    lowp = [None, W.BF16, W.F16][int(rng.integers(0, 3))] if rng.random() < 0.3 else None
    tensors, shifts = [], []
    for k in range(ntensors):
        size = int(rng.choice([0, 1, 7, 8, 9, 63, 64, 65, 1000, 4099, 33000]))
        if rng.random() < 0.3:
            size = int(rng.integers(0, 70000))
        tensors.append(W.TensorSpec(name=f"t{k}", shape=(size,), grad_dtype=str(rng.choice([W.F32, W.BF16, W.F16])),
                                    group=int(rng.integers(0, ngroups)), trainable=bool(rng.random() > 0.1),
                                    owned=bool(rng.random() > 0.2), zero_grad=bool(rng.random() < 0.05),
                                    param_lowp=lowp))
        shifts.append(tuple(int(x) for x in rng.integers(0, 8, size=4)) if rng.random() < 0.4 else (0, 0, 0, 0))
    tuning = None
    if rng.random() < 0.6:
        tuning = dict(update_chunk=int(rng.choice([64, 192, 1024, 8192])),
                      norm_chunk=int(rng.choice([64, 512, 4096, 65536])))
    w = W.Workload(name=f"fuzz{seed}", tensors=tuple(tensors), groups=tuple(groups),
                   grad_divisor=float(rng.choice([1.0, 4.0, 6.0, 64.0])), max_norm=float(rng.choice([0.1, 1.0, 100.0])),
                   steps=2, grad_std=float(rng.choice([0.01, 1.0, 10.0])), seed=100 + seed)
    return w, shifts, tuning


@pytest.mark.parametrize("seed", range(CASES))
def test_random_list(seed):
    w, shifts, tuning = _random_case(seed)
    run_parity(w, shift=shifts, tuning=tuning, tensor_rtol=1e-6)


@pytest.mark.parametrize("seed", range(8))
def test_random_list_graph_replays_equal_regular_steps(seed):
    # The graph step derives each group's constants on the device; on the
    # random lists (beta1 = 0, group divisors, model copies, resumed step
    # counts) its replays must leave the same bits as regular steps.
    import torch
    from parity_harness import DeviceList, make_opt
    w, shifts, tuning = _random_case(seed)
    w = W.with_steps(w, 3)
    finals = []
    for graph_mode in (False, True):
        dl = DeviceList(w, W.draw_params(w, "cpu"), shift=shifts)
        opt = make_opt(w)
        if tuning:
            opt.set_tuning(**tuning)
        for q in range(len(w.groups)):
            opt.set_group_step(q, 1000 * q)
        stream = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        norms = []
        for s in range(1, w.steps + 1):
            dl.load_grads(W.draw_grads(w, s, "cpu"))
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
            norms.append(opt.get_norm(stream))
            torch.cuda.current_stream().wait_stream(stream)
        torch.cuda.synchronize()
        dl.check_guards()
        finals.append((norms, [x.cpu().view(torch.int32) for x in dl.p + dl.m + dl.v]))
        del graph
        opt.close()
    assert finals[0][0] == finals[1][0]
    for k, (a, b) in enumerate(zip(finals[0][1], finals[1][1])):
        assert torch.equal(a, b), k
