"""soma_clip_norm_noalloc against the fp64 oracle and the regular step.

The library's regular entry points allocate device memory on first use.  Some
callers cannot allow that: an application whose own allocator owns the device
heap (an extra cudaMalloc fails or fragments its pool), or a latency-critical
loop where cudaMalloc/cudaFree, which can synchronise the device, are not
allowed.  soma_clip_norm_noalloc gives them the norm and clip coefficient
using only a fixed scratch array inside the library.  Here it is called through
the C ABI on three lists in a row, with nothing in between, and each result
{norm, c} is compared with the oracle's global norm and clip coefficient, and
with what soma_opt_step computes on the same inputs.  The lists cover bf16
gradients with replicated entries, fp32 gradients with frozen and all-zero
entries, and fp16 gradients placed off the 16-byte grid (odd element shifts),
so that the table's unaligned heads are used.

The file name puts it last in collection order, so a run that stops at its
first failure has run every other test before this one.
"""
import ctypes
import dataclasses
import math
import time

import pytest
import torch

import workloads as W
from parity_harness import NORM_RTOL, DeviceList, make_opt, make_oracle
from tensor_grad_clip_gb300 import _abi, build

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    _abi.load()
    oracle.lib()


def _noalloc(tl, divisor, max_norm, out):
    stream = torch.cuda.current_stream().cuda_stream
    return _abi.soma_clip_norm_noalloc(0, tl.pointer(), tl.n, divisor, max_norm, out.data_ptr(), stream)


def _f16_list():
    w = W.with_steps(W.SMALL["action_expert"](), 1)
    return dataclasses.replace(w, name=w.name + "-f16",
                               tensors=tuple(dataclasses.replace(t, grad_dtype=W.F16) for t in w.tensors))


def test_calls_in_a_row_match_the_oracle_and_the_step():
    lists = [W.with_steps(W.SMALL["hsdp_shard"](), 1),   # bf16, replicated entries
             W.with_steps(W.SMALL["many_small"](), 1),   # fp32, frozen and all-zero entries
             _f16_list()]                                # fp16, gradients off the 16-byte grid
    shifts = [None, None, [(0, 1 + k % 7, 0, 0) for k in range(len(lists[2].tensors))]]
    cases = []
    for w, sh in zip(lists, shifts):
        params = W.draw_params(w, "cpu")
        grads = W.draw_grads(w, 1, "cpu")
        dl = DeviceList(w, params, shift=sh)
        dl.load_grads(grads)
        cases.append((w, params, grads, dl))
    outs = [torch.full((2,), float("nan"), dtype=torch.float64, device="cuda") for _ in lists]
    snaps = [dl.snapshot() for _, _, _, dl in cases]
    p_before = [[x.clone() for x in dl.p] for _, _, _, dl in cases]
    # the calls back to back on one stream: each reuses the scratch the previous one left
    for (w, _, _, dl), out in zip(cases, outs):
        assert _noalloc(dl.tl, w.grad_divisor, w.max_norm, out) == _abi.SOMA_OK
    torch.cuda.synchronize()
    for (w, params, grads, dl), out, snap, pb in zip(cases, outs, snaps, p_before):
        got_norm, got_coef = out.cpu().tolist()
        dl.check_snapshot(snap)
        dl.check_guards()
        assert all(torch.equal(a, b) for a, b in zip(pb, dl.p))  # nothing updated
        # the oracle: global norm over trainable, owned entries, then c
        rn = make_oracle(w, params).global_norm(grads, w.grad_divisor)
        rc = oracle.clip_coef(rn, w.max_norm)
        assert rn > 0
        assert math.isclose(got_norm, rn, rel_tol=NORM_RTOL), (w.name, got_norm, rn)
        assert math.isclose(got_coef, rc, rel_tol=NORM_RTOL), (w.name, got_coef, rc)
        if rc == 1.0:
            assert got_coef == 1.0
        # the regular step on the same inputs (its chunks differ: equal within the tolerance)
        opt = make_opt(w)
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
        norm, coef, _ = opt.get_norm()
        opt.close()
        assert math.isclose(got_norm, norm, rel_tol=NORM_RTOL), (w.name, got_norm, norm)
        assert math.isclose(got_coef, coef, rel_tol=NORM_RTOL), (w.name, got_coef, coef)


def test_call_returns_without_waiting_for_the_gpu():
    # A caller in a latency-critical loop enqueues the norm behind work that
    # is still running on the stream (here a timed 0.3 s spin).  The call
    # returns at once (its tables travel in kernel arguments, not through a
    # host buffer that has to outlive the call), and the result is right once
    # the stream gets there.
    w = W.with_steps(W.SMALL["action_expert"](), 1)
    params = W.draw_params(w, "cpu")
    grads = W.draw_grads(w, 1, "cpu")
    dl = DeviceList(w, params)
    dl.load_grads(grads)
    out = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    assert _noalloc(dl.tl, w.grad_divisor, w.max_norm, out) == _abi.SOMA_OK  # first call: set-up
    torch.cuda.synchronize()
    out.fill_(float("nan"))
    torch.cuda._sleep(600_000_000)  # 600 M cycles: about 0.3 s at the SM clock
    t0 = time.perf_counter()
    st = _noalloc(dl.tl, w.grad_divisor, w.max_norm, out)
    dt = time.perf_counter() - t0
    torch.cuda.synchronize()
    t_all = time.perf_counter() - t0
    assert st == _abi.SOMA_OK
    assert t_all > 0.1, t_all  # the spin really ran ahead of the norm on the stream
    assert dt < 0.5 * t_all, (dt, t_all)
    got_norm, got_coef = out.cpu().tolist()
    rn = make_oracle(w, params).global_norm(grads, w.grad_divisor)
    assert math.isclose(got_norm, rn, rel_tol=NORM_RTOL), (got_norm, rn)
    assert math.isclose(got_coef, oracle.clip_coef(rn, w.max_norm), rel_tol=NORM_RTOL)


def test_oversized_list_is_refused_before_any_work():
    # 100 000 one-element entries need 100 000 segments of 64 bytes (6.4 MB)
    # in the segment table alone, more than the 4 MiB array; every entry
    # points into real device memory.
    n = 100_000
    buf = torch.zeros(n, dtype=torch.float32, device="cuda")
    arr = (_abi.soma_tensor_t * n)()
    base = buf.data_ptr()
    for k in range(n):
        e = arr[k]
        e.param = e.exp_avg = e.exp_avg_sq = base + 4 * k
        e.grad = base + 4 * k
        e.numel, e.group, e.grad_dtype, e.trainable, e.owned = 1, 0, _abi.SOMA_DTYPE_F32, 1, 1
    out = torch.full((2,), -1.0, dtype=torch.float64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = _abi.soma_clip_norm_noalloc(0, ctypes.cast(arr, ctypes.POINTER(_abi.soma_tensor_t)), n, 1.0, 1.0,
                                     out.data_ptr(), stream)
    assert st == _abi.SOMA_ERR_LIMIT
    torch.cuda.synchronize()
    assert out.cpu().tolist() == [-1.0, -1.0]  # nothing was enqueued
    assert _abi.soma_clip_norm_noalloc(0, None, 0, 1.0, 1.0, None, stream) == _abi.SOMA_ERR_INVALID_ARG


def test_list_near_the_scratch_capacity():
    # 60 000 small fp32 entries (1-17 elements each, at odd element offsets
    # in one buffer, a tenth of them not owned): 54 000 owned segments of 64
    # bytes, about 3.5 MB of tables in the 4 MiB array, staged by about 115
    # copy launches.  The norm and c match the oracle's sum over the owned
    # entries in list order.
    import numpy as np
    n = 60_000
    rng = np.random.default_rng(5)
    sizes = rng.integers(1, 18, n)
    offs = np.cumsum(np.concatenate([[0], (sizes + rng.integers(0, 4, n))[:-1]]))
    owned = rng.random(n) > 0.1
    g_cpu = torch.randn(int(offs[-1] + sizes[-1]), generator=torch.Generator().manual_seed(6))
    g = g_cpu.cuda()
    arr = (_abi.soma_tensor_t * n)()
    base = g.data_ptr()
    for k in range(n):
        e = arr[k]
        e.param = e.exp_avg = e.exp_avg_sq = e.grad = base + 4 * int(offs[k])
        e.numel, e.group, e.grad_dtype, e.trainable, e.owned = int(sizes[k]), 0, _abi.SOMA_DTYPE_F32, 1, int(owned[k])
    out = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    divisor, max_norm = 4.0, 1.0
    st = _abi.soma_clip_norm_noalloc(0, ctypes.cast(arr, ctypes.POINTER(_abi.soma_tensor_t)), n, divisor, max_norm,
                                     out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == _abi.SOMA_OK
    got_norm, got_coef = out.cpu().tolist()
    idx = np.concatenate([np.arange(o, o + s) for o, s, w in zip(offs, sizes, owned) if w])
    rn = math.sqrt(oracle.tensor_sqsum(g_cpu.numpy()[idx], divisor))
    assert math.isclose(got_norm, rn, rel_tol=NORM_RTOL), (got_norm, rn)
    assert math.isclose(got_coef, oracle.clip_coef(rn, max_norm), rel_tol=NORM_RTOL)
