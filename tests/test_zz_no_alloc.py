"""soma_clip_norm_noalloc against the regular step.

The library's regular entry points allocate device memory on first use.  Some
callers cannot allow that: an application whose own allocator owns the device
heap (an extra cudaMalloc fails or fragments its pool), or a latency-critical
loop where cudaMalloc/cudaFree, which can synchronise the device, are not
allowed.  soma_clip_norm_noalloc gives them the norm and clip coefficient
using only a fixed scratch array inside the library.  Here it is called through
the C ABI twice in a row, on two different lists, and each result is compared
with the norm and coefficient that soma_opt_step computes on the same inputs.

The file name puts it last in collection order, so a run that stops at its
first failure has run every other test before this one.
"""
import ctypes
import math

import pytest
import torch

import workloads as W
from parity_harness import NORM_RTOL, DeviceList, make_opt
from tensor_grad_clip_gb300 import _abi, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    _abi.load()


def _noalloc(tl, divisor, max_norm, out):
    stream = torch.cuda.current_stream().cuda_stream
    return _abi.soma_clip_norm_noalloc(0, tl.pointer(), tl.n, divisor, max_norm, out.data_ptr(), stream)


def _case(w):
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    dl.load_grads(W.draw_grads(w, 1, "cpu"))
    return dl


def test_two_calls_in_a_row_match_the_step():
    lists = [W.with_steps(W.SMALL["hsdp_shard"](), 1),   # bf16, replicated entries
             W.with_steps(W.SMALL["many_small"](), 1)]   # fp32, frozen and all-zero entries
    cases = [_case(w) for w in lists]
    out = torch.full((2,), float("nan"), dtype=torch.float64, device="cuda")
    for w, dl in zip(lists, cases):
        snap = dl.snapshot()
        p_before = [x.clone() for x in dl.p]
        assert _noalloc(dl.tl, w.grad_divisor, w.max_norm, out) == _abi.SOMA_OK
        torch.cuda.synchronize()
        got_norm, got_coef = out.cpu().tolist()
        dl.check_snapshot(snap)
        assert all(torch.equal(a, b) for a, b in zip(p_before, dl.p))  # nothing updated
        opt = make_opt(w)
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
        norm, coef, _ = opt.get_norm()
        opt.close()
        assert math.isclose(got_norm, norm, rel_tol=NORM_RTOL), (w.name, got_norm, norm)
        assert math.isclose(got_coef, coef, rel_tol=NORM_RTOL), (w.name, got_coef, coef)
        assert norm > 0


def test_oversized_list_is_refused_before_any_work():
    # 100 000 one-element entries need about 4.8 MB of segment table, more
    # than the 4 MiB array; every entry points into real device memory.
    n = 100_000
    buf = torch.zeros(n, dtype=torch.float32, device="cuda")
    arr = (_abi.soma_tensor_t * n)()
    base = buf.data_ptr()
    for k in range(n):
        e = arr[k]
        e.param = e.exp_avg = e.exp_avg_sq = base + 4 * k
        e.grad = base + 4 * k
        e.numel, e.group, e.grad_dtype, e.trainable, e.owned = 1, 0, _abi.SOMA_DTYPE_F32, 1, 1
    out = torch.zeros(2, dtype=torch.float64, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    st = _abi.soma_clip_norm_noalloc(0, ctypes.cast(arr, ctypes.POINTER(_abi.soma_tensor_t)), n, 1.0, 1.0,
                                     out.data_ptr(), stream)
    assert st == _abi.SOMA_ERR_LIMIT
    assert _abi.soma_clip_norm_noalloc(0, None, 0, 1.0, 1.0, None, stream) == _abi.SOMA_ERR_INVALID_ARG
