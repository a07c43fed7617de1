"""A device allocation that fails is reported, not fatal: with the GPU's
memory held by other allocations, a step whose tables cannot be allocated
returns SOMA_ERR_OOM and changes nothing (step counts, weights, moments,
the prepared-list cache); once memory is free the same call succeeds.  The
failure is a real cudaMalloc error on the host side; no kernel runs on it."""
import math

import pytest
import torch

from tensor_grad_clip_gb300 import SomaError, SomaOpt, TensorList, _abi, build

pytestmark = pytest.mark.gpu

N = 300_000  # one-element tensors: about 40 MB of segment tables


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _hog(leave_bytes):
    """Device allocations until less than `leave_bytes` stay free."""
    hog = []
    while True:
        free, _ = torch.cuda.mem_get_info()
        if free <= leave_bytes:
            return hog
        n = min(free - leave_bytes // 2, 8 << 30)
        try:
            hog.append(torch.empty(n, dtype=torch.uint8, device="cuda"))
        except torch.cuda.OutOfMemoryError:
            return hog


def test_table_allocation_failure_returns_oom_and_changes_nothing():
    g = torch.Generator(device="cuda").manual_seed(7)
    P = torch.randn(N, device="cuda", generator=g) * 0.02
    G = torch.randn(N, device="cuda", generator=g)
    M = torch.zeros(N, device="cuda")
    V = torch.zeros(N, device="cuda")
    # views 256 B apart would need more memory; one element each is enough
    tl = TensorList([P[k:k + 1] for k in range(N)], [G[k:k + 1] for k in range(N)],
                    [M[k:k + 1] for k in range(N)], [V[k:k + 1] for k in range(N)], groups=[0] * N)
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3, weight_decay=0.01)
    opt.step(TensorList([P[:8]], [G[:8]], [M[:8]], [V[:8]], groups=[0]), 1.0, 1.0)  # device state exists
    torch.cuda.synchronize()
    p_before = P.clone()
    steps_before = opt.get_group_step(0)
    stats_before = opt.cache_stats()
    hog = _hog(leave_bytes=16 << 20)
    try:
        with pytest.raises(SomaError) as e:
            opt.step(tl, 1.0, 1.0)
        assert e.value.status == _abi.SOMA_ERR_OOM, str(e.value)
        assert "cudaMalloc" in str(e.value)
    finally:
        del hog
        torch.cuda.empty_cache()
    torch.cuda.synchronize()
    assert opt.get_group_step(0) == steps_before
    assert opt.cache_stats()["builds"] == stats_before["builds"]
    assert torch.equal(P.view(torch.int32), p_before.view(torch.int32))
    # memory is back: the same call succeeds
    opt.step(tl, 1.0, 1.0)
    norm, coef, nonfinite = opt.get_norm()
    ref = math.sqrt(float((G.double() ** 2).sum()))
    assert not nonfinite and math.isclose(norm, ref, rel_tol=1e-5)
    assert opt.get_group_step(0) == steps_before + 1
    opt.close()


def test_list_too_large_for_free_memory_is_refused_before_allocating(monkeypatch):
    # The flat buffers of a list are checked against the free device memory
    # before any allocation: a list larger than what is free raises
    # MemoryError naming both figures, and nothing is allocated.
    import workloads as W
    from workloads import device as D
    w = W.SMALL["action_expert"]()
    allocated = torch.cuda.memory_allocated()
    monkeypatch.setattr(D.torch.cuda, "mem_get_info", lambda device=None: (1 << 20, 1 << 40))
    monkeypatch.setattr(D.torch.cuda, "memory_reserved", lambda device=None: allocated)  # no cached blocks
    with pytest.raises(MemoryError, match="GB are free"):
        D.FlatBuffers(w, "cuda")
    assert torch.cuda.memory_allocated() == allocated
    monkeypatch.undo()
    fb = D.FlatBuffers(w, "cuda")  # with the real figure it fits
    assert fb.P.numel() >= w.trainable_numel
    del fb
    torch.cuda.empty_cache()
