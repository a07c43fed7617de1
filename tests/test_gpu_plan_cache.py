"""Prepared-list cache: a handle keeps the device tables of its last few
distinct lists, so steps that alternate between lists (gradients written
into two buffers in turn) reuse them.  Every step is still compared with
the fp64 oracle; the cache may change only what the host does, never a
result."""
import math

import pytest
import torch

import workloads as W
from parity_harness import NORM_RTOL, DeviceList, assert_close, make_opt, make_oracle
from tensor_grad_clip_gb300 import TensorList, _abi, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


def _workload(steps):
    T = W.TensorSpec
    tensors = [T("a", (300, 17), W.BF16), T("b", (4099,), W.F32, group=1), T("c", (77,), W.F16, owned=False),
               T("d", (65541,), W.BF16, group=1), T("frozen", (33,), trainable=False)]
    groups = (W.GroupSpec(lr=1e-3, weight_decay=0.01), W.GroupSpec(lr=2e-3, beta1=0.8, beta2=0.99))
    return W.Workload(name="buffers", tensors=tuple(tensors), groups=groups, grad_divisor=4.0,
                      max_norm=1.0, steps=steps, grad_std=1.0)


def _alternating(nbuf, steps):
    """`nbuf` gradient buffer sets used in turn, each with its own list of
    entries over the same weights and moments; compared with the oracle
    after every step.  Returns the handle's cache counters."""
    w = _workload(steps)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    lists = [dl.tl]
    extra = []
    for _ in range(nbuf - 1):
        gs = [torch.empty_like(g) for g in dl.g]
        extra.append(gs)
        lists.append(TensorList(dl.p, gs, dl.m, dl.v, groups=[t.group for t in w.tensors],
                                trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors]))
    bufs = [dl.g] + extra
    opt = make_opt(w)
    orc = make_oracle(w, params)
    for s in range(1, steps + 1):
        grads = W.draw_grads(w, s, "cpu")
        b = (s - 1) % nbuf
        for dst, src in zip(bufs[b], grads):
            dst.copy_(src.reshape(-1))
        opt.step(lists[b], w.grad_divisor, w.max_norm)
        norm, coef, _ = opt.get_norm()
        rn, rc = orc.step(grads, w.grad_divisor, w.max_norm)
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s, norm, rn)
        assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s, coef, rc)
        for k, t in enumerate(w.tensors):
            if t.trainable:
                assert_close(f"step {s} {t.name} p", dl.p[k].cpu().numpy(), orc.params[k])
                assert_close(f"step {s} {t.name} m", dl.m[k].cpu().numpy(), orc.exp_avg[k])
                assert_close(f"step {s} {t.name} v", dl.v[k].cpu().numpy(), orc.exp_avg_sq[k])
    dl.check_guards()
    stats = opt.cache_stats()
    opt.close()
    return stats


def test_double_buffered_gradients_build_tables_once_per_buffer():
    stats = _alternating(2, 8)
    assert stats == {"builds": 2, "reuses": 6, "entries": 2}


def test_as_many_lists_as_the_cache_holds():
    n = _abi.SOMA_PLAN_CACHE
    stats = _alternating(n, 3 * n)
    assert stats == {"builds": n, "reuses": 2 * n, "entries": n}


def test_one_list_more_than_the_cache_holds_evicts_in_lru_order():
    # Cycling through one list more than the cache holds evicts the list
    # needed next every time: every step builds, and results stay exact.
    n = _abi.SOMA_PLAN_CACHE + 1
    stats = _alternating(n, 2 * n)
    assert stats == {"builds": 2 * n, "reuses": 0, "entries": n - 1}


def test_tuning_drops_prepared_lists():
    w = _workload(2)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    opt = make_opt(w)
    orc = make_oracle(w, params)
    for s in (1, 2):
        grads = W.draw_grads(w, s, "cpu")
        dl.load_grads(grads)
        if s == 2:
            opt.set_tuning(update_chunk=512, norm_chunk=1024)
            assert opt.cache_stats()["entries"] == 0
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
        orc.step(grads, w.grad_divisor, w.max_norm)
    assert opt.cache_stats() == {"builds": 2, "reuses": 0, "entries": 1}
    assert opt.plan()["update_chunks"] > 100  # the new chunk size took effect
    for k, t in enumerate(w.tensors):
        if t.trainable:
            assert_close(f"{t.name} p", dl.p[k].cpu().numpy(), orc.params[k])
    opt.close()


def test_pipelined_uploads_equal_serial_steps_bit_for_bit():
    # Gradients arrive from pinned host memory.  Pipelined: two device buffers
    # used in turn; step t+1's upload runs on a copy stream while step t's
    # kernels run, each step waits only for its own upload, and an upload
    # waits for the step that last read its buffer.  Serial: one buffer,
    # copy then step.  Both must leave the same bits.
    w = _workload(6)
    params = W.draw_params(w, "cpu")
    host = [[g.reshape(-1).pin_memory() for g in W.draw_grads(w, s, "cpu")] for s in range(1, w.steps + 1)]
    finals = []
    for pipelined in (False, True):
        dl = DeviceList(w, params)
        opt = make_opt(w)
        main = torch.cuda.current_stream()
        if not pipelined:
            for s in range(w.steps):
                for dst, src in zip(dl.g, host[s]):
                    dst.copy_(src, non_blocking=True)
                opt.step(dl.tl, w.grad_divisor, w.max_norm, main)
        else:
            gs2 = [torch.empty_like(g) for g in dl.g]
            tl2 = TensorList(dl.p, gs2, dl.m, dl.v, groups=[t.group for t in w.tensors],
                             trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors])
            bufs = [(dl.g, dl.tl), (gs2, tl2)]
            cs = torch.cuda.Stream()
            copied = [torch.cuda.Event(), torch.cuda.Event()]
            freed = [torch.cuda.Event(), torch.cuda.Event()]

            def upload(s):
                b = s % 2
                cs.wait_event(freed[b])
                with torch.cuda.stream(cs):
                    for dst, src in zip(bufs[b][0], host[s]):
                        dst.copy_(src, non_blocking=True)
                copied[b].record(cs)

            cs.wait_stream(main)
            upload(0)
            for s in range(w.steps):
                b = s % 2
                main.wait_event(copied[b])
                opt.step(bufs[b][1], w.grad_divisor, w.max_norm, main)
                freed[b].record(main)
                if s + 1 < w.steps:
                    upload(s + 1)
            assert opt.cache_stats()["builds"] == 2
        torch.cuda.synchronize()
        dl.check_guards()
        finals.append([x.cpu().view(torch.int32) for x in dl.p + dl.m + dl.v])
        opt.close()
    for k, (a, b) in enumerate(zip(*finals)):
        assert torch.equal(a, b), k


@pytest.mark.parametrize("which", ["many_small", "hsdp_shard", "unaligned"])
def test_segment_tables_tile_every_tensor(which):
    # soma_opt_get_segments on the list the last step ran: both tables cover
    # their tensors exactly once, in list order, in chunks of at most 64
    # segments; a segment's vector body follows its head and is 16-byte
    # aligned in the gradient.
    import numpy as np
    if which == "unaligned":
        w = _workload(1)
        shift = [(k % 3, 1 + k % 5, (k + 1) % 2, 0) for k in range(len(w.tensors))]
    else:
        w = W.with_steps(W.SMALL[which](), 1)
        shift = None
    dl = DeviceList(w, W.draw_params(w, "cpu"), shift=shift)
    dl.load_grads(W.draw_grads(w, 1, "cpu"))
    opt = make_opt(w)
    opt.set_single_launch(0)  # the tables the two kernels use
    opt.step(dl.tl, w.grad_divisor, w.max_norm)
    plan = opt.plan()
    starts = {dl.g[k].data_ptr(): k for k in range(len(w.tensors)) if w.tensors[k].numel}
    for which_tab, want in (("update", lambda t: t.trainable), ("norm", lambda t: t.trainable and t.owned)):
        seg = opt.segments(which_tab)
        assert seg["len"].size == plan[f"{which_tab}_segments"]
        chunks = seg["chunk"]
        assert chunks[0] == 0 and np.all(np.diff(chunks) >= 0) and np.all(np.diff(chunks) <= 1)
        assert chunks[-1] + 1 == plan[f"{which_tab}_chunks"]
        assert np.bincount(chunks).max() <= 64
        covered = {}
        k = -1
        for a, n, h, nv, grp in zip(seg["grad"], seg["len"], seg["head"], seg["nvec"], seg["group"]):
            a, n, h, nv, grp = int(a), int(n), int(h), int(nv), int(grp)
            if a in starts:  # the first segment of a tensor
                k = starts[a]
                off = 0
            esz = dl.g[k].element_size()
            assert a == dl.g[k].data_ptr() + off * esz, (which_tab, k, off)
            assert grp == w.tensors[k].group
            assert 0 <= h <= n and h + 8 * nv <= n
            if nv:
                assert (a + h * esz) % 16 == 0
            off += n
            covered[k] = off
        expect = {k: t.numel for k, t in enumerate(w.tensors) if want(t) and t.numel}
        assert covered == expect, which_tab
    opt.close()
