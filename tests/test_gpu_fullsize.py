"""Parity at full size, in the layout and launch configuration bench.py times.

Every element, after each chained step:

* the action-expert list (302 M parameters) and the flat list (1.5 G + 256):
  10 steps, the fp64 oracle state of every element kept on the host
  (7.2 GB and 36 GB) and updated by the oracle's own per-tensor function on
  slices of 1 Mi elements over a thread pool;
* the 20 000-tensor list (104 M): 10 steps through the oracle's whole step.

The 7B shard view (6.48 G) would need 155 GB of fp64 state to check every
element after each of its 10 steps.  It is checked instead on every element
after its first step and after its tenth, with each tensor's oracle chain run
on its own (it depends only on that tensor's state, its gradients and each
step's clip coefficient), and after each step on:

* every element of its first and last block (16 tensors, both groups, owned
  and replicated ones: 404 M elements);
* a 64-element window around the start of every segment of both tables
  (soma_opt_get_segments), so that every chunk boundary, every cut of a
  large tensor and every tensor's first and last elements are seen
  (about 25 M elements);
* 128 random elements per tensor.

For every list the norm is the oracle's fp64 sum over every owned gradient
(in pieces of at most 2^26 elements, added in list order), the gradients are
bit-unchanged and the sentinel gaps between tensors are intact.  A single
tensor of more than 2^31 elements covers 64-bit offsets.
"""
import math
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from parity_harness import ATOL, NORM_RTOL, RTOL, assert_close
from tensor_grad_clip_gb300 import SomaOpt, TensorList, build

pytestmark = pytest.mark.gpu

SLICE = 1 << 20
POOL = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()
    oracle.lib()


def divisor_of(w, k):
    """Tensor k's effective-batch divisor: its group's own, else the list's."""
    return w.groups[w.tensors[k].group].divisor or w.grad_divisor


def oracle_norm(w, host_g, pool):
    """sqrt of the oracle's sum of (g/d)^2 over owned tensors, d each
    tensor's divisor; large tensors are summed in pieces of 2^26 elements,
    pieces added in list order."""
    piece = 1 << 26
    tasks = [(k, a) for k, t in enumerate(w.tensors) if t.trainable and t.owned
             for a in range(0, t.numel, piece)]
    total = 0.0
    for x in pool.map(lambda ka: oracle.tensor_sqsum(host_g[ka[0]][ka[1]:ka[1] + piece], divisor_of(w, ka[0])),
                      tasks):
        total += x
    return math.sqrt(total)


def _bad(got, ref):
    """Elements outside |got - ref| <= RTOL |ref| + ATOL (NaN counts as out)."""
    got = got.astype(np.float64)
    err = np.abs(got - ref)
    bound = np.abs(ref)
    bound *= RTOL
    bound += ATOL
    return ~(err <= bound)


def _segment_starts(opt, fb, w):
    """Per tensor, the element offsets at which a segment of either table
    starts (from the segment tables the last step ran).  Also checks that the
    segments tile each table's tensors exactly: every segment inside its
    tensor, consecutive within it, covering it once."""
    esize = fb.G.element_size()
    base = fb.G.data_ptr()
    offs = np.asarray(fb.offsets, dtype=np.int64)
    numel = np.asarray([t.numel for t in w.tensors], dtype=np.int64)
    starts = [[] for _ in w.tensors]
    for which in ("update", "norm"):
        seg = opt.segments(which)
        e = (seg["grad"].astype(np.int64) - base) // esize
        k = np.searchsorted(offs, e, side="right") - 1
        off = e - offs[k]
        assert np.all((off >= 0) & (off + seg["len"] <= numel[k])), which
        covered = np.bincount(k, weights=seg["len"], minlength=len(w.tensors)).astype(np.int64)
        want = np.asarray([t.numel if t.trainable and (which == "update" or t.owned) else 0
                           for t in w.tensors], dtype=np.int64)
        assert np.array_equal(covered, want), which
        for kk in np.unique(k):
            sk = off[k == kk]
            assert np.all(np.diff(sk) > 0) and sk[0] == 0, which  # in order, from the tensor's start
            starts[kk].append(sk)
    return [np.unique(np.concatenate(s)) if s else np.zeros(0, np.int64) for s in starts]


def _windows(starts, numel, half=32):
    if numel == 0 or starts.size == 0:
        return np.zeros(0, np.int64)
    ix = (starts[:, None] + np.arange(-half, half)[None, :]).reshape(-1)
    return np.unique(ix[(ix >= 0) & (ix < numel)])


def run_full(w, steps, select=None, graph=False, extra_idx=None):
    """Chained steps of `w` at full size against the fp64 oracle.

    select(opt, fb) -> per tensor None (every element) or an index array,
    called once after the first step (the segment tables exist then); None
    checks every element of every tensor.  extra_idx is added to every
    sampled tensor."""
    dev = torch.device("cuda", 0)
    fb = W.FlatBuffers(w, dev, grad_step=1)
    opt = SomaOpt(0)
    for i, q in enumerate(w.groups):
        opt.add_group(lr=q.lr, betas=(q.beta1, q.beta2), eps=q.eps, weight_decay=q.weight_decay)
        if q.divisor:
            opt.set_group_divisor(i, q.divisor)
    tl = TensorList(fb.p, fb.g, fb.m, fb.v, groups=[t.group for t in w.tensors],
                    trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors],
                    params_lowp=fb.plow)
    p0 = [x.cpu() for x in fb.p]  # initial weights: fp32, converted to fp64 per checked element
    pool = ThreadPoolExecutor(POOL)
    stream = torch.cuda.Stream() if graph else None
    cuda_graph = torch.cuda.CUDAGraph() if graph else None
    gbits = torch.int16 if fb.G.element_size() == 2 else torch.int32
    idx = idx_t = state = host = None
    checked = 0
    for s in range(1, steps + 1):
        if s > 1:
            fb.load_grads(s)
        lrs = w.group_lrs(s)
        for q, lr in enumerate(lrs):
            opt.set_lr(q, lr)
        g_before = fb.G.view(gbits).clone()
        # every gradient of this step on the host, for the norm and the update
        host_g = [x.cpu() for x in fb.g]
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
        rn = oracle_norm(w, host_g, pool)
        rc = oracle.clip_coef(rn, w.max_norm)
        assert not nonfinite
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s, norm, rn)
        assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s, coef, rc)
        if rc == 1.0:
            assert coef == 1.0
        assert torch.equal(fb.G.view(gbits), g_before), "gradients changed"
        del g_before
        for k, low in enumerate(fb.plow):  # 16-bit model copies: the round-to-nearest-even of the GPU's master
            if low is not None:
                assert torch.equal(low.view(torch.int16), fb.p[k].to(low.dtype).view(torch.int16)), (s, k)

        if idx is None:  # after the first step: choose the checked elements, seed their fp64 state
            sel = select(opt, fb) if select is not None else [None] * len(w.tensors)
            idx, idx_t, state, host = [], [], [], []
            for k, t in enumerate(w.tensors):
                ix = sel[k]
                if ix is not None and extra_idx is not None:
                    ix = np.unique(np.concatenate([ix, extra_idx[(extra_idx >= 0) & (extra_idx < t.numel)]]))
                idx.append(ix)
                idx_t.append(None if ix is None else torch.from_numpy(ix).to(dev))
                n = t.numel if ix is None else ix.size
                pk = p0[k].numpy() if ix is None else p0[k].numpy()[ix]
                state.append([pk.astype(np.float64), np.zeros(n), np.zeros(n)])
                host.append([torch.empty(n, dtype=torch.float32, pin_memory=True) for _ in range(3)])
                checked += n if t.trainable else 0
            del p0

        # the oracle's update of every checked element, slice by slice
        tasks = []
        for k, t in enumerate(w.tensors):
            if not t.trainable:
                continue
            gk = host_g[k] if idx[k] is None else host_g[k][torch.from_numpy(idx[k])]
            for src, dst in zip((fb.p[k], fb.m[k], fb.v[k]), host[k]):
                dst.copy_(src if idx_t[k] is None else src[idx_t[k]])
            for lo in range(0, gk.numel(), SLICE):
                tasks.append((k, lo, min(gk.numel(), lo + SLICE), gk))

        def one(task):
            k, lo, hi, gk = task
            t = w.tensors[k]
            q = w.groups[t.group]
            p_s, m_s, v_s = (x[lo:hi] for x in state[k])
            oracle.adamw_update(p_s, gk[lo:hi], m_s, v_s, lr=lrs[t.group], beta1=q.beta1, beta2=q.beta2, eps=q.eps,
                                weight_decay=q.weight_decay, step=s, c=rc, divisor=divisor_of(w, k))
            out = []
            for nm, got, ref in zip("pmv", host[k], (p_s, m_s, v_s)):
                bad = _bad(got[lo:hi].numpy(), ref)
                if bad.any():
                    out.append((nm, k, lo, np.flatnonzero(bad)))
            return out

        for res in pool.map(one, tasks):
            for nm, k, lo, where in res:
                j = int(where[0])
                ref = state[k]["pmv".index(nm)][lo:lo + j + 1]
                got = host[k]["pmv".index(nm)][lo:lo + j + 1].numpy()
                at = lo + j if idx[k] is None else int(idx[k][lo + j])
                assert_close(f"step {s} {w.tensors[k].name} {nm} (element {at}, {where.size} bad in its slice)",
                             got, ref)
        del host_g
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
    return plan, checked


def sample_indices(numel, seed, k):
    rng = np.random.default_rng(seed * 1000 + k)
    head = np.arange(min(32, numel))
    tail = np.arange(max(0, numel - 32), numel)
    rand = rng.integers(0, numel, size=min(128, numel))
    return np.unique(np.concatenate([head, tail, rand]))


def sampled(w):
    return lambda opt, fb: [sample_indices(t.numel, w.seed, k) for k, t in enumerate(w.tensors)]


@pytest.mark.parametrize("name", ["action_expert", "flat"])
def test_full_size_every_element(name):
    w = W.FULL[name]()
    plan, checked = run_full(w, steps=10)
    assert checked == w.trainable_numel
    assert plan["trainable_numel"] == w.trainable_numel
    assert plan["owned_numel"] == w.owned_numel


def test_full_size_fp16_grads_master_copies_group_divisor():
    # The action-expert list at full size with fp16 gradients, bf16 model
    # copies rewritten from the fp32 master weights in the same pass, and the
    # norm-weight group on its own effective-batch divisor (16 against the
    # list's 64): the kernels' group-divisor variants and the large-list norm
    # table that starts a chunk at every group change.  Every element after
    # each of 3 chained steps; each bf16 copy bit for bit the rounding of the
    # GPU's own master weights.
    import dataclasses
    w = W.action_expert(master=True, steps=3)
    w = dataclasses.replace(
        w, name=w.name + "-f16-groupdiv",
        tensors=tuple(dataclasses.replace(t, grad_dtype=W.F16) for t in w.tensors),
        groups=(w.groups[0], dataclasses.replace(w.groups[1], divisor=16.0)))
    plan, checked = run_full(w, steps=3)
    assert checked == w.trainable_numel


def test_full_size_hsdp_shard_blocks_and_every_chunk_boundary():
    w = W.FULL["hsdp_shard"]()
    per_block = 8

    def select(opt, fb):
        starts = _segment_starts(opt, fb, w)
        out = []
        for k, t in enumerate(w.tensors):
            if k < per_block or k >= len(w.tensors) - per_block:  # first and last block: every element
                out.append(None)
            else:
                out.append(np.unique(np.concatenate([_windows(starts[k], t.numel),
                                                     sample_indices(t.numel, w.seed, k)])))
        return out

    plan, checked = run_full(w, steps=10, select=select)
    assert plan["trainable_numel"] == w.trainable_numel
    assert plan["owned_numel"] == w.owned_numel


def test_full_size_hsdp_shard_run_to_run_bitwise_identical():
    # The step is reproducible at full size: two runs of two chained steps
    # from the same state, on two copies of the weights and moments at
    # different addresses (same alignment), each through a fresh handle,
    # give the same norms and the same p, m and v bit for bit.  The norm is
    # the only reduction; its fixed-order sum of chunk partials does not
    # depend on which CTA finishes last.
    w = W.FULL["hsdp_shard"]()
    dev = torch.device("cuda", 0)
    fb = W.FlatBuffers(w, dev, grad_step=1)
    P2, M2, V2 = fb.P.clone(), fb.M.clone(), fb.V.clone()  # the same initial state, 78 GB

    def views(buf):
        return [buf[fb.offsets[k]:fb.offsets[k] + t.numel] for k, t in enumerate(w.tensors)]

    def run(p, m, v):
        opt = SomaOpt(0)
        for q in w.groups:
            opt.add_group(lr=q.lr, betas=(q.beta1, q.beta2), eps=q.eps, weight_decay=q.weight_decay)
        tl = TensorList(p, fb.g, m, v, groups=[t.group for t in w.tensors],
                        trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors])
        norms = []
        for s in (1, 2):
            fb.load_grads(s)
            for q, lr in enumerate(w.group_lrs(s)):
                opt.set_lr(q, lr)
            opt.step(tl, w.grad_divisor, w.max_norm)
            norms.append(opt.get_norm()[0])
        opt.close()
        return norms

    a = run(fb.p, fb.m, fb.v)
    b = run(views(P2), views(M2), views(V2))
    torch.cuda.synchronize()
    assert [x.hex() for x in a] == [x.hex() for x in b]
    for x, y in ((fb.P, P2), (fb.M, M2), (fb.V, V2)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32))
    assert fb.gaps_intact()


def test_full_size_hsdp_shard_first_step_every_element():
    # Every element of the 7B shard view after its first step: the oracle
    # starts from the same seeded weights with zero moments, so each tensor
    # can be checked on its own, slice by slice, without carrying fp64 state
    # for the whole list (the 10-step chain above is sampled instead).
    w = W.FULL["hsdp_shard"]()
    dev = torch.device("cuda", 0)
    fb = W.FlatBuffers(w, dev, grad_step=1)
    opt = SomaOpt(0)
    for q in w.groups:
        opt.add_group(lr=q.lr, betas=(q.beta1, q.beta2), eps=q.eps, weight_decay=q.weight_decay)
    tl = TensorList(fb.p, fb.g, fb.m, fb.v, groups=[t.group for t in w.tensors],
                    trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors])
    p0 = [x.cpu() for x in fb.p]
    host_g = [x.cpu() for x in fb.g]
    lrs = w.group_lrs(1)
    for q, lr in enumerate(lrs):
        opt.set_lr(q, lr)
    opt.step(tl, w.grad_divisor, w.max_norm)
    norm, coef, nonfinite = opt.get_norm()
    pool = ThreadPoolExecutor(POOL)
    rn = oracle_norm(w, host_g, pool)
    rc = oracle.clip_coef(rn, w.max_norm)
    assert not nonfinite
    assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (norm, rn)
    assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (coef, rc)
    checked = 0
    for k, t in enumerate(w.tensors):
        q = w.groups[t.group]
        got = [x.cpu().numpy() for x in (fb.p[k], fb.m[k], fb.v[k])]

        def one(lo, k=k, t=t, q=q, got=got):
            hi = min(t.numel, lo + SLICE)
            p_s = p0[k].numpy()[lo:hi].astype(np.float64)
            m_s, v_s = np.zeros_like(p_s), np.zeros_like(p_s)
            oracle.adamw_update(p_s, host_g[k][lo:hi], m_s, v_s, lr=lrs[t.group], beta1=q.beta1, beta2=q.beta2,
                                eps=q.eps, weight_decay=q.weight_decay, step=1, c=rc, divisor=divisor_of(w, k))
            out = []
            for nm, g_, r_ in zip("pmv", got, (p_s, m_s, v_s)):
                bad = np.flatnonzero(_bad(g_[lo:hi], r_))
                if bad.size:
                    out.append((nm, lo, bad[:1]))
            return out

        for res in pool.map(one, range(0, t.numel, SLICE)):
            for nm, lo, where in res:
                j = lo + int(where[0])
                raise AssertionError(f"step 1 {t.name} {nm}: element {j} out of tolerance "
                                     f"(got {got['pmv'.index(nm)][j]!r})")
        checked += t.numel
        del got
    assert checked == w.trainable_numel
    gbits = torch.int16
    assert all(torch.equal(fb.g[k].cpu().view(gbits), host_g[k].view(gbits)) for k in range(len(w.tensors)))
    torch.cuda.synchronize()
    assert fb.gaps_intact(), "a write landed outside a tensor"
    opt.close()
    pool.shutdown()
    del fb, p0, host_g
    torch.cuda.empty_cache()


def test_full_size_hsdp_shard_ten_steps_every_element():
    # Every element of the 7B shard view after its 10 chained steps.  Each
    # tensor's oracle chain depends only on its own weights, its gradients
    # and each step's clip coefficient, so the GPU runs the whole chain first
    # (the oracle's norm and c of every step checked and kept), its final
    # p, m, v come back to the host, and the oracle then replays the chain
    # tensor by tensor in fp64.  Weights and gradients are drawn again on the
    # device with the seeds the buffers were filled from (the same values).
    w = W.FULL["hsdp_shard"]()
    dev = torch.device("cuda", 0)
    fb = W.FlatBuffers(w, dev, grad_step=1)
    opt = SomaOpt(0)
    for q in w.groups:
        opt.add_group(lr=q.lr, betas=(q.beta1, q.beta2), eps=q.eps, weight_decay=q.weight_decay)
    tl = TensorList(fb.p, fb.g, fb.m, fb.v, groups=[t.group for t in w.tensors],
                    trainable=[t.trainable for t in w.tensors], owned=[t.owned for t in w.tensors])
    pool = ThreadPoolExecutor(POOL)
    coefs = []
    for s_ in range(1, w.steps + 1):
        if s_ > 1:
            fb.load_grads(s_)
        for q, lr in enumerate(w.group_lrs(s_)):
            opt.set_lr(q, lr)
        opt.step(tl, w.grad_divisor, w.max_norm)
        norm, coef, nonfinite = opt.get_norm()
        host_g = [x.cpu() for x in fb.g]
        rn = oracle_norm(w, host_g, pool)
        del host_g
        rc = oracle.clip_coef(rn, w.max_norm)
        assert not nonfinite
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL), (s_, norm, rn)
        assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s_, coef, rc)
        coefs.append(rc)
    for q in range(len(w.groups)):
        assert opt.get_group_step(q) == w.steps
    torch.cuda.synchronize()
    assert fb.gaps_intact(), "a write landed outside a tensor"
    opt.close()

    # each tensor's final state comes back only when it is checked, so the
    # host holds one tensor's p, m, v at a time (the list's are 78 GB)
    checked = 0
    for k, t in enumerate(w.tensors):
        final_k = [x.cpu().numpy() for x in (fb.p[k], fb.m[k], fb.v[k])]
        q = w.groups[t.group]
        state = [W.draw_param(w, k, dev).reshape(-1).cpu().numpy().astype(np.float64)]
        state += [np.zeros_like(state[0]), np.zeros_like(state[0])]
        slices = range(0, t.numel, SLICE)
        for s_ in range(1, w.steps + 1):
            g = W.draw_grad(w, k, s_, dev).reshape(-1).cpu()
            lr = w.group_lrs(s_)[t.group]

            def upd(lo, s_=s_, g=g, lr=lr, q=q, state=state, n=t.numel):
                hi = min(n, lo + SLICE)
                oracle.adamw_update(state[0][lo:hi], g[lo:hi], state[1][lo:hi], state[2][lo:hi], lr=lr,
                                    beta1=q.beta1, beta2=q.beta2, eps=q.eps, weight_decay=q.weight_decay, step=s_,
                                    c=coefs[s_ - 1], divisor=divisor_of(w, k))
            list(pool.map(upd, slices))
            del g

        def cmp(lo, final_k=final_k, state=state, n=t.numel):
            hi = min(n, lo + SLICE)
            for nm, got, ref in zip("pmv", final_k, state):
                bad = np.flatnonzero(_bad(got[lo:hi], ref[lo:hi]))
                if bad.size:
                    return nm, lo + int(bad[0])
            return None

        for res in pool.map(cmp, slices):
            if res is not None:
                nm, j = res
                i = "pmv".index(nm)
                raise AssertionError(f"after {w.steps} steps {t.name} {nm}: element {j} got {final_k[i][j]!r} "
                                     f"oracle {state[i][j]!r}")
        checked += t.numel
        del state, final_k
    assert checked == w.trainable_numel
    pool.shutdown()
    del fb, tl
    torch.cuda.empty_cache()


def test_full_size_graph_replays():
    # The graph-capturable step at full size: one capture, replays with the
    # lr pushed each step (the flat list's cosine schedule), sampled against
    # the oracle like the regular step.
    w = W.with_steps(W.FULL["flat"](), 4)
    run_full(w, steps=4, select=sampled(w), graph=True)
    w = W.with_steps(W.FULL["action_expert"](), 3)
    run_full(w, steps=3, select=sampled(w), graph=True)


def test_tensor_beyond_2_pow_31_elements():
    n = (1 << 31) + 13
    w = W.Workload(name="huge", tensors=(W.TensorSpec("huge", (n,), W.BF16),),
                   groups=(W.GroupSpec(lr=1e-4, weight_decay=0.01),), grad_divisor=4.0, max_norm=1.0,
                   steps=2, grad_std=1e-3, seed=77)
    around = np.arange((1 << 31) - 20, (1 << 31) + 13)
    run_full(w, steps=2, select=sampled(w), extra_idx=around)


def test_full_size_many_small_every_element():
    # The 20 000-tensor list at full size (104 M trainable elements), every
    # element against the oracle after each of its 10 chained steps.  The flat
    # buffers come back to the host once per step and are sliced per tensor.
    from parity_harness import make_oracle
    w = W.FULL["many_small"]()
    assert w.steps == 10
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
