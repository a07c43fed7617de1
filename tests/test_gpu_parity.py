"""GPU parity: the sm_103a kernels through the C ABI against the fp64 oracle,
after every chained step, on reduced-size workloads that still span many
chunks and end in ragged tails, plus the edge cases of the method."""
import math

import numpy as np
import pytest
import torch

import golden_fixture
import workloads as W
from parity_harness import (NORM_RTOL, DeviceList, assert_close, make_opt, make_oracle, run_parity,
                            sixty_four_groups)
from tensor_grad_clip_gb300 import SomaOpt, TensorList, _abi, build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    build.build()


@pytest.mark.parametrize("name", ["tiny", "action_expert", "many_small", "hsdp_shard", "flat"])
def test_workload_parity(name):
    w = W.SMALL[name]()
    res = run_parity(w)
    if name == "tiny":
        assert all(rc < 1.0 for _, _, _, rc in res)  # clipping fires on the tiny list
    if name == "flat":
        assert all(rc == 1.0 for _, _, _, rc in res)  # no-clip path: c is exactly 1


def test_many_chunks_and_persistent_grid():
    # Tiny chunks force hundreds of chunks and segments that straddle tensors;
    # a persistent grid (fewer CTAs than chunks) must give the same bits.
    w = W.with_steps(W.SMALL["action_expert"](), 3)
    run_parity(w, tuning=dict(update_chunk=640, norm_chunk=1024))
    a = _final_state(w, dict(update_chunk=2048, norm_chunk=4096))
    b = _final_state(w, dict(update_chunk=2048, norm_chunk=4096, update_ctas_per_sm=1, norm_ctas_per_sm=1))
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def _final_state(w, tuning=None, shift=None):
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params, shift=shift)
    opt = make_opt(w)
    if tuning:
        opt.set_tuning(**tuning)
    norms = []
    for s in range(1, w.steps + 1):
        dl.load_grads(W.draw_grads(w, s, "cpu"))
        for q, lr in enumerate(w.group_lrs(s)):
            opt.set_lr(q, lr)
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
        norms.append(opt.get_norm()[0])
    torch.cuda.synchronize()
    opt.close()
    return [torch.tensor(norms, dtype=torch.float64)] + [x.cpu().clone() for x in dl.p + dl.m + dl.v]


@pytest.mark.parametrize("name", ["tiny", "action_expert", "many_small", "hsdp_shard", "flat"])
def test_run_to_run_bitwise_identical(name):
    w = W.with_steps(W.SMALL[name](), 3)
    a = _final_state(w)
    b = _final_state(w)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_checkpoint_resume_bitwise_equal_to_an_uninterrupted_run():
    # A checkpoint after step k holds the caller's weights and moments (its
    # own buffers) and the handle's state_dict (group settings, divisors and
    # step counts; bias corrections depend on the counts).  A fresh handle
    # restored from it, on fresh buffers loaded from the checkpoint, runs the
    # remaining steps: norms, weights and moments equal a run that never
    # stopped, bit for bit.
    import json
    from dataclasses import replace
    w = W.with_steps(W.SMALL["hsdp_shard"](), 6)  # two groups, replicated tensors
    w = replace(w, groups=(replace(w.groups[0], divisor=3.0), w.groups[1]))  # one group on its own divisor
    k = 3
    whole = _final_state(w)
    params = W.draw_params(w, "cpu")

    def run(opt, dl, steps):
        norms = []
        for s in steps:
            dl.load_grads(W.draw_grads(w, s, "cpu"))
            for q, lr in enumerate(w.group_lrs(s)):
                opt.set_lr(q, lr)
            opt.step(dl.tl, w.grad_divisor, w.max_norm)
            norms.append(opt.get_norm()[0])
        return norms

    dl = DeviceList(w, params)
    opt = make_opt(w)
    norms = run(opt, dl, range(1, k + 1))
    torch.cuda.synchronize()
    state = json.loads(json.dumps(opt.state_dict()))  # as a checkpoint file holds it
    saved = [x.cpu().clone() for x in dl.p + dl.m + dl.v]
    opt.close()
    del dl
    dl2 = DeviceList(w, params)  # new buffers, at other addresses
    for dst, src in zip(dl2.p + dl2.m + dl2.v, saved):
        dst.copy_(src)
    opt2 = SomaOpt(0)
    opt2.load_state_dict(state)
    assert [opt2.get_group_step(q) for q in range(len(w.groups))] == [k] * len(w.groups)
    norms += run(opt2, dl2, range(k + 1, w.steps + 1))
    torch.cuda.synchronize()
    resumed = [torch.tensor(norms, dtype=torch.float64)] + [x.cpu().clone() for x in dl2.p + dl2.m + dl2.v]
    opt2.close()
    for x, y in zip(whole, resumed):
        assert torch.equal(x.view(torch.int64) if x.dtype == torch.float64 else x.view(torch.int32),
                           y.view(torch.int64) if y.dtype == torch.float64 else y.view(torch.int32))


@pytest.mark.parametrize("pattern", ["same_offset", "mixed_offset"])
def test_unaligned_views(pattern):
    # same_offset: every buffer one element off the 16-byte grid (vector body
    # after a scalar head); mixed_offset: buffers misaligned differently, so
    # some tensors run the element-wise path.
    w = W.with_steps(W.SMALL["hsdp_shard"](), 2)
    shifts = []
    for k, t in enumerate(w.tensors):
        if pattern == "same_offset":
            shifts.append((1, 1, 1, 1))
        else:
            shifts.append((k % 3, (k * 5) % 7, (k + 1) % 2, 0))
    run_parity(w, shift=shifts)


def _custom(tensors, groups=None, divisor=2.0, max_norm=1.0, steps=2, grad_std=1.0):
    groups = groups or (W.GroupSpec(lr=1e-3, weight_decay=0.01),)
    return W.Workload(name="custom", tensors=tuple(tensors), groups=tuple(groups), grad_divisor=divisor,
                      max_norm=max_norm, steps=steps, grad_std=grad_std)


def test_edge_shapes_mixed_dtypes_and_groups():
    T = W.TensorSpec
    tensors = [T("one", (1,)), T("empty", (0,)), T("seven", (7,), W.BF16), T("eight", (8,), W.BF16, group=1),
               T("nine", (9,), W.F32, owned=False), T("frozen", (33,), trainable=False),
               T("big", (70001,), W.BF16, group=2), T("z", (5,), zero_grad=True),
               T("rep_bf16", (4099,), W.BF16, owned=False, group=1), T("empty_frozen", (0,), trainable=False)]
    groups = (W.GroupSpec(lr=1e-3, weight_decay=0.01), W.GroupSpec(lr=2e-3, beta1=0.8, beta2=0.99, eps=1e-6),
              W.GroupSpec(lr=5e-4, weight_decay=0.1), W.GroupSpec(lr=1.0))  # group 3 has no tensors
    w = _custom(tensors, groups, steps=3)
    run_parity(w)
    run_parity(w, frozen_null=True, tuning=dict(update_chunk=64, norm_chunk=64))


@pytest.mark.parametrize("single", [False, True], ids=["two_kernels", "single_launch"])
def test_sixty_four_groups(single):
    # Group ids up to the limit: each group's constants reach its tensors,
    # on the two-kernel path and in the single-launch step.
    w = sixty_four_groups()
    assert len(w.groups) == _abi.SOMA_MAX_GROUPS
    run_parity(w, single_launch=None if single else 0, expect_launches=1 if single else 2)


def test_nothing_owned_and_all_frozen():
    T = W.TensorSpec
    w = _custom([T("a", (100,), owned=False), T("b", (31,), W.BF16, owned=False)])
    res = run_parity(w)
    assert all(n == 0.0 and c == 1.0 for n, _, c, _ in res)
    w = _custom([T("a", (100,), trainable=False), T("b", (31,), W.BF16, trainable=False)])
    run_parity(w)


def test_empty_list():
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    tl = TensorList([], [], [], [], groups=[])
    opt.step(tl, 4.0, 1.0)
    assert opt.get_norm() == (0.0, 1.0, False)
    assert opt.get_group_step(0) == 0
    p = opt.plan()
    assert p["update_chunks"] == 0 and p["launches_per_step"] == 1
    opt.close()


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_gradient(bad):
    T = W.TensorSpec
    w = _custom([T("a", (1000,)), T("b", (64,), W.BF16)], steps=1)
    params = W.draw_params(w, "cpu")
    grads = W.draw_grads(w, 1, "cpu")
    grads[0][17] = bad
    dl = DeviceList(w, params)
    dl.load_grads(grads)
    opt = make_opt(w)
    opt.step(dl.tl, w.grad_divisor, w.max_norm)
    norm, coef, nonfinite = opt.get_norm()
    orc = make_oracle(w, params)
    rn, rc = orc.step(grads, w.grad_divisor, w.max_norm)
    assert nonfinite
    if bad != bad:
        assert math.isnan(norm) and math.isnan(coef) and math.isnan(rc)
    else:
        assert norm == math.inf and coef == 0.0 and rc == 0.0
    for k in range(2):
        got = dl.p[k].cpu().double().numpy()
        np.testing.assert_array_equal(np.isnan(got), np.isnan(orc.params[k]))
        fin = ~np.isnan(got)
        assert_close("p", got[fin], orc.params[k][fin])
    opt.close()


def test_nonfinite_steps_are_counted_until_read():
    # A loop that reads the norm only now and then still learns of a step
    # whose norm was not finite: get_norm counts such steps since its last call.
    T = W.TensorSpec
    w = _custom([T("a", (1000,)), T("b", (64,), W.BF16)], steps=4)
    dl = DeviceList(w, W.draw_params(w, "cpu"))
    opt = make_opt(w)
    for s, bad in ((1, False), (2, True), (3, False), (4, True)):
        grads = W.draw_grads(w, s, "cpu")
        if bad:
            grads[0][5] = float("nan")
        dl.load_grads(grads)
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
        if s == 3:
            norm, coef, nonfinite = opt.get_norm()
            assert math.isfinite(norm) and nonfinite == 1  # step 2, not the last one
    norm, coef, nonfinite = opt.get_norm()
    assert math.isnan(norm) and nonfinite == 1  # step 4 only
    assert opt.get_norm()[2] == 0               # nothing new since
    opt.close()


def test_golden_example_on_gpu():
    g = golden_fixture.load()
    params = [torch.tensor(t["p0"], dtype=torch.float32) for t in g.tensors]
    T = W.TensorSpec
    w = W.Workload(name="golden", tensors=tuple(
        T(t["name"], (len(t["p0"]),), W.BF16 if t["dtype"] == "bf16" else W.F32, t["group"], t["trainable"],
          t["owned"]) for t in g.tensors),
        groups=tuple(W.GroupSpec(**q) for q in g.groups), grad_divisor=g.divisor, max_norm=g.max_norm,
        steps=len(g.grads), grad_std=1.0)
    dl = DeviceList(w, params)
    opt = make_opt(w)
    for s in sorted(g.grads):
        grads = [torch.tensor(v, dtype=torch.float32).to(W.torch_dtype(w.tensors[k].grad_dtype))
                 for k, v in enumerate(g.grads[s])]
        dl.load_grads(grads)
        opt.step(dl.tl, g.divisor, g.max_norm)
        norm, coef, _ = opt.get_norm()
        assert math.isclose(norm, g.expect[s]["norm"], rel_tol=NORM_RTOL)
        assert math.isclose(coef, g.expect[s]["coef"], rel_tol=NORM_RTOL)
        for k, t in enumerate(g.tensors):
            assert_close(f"{s} {t['name']} p", dl.p[k].cpu().numpy(), g.expect[s][(t["name"], "p")])
            assert_close(f"{s} {t['name']} m", dl.m[k].cpu().numpy(), g.expect[s][(t["name"], "m")])
            assert_close(f"{s} {t['name']} v", dl.v[k].cpu().numpy(), g.expect[s][(t["name"], "v")])
    opt.close()


def test_side_stream_and_handoff_between_streams():
    w = W.with_steps(W.SMALL["action_expert"](), 2)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    opt = make_opt(w)
    orc = make_oracle(w, params)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for step, stream in ((1, s1), (2, s2)):
        grads = W.draw_grads(w, step, "cpu")
        dl.load_grads(grads)
        s1.wait_stream(torch.cuda.current_stream())
        s2.wait_stream(torch.cuda.current_stream())
        opt.step(dl.tl, w.grad_divisor, w.max_norm, stream=stream)
        norm, coef, _ = opt.get_norm(stream=stream)
        rn, rc = orc.step(grads, w.grad_divisor, w.max_norm)
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL)
        torch.cuda.current_stream().wait_stream(stream)
    for k in range(len(w.tensors)):
        assert_close("p", dl.p[k].cpu().numpy(), orc.params[k])
    opt.close()


def test_list_change_rebuilds_tables():
    # Alternate between two lists on one handle; each must update only its own tensors.
    wa = W.with_steps(W.SMALL["tiny"](), 1)
    wb = _custom([W.TensorSpec("x", (3000,), W.BF16)], steps=1)
    pa, pb = W.draw_params(wa, "cpu"), W.draw_params(wb, "cpu")
    da, db = DeviceList(wa, pa), DeviceList(wb, pb)
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3, weight_decay=0.01)
    oa, ob = make_oracle(wa, pa), make_oracle(wb, pb)
    for s in (1, 2, 3):
        for w, d, o in ((wa, da, oa), (wb, db, ob)):
            grads = W.draw_grads(w, s, "cpu")
            d.load_grads(grads)
            opt.step(d.tl, w.grad_divisor, w.max_norm)
            norm, _, _ = opt.get_norm()
            rn, _ = o.step(grads, w.grad_divisor, w.max_norm)
            assert math.isclose(norm, rn, rel_tol=NORM_RTOL)
    for w, d, o in ((wa, da, oa), (wb, db, ob)):
        for k, t in enumerate(w.tensors):
            if t.trainable:
                # this handle's single step count advanced on both lists (6 steps);
                # the oracles stepped 3 times each, so only m (no bias correction) matches
                assert_close("m", d.m[k].cpu().numpy(), o.exp_avg[k])
    assert opt.get_group_step(0) == 6
    # both lists stay prepared: two table builds, four steps that reused one
    assert opt.cache_stats() == {"builds": 2, "reuses": 4, "entries": 2}
    opt.close()


def test_timing_counts_steps():
    w = W.with_steps(W.SMALL["flat"](), 3)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    opt = make_opt(w)
    opt.set_timing(True)
    for s in range(1, 4):
        dl.load_grads(W.draw_grads(w, s, "cpu"))
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
    a, b, n = opt.read_timing()
    assert n == 3 and a > 0 and b > 0
    assert opt.read_timing() == (0.0, 0.0, 0)
    opt.close()


@pytest.mark.parametrize("grad_dt,low_dt", [(W.F16, None), (W.BF16, W.BF16), (W.F16, W.F16), (W.F32, W.BF16),
                                            (W.BF16, W.F16)])
def test_fp16_grads_and_master_weight_copies(grad_dt, low_dt):
    # fp16 gradients, and bf16/fp16 model weights rewritten from the fp32
    # master copy in the same pass (the RLinf page's FP32MasterAdamW): the
    # master weights follow the oracle, each copy is its exact rounding.
    T = W.TensorSpec
    tensors = [T("a", (96, 80), grad_dt, param_lowp=low_dt), T("b", (80,), grad_dt, group=1, param_lowp=low_dt),
               T("c", (5003,), grad_dt, param_lowp=low_dt, owned=False), T("d", (7,), grad_dt, param_lowp=low_dt),
               T("e", (70001,), grad_dt, param_lowp=low_dt, group=1),
               T("frozen", (33,), grad_dt, trainable=False, param_lowp=low_dt)]
    groups = (W.GroupSpec(lr=1e-3, weight_decay=0.01), W.GroupSpec(lr=2e-3, beta1=0.8, beta2=0.99))
    w = _custom(tensors, groups, steps=4, grad_std=0.5)
    run_parity(w)
    run_parity(w, shift=[(1, 1, 1, 1)] * len(tensors), tuning=dict(update_chunk=1024, norm_chunk=2048))


def test_group_divisors():
    # Each group normalizes by its own divisor (3 is not a power of two);
    # small chunks put several groups in one chunk.
    T = W.TensorSpec
    tensors = [T("a", (300, 17), W.BF16), T("b", (4099,), W.F32, group=1),
               T("c", (77,), W.F16, group=2, owned=False), T("d", (65541,), W.BF16, group=1),
               T("e", (9,), W.F32, group=2)]
    groups = (W.GroupSpec(lr=1e-3, weight_decay=0.01), W.GroupSpec(lr=2e-3, divisor=3.0),
              W.GroupSpec(lr=5e-4, weight_decay=0.1, divisor=16.0))
    w = _custom(tensors, groups, divisor=4.0, steps=3, grad_std=2.0)
    res = run_parity(w)
    assert all(rc < 1.0 for _, _, _, rc in res)
    run_parity(w, tuning=dict(update_chunk=512, norm_chunk=1024))


def test_degenerate_hyperparameters():
    # lr = 0 leaves the weights bit-unchanged (decay factor exactly 1, step
    # size exactly 0) while the moments still advance; beta1 = beta2 = 0
    # makes m = g' and v = g'^2 with bias corrections of exactly 1; a large
    # eps dominates sqrt(v).
    T = W.TensorSpec
    tensors = [T("frozen_lr", (4099,), W.BF16), T("b0", (3001,), W.F32, group=1),
               T("eps", (777,), W.F16, group=2), T("frozen_lr_rep", (65,), W.F32, owned=False)]
    groups = (W.GroupSpec(lr=0.0, weight_decay=0.5), W.GroupSpec(lr=1e-3, beta1=0.0, beta2=0.0, weight_decay=0.01),
              W.GroupSpec(lr=1e-2, eps=1.0))
    w = _custom(tensors, groups, steps=3, grad_std=0.3)
    run_parity(w)
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params)
    opt = make_opt(w)
    before = [p.clone() for p in dl.p]
    for s in (1, 2):
        dl.load_grads(W.draw_grads(w, s, "cpu"))
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
    torch.cuda.synchronize()
    for k in (0, 3):
        assert torch.equal(before[k].view(torch.int32), dl.p[k].view(torch.int32))
        assert dl.m[k].abs().max().item() > 0
    opt.close()


def test_two_handles_on_two_streams_concurrently():
    # Handles share no state: two lists stepped at the same time on unordered
    # streams each match their own oracle.
    wa = W.with_steps(W.SMALL["action_expert"](), 3)
    wb = W.with_steps(W.SMALL["many_small"](), 3)
    runs = []
    for w in (wa, wb):
        params = W.draw_params(w, "cpu")
        runs.append((w, DeviceList(w, params), make_opt(w), make_oracle(w, params), torch.cuda.Stream()))
    for s in range(1, 4):
        grads = []
        for w, dl, opt, orc, st in runs:
            g = W.draw_grads(w, s, "cpu")
            dl.load_grads(g)
            grads.append(g)
        torch.cuda.synchronize()
        for w, dl, opt, orc, st in runs:  # both enqueued before either is waited on
            opt.step(dl.tl, w.grad_divisor, w.max_norm, st)
        for (w, dl, opt, orc, st), g in zip(runs, grads):
            norm, coef, _ = opt.get_norm(st)
            rn, rc = orc.step(g, w.grad_divisor, w.max_norm)
            assert math.isclose(norm, rn, rel_tol=NORM_RTOL) and math.isclose(coef, rc, rel_tol=NORM_RTOL)
    torch.cuda.synchronize()
    for w, dl, opt, orc, st in runs:
        for k, t in enumerate(w.tensors):
            if t.trainable:
                assert_close(f"{w.name} {t.name} p", dl.p[k].cpu().numpy(), orc.params[k])
                assert_close(f"{w.name} {t.name} v", dl.v[k].cpu().numpy(), orc.exp_avg_sq[k])
        dl.check_guards()
        opt.close()
