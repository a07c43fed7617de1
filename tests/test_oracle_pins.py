"""Pins of the fp64 oracle to facts outside itself: closed forms of AdamW,
the clipping identity, exact brute force on tiny inputs, invariants the
SomaSpeed optimizer paragraphs state, and the library special case
(torch.nn.utils clipping + torch.optim.AdamW in float64, the unfused step of
the veRL write-up, 4.2 PPO Update).  CPU only."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import OracleOptimizer, GroupState


def f32(x):
    return np.asarray(x, dtype=np.float32)


def one_tensor_opt(p0, lr, wd, beta1=0.9, beta2=0.999, eps=1e-8):
    return OracleOptimizer([np.asarray(p0, dtype=np.float64)], [(0, True, True)],
                           [GroupState(lr=lr, beta1=beta1, beta2=beta2, eps=eps, weight_decay=wd)])


# --- norm and clip coefficient -------------------------------------------

def test_norm_three_four_five():
    # g = [3, 4], d = 1: the norm is 5 exactly, clip fires with c = 1/(5 + 1e-6).
    assert oracle.tensor_sqsum(f32([3, 4]), 1.0) == 25.0
    opt = one_tensor_opt([0.0, 0.0], lr=0.0, wd=0.0)
    norm, c = opt.step([f32([3, 4])], divisor=1.0, max_norm=1.0)
    assert norm == 5.0
    assert c == 1.0 / 5.000001


def test_norm_uses_normalized_gradient():
    # d = 2 halves the norm: ||[3,4]/2|| = 2.5.
    opt = one_tensor_opt([0.0, 0.0], lr=0.0, wd=0.0)
    norm, c = opt.step([f32([3, 4])], divisor=2.0, max_norm=10.0)
    assert norm == 2.5
    assert c == 1.0  # 10 / 2.500001 > 1 is clamped


def test_clip_coef_clamp_and_epsilon():
    assert oracle.clip_coef(0.0, 1.0) == 1.0
    assert oracle.clip_coef(0.5, 1.0) == 1.0
    assert oracle.clip_coef(1.0 - 1e-6, 1.0) == 1.0  # exactly at the threshold
    assert oracle.clip_coef(3.0, 1.5) == 1.5 / 3.000001


def test_norm_brute_force_exact():
    # Exact rational sum of squares of the exact fp32 inputs, sqrt to 40 digits.
    rng = np.random.default_rng(7)
    gs = [f32(rng.standard_normal(n) * s) for n, s in ((1, 1.0), (3, 1e-3), (5, 20.0))]
    d = 3.0
    exact = sum(Fraction(float(x)) ** 2 for g in gs for x in g) / Fraction(d) ** 2
    from decimal import Decimal, getcontext
    getcontext().prec = 40
    ref = float((Decimal(exact.numerator) / Decimal(exact.denominator)).sqrt())
    opt = OracleOptimizer([np.zeros(g.size) for g in gs], [(0, True, True)] * 3,
                          [GroupState(lr=0.0)])
    assert math.isclose(opt.global_norm(gs, d), ref, rel_tol=1e-15)


def test_bf16_words_widen_exactly():
    # bf16 words: 0x3F80 = 1.0, 0xC000 = -2.0, 0x3E80 = 0.25, 0x0001 = 2^-133.
    words = np.array([0x3F80, 0xC000, 0x3E80, 0x0001], dtype=np.uint16)
    assert oracle.tensor_sqsum(words, 1.0) == 1.0 + 4.0 + 0.0625 + 2.0 ** -266
    t = torch.tensor([1.0, -2.0, 0.25, 3.0e-3], dtype=torch.bfloat16)
    assert oracle.tensor_sqsum(t, 1.0) == sum(float(x) ** 2 for x in t.float())


def test_post_clip_norm_equals_max_norm():
    # When clipping fires, ||c g / d|| = max_norm * norm / (norm + 1e-6).
    rng = np.random.default_rng(11)
    g = f32(rng.standard_normal(1000))
    d, mx = 4.0, 1.0
    opt = one_tensor_opt(np.zeros(1000), lr=0.0, wd=0.0)
    norm, c = opt.step([g], d, mx)
    clipped = np.linalg.norm(g.astype(np.float64) / d * c)
    assert c < 1.0
    assert math.isclose(clipped, mx * norm / (norm + 1e-6), rel_tol=1e-13)
    assert math.isclose(clipped, mx, rel_tol=1e-6)


def test_no_clip_coefficient_is_exactly_one():
    rng = np.random.default_rng(12)
    g = f32(rng.standard_normal(1000) * 1e-3)
    opt = one_tensor_opt(np.zeros(1000), lr=0.0, wd=0.0)
    norm, c = opt.step([g], 1.0, 1.0)
    assert norm < 1.0 and c == 1.0


# --- AdamW closed forms --------------------------------------------------

def test_first_step_closed_form():
    # t = 1, m0 = v0 = 0: m_hat = g', v_hat = g'^2, so
    # p1 = p0 (1 - lr wd) - lr g' / (|g'| + eps).
    rng = np.random.default_rng(3)
    n = 257
    p0 = rng.standard_normal(n) * 0.02
    g = f32(rng.standard_normal(n))
    lr, wd, eps, d = 1e-3, 0.01, 1e-8, 4.0
    opt = one_tensor_opt(p0, lr=lr, wd=wd, eps=eps)
    norm, c = opt.step([g], d, 1.0)
    gp = g.astype(np.float64) / d * c
    expect = p0 * (1 - lr * wd) - lr * gp / (np.abs(gp) + eps)
    np.testing.assert_allclose(opt.params[0], expect, rtol=1e-14, atol=1e-18)
    # and each weight moved by about lr * sign(g) beyond the decay
    np.testing.assert_allclose(p0 * (1 - lr * wd) - opt.params[0], lr * np.sign(gp), rtol=1e-4)


def test_eps_sits_outside_the_square_root():
    # |g'| = eps at t = 1: the step is lr * eps / (eps + eps) = lr / 2.
    eps = 1e-3
    opt = one_tensor_opt([0.0], lr=0.5, wd=0.0, eps=eps)
    opt.step([f32([eps])], 1.0, 1e9)
    assert math.isclose(opt.params[0][0], -0.25, rel_tol=1e-6)


def test_constant_gradient_closed_form():
    # Constant g': m_t = (1 - b1^t) g' and v_t = (1 - b2^t) g'^2, so the bias
    # corrected moments are exactly g' and g'^2 at every t:
    # p_t = p_{t-1} (1 - lr wd) - lr g'/(|g'| + eps).
    lr, wd, eps = 0.01, 0.1, 1e-8
    g = f32([0.5, -0.25, 2.0])
    opt = one_tensor_opt([0.3, -0.2, 0.1], lr=lr, wd=wd, beta1=0.8, beta2=0.95, eps=eps)
    p = np.array([0.3, -0.2, 0.1])
    gp = g.astype(np.float64)
    for t in range(1, 8):
        opt.step([g], 1.0, 1e9)
        p = p * (1 - lr * wd) - lr * gp / (np.abs(gp) + eps)
        np.testing.assert_allclose(opt.params[0], p, rtol=1e-13)
        np.testing.assert_allclose(opt.exp_avg[0], (1 - 0.8 ** t) * gp, rtol=1e-13)
        np.testing.assert_allclose(opt.exp_avg_sq[0], (1 - 0.95 ** t) * gp * gp, rtol=1e-13)


def test_alternating_gradient_closed_form():
    # g' = +a then -a: m_hat_2 = -(1-b1) a / (1+b1), v_hat_2 = a^2.  A swap of
    # b1 and b2 or a wrong bias-correction exponent breaks this.
    a, b1, b2, lr, eps = 0.5, 0.9, 0.999, 0.1, 1e-12
    opt = one_tensor_opt([0.0], lr=lr, wd=0.0, beta1=b1, beta2=b2, eps=eps)
    opt.step([f32([a])], 1.0, 1e9)
    p1 = -lr * a / (a + eps)
    assert math.isclose(opt.params[0][0], p1, rel_tol=1e-14)
    opt.step([f32([-a])], 1.0, 1e9)
    p2 = p1 - lr * (-(1 - b1) * a / (1 + b1)) / (a + eps)
    assert math.isclose(opt.params[0][0], p2, rel_tol=1e-12)


def test_zero_gradients_leave_only_decay():
    lr, wd = 1e-3, 0.1
    p0 = np.array([0.5, -0.125, 3.0])
    opt = one_tensor_opt(p0, lr=lr, wd=wd)
    for t in range(1, 6):
        norm, c = opt.step([f32([0, 0, 0])], 8.0, 1.0)
        assert norm == 0.0 and c == 1.0
        assert not opt.exp_avg[0].any() and not opt.exp_avg_sq[0].any()
        np.testing.assert_allclose(opt.params[0], p0 * (1 - lr * wd) ** t, rtol=1e-15)
    # wd = 0: the weights do not move at all
    opt = one_tensor_opt(p0, lr=lr, wd=0.0)
    opt.step([f32([0, 0, 0])], 8.0, 1.0)
    assert np.array_equal(opt.params[0], p0)


# --- ownership, frozen tensors, step counts ------------------------------

def _three_tensor_case(owned=(True, False, True), trainable=(True, True, False)):
    rng = np.random.default_rng(5)
    sizes = (40, 30, 20)
    params = [rng.standard_normal(n) * 0.02 for n in sizes]
    grads = [f32(rng.standard_normal(n)) for n in sizes]
    flags = [(0, t, o) for t, o in zip(trainable, owned)]
    return params, grads, flags


def test_unowned_and_frozen_gradients_do_not_enter_the_norm():
    params, grads, flags = _three_tensor_case()
    opt = OracleOptimizer(params, flags, [GroupState(lr=1e-3)])
    base = opt.global_norm(grads, 2.0)
    assert math.isclose(base, np.linalg.norm(grads[0].astype(np.float64) / 2.0), rel_tol=1e-14)
    changed = [grads[0], grads[1] * 7, grads[2] * 9]
    assert opt.global_norm(changed, 2.0) == base
    # every trainable tensor owned: the plain norm over trainable tensors
    opt2 = OracleOptimizer(params, [(0, True, True), (0, True, True), (0, False, True)],
                           [GroupState(lr=1e-3)])
    plain = np.linalg.norm(np.concatenate([grads[0], grads[1]]).astype(np.float64) / 2.0)
    assert math.isclose(opt2.global_norm(grads, 2.0), plain, rel_tol=1e-14)


def test_unowned_tensor_updated_with_the_same_coefficient():
    # Two copies of one tensor, one owned and one replicated, step the same.
    rng = np.random.default_rng(9)
    p = rng.standard_normal(64) * 0.02
    g = f32(rng.standard_normal(64))
    opt = OracleOptimizer([p, p], [(0, True, True), (0, True, False)],
                          [GroupState(lr=1e-3, weight_decay=0.01)])
    norm, c = opt.step([g, g], 4.0, 1.0)
    assert math.isclose(norm, np.linalg.norm(g.astype(np.float64) / 4.0), rel_tol=1e-14)
    assert c < 1.0
    assert np.array_equal(opt.params[0], opt.params[1])
    assert np.array_equal(opt.exp_avg_sq[0], opt.exp_avg_sq[1])


def test_frozen_tensor_untouched():
    params, grads, flags = _three_tensor_case()
    opt = OracleOptimizer(params, flags, [GroupState(lr=1e-3, weight_decay=0.5)])
    g_before = [g.copy() for g in grads]
    opt.step(grads, 2.0, 1.0)
    assert np.array_equal(opt.params[2], params[2])
    assert not opt.exp_avg[2].any() and not opt.exp_avg_sq[2].any()
    for a, b in zip(grads, g_before):
        assert np.array_equal(a, b)  # gradients are read only


def test_group_step_counts_and_hyperparameters():
    # group 1 owns only a frozen tensor: its count stays 0.
    rng = np.random.default_rng(2)
    params = [rng.standard_normal(8), rng.standard_normal(8), rng.standard_normal(8)]
    grads = [f32(rng.standard_normal(8)) for _ in range(3)]
    flags = [(0, True, True), (1, False, True), (2, True, True)]
    groups = [GroupState(lr=1e-2), GroupState(lr=1e-2), GroupState(lr=1e-3, beta1=0.5, weight_decay=0.2)]
    opt = OracleOptimizer(params, flags, groups)
    for _ in range(3):
        opt.step(grads, 1.0, 1e9)
    assert [g.step for g in opt.groups] == [3, 0, 3]
    with pytest.raises(ValueError):
        OracleOptimizer([np.zeros(2)], [(5, True, True)], [GroupState(lr=1.0)]).step([f32([1, 2])], 1.0, 1.0)


def test_divisor_nearly_irrelevant_under_strong_clipping():
    # c g / d = max_norm g / (||g|| + d 1e-6): with norm >> 1, updates barely depend on d.
    rng = np.random.default_rng(4)
    p = rng.standard_normal(500) * 0.02
    g = f32(rng.standard_normal(500) * 10)
    outs = []
    for d in (1.0, 4.0, 64.0):
        opt = one_tensor_opt(p, lr=1e-3, wd=0.0)
        opt.step([g], d, 1.0)
        outs.append(opt.exp_avg[0].copy())
    np.testing.assert_allclose(outs[1], outs[0], rtol=1e-6)
    np.testing.assert_allclose(outs[2], outs[0], rtol=1e-5)


def test_deterministic():
    params, grads, flags = _three_tensor_case()
    a = OracleOptimizer(params, flags, [GroupState(lr=1e-3)])
    b = OracleOptimizer(params, flags, [GroupState(lr=1e-3)])
    for _ in range(3):
        ra, rb = a.step(grads, 3.0, 1.0), b.step(grads, 3.0, 1.0)
        assert ra == rb
    for x, y in zip(a.params, b.params):
        assert np.array_equal(x, y)


# --- library special case: torch clipping + torch.optim.AdamW in float64 --

def _torch_reference_run(params, grads_per_step, flags, groups, divisor, max_norm, lrs_per_step):
    """The unfused step with PyTorch library routines in float64: the norm
    over owned gradients, every trainable gradient scaled by the one
    coefficient, then torch.optim.AdamW (single-tensor path)."""
    tp = [torch.tensor(p, dtype=torch.float64, requires_grad=True) for p in params]
    by_group = {}
    for k, (grp, tr, _) in enumerate(flags):
        if tr:
            by_group.setdefault(grp, []).append(tp[k])
    pg = [dict(params=by_group[q], lr=g.lr, betas=(g.beta1, g.beta2), eps=g.eps,
               weight_decay=g.weight_decay) for q, g in enumerate(groups) if q in by_group]
    gidx = [q for q in range(len(groups)) if q in by_group]
    opt = torch.optim.AdamW(pg, foreach=False, fused=False)
    norms = []
    for step, grads in enumerate(grads_per_step):
        for i, q in enumerate(gidx):
            opt.param_groups[i]["lr"] = lrs_per_step[step][q]
        for k, g in enumerate(grads):
            tp[k].grad = torch.tensor(np.asarray(g, dtype=np.float64), dtype=torch.float64) / divisor
        owned = [tp[k].grad for k, (_, tr, o) in enumerate(flags) if tr and o]
        total = torch.nn.utils.get_total_norm(owned, norm_type=2.0)
        trainable = [tp[k] for k, (_, tr, _) in enumerate(flags) if tr]
        torch.nn.utils.clip_grads_with_norm_(trainable, max_norm, total)
        opt.step()
        norms.append(float(total))
    state = opt.state
    return ([p.detach().numpy() for p in tp],
            [state[p]["exp_avg"].numpy() if p in state else None for p in tp],
            [state[p]["exp_avg_sq"].numpy() if p in state else None for p in tp], norms)


@pytest.mark.parametrize("divisor,max_norm,grad_scale", [(4.0, 1.0, 1.0), (8.0, 1.0, 1e-3), (3.0, 0.5, 0.3)])
def test_matches_torch_library_special_case(divisor, max_norm, grad_scale):
    rng = np.random.default_rng(21)
    sizes = (31, 64, 7, 100, 1, 16)
    params = [rng.standard_normal(n) * 0.02 for n in sizes]
    flags = [(0, True, True), (1, True, True), (0, True, False), (0, True, True), (1, True, False),
             (1, False, True)]
    groups = [GroupState(lr=1e-3, weight_decay=0.01), GroupState(lr=2e-3, beta1=0.8, beta2=0.99,
                                                                  eps=1e-6, weight_decay=0.0)]
    steps = 5
    grads_per_step = [[f32(rng.standard_normal(n) * grad_scale) for n in sizes] for _ in range(steps)]
    lrs = [(1e-3 * (1 + 0.5 * s), 2e-3 / (1 + s)) for s in range(steps)]
    ref_p, ref_m, ref_v, ref_norms = _torch_reference_run(params, grads_per_step, flags, groups,
                                                          divisor, max_norm, lrs)
    opt = OracleOptimizer(params, flags, [GroupState(**vars(g)) for g in groups])
    for s in range(steps):
        for q in range(2):
            opt.set_lr(q, lrs[s][q])
        norm, c = opt.step(grads_per_step[s], divisor, max_norm)
        assert math.isclose(norm, ref_norms[s], rel_tol=1e-13)
    for k, (_, tr, _) in enumerate(flags):
        np.testing.assert_allclose(opt.params[k], ref_p[k], rtol=1e-12, atol=1e-18)
        if tr:
            np.testing.assert_allclose(opt.exp_avg[k], ref_m[k], rtol=1e-11, atol=1e-20)
            np.testing.assert_allclose(opt.exp_avg_sq[k], ref_v[k], rtol=1e-11, atol=1e-24)
        else:
            assert np.array_equal(opt.params[k], params[k])


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_gradient_follows_the_library(bad):
    # Not covered by the pages; the reading is clip_grad_norm_'s default
    # (no error): a NaN norm propagates into every update, an infinite norm
    # gives c = 0.
    rng = np.random.default_rng(31)
    sizes = (9, 4)
    params = [rng.standard_normal(n) * 0.02 for n in sizes]
    flags = [(0, True, True), (0, True, True)]
    grads = [f32(rng.standard_normal(n)) for n in sizes]
    grads[1][2] = bad
    groups = [GroupState(lr=1e-3, weight_decay=0.01)]
    ref_p, ref_m, ref_v, ref_norms = _torch_reference_run(params, [grads], flags, groups, 2.0, 1.0, [(1e-3,)])
    opt = OracleOptimizer(params, flags, [GroupState(**vars(g)) for g in groups])
    norm, c = opt.step(grads, 2.0, 1.0)
    if bad != bad:
        assert math.isnan(norm) and math.isnan(c)
    else:
        assert norm == float("inf") and c == 0.0
    for k in range(2):
        np.testing.assert_allclose(opt.params[k], ref_p[k], rtol=1e-12, equal_nan=True)
        np.testing.assert_allclose(opt.exp_avg[k], ref_m[k], rtol=1e-12, equal_nan=True)


def test_binary16_decoder_all_words():
    # Every one of the 65 536 binary16 words against numpy's float16 (NaN
    # words must decode to NaN, signed zeros keep their sign).
    words = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f64(words)
    ref = words.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))
    t = torch.tensor([1.0, -2.5, 6.1e-5, 65504.0], dtype=torch.float16)
    assert oracle.tensor_sqsum(t, 2.0) == sum((float(x) / 2.0) ** 2 for x in t.float())


def test_group_divisors_match_the_library_with_pre_divided_gradients():
    # A group's own divisor d_q normalizes its gradients before the norm and
    # the update: the same as torch with each group's gradients divided by
    # d_q and a step divisor of 1.
    rng = np.random.default_rng(41)
    sizes = (33, 64, 10, 7)
    params = [rng.standard_normal(n) * 0.02 for n in sizes]
    flags = [(0, True, True), (1, True, True), (1, True, False), (2, True, True)]
    divs = (0.0, 3.0, 16.0)  # group 0 keeps the step's divisor
    step_d = 4.0
    groups = [GroupState(lr=1e-3, weight_decay=0.01, divisor=divs[0]),
              GroupState(lr=2e-3, beta1=0.8, divisor=divs[1]),
              GroupState(lr=5e-4, weight_decay=0.1, divisor=divs[2])]
    steps = 3
    grads = [[f32(rng.standard_normal(n)) for n in sizes] for _ in range(steps)]
    eff = [step_d if divs[g] == 0.0 else divs[g] for g, _, _ in flags]
    pre = [[(g.astype(np.float64) / eff[k]) for k, g in enumerate(gs)] for gs in grads]
    ref_p, ref_m, ref_v, ref_norms = _torch_reference_run(params, pre, flags, groups, 1.0, 1.0,
                                                          [(1e-3, 2e-3, 5e-4)] * steps)
    opt = OracleOptimizer(params, flags, [GroupState(**vars(g)) for g in groups])
    for s in range(steps):
        norm, c = opt.step(grads[s], step_d, 1.0)
        assert math.isclose(norm, ref_norms[s], rel_tol=1e-13)
    for k in range(len(sizes)):
        np.testing.assert_allclose(opt.params[k], ref_p[k], rtol=1e-12)
        np.testing.assert_allclose(opt.exp_avg[k], ref_m[k], rtol=1e-11)
