"""GPU-vs-oracle harness shared by the parity tests.

Device buffers are carved out of larger allocations with a sentinel guard
band before and after every tensor; after each step the bands must be
bit-unchanged (an out-of-bounds write shows up there).  Gradients and frozen
tensors are compared bit for bit with copies taken before the step.

Tolerances (per element, after every chained step): norm within 1e-5
relative; p, m, v within 2e-6 * |ref| + 1e-8 of the fp64 oracle.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import workloads as W
from oracle import GroupState, OracleOptimizer
from tensor_grad_clip_gb300 import SomaOpt, TensorList

NORM_RTOL = 1e-5
RTOL = 2e-6
ATOL = 1e-8
PAD = 64                      # guard elements on each side (256 B for fp32)
SENTINEL_F32 = 0x7FC0DEAD     # a NaN payload no computation produces
SENTINEL_BF16 = 0x7FAD


def assert_close(name, got, ref, rtol=RTOL, atol=ATOL, tensor_rtol=0.0):
    """Per element |got - ref| <= rtol |ref| + atol, plus tensor_rtol times
    the tensor's largest |ref| when given (see run_parity)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bound = rtol * np.abs(ref) + atol
    if tensor_rtol and ref.size:
        bound = bound + tensor_rtol * float(np.max(np.abs(ref)))
    bad = ~(err <= bound)
    if bad.any():
        i = int(np.argmax(np.where(bad, err / bound, 0)))
        raise AssertionError(f"{name}: {int(bad.sum())} of {got.size} elements out of tolerance; worst at "
                             f"{i}: got {got.flat[i]!r} ref {ref.flat[i]!r} err {err.flat[i]:.3e} "
                             f"bound {bound.flat[i]:.3e}")


class DeviceList:
    """Device copies of a workload's weights, zero moments and gradient
    buffers, each inside a guard-banded allocation.  `shift` moves every
    buffer of tensor k by shift[k] = (p, g, m, v) elements off the 256-byte
    grid (to exercise unaligned heads)."""

    def __init__(self, w: W.Workload, params_cpu, device="cuda", shift=None, frozen_null=False):
        self.w = w
        self.device = device
        self.bufs = []      # (full buffer, sentinel word, view slice)
        self.p, self.g, self.m, self.v, self.plow = [], [], [], [], []
        for k, t in enumerate(w.tensors):
            sp, sg, sm, sv = shift[k] if shift is not None else (0, 0, 0, 0)
            gdt = W.torch_dtype(t.grad_dtype)
            p = self._alloc(t.numel, torch.float32, sp)
            p.copy_(params_cpu[k].reshape(-1).to(device))
            if t.param_lowp:
                lp = self._alloc(t.numel, W.torch_dtype(t.param_lowp), sp)
                lp.copy_(p.to(lp.dtype))
                self.plow.append(lp)
            else:
                self.plow.append(None)
            g = self._alloc(t.numel, gdt, sg)
            m = self._alloc(t.numel, torch.float32, sm)
            v = self._alloc(t.numel, torch.float32, sv)
            m.zero_()
            v.zero_()
            self.p.append(p)
            self.g.append(g)
            self.m.append(m)
            self.v.append(v)
        trainable = [t.trainable for t in w.tensors]
        if frozen_null:
            none = lambda xs: [x if tr else None for x, tr in zip(xs, trainable)]
            self.tl = TensorList(self.p, none(self.g), none(self.m), none(self.v),
                                 groups=[t.group for t in w.tensors], trainable=trainable,
                                 owned=[t.owned for t in w.tensors], params_lowp=self.plow)
        else:
            self.tl = TensorList(self.p, self.g, self.m, self.v, groups=[t.group for t in w.tensors],
                                 trainable=trainable, owned=[t.owned for t in w.tensors],
                                 params_lowp=self.plow)

    def _alloc(self, numel, dtype, shift):
        full = torch.empty(numel + 2 * PAD + 8, dtype=dtype, device=self.device)
        word = SENTINEL_F32 if dtype == torch.float32 else SENTINEL_BF16
        iview = full.view(torch.int32 if dtype == torch.float32 else torch.int16)
        iview.fill_(word)
        lo = PAD + shift
        self.bufs.append((full, iview.clone(), lo, numel))
        return full[lo:lo + numel]

    def load_grads(self, grads):
        for dst, src in zip(self.g, grads):
            dst.copy_(src.reshape(-1))

    def check_guards(self):
        for full, pattern, lo, numel in self.bufs:
            iv = full.view(pattern.dtype)
            if not torch.equal(iv[:lo], pattern[:lo]) or not torch.equal(iv[lo + numel:], pattern[lo + numel:]):
                raise AssertionError("a guard band around a tensor was overwritten")

    def snapshot(self):
        """Bit copies of every gradient and of frozen tensors' p, m, v."""
        snap = {"g": [x.clone() for x in self.g]}
        snap["frozen"] = [(k, self.p[k].clone(), self.m[k].clone(), self.v[k].clone())
                          for k, t in enumerate(self.w.tensors) if not t.trainable]
        snap["frozen_lowp"] = [(k, self.plow[k].clone()) for k, t in enumerate(self.w.tensors)
                               if not t.trainable and self.plow[k] is not None]
        return snap

    def check_lowp_copies(self):
        """Each model copy is the round-to-nearest-even image of the fp32
        weights the kernel just wrote (torch's CPU conversion as reference)."""
        for k, t in enumerate(self.w.tensors):
            lp = self.plow[k]
            if lp is None or not t.trainable:
                continue
            ref = self.p[k].cpu().to(lp.dtype)
            if not torch.equal(lp.cpu().view(torch.int16), ref.view(torch.int16)):
                raise AssertionError(f"tensor {k}: {lp.dtype} copy is not the rounded fp32 weights")

    def check_snapshot(self, snap):
        bits = lambda x: x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32)
        for k, (a, b) in enumerate(zip(snap["g"], self.g)):
            if not torch.equal(bits(a), bits(b)):
                raise AssertionError(f"gradient {k} changed")
        for k, p, m, v in snap["frozen"]:
            for x, y in ((p, self.p[k]), (m, self.m[k]), (v, self.v[k])):
                if not torch.equal(x.view(torch.int32), y.view(torch.int32)):
                    raise AssertionError(f"frozen tensor {k} changed")
        for k, lp in snap.get("frozen_lowp", []):
            if not torch.equal(lp.view(torch.int16), self.plow[k].view(torch.int16)):
                raise AssertionError(f"frozen tensor {k}'s model copy changed")


def sixty_four_groups(steps=3) -> W.Workload:
    """A list at the group limit (SOMA_MAX_GROUPS = 64): tensor k in group k,
    every group with its own lr, betas, eps and weight decay, every fifth on
    its own divisor; fp32, bf16 and fp16 gradients in turn, some replicated
    (not owned) and some frozen entries (their groups do not step).  59,168
    trainable-or-frozen elements in all, small enough for the single-launch
    step."""
    T = W.TensorSpec
    dts = (W.F32, W.BF16, W.F16)
    tensors = tuple(T(f"t{k}", (200 + 23 * k,), dts[k % 3], group=k, owned=(k % 7 != 3),
                      trainable=(k % 11 != 5)) for k in range(64))
    groups = tuple(W.GroupSpec(lr=1e-3 * (1 + k / 64), beta1=0.8 + 0.003 * k, beta2=0.95 + 0.0007 * k,
                               eps=1e-8 * (1 + k), weight_decay=0.002 * k,
                               divisor=(2.0 + k % 3) if k % 5 == 0 else 0.0) for k in range(64))
    return W.Workload(name="groups64", tensors=tensors, groups=groups, grad_divisor=2.0, max_norm=1.0,
                      steps=steps, grad_std=1.0)


def make_opt(w: W.Workload, device_index=0) -> SomaOpt:
    opt = SomaOpt(device_index)
    for q, g in enumerate(w.groups):
        opt.add_group(lr=g.lr, betas=(g.beta1, g.beta2), eps=g.eps, weight_decay=g.weight_decay)
        if g.divisor:
            opt.set_group_divisor(q, g.divisor)
    return opt


def make_oracle(w: W.Workload, params_cpu) -> OracleOptimizer:
    flags = [(t.group, t.trainable, t.owned) for t in w.tensors]
    groups = [GroupState(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps, weight_decay=g.weight_decay,
                         divisor=g.divisor) for g in w.groups]
    return OracleOptimizer([p.double().numpy().reshape(-1) for p in params_cpu], flags, groups)


def run_parity(w: W.Workload, steps=None, shift=None, frozen_null=False, tuning=None, check_every_step=True,
               tensor_rtol=0.0, single_launch=None, expect_launches=None):
    """Chained steps of `w` on the GPU and in the oracle, compared after
    every step.  Returns the list of (gpu_norm, oracle_norm, gpu_coef,
    oracle_coef) per step.

    tensor_rtol adds that fraction of each tensor's largest |value| to the
    per-element bound.  fp32 evaluation of m = beta1 m + (1 - beta1) g' errs
    by about 2^-24 of its two terms, not of their difference: where they
    cancel, the element-relative bound cannot hold whatever the kernel does.
    The workloads' gradients keep the terms small enough that it does; lists
    with large gradients need this term.

    single_launch: when set, the handle's single-launch limit
    (soma_opt_set_single_launch); expect_launches: when set, the kernels every
    step must have launched (1 = the single-launch step)."""
    steps = w.steps if steps is None else steps
    params = W.draw_params(w, "cpu")
    dl = DeviceList(w, params, shift=shift, frozen_null=frozen_null)
    opt = make_opt(w)
    if tuning:
        opt.set_tuning(**tuning)
    if single_launch is not None:
        opt.set_single_launch(single_launch)
    orc = make_oracle(w, params)
    out = []
    for s in range(1, steps + 1):
        grads = W.draw_grads(w, s, "cpu")
        dl.load_grads(grads)
        lrs = w.group_lrs(s)
        for q, lr in enumerate(lrs):
            opt.set_lr(q, lr)
            orc.set_lr(q, lr)
        snap = dl.snapshot()
        opt.step(dl.tl, w.grad_divisor, w.max_norm)
        norm, coef, nonfinite = opt.get_norm()
        if expect_launches is not None:
            assert opt.plan()["launches_per_step"] == expect_launches, opt.plan()
        rn, rc = orc.step(grads, w.grad_divisor, w.max_norm)
        out.append((norm, rn, coef, rc))
        assert not nonfinite
        assert math.isclose(norm, rn, rel_tol=NORM_RTOL, abs_tol=1e-30), (s, norm, rn)
        assert math.isclose(coef, rc, rel_tol=NORM_RTOL), (s, coef, rc)
        if rc == 1.0:
            assert coef == 1.0
        dl.check_snapshot(snap)
        dl.check_guards()
        dl.check_lowp_copies()
        if check_every_step or s == steps:
            for k, t in enumerate(w.tensors):
                if not t.trainable:
                    continue
                assert_close(f"step {s} {t.name} p", dl.p[k].cpu().numpy(), orc.params[k], tensor_rtol=tensor_rtol)
                assert_close(f"step {s} {t.name} m", dl.m[k].cpu().numpy(), orc.exp_avg[k], tensor_rtol=tensor_rtol)
                assert_close(f"step {s} {t.name} v", dl.v[k].cpu().numpy(), orc.exp_avg_sq[k], tensor_rtol=tensor_rtol)
        for q in range(len(w.groups)):
            assert opt.get_group_step(q) == orc.groups[q].step
    opt.close()
    return out
