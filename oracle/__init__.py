"""ctypes front end of the fp64 oracle (oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline leg use it; the product library never imports it.  Nothing here
imports the product package.

Gradients are handed over in their stored type (fp32, or bf16 / fp16 as raw
16-bit words), weights and moments as fp64 numpy arrays that the oracle
updates in place.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from . import build as _build

GRAD_F32 = 0
GRAD_BF16 = 1
GRAD_F16 = 2

_lib = None


class _Tensor(ctypes.Structure):
    _fields_ = [
        ("param", ctypes.POINTER(ctypes.c_double)),
        ("grad", ctypes.c_void_p),
        ("grad_dtype", ctypes.c_int32),
        ("group", ctypes.c_int32),
        ("exp_avg", ctypes.POINTER(ctypes.c_double)),
        ("exp_avg_sq", ctypes.POINTER(ctypes.c_double)),
        ("numel", ctypes.c_int64),
        ("trainable", ctypes.c_int32),
        ("owned", ctypes.c_int32),
    ]


class _Group(ctypes.Structure):
    _fields_ = [
        ("lr", ctypes.c_double),
        ("beta1", ctypes.c_double),
        ("beta2", ctypes.c_double),
        ("eps", ctypes.c_double),
        ("weight_decay", ctypes.c_double),
        ("step", ctypes.c_int64),
        ("divisor", ctypes.c_double),
    ]


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_build.build())
        dp = ctypes.POINTER(ctypes.c_double)
        L.oracle_tensor_sqsum.restype = ctypes.c_double
        L.oracle_tensor_sqsum.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_double]
        L.oracle_global_norm.restype = ctypes.c_double
        L.oracle_global_norm.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_int64, ctypes.c_double]
        L.oracle_clip_coef.restype = ctypes.c_double
        L.oracle_clip_coef.argtypes = [ctypes.c_double, ctypes.c_double]
        L.oracle_adamw_update.restype = None
        L.oracle_adamw_update.argtypes = [dp, ctypes.c_void_p, ctypes.c_int32, dp, dp, ctypes.c_int64,
                                          ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                          ctypes.c_double, ctypes.c_double, ctypes.c_int64,
                                          ctypes.c_double, ctypes.c_double]
        L.oracle_f16_to_f64.restype = None
        L.oracle_f16_to_f64.argtypes = [ctypes.c_void_p, dp, ctypes.c_int64]
        L.oracle_step.restype = ctypes.c_int
        L.oracle_step.argtypes = [ctypes.POINTER(_Tensor), ctypes.c_int64, ctypes.POINTER(_Group),
                                  ctypes.c_int32, ctypes.c_double, ctypes.c_double, dp, dp]
        _lib = L
    return _lib


def grad_words(g) -> tuple:
    """(numpy array, dtype code) for a CPU gradient given as a torch tensor
    (float32, bfloat16 or float16) or a numpy array (float32, float16, or
    uint16 bf16 words)."""
    try:
        import torch
        if isinstance(g, torch.Tensor):
            g = g.detach().contiguous().reshape(-1)
            if g.dtype == torch.float32:
                return g.numpy(), GRAD_F32
            if g.dtype == torch.bfloat16:
                return g.view(torch.int16).numpy().view(np.uint16), GRAD_BF16
            if g.dtype == torch.float16:
                return g.view(torch.int16).numpy().view(np.uint16), GRAD_F16
            raise TypeError(f"unsupported gradient dtype {g.dtype}")
    except ImportError:  # pragma: no cover
        pass
    g = np.ascontiguousarray(g).reshape(-1)
    if g.dtype == np.float32:
        return g, GRAD_F32
    if g.dtype == np.uint16:
        return g, GRAD_BF16
    if g.dtype == np.float16:
        return g.view(np.uint16), GRAD_F16
    raise TypeError(f"unsupported gradient dtype {g.dtype}")


def f16_to_f64(words) -> np.ndarray:
    """binary16 words (uint16) to fp64 through the oracle's own decoder."""
    w = np.ascontiguousarray(words, dtype=np.uint16).reshape(-1)
    out = np.empty(w.size, dtype=np.float64)
    lib().oracle_f16_to_f64(w.ctypes.data, _dptr(out), w.size)
    return out


def _dptr(a: np.ndarray):
    assert a.dtype == np.float64 and a.flags.c_contiguous
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def tensor_sqsum(grad, divisor: float) -> float:
    """sum_i (g_i / d)^2 over one gradient tensor."""
    a, code = grad_words(grad)
    return lib().oracle_tensor_sqsum(a.ctypes.data, code, a.size, float(divisor))


def clip_coef(norm: float, max_norm: float) -> float:
    return lib().oracle_clip_coef(float(norm), float(max_norm))


def adamw_update(p, grad, m, v, *, lr, beta1, beta2, eps, weight_decay, step, c, divisor):
    """In-place AdamW on fp64 arrays p, m, v with gradient g * c / d."""
    a, code = grad_words(grad)
    assert p.size == a.size == m.size == v.size
    lib().oracle_adamw_update(_dptr(p), a.ctypes.data, code, _dptr(m), _dptr(v), a.size,
                              lr, beta1, beta2, eps, weight_decay, int(step), float(c), float(divisor))


@dataclass
class GroupState:
    lr: float
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.0
    step: int = 0
    divisor: float = 0.0  # the group's own effective-batch divisor; 0 = the step's


class OracleOptimizer:
    """fp64 state (weights, moments, group step counts) of one tensor list.

    `flags` is a list of (group, trainable, owned) per tensor; `params` the
    initial weights (any float array-like, widened to fp64)."""

    def __init__(self, params, flags, groups):
        self.params = [np.array(np.asarray(p, dtype=np.float64).reshape(-1), copy=True) for p in params]
        self.exp_avg = [np.zeros_like(p) for p in self.params]
        self.exp_avg_sq = [np.zeros_like(p) for p in self.params]
        self.flags = [(int(g), bool(t), bool(o)) for g, t, o in flags]
        self.groups = [GroupState(**g) if isinstance(g, dict) else g for g in groups]
        assert len(self.flags) == len(self.params)

    def set_lr(self, group: int, lr: float):
        self.groups[group].lr = float(lr)

    def _tensor_array(self, grads):
        keep = []
        arr = (_Tensor * max(1, len(self.params)))()
        for k, (p, g) in enumerate(zip(self.params, grads)):
            grp, tr, own = self.flags[k]
            if g is None:
                a, code = np.zeros(p.size, dtype=np.float32), GRAD_F32
            else:
                a, code = grad_words(g)
            assert a.size == p.size, (k, a.size, p.size)
            keep.append(a)
            arr[k] = _Tensor(_dptr(p), a.ctypes.data, code, grp, _dptr(self.exp_avg[k]),
                             _dptr(self.exp_avg_sq[k]), p.size, int(tr), int(own))
        return arr, keep

    def global_norm(self, grads, divisor: float) -> float:
        arr, keep = self._tensor_array(grads)
        return lib().oracle_global_norm(arr, len(self.params), float(divisor))

    def step(self, grads, divisor: float, max_norm: float):
        """One step; returns (norm, c)."""
        arr, keep = self._tensor_array(grads)
        garr = (_Group * max(1, len(self.groups)))()
        for q, g in enumerate(self.groups):
            garr[q] = _Group(g.lr, g.beta1, g.beta2, g.eps, g.weight_decay, g.step, g.divisor)
        norm = ctypes.c_double()
        coef = ctypes.c_double()
        rc = lib().oracle_step(arr, len(self.params), garr, len(self.groups), float(divisor),
                               float(max_norm), ctypes.byref(norm), ctypes.byref(coef))
        if rc != 0:
            raise ValueError("oracle_step: a trainable tensor names an unknown group")
        for q, g in enumerate(self.groups):
            g.step = int(garr[q].step)
        del keep
        return norm.value, coef.value
