"""GB300-native fused optimizer step: normalize gradients by the effective
batch, one global L2 norm over owned shards, one clip coefficient, and
AdamW on fp32 weights and moments, in two sm_103a kernels behind a C ABI
(include/soma_opt.h).

This module only marshals arguments for that ABI; torch supplies device
memory and streams.  Typical use::

    opt = SomaOpt(device=0)
    g_mat = opt.add_group(lr=5e-6, weight_decay=0.01)
    tl = TensorList(params, grads, exp_avgs, exp_avg_sqs, groups=[g_mat, ...])
    opt.step(tl, grad_divisor=64.0, max_norm=1.0)      # async on the current stream
    norm, coef, nonfinite = opt.get_norm()            # waits
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

from . import _abi
from ._abi import (SOMA_DTYPE_BF16, SOMA_DTYPE_F16, SOMA_DTYPE_F32, SOMA_MAX_GROUPS,  # noqa: F401
                   soma_plan_t, soma_tensor_t)

__all__ = ["SomaOpt", "TensorList", "SomaError", "load", "soma_tensor_t", "soma_plan_t"]


def load():
    return _abi.load()


class SomaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def _grad_code(dtype) -> int:
    import torch
    if dtype == torch.float32:
        return SOMA_DTYPE_F32
    if dtype == torch.bfloat16:
        return SOMA_DTYPE_BF16
    if dtype == torch.float16:
        return SOMA_DTYPE_F16
    raise TypeError(f"unsupported gradient dtype {dtype} (float32, bfloat16 or float16)")


def _lowp_code(dtype) -> int:
    import torch
    if dtype == torch.bfloat16:
        return SOMA_DTYPE_BF16
    if dtype == torch.float16:
        return SOMA_DTYPE_F16
    raise TypeError(f"unsupported model-weight dtype {dtype} (bfloat16 or float16)")


def _stream_handle(stream) -> int:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_f64_out(t, n):
    import torch
    if t.dtype != torch.float64 or not t.is_cuda or not t.is_contiguous() or t.numel() < n:
        raise ValueError("expected a contiguous float64 CUDA tensor")


class TensorList:
    """The soma_tensor_t array for lists of torch tensors, built once and
    reused every step (the tensors must stay alive and keep their storage).

    params / exp_avgs / exp_avg_sqs: contiguous float32 tensors.
    grads: contiguous float32, bfloat16 or float16 tensors (never written).
    groups: group id per tensor.  trainable / owned: bools per tensor
    (default all True).  Frozen entries may pass None buffers.
    params_lowp: optional bfloat16/float16 model weights per tensor (or None
    entries), rewritten each step from the updated fp32 master `params`."""

    def __init__(self, params: Sequence, grads: Sequence, exp_avgs: Sequence, exp_avg_sqs: Sequence,
                 groups: Sequence[int], trainable: Optional[Sequence[bool]] = None,
                 owned: Optional[Sequence[bool]] = None, params_lowp: Optional[Sequence] = None):
        import torch
        n = len(params)
        if not (len(grads) == len(exp_avgs) == len(exp_avg_sqs) == len(groups) == n):
            raise ValueError("all per-tensor sequences must have the same length")
        trainable = [True] * n if trainable is None else list(trainable)
        owned = [True] * n if owned is None else list(owned)
        params_lowp = [None] * n if params_lowp is None else list(params_lowp)
        if len(params_lowp) != n:
            raise ValueError("params_lowp must have one entry per tensor")
        self.lowp = params_lowp  # keep alive
        self.n = n
        self.array = (soma_tensor_t * max(n, 1))()
        self.tensors = list(zip(params, grads, exp_avgs, exp_avg_sqs))  # keep alive

        def ptr(t, dtype=None):
            if t is None:
                return None
            if not t.is_contiguous():
                raise ValueError("tensors must be contiguous")
            if dtype is not None and t.dtype != dtype:
                raise TypeError(f"expected {dtype}, got {t.dtype}")
            return t.data_ptr()

        for k, (p, g, m, v) in enumerate(self.tensors):
            tr = bool(trainable[k])
            e = self.array[k]
            numel = p.numel() if p is not None else (g.numel() if g is not None else 0)
            if tr:
                for other in (g, m, v):
                    if other is None or other.numel() != numel:
                        raise ValueError(f"tensor {k}: param, grad, exp_avg, exp_avg_sq must have equal numel")
            e.param = ptr(p, torch.float32)
            e.grad = ptr(g)
            e.exp_avg = ptr(m, torch.float32)
            e.exp_avg_sq = ptr(v, torch.float32)
            lp = params_lowp[k]
            if lp is not None and tr and lp.numel() != numel:
                raise ValueError(f"tensor {k}: params_lowp must have the param's numel")
            e.param_lowp = ptr(lp) if (lp is not None and tr) else None
            e.lowp_dtype = _lowp_code(lp.dtype) if (lp is not None and tr) else 0
            e.numel = numel
            e.group = int(groups[k])
            e.grad_dtype = _grad_code(g.dtype) if (tr and g is not None) else 0
            e.trainable = 1 if tr else 0
            e.owned = 1 if owned[k] else 0

    def pointer(self):
        return ctypes.cast(self.array, ctypes.POINTER(soma_tensor_t))


class SomaOpt:
    """A handle of the C library (soma_opt_create ... soma_opt_destroy)."""

    def __init__(self, device: int = 0):
        self._lib = _abi.load()
        h = _abi.soma_opt_t()
        st = _abi.soma_opt_create(ctypes.byref(h), int(device))
        if st != 0:
            raise SomaError(st, _abi.soma_opt_last_error(None).decode())
        self._h = h
        self.device = int(device)
        self._ngroups = 0

    def _check(self, st: int):
        if st != 0:
            raise SomaError(st, _abi.soma_opt_last_error(self._h).decode())

    @property
    def handle(self):
        return self._h

    def add_group(self, lr: float, betas=(0.9, 0.999), eps: float = 1e-8, weight_decay: float = 0.0) -> int:
        gid = ctypes.c_int32()
        self._check(_abi.soma_opt_add_group(self._h, lr, betas[0], betas[1], eps, weight_decay,
                                            ctypes.byref(gid)))
        self._ngroups = gid.value + 1
        return gid.value

    @property
    def num_groups(self) -> int:
        return self._ngroups

    def state_dict(self) -> dict:
        """What the library holds for a checkpoint: each group's
        hyperparameters, own divisor and step count (weights and moments are
        the caller's tensors).  After graph-capturable steps, call
        pull_groups first: their step counts live on the device."""
        groups = []
        for q in range(self._ngroups):
            g = self.get_group(q)
            groups.append(dict(lr=g["lr"], betas=list(g["betas"]), eps=g["eps"], weight_decay=g["weight_decay"],
                               divisor=self.get_group_divisor(q), step=self.get_group_step(q)))
        return {"groups": groups}  # plain numbers and lists: JSON round-trips it unchanged

    def load_state_dict(self, state: dict):
        """Restore state_dict() output: creates the groups on a handle that
        has none, else overwrites as many groups as it has (the counts must
        match).  Before graph-capturable steps, call push_groups after this."""
        groups = state["groups"]
        if self._ngroups == 0:
            for g in groups:
                self.add_group(g["lr"], tuple(g["betas"]), g["eps"], g["weight_decay"])
        elif self._ngroups != len(groups):
            raise ValueError(f"state has {len(groups)} groups, this handle {self._ngroups}")
        for q, g in enumerate(groups):
            self.set_group(q, g["lr"], tuple(g["betas"]), g["eps"], g["weight_decay"])
            self.set_group_divisor(q, g["divisor"])
            self.set_group_step(q, int(g["step"]))

    def set_lr(self, group: int, lr: float):
        self._check(_abi.soma_opt_set_lr(self._h, group, lr))

    def get_group(self, group: int) -> dict:
        vals = [ctypes.c_double() for _ in range(5)]
        self._check(_abi.soma_opt_get_group(self._h, group, *[ctypes.byref(v) for v in vals]))
        lr, b1, b2, eps, wd = (v.value for v in vals)
        return dict(lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd)

    def set_group(self, group: int, lr: float, betas=(0.9, 0.999), eps: float = 1e-8,
                  weight_decay: float = 0.0):
        self._check(_abi.soma_opt_set_group(self._h, group, lr, betas[0], betas[1], eps, weight_decay))

    def set_group_divisor(self, group: int, divisor: float):
        """The group's own effective-batch divisor (0 = the step's)."""
        self._check(_abi.soma_opt_set_group_divisor(self._h, group, divisor))

    def get_group_divisor(self, group: int) -> float:
        d = ctypes.c_double()
        self._check(_abi.soma_opt_get_group_divisor(self._h, group, ctypes.byref(d)))
        return d.value

    def get_group_step(self, group: int) -> int:
        t = ctypes.c_int64()
        self._check(_abi.soma_opt_get_group_step(self._h, group, ctypes.byref(t)))
        return t.value

    def set_group_step(self, group: int, t: int):
        self._check(_abi.soma_opt_set_group_step(self._h, group, t))

    def step(self, tensors: TensorList, grad_divisor: float, max_norm: float, stream=None):
        self._check(_abi.soma_opt_step(self._h, tensors.pointer(), tensors.n, grad_divisor, max_norm,
                                       _stream_handle(stream)))

    def sumsq(self, tensors: TensorList, grad_divisor: float, out, stream=None):
        """This rank's sum of (g/d)^2 over owned entries into `out` (a float64
        CUDA tensor with at least one element; written at out[0])."""
        _check_f64_out(out, 1)
        self._check(_abi.soma_opt_sumsq(self._h, tensors.pointer(), tensors.n, grad_divisor, out.data_ptr(),
                                        _stream_handle(stream)))

    def step_from_sumsq(self, tensors: TensorList, grad_divisor: float, max_norm: float, rank_sumsq,
                        stream=None):
        """The update with the global norm from all ranks' sums (a float64
        CUDA tensor, rank r at index r)."""
        _check_f64_out(rank_sumsq, 1)
        self._check(_abi.soma_opt_step_from_sumsq(self._h, tensors.pointer(), tensors.n, grad_divisor, max_norm,
                                                  rank_sumsq.data_ptr(), rank_sumsq.numel(),
                                                  _stream_handle(stream)))

    def step_graph(self, tensors: TensorList, grad_divisor: float, max_norm: float, stream=None):
        """The graph-capturable step (soma_opt_step_graph): may be called
        inside torch.cuda.graph capture once it has run outside capture."""
        self._check(_abi.soma_opt_step_graph(self._h, tensors.pointer(), tensors.n, grad_divisor, max_norm,
                                             _stream_handle(stream)))

    def push_groups(self, stream=None):
        self._check(_abi.soma_opt_push_groups(self._h, _stream_handle(stream)))

    def pull_groups(self, stream=None):
        self._check(_abi.soma_opt_pull_groups(self._h, _stream_handle(stream)))

    def device_groups(self) -> int:
        """Device address of the soma_device_group_t table."""
        p = ctypes.c_void_p()
        self._check(_abi.soma_opt_device_groups(self._h, ctypes.byref(p)))
        return p.value

    def get_norm(self, stream=None):
        """(norm, clip_coef, nonfinite) of the last step; waits for it.
        nonfinite: steps since the previous call whose norm was not finite."""
        n, c, f = ctypes.c_double(), ctypes.c_double(), ctypes.c_int32()
        self._check(_abi.soma_opt_get_norm(self._h, ctypes.byref(n), ctypes.byref(c), ctypes.byref(f),
                                           _stream_handle(stream)))
        return n.value, c.value, int(f.value)

    def set_timing(self, enable: bool):
        self._check(_abi.soma_opt_set_timing(self._h, 1 if enable else 0))

    def read_timing(self):
        """(norm_kernel_ms, update_kernel_ms, steps) summed since the last read."""
        a, b, s = ctypes.c_double(), ctypes.c_double(), ctypes.c_int64()
        self._check(_abi.soma_opt_read_timing(self._h, ctypes.byref(a), ctypes.byref(b), ctypes.byref(s)))
        return a.value, b.value, s.value

    def plan(self) -> dict:
        p = soma_plan_t()
        self._check(_abi.soma_opt_get_plan(self._h, ctypes.byref(p)))
        return {name: getattr(p, name) for name, _ in soma_plan_t._fields_}

    def segments(self, which: str = "update") -> dict:
        """Segment table of the last step's list ("update" or "norm") as
        numpy arrays: grad (address of the first gradient element), chunk,
        len, head, nvec, group.  Waits for the last step."""
        import numpy as np
        code = {"update": 0, "norm": 1}[which]
        n = ctypes.c_int64()
        self._check(_abi.soma_opt_get_segments(self._h, code, None, 0, ctypes.byref(n)))
        arr = (_abi.soma_segment_t * max(1, n.value))()
        self._check(_abi.soma_opt_get_segments(self._h, code, arr, n.value, ctypes.byref(n)))
        raw = np.frombuffer(arr, dtype=np.dtype([("grad", "<u8"), ("chunk", "<i8"), ("len", "<i4"), ("head", "<i4"),
                                                 ("nvec", "<i4"), ("group", "<i4")]))[:n.value]
        return {name: raw[name].copy() for name in raw.dtype.names}

    def cache_stats(self) -> dict:
        """Prepared-list cache: table builds, steps that reused a prepared
        list, lists held now."""
        b, r, e = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int32()
        self._check(_abi.soma_opt_get_cache_stats(self._h, ctypes.byref(b), ctypes.byref(r), ctypes.byref(e)))
        return {"builds": b.value, "reuses": r.value, "entries": e.value}

    def set_tuning(self, update_chunk: int = 0, norm_chunk: int = 0, update_ctas_per_sm: int = 0,
                   norm_ctas_per_sm: int = 0):
        self._check(_abi.soma_opt_set_tuning(self._h, update_chunk, norm_chunk, update_ctas_per_sm,
                                             norm_ctas_per_sm))

    def set_single_launch(self, max_elements: int = -1):
        """Regular steps of lists with at most max_elements trainable elements
        run as one kernel (one thread-block cluster); -1 = automatic, 0 = never."""
        self._check(_abi.soma_opt_set_single_launch(self._h, max_elements))

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _abi.soma_opt_destroy(self._h)
            self._h = _abi.soma_opt_t()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
