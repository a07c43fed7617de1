"""ctypes declarations of include/soma_opt.h, one Python name per C name.

Loading fails loudly when libsoma_opt.so has not been built: there is no
fallback implementation of the step anywhere in this package.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

SOMA_OK = 0
SOMA_ERR_INVALID_ARG = 1
SOMA_ERR_BAD_GROUP = 2
SOMA_ERR_DTYPE = 3
SOMA_ERR_ALIGNMENT = 4
SOMA_ERR_OOM = 5
SOMA_ERR_CUDA = 6
SOMA_ERR_STATE = 7
SOMA_ERR_LIMIT = 8

SOMA_DTYPE_F32 = 0
SOMA_DTYPE_BF16 = 1
SOMA_DTYPE_F16 = 2
SOMA_MAX_GROUPS = 64
SOMA_ABI_VERSION = 5
SOMA_MAX_RANKS = 65536
SOMA_PLAN_CACHE = 4

soma_status_t = ctypes.c_int32
soma_opt_t = ctypes.c_void_p


class soma_tensor_t(ctypes.Structure):
    _fields_ = [
        ("param", ctypes.c_void_p),
        ("grad", ctypes.c_void_p),
        ("exp_avg", ctypes.c_void_p),
        ("exp_avg_sq", ctypes.c_void_p),
        ("param_lowp", ctypes.c_void_p),
        ("numel", ctypes.c_int64),
        ("group", ctypes.c_int32),
        ("grad_dtype", ctypes.c_uint8),
        ("trainable", ctypes.c_uint8),
        ("owned", ctypes.c_uint8),
        ("lowp_dtype", ctypes.c_uint8),
    ]


assert ctypes.sizeof(soma_tensor_t) == 56


class soma_plan_t(ctypes.Structure):
    _fields_ = [
        ("norm_chunks", ctypes.c_int64),
        ("norm_segments", ctypes.c_int64),
        ("update_chunks", ctypes.c_int64),
        ("update_segments", ctypes.c_int64),
        ("norm_grid", ctypes.c_int32),
        ("norm_block", ctypes.c_int32),
        ("update_grid", ctypes.c_int32),
        ("update_block", ctypes.c_int32),
        ("trainable_numel", ctypes.c_int64),
        ("owned_numel", ctypes.c_int64),
        ("launches_per_step", ctypes.c_int32),
        ("single_launch_ctas", ctypes.c_int32),
    ]


class soma_segment_t(ctypes.Structure):
    _fields_ = [("grad", ctypes.c_void_p), ("chunk", ctypes.c_int64), ("len", ctypes.c_int32),
                ("head", ctypes.c_int32), ("nvec", ctypes.c_int32), ("group", ctypes.c_int32)]


assert ctypes.sizeof(soma_segment_t) == 32


class soma_device_group_t(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double), ("beta2", ctypes.c_double),
                ("eps", ctypes.c_double), ("weight_decay", ctypes.c_double), ("step", ctypes.c_int64),
                ("reserved", ctypes.c_int64 * 2)]


assert ctypes.sizeof(soma_device_group_t) == 64

_D = ctypes.c_double
_DP = ctypes.POINTER(ctypes.c_double)
_I32 = ctypes.c_int32
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64 = ctypes.c_int64
_I64P = ctypes.POINTER(ctypes.c_int64)

# name -> (restype, argtypes); every function the header declares.
SIGNATURES = {
    "soma_opt_create": (soma_status_t, [ctypes.POINTER(soma_opt_t), _I32]),
    "soma_opt_add_group": (soma_status_t, [soma_opt_t, _D, _D, _D, _D, _D, _I32P]),
    "soma_opt_set_lr": (soma_status_t, [soma_opt_t, _I32, _D]),
    "soma_opt_get_group": (soma_status_t, [soma_opt_t, _I32, _DP, _DP, _DP, _DP, _DP]),
    "soma_opt_set_group": (soma_status_t, [soma_opt_t, _I32, _D, _D, _D, _D, _D]),
    "soma_opt_set_group_divisor": (soma_status_t, [soma_opt_t, _I32, _D]),
    "soma_opt_get_group_divisor": (soma_status_t, [soma_opt_t, _I32, _DP]),
    "soma_opt_get_group_step": (soma_status_t, [soma_opt_t, _I32, _I64P]),
    "soma_opt_set_group_step": (soma_status_t, [soma_opt_t, _I32, _I64]),
    "soma_opt_step": (soma_status_t, [soma_opt_t, ctypes.POINTER(soma_tensor_t), _I64, _D, _D,
                                      ctypes.c_void_p]),
    "soma_opt_get_norm": (soma_status_t, [soma_opt_t, _DP, _DP, _I32P, ctypes.c_void_p]),
    "soma_opt_set_timing": (soma_status_t, [soma_opt_t, _I32]),
    "soma_opt_read_timing": (soma_status_t, [soma_opt_t, _DP, _DP, _I64P]),
    "soma_opt_get_plan": (soma_status_t, [soma_opt_t, ctypes.POINTER(soma_plan_t)]),
    "soma_opt_get_cache_stats": (soma_status_t, [soma_opt_t, _I64P, _I64P, _I32P]),
    "soma_opt_get_segments": (soma_status_t, [soma_opt_t, _I32, ctypes.POINTER(soma_segment_t), _I64, _I64P]),
    "soma_opt_set_tuning": (soma_status_t, [soma_opt_t, _I32, _I32, _I32, _I32]),
    "soma_opt_set_single_launch": (soma_status_t, [soma_opt_t, _I64]),
    "soma_status_string": (ctypes.c_char_p, [soma_status_t]),
    "soma_opt_last_error": (ctypes.c_char_p, [soma_opt_t]),
    "soma_abi_version": (_I32, []),
    "soma_opt_destroy": (None, [soma_opt_t]),
    "soma_opt_sumsq": (soma_status_t, [soma_opt_t, ctypes.POINTER(soma_tensor_t), _I64, _D, ctypes.c_void_p,
                                       ctypes.c_void_p]),
    "soma_opt_step_from_sumsq": (soma_status_t, [soma_opt_t, ctypes.POINTER(soma_tensor_t), _I64, _D, _D,
                                                 ctypes.c_void_p, _I32, ctypes.c_void_p]),
    "soma_opt_step_graph": (soma_status_t, [soma_opt_t, ctypes.POINTER(soma_tensor_t), _I64, _D, _D,
                                            ctypes.c_void_p]),
    "soma_opt_push_groups": (soma_status_t, [soma_opt_t, ctypes.c_void_p]),
    "soma_opt_pull_groups": (soma_status_t, [soma_opt_t, ctypes.c_void_p]),
    "soma_opt_device_groups": (soma_status_t, [soma_opt_t, ctypes.POINTER(ctypes.c_void_p)]),
    "soma_clip_norm_noalloc": (soma_status_t, [_I32, ctypes.POINTER(soma_tensor_t), _I64, _D, _D,
                                               ctypes.c_void_p, ctypes.c_void_p]),
}
SOMA_NOALLOC_SCRATCH_BYTES = 4 << 20

_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libsoma_opt.so (built by tensor_grad_clip_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m tensor_grad_clip_gb300.build` "
                           "(there is no fallback implementation)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
        globals()[name] = fn
    if lib.soma_abi_version() != SOMA_ABI_VERSION:
        raise RuntimeError(f"{path}: ABI version {lib.soma_abi_version()}, expected {SOMA_ABI_VERSION}")
    _lib = lib
    return lib
