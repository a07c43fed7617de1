"""Host-side behaviour of the C ABI: the library loads, exports every function
include/soma_opt.h declares, and rejects bad arguments with a status and no
state change.  Every list passed here is invalid in at least one respect (or
the process has no GPU), so no kernel is ever launched on fake pointers."""
import ctypes
import os
import re

import pytest
import torch

from tensor_grad_clip_gb300 import SomaError, SomaOpt, _abi, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "soma_opt.h")


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return _abi.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(soma_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "soma_opt_step" in names and len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_abi.SIGNATURES), "binding and header disagree"
    assert lib.soma_abi_version() == _abi.SOMA_ABI_VERSION


def test_struct_layout():
    assert ctypes.sizeof(_abi.soma_plan_t) == 72 and _abi.soma_plan_t.single_launch_ctas.offset == 68
    assert ctypes.sizeof(_abi.soma_tensor_t) == 56
    assert _abi.soma_tensor_t.param_lowp.offset == 32
    assert _abi.soma_tensor_t.numel.offset == 40 and _abi.soma_tensor_t.group.offset == 48
    assert _abi.soma_tensor_t.lowp_dtype.offset == 55


def test_status_strings(lib):
    for s in range(9):
        assert _abi.soma_status_string(s)
    assert b"unknown" in _abi.soma_status_string(99)


def test_create_rejects_bad_arguments(lib):
    assert _abi.soma_opt_create(None, 0) == _abi.SOMA_ERR_INVALID_ARG
    h = _abi.soma_opt_t(12345)
    assert _abi.soma_opt_create(ctypes.byref(h), -1) == _abi.SOMA_ERR_INVALID_ARG
    assert h.value is None  # *out cleared on failure
    assert b"device" in _abi.soma_opt_last_error(None)


def test_groups_and_step_counts():
    opt = SomaOpt(0)  # makes no CUDA call
    g0 = opt.add_group(lr=1e-3, weight_decay=0.01)
    g1 = opt.add_group(lr=5e-6, betas=(0.8, 0.99), eps=1e-6)
    assert (g0, g1) == (0, 1)
    assert opt.get_group(1) == dict(lr=5e-6, betas=(0.8, 0.99), eps=1e-6, weight_decay=0.0)
    opt.set_lr(0, 2e-3)
    assert opt.get_group(0)["lr"] == 2e-3
    assert opt.get_group_step(0) == 0
    opt.set_group_step(1, 41)
    assert opt.get_group_step(1) == 41
    for bad in (dict(lr=-1.0), dict(lr=float("nan")), dict(lr=1e-3, betas=(1.0, 0.9)),
                dict(lr=1e-3, betas=(0.9, -0.1)), dict(lr=1e-3, eps=0.0), dict(lr=1e-3, weight_decay=-0.5),
                dict(lr=1e-3, weight_decay=float("inf"))):
        with pytest.raises(SomaError) as e:
            opt.add_group(**bad)
        assert e.value.status == _abi.SOMA_ERR_INVALID_ARG
    with pytest.raises(SomaError) as e:
        opt.set_lr(7, 1.0)
    assert e.value.status == _abi.SOMA_ERR_BAD_GROUP
    with pytest.raises(SomaError):
        opt.set_group_step(0, -1)
    opt.close()


def test_group_limit():
    opt = SomaOpt(0)
    for _ in range(_abi.SOMA_MAX_GROUPS):
        opt.add_group(lr=1e-3)
    with pytest.raises(SomaError) as e:
        opt.add_group(lr=1e-3)
    assert e.value.status == _abi.SOMA_ERR_LIMIT
    opt.close()


def _entry(**kw):
    e = _abi.soma_tensor_t()
    e.param, e.grad, e.exp_avg, e.exp_avg_sq = 0x10000, 0x20000, 0x30000, 0x40000
    e.param_lowp = 0
    e.numel, e.group, e.grad_dtype, e.trainable, e.owned, e.lowp_dtype = 8, 0, 0, 1, 1, 0
    for k, v in kw.items():
        setattr(e, k, v)
    return e


def _step(opt, entries, divisor=1.0, max_norm=1.0, n=None):
    arr = (_abi.soma_tensor_t * max(1, len(entries)))(*entries)
    return _abi.soma_opt_step(opt.handle, arr, len(entries) if n is None else n, divisor, max_norm, None)


@pytest.mark.parametrize("entry,status", [
    (dict(lowp_dtype=1), _abi.SOMA_ERR_DTYPE),                      # dtype without a copy
    (dict(param_lowp=0x50000), _abi.SOMA_ERR_DTYPE),                # copy without a dtype
    (dict(param_lowp=0x50000, lowp_dtype=3), _abi.SOMA_ERR_DTYPE),
    (dict(param_lowp=0x50001, lowp_dtype=1), _abi.SOMA_ERR_ALIGNMENT),
    (dict(grad=0x20001, grad_dtype=2), _abi.SOMA_ERR_ALIGNMENT),    # fp16 grad on an odd address
    (dict(trainable=2), _abi.SOMA_ERR_INVALID_ARG),
    (dict(owned=3), _abi.SOMA_ERR_INVALID_ARG),
    (dict(numel=-1), _abi.SOMA_ERR_INVALID_ARG),
    (dict(group=1), _abi.SOMA_ERR_BAD_GROUP),
    (dict(group=-1), _abi.SOMA_ERR_BAD_GROUP),
    (dict(grad_dtype=7), _abi.SOMA_ERR_DTYPE),
    (dict(param=0), _abi.SOMA_ERR_INVALID_ARG),
    (dict(grad=0), _abi.SOMA_ERR_INVALID_ARG),
    (dict(exp_avg_sq=0), _abi.SOMA_ERR_INVALID_ARG),
    (dict(param=0x10002), _abi.SOMA_ERR_ALIGNMENT),
    (dict(grad=0x20002), _abi.SOMA_ERR_ALIGNMENT),          # fp32 grad on a 2-byte boundary
    (dict(grad=0x20001, grad_dtype=1), _abi.SOMA_ERR_ALIGNMENT),  # bf16 grad on an odd address
])
def test_step_rejects_bad_entries_without_state_change(entry, status):
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    good = _entry()
    bad = _entry(**entry)
    assert _step(opt, [good, bad]) == status
    assert opt.get_group_step(0) == 0
    assert f"list[1]".encode() in _abi.soma_opt_last_error(opt.handle)
    opt.close()


@pytest.mark.parametrize("divisor,max_norm", [(0.0, 1.0), (-2.0, 1.0), (float("nan"), 1.0),
                                              (float("inf"), 1.0), (1.0, 0.0), (1.0, -1.0),
                                              (1.0, float("nan"))])
def test_step_rejects_bad_scalars(divisor, max_norm):
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    assert _step(opt, [_entry(group=5)], divisor, max_norm) == _abi.SOMA_ERR_INVALID_ARG
    assert opt.get_group_step(0) == 0
    opt.close()


def test_step_rejects_null_list_and_negative_count():
    opt = SomaOpt(0)
    assert _abi.soma_opt_step(opt.handle, None, 3, 1.0, 1.0, None) == _abi.SOMA_ERR_INVALID_ARG
    assert _step(opt, [_entry()], n=-1) == _abi.SOMA_ERR_INVALID_ARG
    opt.close()


def test_empty_entry_may_have_null_buffers_and_a_copy_dtype():
    # an empty torch tensor has no storage: data_ptr() is 0 for every buffer
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    empty = _entry(param=0, grad=0, exp_avg=0, exp_avg_sq=0, numel=0, lowp_dtype=1)
    bad = _entry(grad_dtype=9)
    # the empty entry passes validation; the second entry is what fails
    assert _step(opt, [empty, bad]) == _abi.SOMA_ERR_DTYPE
    assert b"list[1]" in _abi.soma_opt_last_error(opt.handle)
    # a copy dtype without a copy stays an error for a non-empty entry
    assert _step(opt, [_entry(lowp_dtype=1), bad]) == _abi.SOMA_ERR_DTYPE
    assert b"list[0]" in _abi.soma_opt_last_error(opt.handle)
    opt.close()


def test_frozen_entries_may_have_null_buffers_and_any_group():
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    frozen = _entry(param=0, grad=0, exp_avg=0, exp_avg_sq=0, group=99, grad_dtype=9, trainable=0)
    bad = _entry(grad_dtype=9)
    # the frozen entry passes validation; the second entry is what fails
    assert _step(opt, [frozen, bad]) == _abi.SOMA_ERR_DTYPE
    opt.close()


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_step_without_a_gpu_reports_cuda_error():
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    assert _step(opt, [_entry()]) == _abi.SOMA_ERR_CUDA
    assert b"CUDA" in _abi.soma_opt_last_error(opt.handle)
    assert opt.get_group_step(0) == 0
    with pytest.raises(SomaError) as e:
        opt.get_norm(stream=0)
    assert e.value.status == _abi.SOMA_ERR_STATE
    opt.close()


def test_use_after_destroy_and_null_handle():
    opt = SomaOpt(0)
    h = opt.handle.value
    opt.close()
    dead = _abi.soma_opt_t(h)
    i = ctypes.c_int32()
    assert _abi.soma_opt_add_group(dead, 1e-3, 0.9, 0.999, 1e-8, 0.0, ctypes.byref(i)) == _abi.SOMA_ERR_STATE
    assert _abi.soma_opt_step(dead, None, 0, 1.0, 1.0, None) == _abi.SOMA_ERR_STATE
    assert _abi.soma_opt_set_timing(None, 1) == _abi.SOMA_ERR_STATE
    assert _abi.soma_opt_last_error(dead) == b"invalid handle"
    _abi.soma_opt_destroy(dead)  # ignored
    _abi.soma_opt_destroy(None)


def test_tuning_and_timing_arguments():
    opt = SomaOpt(0)
    opt.set_tuning(update_chunk=4096, norm_chunk=8192, update_ctas_per_sm=2, norm_ctas_per_sm=4)
    for bad in (dict(update_chunk=10), dict(norm_chunk=1 << 27), dict(update_ctas_per_sm=-1),
                dict(norm_ctas_per_sm=65)):
        with pytest.raises(SomaError):
            opt.set_tuning(**bad)
    assert _abi.soma_opt_set_timing(opt.handle, 2) == _abi.SOMA_ERR_INVALID_ARG
    opt.set_timing(True)
    assert opt.read_timing() == (0.0, 0.0, 0)
    for ok in (-1, 0, 1, 1 << 40):
        opt.set_single_launch(ok)
    assert _abi.soma_opt_set_single_launch(opt.handle, -2) == _abi.SOMA_ERR_INVALID_ARG
    opt.close()
    assert _abi.soma_opt_set_single_launch(opt.handle, 0) == _abi.SOMA_ERR_STATE


def test_tensor_list_marshalling_checks():
    from tensor_grad_clip_gb300 import TensorList
    p = torch.zeros(4, 4)
    g = torch.zeros(4, 4, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        TensorList([p.t()], [g], [p], [p], groups=[0])  # non-contiguous
    with pytest.raises(TypeError):
        TensorList([p], [g.double()], [p], [p], groups=[0])
    with pytest.raises(TypeError):
        TensorList([p], [g], [p], [p], groups=[0], params_lowp=[p])  # fp32 is not a 16-bit copy
    tl16 = TensorList([p], [g.half()], [p], [p], groups=[0], params_lowp=[g])
    assert tl16.array[0].grad_dtype == _abi.SOMA_DTYPE_F16 and tl16.array[0].lowp_dtype == _abi.SOMA_DTYPE_BF16
    with pytest.raises(ValueError):
        TensorList([p], [torch.zeros(3)], [p], [p], groups=[0])
    tl = TensorList([p, p], [g, None], [p, None], [p, None], groups=[0, 0], trainable=[True, False])
    assert tl.array[0].grad_dtype == _abi.SOMA_DTYPE_BF16 and tl.array[1].trainable == 0
    assert tl.array[1].grad is None and tl.array[0].numel == 16


def test_multirank_entry_points_reject_bad_arguments():
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    arr = (_abi.soma_tensor_t * 1)(_entry())
    h = opt.handle
    assert _abi.soma_opt_sumsq(h, arr, 1, 1.0, None, None) == _abi.SOMA_ERR_INVALID_ARG
    assert _abi.soma_opt_sumsq(h, arr, 1, 1.0, 0x1004, None) == _abi.SOMA_ERR_INVALID_ARG  # not 8-byte aligned
    assert _abi.soma_opt_sumsq(h, arr, 1, 0.0, 0x1000, None) == _abi.SOMA_ERR_INVALID_ARG  # divisor
    f = _abi.soma_opt_step_from_sumsq
    assert f(h, arr, 1, 1.0, 1.0, None, 1, None) == _abi.SOMA_ERR_INVALID_ARG
    assert f(h, arr, 1, 1.0, 1.0, 0x1000, 0, None) == _abi.SOMA_ERR_INVALID_ARG
    assert f(h, arr, 1, 1.0, 1.0, 0x1000, _abi.SOMA_MAX_RANKS + 1, None) == _abi.SOMA_ERR_INVALID_ARG
    bad = (_abi.soma_tensor_t * 1)(_entry(group=4))
    assert f(h, bad, 1, 1.0, 1.0, 0x1000, 2, None) == _abi.SOMA_ERR_BAD_GROUP
    assert opt.get_group_step(0) == 0
    opt.close()


def test_owned_flags_count_every_entry_once():
    from tensor_grad_clip_gb300.sharded import owned_flags
    sharded = [True, False, False, True, False]
    world = 3
    flags = [owned_flags(5, r, world, sharded) for r in range(world)]
    for k in range(5):
        owners = [r for r in range(world) if flags[r][k]]
        assert owners == (list(range(world)) if sharded[k] else [k % world])
    with pytest.raises(ValueError):
        owned_flags(5, 3, 3, sharded)


def test_group_divisor_arguments():
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    assert opt.get_group_divisor(0) == 0.0
    opt.set_group_divisor(0, 3.0)
    assert opt.get_group_divisor(0) == 3.0
    for bad in (-1.0, float("nan"), float("inf")):
        with pytest.raises(SomaError) as e:
            opt.set_group_divisor(0, bad)
        assert e.value.status == _abi.SOMA_ERR_INVALID_ARG
    with pytest.raises(SomaError) as e:
        opt.set_group_divisor(1, 2.0)
    assert e.value.status == _abi.SOMA_ERR_BAD_GROUP
    opt.set_group_divisor(0, 0.0)  # back to the step's divisor
    assert opt.get_group_divisor(0) == 0.0
    opt.close()


def test_header_constants_match_the_binding():
    text = open(HEADER).read()
    defs = {k: v.strip() for k, v in re.findall(r"#define\s+(SOMA_\w+)[ \t]+([^/\n]+)", text)}
    for name, value in defs.items():
        if name.endswith("_H") or not hasattr(_abi, name):
            continue
        assert eval(value.replace("u", "")) == getattr(_abi, name), name
    assert "SOMA_PLAN_CACHE" in defs and "SOMA_ABI_VERSION" in defs


def test_cache_stats_of_a_fresh_handle_and_after_a_failed_step():
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    assert opt.cache_stats() == {"builds": 0, "reuses": 0, "entries": 0}
    assert _step(opt, [_entry(grad_dtype=9)]) == _abi.SOMA_ERR_DTYPE
    assert opt.cache_stats() == {"builds": 0, "reuses": 0, "entries": 0}
    assert _abi.soma_opt_get_cache_stats(opt.handle, None, None, None) == _abi.SOMA_OK
    opt.close()


def test_state_dict_round_trip():
    # The library's whole state (group hyperparameters, divisors, step
    # counts) survives a checkpoint into a fresh handle; no GPU needed.
    import json
    a = SomaOpt(0)
    a.add_group(lr=1e-3, betas=(0.8, 0.99), eps=1e-6, weight_decay=0.1)
    a.add_group(lr=5e-6)
    a.set_group_divisor(1, 3.0)
    a.set_group_step(0, 1234)
    a.set_group_step(1, 7)
    state = json.loads(json.dumps(a.state_dict()))  # as a checkpoint file would hold it
    b = SomaOpt(0)
    b.load_state_dict(state)
    assert b.num_groups == 2
    assert b.state_dict() == state
    assert b.get_group_step(0) == 1234 and b.get_group_divisor(1) == 3.0
    c = SomaOpt(0)
    c.add_group(lr=1.0)
    with pytest.raises(ValueError):
        c.load_state_dict(state)
    for o in (a, b, c):
        o.close()


def _noalloc_list(numels, dtype=_abi.SOMA_DTYPE_F32):
    """Entries at distinct fake 256-byte-aligned addresses (never dereferenced:
    the size check runs before any CUDA call)."""
    arr = (_abi.soma_tensor_t * len(numels))()
    addr = 1 << 40
    for k, n in enumerate(numels):
        e = arr[k]
        e.param = e.exp_avg = e.exp_avg_sq = e.grad = addr
        e.numel, e.group, e.grad_dtype, e.trainable, e.owned = n, 0, dtype, 1, 1
        addr += (n * 4 + 255) // 256 * 256
    return ctypes.cast(arr, ctypes.POINTER(_abi.soma_tensor_t)), arr


@pytest.mark.skipif(torch.cuda.is_available(), reason="a list that fits would be launched on fake pointers")
def test_noalloc_capacity_matches_the_header():
    # The header promises at least 26 000 owned entries of any sizes (one
    # 2^40-element entry forces the most chunks a list can have, 32 768 full
    # ones, plus the tiny entries' own segments) and about 65 000 tiny ones.
    # A list that fits passes the size check and then fails on this machine's
    # missing GPU (SOMA_ERR_CUDA); one that does not fit gets SOMA_ERR_LIMIT.
    out = 1 << 41  # 8-byte aligned, never written: no device here
    def status(numels):
        ptr, keep = _noalloc_list(numels)
        return _abi.soma_clip_norm_noalloc(0, ptr, len(numels), 1.0, 1.0, out, None)
    assert status([1 << 40] + [1] * 25_999) == _abi.SOMA_ERR_CUDA
    assert status([1 << 40] + [1] * 26_599) == _abi.SOMA_ERR_LIMIT
    assert status([1] * 65_000) == _abi.SOMA_ERR_CUDA
    assert status([1] * 65_400) == _abi.SOMA_ERR_LIMIT
    assert status([1 << 20] * 26_000) == _abi.SOMA_ERR_CUDA  # 26 000 entries of 1 Mi elements each


def test_get_segments_arguments_and_state():
    # the segment tables exist only once a step has built them
    opt = SomaOpt(0)
    opt.add_group(lr=1e-3)
    n = ctypes.c_int64(-1)
    assert _abi.soma_opt_get_segments(opt.handle, 0, None, 0, ctypes.byref(n)) == _abi.SOMA_ERR_STATE
    with pytest.raises(SomaError) as e:
        opt.segments("update")
    assert e.value.status == _abi.SOMA_ERR_STATE
    assert _abi.soma_opt_get_segments(opt.handle, 2, None, 0, ctypes.byref(n)) == _abi.SOMA_ERR_INVALID_ARG
    assert _abi.soma_opt_get_segments(opt.handle, 0, None, 0, None) == _abi.SOMA_ERR_INVALID_ARG
    assert _abi.soma_opt_get_segments(opt.handle, 0, None, 5, ctypes.byref(n)) == _abi.SOMA_ERR_INVALID_ARG
    assert _abi.soma_opt_get_segments(opt.handle, 0, None, -1, ctypes.byref(n)) == _abi.SOMA_ERR_INVALID_ARG
    assert n.value == -1  # nothing written on failure
    opt.close()
    assert _abi.soma_opt_get_segments(None, 0, None, 0, ctypes.byref(n)) == _abi.SOMA_ERR_STATE
