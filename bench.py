#!/usr/bin/env python
"""Throughput of the fused normalize -> global-norm clip -> AdamW step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload hsdp_shard|action_expert|flat|many_small|tiny]
                    [--per-config LIST]

A step is one soma_opt_step over the whole tensor list (square-sum kernel +
fused update kernel).  Default workload: the 7B-parameter HSDP shard view
(32 blocks at width 4096, MLP 11008: 256 tensors, 6,476,136,448 fp32
parameters, bf16 gradients, a quarter of the tensors replicated, 2 groups,
divisor 128, max_norm 1), the largest list that fits one GPU.  Inputs are
synthetic and resident in HBM; p, m and v far exceed the 129 MB L2, so no
flush is needed between steps.

Prints one JSON line (rank 0): value = trainable parameter elements updated
per second over all ranks, plus the effective HBM bandwidth under the stated
accounting (28 B per element with bf16 gradients, 32 B with fp32), a
roofline entry for the update kernel, the oracle's CPU throughput, an
end-to-end number through the C ABI with host-resident gradients, and the SM
clocks seen during the timed region.  `per_config` holds the same
device-side measurement for the other lists (by default the action-expert,
flat, 20 000-tensor and tiny lists, the action-expert list with bf16 model
copies of fp32 master weights, and graph replays of the 20 000-tensor and
tiny lists), each set up after the previous list's buffers were freed, in
the same process.

--impl reference times the fp64 CPU oracle (the only other implementation of
this step available here) on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "param-elements updated/sec and effective HBM GB/s (% of GB300 peak) per step"
UNIT = "param-elements/s"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20
DEFAULT_WORKLOAD = "hsdp_shard"
# list[:mode]: master = bf16 model weights rewritten from fp32 master weights
# in the same pass; graph = one captured step (soma_opt_step_graph) replayed
DEFAULT_PER_CONFIG = "action_expert,flat,many_small,tiny,action_expert:master,many_small:graph,tiny:graph"
PER_CONFIG_MIN_S = 0.5   # timed seconds per per-config list, at least


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1, help="GPUs (one rank each under torchrun)")
    ap.add_argument("--steps", type=int, default=200, help="timed steps")
    ap.add_argument("--warmup", type=int, default=20, help="untimed steps first")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours",
                    help="reference: the fp64 CPU oracle on bounded samples of the same list")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    help="tiny, action_expert, many_small, hsdp_shard or flat")
    ap.add_argument("--per-config", default=None,
                    help="comma-separated further workloads measured after the main one, device side only "
                         f"(default with the default workload: {DEFAULT_PER_CONFIG}; 'none' = skip)")
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="steps per end-to-end window (gradients uploaded from pinned host memory)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end runs")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip timing the CPU oracle")
    ap.add_argument("--tuning", default="",
                    help="update_chunk,norm_chunk,update_ctas_per_sm,norm_ctas_per_sm (0 = default)")
    ap.add_argument("--single-launch", type=int, default=-1,
                    help="lists with at most this many trainable elements run as one cluster launch "
                         "(-1 = automatic, 0 = always the two kernels)")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step (soma_opt_step_graph) in a CUDA graph and time its replays")
    ap.add_argument("--master", action="store_true",
                    help="action-expert list with bf16 model weights rewritten from fp32 master weights")
    ap.add_argument("--blocks", type=int, default=0,
                    help="transformer blocks of the action-expert / shard-view lists (0 = full size)")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x, device):
    """Largest value of x over the ranks (x itself on one rank).  NCCL
    reduces device tensors, gloo host ones."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", d
    except Exception:
        return FALLBACK_HBM_GBS, "fallback", {}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period = period_ms
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=self.file, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(", ") for r in self.file.read().strip().splitlines() if r.strip()]
        self.file.close()
        os.unlink(self.file.name)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for nm, val in zip(names, r[5:9]):
                    if val.strip() == "Active":
                        reasons.add(nm)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def workload(name, blocks=0, master=False):
    import workloads as W
    if name not in W.FULL:
        raise SystemExit(f"unknown workload {name}; choose from {sorted(W.FULL)}")
    if name == "action_expert" and (blocks or master):
        return W.action_expert(n_blocks=blocks or 18, master=master)
    if blocks and name == "hsdp_shard":
        return W.hsdp_shard_view(n_blocks=blocks)
    return W.FULL[name]()


def describe(w):
    import workloads as W
    dts = sorted({t.grad_dtype for t in w.tensors if t.trainable})
    return {
        "workload": f"{w.name}: {len(w.tensors)} tensors, {w.trainable_numel:,} trainable fp32 params, "
                    f"{'/'.join(dts)} grads, {len(w.groups)} groups, divisor {w.grad_divisor:g}, "
                    f"max_norm {w.max_norm:g}",
        "tensors": len(w.tensors),
        "trainable_params": w.trainable_numel,
        "owned_params": w.owned_numel,
        "grad_dtype": "/".join(dts),
        "effective_bytes_per_step": w.effective_bytes_per_step(),
        "algorithmic_bytes_per_step": w.algorithmic_bytes_per_step(),
        "l2": "no flush: p, m, v and g exceed the 129 MB L2" if w.trainable_numel * 4 > 4 * L2_BYTES
        else "working set may fit in L2 (small workload)",
    }


def _code_only(text):
    """C++ source without comments and with whitespace collapsed (string
    literals kept): a comment edit leaves the hash of the code unchanged."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
        elif text.startswith("/*", i):
            i = text.find("*/", i + 2)
            i = n if i < 0 else i + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash():
    """Hash of the kernels' code and of the host code that cuts the lists
    into chunks (comments and layout ignored): the ncu traffic record applies
    only to the code and launch shapes it was measured on."""
    h = hashlib.sha256()
    for f in ("kernels.cu", "soma_kernels.h", "soma_opt.cpp"):
        with open(os.path.join(ROOT, "tensor_grad_clip_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def profile_json(key):
    """Committed ncu traffic record of the update kernel on workload `key`."""
    return os.path.join(ROOT, "profiles", f"update_kernel_{key}.json")


def ncu_traffic(key, workload_name):
    """DRAM bytes per update-kernel launch from the committed ncu summary,
    if it was taken on this workload and on the current kernel source."""
    try:
        with open(profile_json(key)) as f:
            d = json.load(f)
    except Exception:
        return None
    if d.get("kernel_sha") != kernel_source_hash() or d.get("workload") != workload_name:
        return None
    return d.get("dram_bytes_per_launch")


def cpu_baseline(w, budget_s=10.0):
    """The fp64 oracle (single thread, as it stands) on the first tensors of
    the workload, repeated until about `budget_s` seconds have passed."""
    import oracle
    import workloads as W
    from oracle import GroupState, OracleOptimizer
    oracle.lib()
    idx, n = [], 0
    for k, t in enumerate(w.tensors):
        if t.trainable and n < 8_500_000:
            idx.append(k)
            n += t.numel
    params = [W.draw_param(w, k, "cpu") for k in idx]
    grads = [W.draw_grad(w, k, 1, "cpu") for k in idx]
    orc = OracleOptimizer([p.double().numpy().reshape(-1) for p in params],
                          [(w.tensors[k].group, True, w.tensors[k].owned) for k in idx],
                          [GroupState(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                                      weight_decay=g.weight_decay) for g in w.groups])
    steps, t0 = 0, time.perf_counter()
    while True:
        orc.step(grads, w.grad_divisor, w.max_norm)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": n * steps / el, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{len(idx)} tensors ({n:,} params) of {w.name}, {steps} full oracle steps "
                      f"(norm + update) in {el:.1f} s, fp64, one thread"}


def cpu_baseline_all_cores(w, budget_s=10.0):
    """The same oracle functions on every host core: the step's two passes
    (square-sums, then the update) split into slices of at most 1 Mi
    elements and run on a thread pool (ctypes releases the GIL during each
    call); square-sums are added in list order on one thread, as in the
    oracle's own step."""
    import concurrent.futures as cf
    import math

    import numpy as np

    import oracle
    import workloads as W
    oracle.lib()
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    idx, n = [], 0
    for k, t in enumerate(w.tensors):
        if t.trainable and n < 17_000_000:
            idx.append(k)
            n += t.numel
    slices = []  # (p, g, m, v, group, owned) per slice, p/m/v fp64 views
    for k in idx:
        t = w.tensors[k]
        p = W.draw_param(w, k, "cpu").double().numpy().reshape(-1).copy()
        g = W.draw_grad(w, k, 1, "cpu").reshape(-1)
        m, v = np.zeros_like(p), np.zeros_like(p)
        for lo in range(0, t.numel, 1 << 20):
            hi = min(t.numel, lo + (1 << 20))
            slices.append((p[lo:hi], g[lo:hi], m[lo:hi], v[lo:hi], t.group, t.owned))
    steps = [0] * len(w.groups)

    def one_step(pool):
        sq = list(pool.map(lambda s: oracle.tensor_sqsum(s[1], w.grad_divisor) if s[5] else 0.0, slices))
        c = oracle.clip_coef(math.sqrt(sum(sq)), w.max_norm)
        for q in {s[4] for s in slices}:
            steps[q] += 1

        def upd(s):
            g = w.groups[s[4]]
            oracle.adamw_update(s[0], s[1], s[2], s[3], lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                                weight_decay=g.weight_decay, step=steps[s[4]], c=c, divisor=w.grad_divisor)
        list(pool.map(upd, slices))

    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        one_step(pool)  # warm-up
        count, t0 = 0, time.perf_counter()
        while True:
            one_step(pool)
            count += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    return {"value": n * count / el, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{len(idx)} tensors ({n:,} params) of {w.name} in {len(slices)} slices, {count} steps "
                      f"(square-sums, then update) in {el:.1f} s, fp64, {cores} threads"}


def run_reference(args):
    """The oracle as the reference arm: K timed steps after W warm-ups, each
    a bounded sample of the workload, sized to finish within minutes."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    import workloads as W
    from oracle import GroupState, OracleOptimizer
    w = workload(args.workload, args.blocks)
    oracle.lib()
    # calibrate: elements per second on one tensor, then size the per-step sample
    k0 = next(k for k, t in enumerate(w.tensors) if t.trainable)
    cal_p = W.draw_param(w, k0, "cpu")
    cal_g = W.draw_grad(w, k0, 1, "cpu")
    cal = OracleOptimizer([cal_p.double().numpy().reshape(-1)], [(w.tensors[k0].group, True, True)],
                          [GroupState(lr=g.lr) for g in w.groups])
    t0 = time.perf_counter()
    cal.step([cal_g], w.grad_divisor, w.max_norm)
    rate = cal_p.numel() / max(time.perf_counter() - t0, 1e-6)
    per_step = min(17_000_000, max(1, int(rate * 120.0 / max(1, args.steps + args.warmup))))
    idx, n = [], 0
    for k, t in enumerate(w.tensors):
        if t.trainable and (n == 0 or n + t.numel <= per_step):
            idx.append(k)
            n += t.numel
    params = [W.draw_param(w, k, "cpu") for k in idx]
    grads = [W.draw_grad(w, k, 1, "cpu") for k in idx]
    orc = OracleOptimizer([p.double().numpy().reshape(-1) for p in params],
                          [(w.tensors[k].group, True, w.tensors[k].owned) for k in idx],
                          [GroupState(lr=g.lr, beta1=g.beta1, beta2=g.beta2, eps=g.eps,
                                      weight_decay=g.weight_decay) for g in w.groups])
    for _ in range(args.warmup):
        orc.step(grads, w.grad_divisor, w.max_norm)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        orc.step(grads, w.grad_divisor, w.max_norm)
    el = time.perf_counter() - t0
    value = n * args.steps / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": describe(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{len(idx)} tensors ({n:,} params) of {w.name} per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def e2e_runs(args, w, fb, tl, owned, step_on, stream, device, barrier, world):
    """The step through the public API with the gradients arriving from
    pinned host memory every step, timed twice:

    - pipelined (the reported value): two device gradient buffers used in
      turn.  Step t+1's upload runs on a copy stream while step t's kernels
      run; each step waits only for its own upload, and an upload waits for
      the step that last read its buffer.  The handle keeps both lists
      prepared, so switching between them costs nothing on the host.
    - serial: one buffer; copy, step and norm read strictly in sequence.

    Each step's norm is read back (a device-to-host copy and a wait) before
    the next step is enqueued; only the next upload is already queued then.
    Each mode is timed over three windows and the median window reported."""
    import torch
    from tensor_grad_clip_gb300 import TensorList
    G = fb.G
    host_g = torch.empty(G.shape, dtype=G.dtype, pin_memory=True)
    host_g.copy_(G)
    G2 = G.clone()
    tl2 = TensorList(fb.p, [G2[fb.offsets[k]:fb.offsets[k] + t.numel] for k, t in enumerate(w.tensors)], fb.m,
                     fb.v, groups=[t.group for t in w.tensors], trainable=[t.trainable for t in w.tensors],
                     owned=owned, params_lowp=fb.plow)
    bufs = [(G, tl), (G2, tl2)]
    cs = torch.cuda.Stream(device)
    copied = [torch.cuda.Event() for _ in bufs]
    freed = [torch.cuda.Event() for _ in bufs]
    torch.cuda.synchronize()

    def upload(t):
        b = t % 2
        cs.wait_event(freed[b])  # the step that last read buffer b has finished
        with torch.cuda.stream(cs):
            bufs[b][0].copy_(host_g, non_blocking=True)
        copied[b].record(cs)

    def pipelined(n):
        cs.wait_stream(stream)
        upload(0)
        for t in range(n):
            b = t % 2
            stream.wait_event(copied[b])
            opt = step_on(bufs[b][1])
            freed[b].record(stream)
            if t + 1 < n:
                upload(t + 1)
            opt.get_norm(stream)

    upload_ms = []  # each upload of the serial mode, from events on the copy stream

    def serial(n):
        for _ in range(n):
            cs.wait_stream(stream)
            u0, u1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            u0.record(cs)
            upload(0)
            u1.record(cs)  # right behind the copy on the copy stream
            upload_ms.append((u0, u1))
            stream.wait_event(copied[0])
            opt = step_on(tl)
            freed[0].record(stream)
            opt.get_norm(stream)

    def timed(fn, n):
        fn(2)  # warm-up: both lists prepared
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        fn(n)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier()
        ms = max(e0.elapsed_time(e1), (time.perf_counter() - t0) * 1e3)
        return max_over_ranks(ms, device)

    # the host link on its own: one gradient upload, no kernels
    torch.cuda.synchronize()
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(cs)
    with torch.cuda.stream(cs):
        for _ in range(5):
            G2.copy_(host_g, non_blocking=True)
    l1.record(cs)
    torch.cuda.synchronize()
    link_gbs = 5 * G.numel() * G.element_size() / (l0.elapsed_time(l1) / 1e3) / 1e9
    G2.copy_(G)

    # Three timed windows of n steps each; the median window is reported (the
    # host link is shared, and one window can catch contention), all three listed.
    n = args.e2e_steps
    elems = w.trainable_numel * world
    p_all = [timed(pipelined, n) / n for _ in range(3)]
    s_all = [timed(serial, n) / n for _ in range(3)]
    p_ms, s_ms = statistics.median(p_all), statistics.median(s_all)
    torch.cuda.synchronize()
    up_ms = statistics.median(a.elapsed_time(b) for a, b in upload_ms[-n:])
    return {"value": elems / (p_ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": G.numel() * G.element_size(), "d2h_bytes_per_step": 48,
            "steps": n, "ms_per_step": p_ms, "windows_ms_per_step": p_all,
            "mode": "pipelined: two device gradient buffers, upload of step t+1 overlaps step t; "
                    "median of three windows",
            "h2d_link_gbs": link_gbs,
            # the upload alone at the link rate measured above: no step can be faster
            "link_floor_ms": G.numel() * G.element_size() / (link_gbs * 1e9) * 1e3,
            "frac_of_link_floor": (G.numel() * G.element_size() / (link_gbs * 1e9) * 1e3) / p_ms,
            "serial": {"value": elems / (s_ms / 1e3), "ms_per_step": s_ms, "windows_ms_per_step": s_all,
                       # the upload alone inside the serial loop, against the link test above
                       "upload_ms_median": up_ms, "upload_gbs": G.numel() * G.element_size() / (up_ms * 1e6)}}


def kernel_bytes(w):
    """Algorithmic bytes of one update launch (g 2/4 B, p, m, v read and
    written: 26/28 B per trainable element, +2 B with a 16-bit model copy) and
    of one square-sum launch (each owned gradient read once)."""
    gsz = lambda t: 4 if t.grad_dtype == "f32" else 2
    upd = sum(t.numel * (gsz(t) + 24 + (2 if t.param_lowp else 0)) for t in w.tensors if t.trainable)
    nrm = sum(t.numel * gsz(t) for t in w.tensors if t.trainable and t.owned)
    return upd, nrm


class Setup:
    """One list on the device: flat buffers, a handle with the list's groups,
    and the tensor list.  Under several ranks each rank holds its own shards
    of the sharded tensors (own seeds) and the replicated ones, and owns a
    replicated tensor only if it is that tensor's round-robin owner, so the
    global norm counts every entry once."""

    def __init__(self, args, w, local, rank, world):
        import workloads as W
        from tensor_grad_clip_gb300 import SomaOpt, TensorList
        from tensor_grad_clip_gb300.sharded import owned_flags
        self.w = w
        self.fb = W.FlatBuffers(w, torch_device(local), shard_rank=rank if world > 1 else 0)
        self.owned = ([t.owned for t in w.tensors] if world == 1
                      else owned_flags(len(w.tensors), rank, world, [t.owned for t in w.tensors]))
        self.opt = SomaOpt(local)
        for q in w.groups:
            self.opt.add_group(lr=q.lr, betas=(q.beta1, q.beta2), eps=q.eps, weight_decay=q.weight_decay)
        if args.tuning:
            self.opt.set_tuning(*(int(x) for x in args.tuning.split(",")))
        if args.single_launch != -1:
            self.opt.set_single_launch(args.single_launch)
        fb = self.fb
        self.tl = TensorList(fb.p, fb.g, fb.m, fb.v, groups=[t.group for t in w.tensors],
                             trainable=[t.trainable for t in w.tensors], owned=self.owned, params_lowp=fb.plow)

    def close(self):
        import torch
        self.opt.close()
        del self.fb, self.tl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def torch_device(local):
    import torch
    return torch.device("cuda", local)


def measure(args, S, stream, world, steps, warmup, graph_mode, timing_steps):
    """Warm-up steps, then `steps` timed steps between CUDA events on the
    step's stream (a barrier and a device synchronize on both sides, the
    maximum over ranks), with the SM clocks sampled meanwhile; then a pass
    with the handle's kernel timing on for per-kernel durations."""
    import torch
    import torch.distributed as dist
    w, opt, tl = S.w, S.opt, S.tl
    device = stream.device
    sharded_step = None
    if world > 1:
        # one float64 per rank per step (the owned square-sums) for the global norm
        from tensor_grad_clip_gb300.sharded import ShardedStep
        sharded_step = ShardedStep(opt)

    def step_on(lst):
        if sharded_step is not None:
            sharded_step(lst, w.grad_divisor, w.max_norm)
        else:
            opt.step(lst, w.grad_divisor, w.max_norm, stream)
        return opt

    def barrier():
        if world > 1:
            dist.barrier()

    def set_lrs(t):
        for q, lr in enumerate(w.group_lrs(t)):
            opt.set_lr(q, lr)

    torch.cuda.synchronize()
    graph = None
    if graph_mode:
        # one step captured on a side stream; replays read lr and step counts
        # from the library's device table
        opt.push_groups(stream)
        opt.step_graph(tl, w.grad_divisor, w.max_norm, stream)
        side = torch.cuda.Stream(device)
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(graph, stream=side):
                opt.step_graph(tl, w.grad_divisor, w.max_norm, side)
        torch.cuda.synchronize()
        for i in range(warmup):
            graph.replay()
    else:
        for i in range(warmup):
            set_lrs(i % w.steps + 1)
            step_on(tl)
    torch.cuda.synchronize()
    plan = opt.plan()

    sampler = ClockSampler(device.index)
    sampler.start()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        if graph is not None:
            graph.replay()
            continue
        if w.lr_at is not None:
            set_lrs(i % w.steps + 1)
        step_on(tl)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clocks = sampler.stop()
    elapsed_ms = e0.elapsed_time(e1)
    # Per-step distribution: a separate pass with an event after every step
    # (events between steps keep a step's square-sum kernel from starting
    # under the previous update kernel's tail, so this pass is not the
    # headline number either).
    per_step = None
    if graph is None and timing_steps > 0:
        n_ps = max(1, min(steps, 50))
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_ps + 1)]
        evs[0].record(stream)
        for i in range(n_ps):
            if w.lr_at is not None:
                set_lrs(i % w.steps + 1)
            step_on(tl)
            evs[i + 1].record(stream)
        torch.cuda.synchronize()
        ts = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(n_ps))
        per_step = {"steps": n_ps, "median_ms": statistics.median(ts), "min_ms": ts[0], "max_ms": ts[-1]}
    # Per-kernel durations for the roofline: a second pass over the same
    # steps with CUDA events recorded between the two kernels (an event there
    # also stops the update kernel from overlapping the square-sum's tail, and
    # a list small enough for the single-launch step runs this pass as the two
    # kernels, so this pass is not the one the headline number comes from).
    norm_ms = upd_ms = 0.0
    nsteps = 0
    if graph is None:
        opt.set_timing(True)
        opt.read_timing()
        for i in range(min(steps, timing_steps)):
            step_on(tl)
        torch.cuda.synchronize()
        norm_ms, upd_ms, nsteps = opt.read_timing()
        opt.set_timing(False)
    # The square-sum kernel on its own, launched back to back (soma_opt_sumsq
    # runs the step's first kernel and stores the square-sum): events around
    # a single launch also time the gap before it starts, which is a large
    # part of a 0.1 ms launch.
    chained_ms = None
    if graph is None and world == 1 and timing_steps > 0:
        out = torch.zeros(1, dtype=torch.float64, device=device)
        opt.sumsq(tl, w.grad_divisor, out, stream)
        n_chain = max(5, min(steps, timing_steps))
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(n_chain):
            opt.sumsq(tl, w.grad_divisor, out, stream)
        c1.record(stream)
        torch.cuda.synchronize()
        chained_ms = c0.elapsed_time(c1) / n_chain
        step_on(tl)  # leave the handle's last result a full step's
    elapsed_ms = max_over_ranks(elapsed_ms, device)
    norm, coef, nonfinite = opt.get_norm(stream)
    if graph is not None:  # no per-kernel events inside a graph: attribute the whole step
        upd_ms, norm_ms, nsteps = elapsed_ms, 0.0, steps
        del graph
    return {"elapsed_ms": elapsed_ms, "steps": steps, "plan": plan, "clocks": clocks, "norm_ms": norm_ms,
            "upd_ms": upd_ms, "timing_steps": nsteps, "norm_chained_ms": chained_ms, "per_step": per_step,
            "norm": norm, "coef": coef,
            "nonfinite": nonfinite, "step_on": step_on, "barrier": barrier}


def summarize(w, r, world, hbm_peak):
    """Throughput and bandwidth figures of one measured list."""
    ms = r["elapsed_ms"] / r["steps"]
    eff = w.effective_bytes_per_step() / (ms / 1e3) / 1e9
    alg = w.algorithmic_bytes_per_step() / (ms / 1e3) / 1e9
    upd_bytes, norm_bytes = kernel_bytes(w)
    n = max(r["timing_steps"], 1)
    upd_ms, norm_ms = r["upd_ms"] / n, r["norm_ms"] / n
    return {
        "ms_per_step": ms, "steps": r["steps"], "per_step_ms": r["per_step"],
        "value": w.trainable_numel * world / (ms / 1e3),
        "effective_hbm_gbs": eff * world, "effective_hbm_frac_of_peak": eff / hbm_peak,
        "effective_hbm_frac_of_8tbs": eff / 8000.0,
        "algorithmic_hbm_gbs": alg * world, "algorithmic_hbm_frac_of_8tbs": alg / 8000.0,
        "update_kernel_ms": upd_ms, "norm_kernel_ms": norm_ms,
        "update_kernel_gbs": upd_bytes / (upd_ms / 1e3) / 1e9 if upd_ms > 0 else None,
        "norm_kernel_gbs": norm_bytes / (norm_ms / 1e3) / 1e9 if norm_ms > 0 and world == 1 else None,
        "norm_kernel_chained_ms": r["norm_chained_ms"],
        "norm_kernel_chained_gbs": norm_bytes / (r["norm_chained_ms"] / 1e3) / 1e9 if r["norm_chained_ms"] else None,
        "launches_per_step": r["plan"]["launches_per_step"],
        "clocks": r["clocks"], "last_norm": r["norm"], "last_clip_coef": r["coef"], "nonfinite": r["nonfinite"],
    }


def run_ours(args):
    import torch
    import torch.distributed as dist
    world, rank, local = dist_env()
    if world > 1:
        # one rank per GPU over NCCL; ranks that share a GPU (fewer GPUs than
        # ranks: NCCL refuses two ranks on one device) exchange over gloo
        backend = "nccl" if torch.cuda.device_count() >= world else "gloo"
        dist.init_process_group(backend=backend, init_method="env://")
        local = local % torch.cuda.device_count()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import tensor_grad_clip_gb300
    tensor_grad_clip_gb300.load()
    hbm_peak, peak_kind, _ = peaks()
    stream = torch.cuda.current_stream(device)

    w = workload(args.workload, args.blocks, args.master)
    S = Setup(args, w, local, rank, world)
    r = measure(args, S, stream, world, args.steps, args.warmup, args.graph, 300)
    head = summarize(w, r, world, hbm_peak)
    plan = r["plan"]

    # dominant kernel: the fused update (26 B/elem bf16 grads, 28 B/elem fp32)
    upd_bytes, norm_bytes = kernel_bytes(w)
    upd_avg_ms, norm_avg_ms = head["update_kernel_ms"], head["norm_kernel_ms"]
    achieved = upd_bytes / (upd_avg_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "kernel": "update_kernel", "achieved": achieved, "peak": hbm_peak,
                "unit": "GB/s", "frac": achieved / hbm_peak, "peak_kind": f"{peak_kind} copy bandwidth",
                "traffic": ncu_traffic(args.workload, w.name) if not (args.blocks or args.master) else None,
                "algorithmic_bytes_per_launch": upd_bytes, "avg_launch_ms": upd_avg_ms,
                "norm_kernel": {"achieved": head["norm_kernel_gbs"], "avg_launch_ms": norm_avg_ms,
                                "algorithmic_bytes_per_launch": norm_bytes,
                                "note": "events around each launch in the kernel-timing pass (they also time the "
                                        "gap before the launch starts); chained: the same kernel launched back to "
                                        "back through soma_opt_sumsq",
                                "chained_launch_ms": head["norm_kernel_chained_ms"],
                                "achieved_chained": head["norm_kernel_chained_gbs"]}}
    if world > 1:
        roofline["norm_kernel"]["note"] = ("several ranks: the square-sum runs in soma_opt_sumsq before the "
                                           "all-gather; the events time the finish kernel")

    e2e = None
    if not args.no_e2e and not args.graph:
        # End to end through the C ABI: every step copies that step's gradients
        # from pinned host memory into a device gradient buffer, runs the step
        # and reads the norm back to the host.
        e2e = e2e_runs(args, w, S.fb, S.tl, S.owned, r["step_on"], stream, device, r["barrier"], world)
    S.close()
    del S

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)
        cpu["all_cores"] = cpu_baseline_all_cores(w)

    # The other lists, device side only, each on a fresh handle after the
    # previous list's buffers were freed.  Each is timed for at least
    # PER_CONFIG_MIN_S seconds (and at least --steps steps).
    per = {}
    names = args.per_config
    if names is None:
        names = DEFAULT_PER_CONFIG if (args.workload == DEFAULT_WORKLOAD and not args.blocks) else "none"
    for name in [x for x in names.split(",") if x and x != "none" and x != args.workload]:
        base, _, mode = name.partition(":")
        if mode not in ("", "master", "graph"):
            raise SystemExit(f"unknown mode {mode!r} in --per-config {name}")
        graph_k = mode == "graph" and world == 1  # (graph-capturable steps have no multi-rank form)
        wk = workload(base, master=mode == "master")
        Sk = Setup(args, wk, local, rank, world)
        probe = measure(args, Sk, stream, world, max(3, args.warmup), max(3, args.warmup), graph_k, 0)
        est_ms = probe["elapsed_ms"] / probe["steps"]
        k = max(args.steps, min(20000, int(PER_CONFIG_MIN_S * 1e3 / max(est_ms, 1e-3)) + 1))
        rk = measure(args, Sk, stream, world, k, 0, graph_k, min(k, 300))
        ent = summarize(wk, rk, world, hbm_peak)
        if graph_k:  # a graph replay has no per-kernel events: drop the kernel fields
            for f in ("update_kernel_ms", "norm_kernel_ms", "update_kernel_gbs", "norm_kernel_gbs"):
                ent[f] = None
        ent["mode"] = ("CUDA-graph replay of one step" if graph_k else "soma_opt_step per step") + \
            (", bf16 model copies of fp32 master weights" if mode == "master" else "")
        per[name] = {"config": describe(wk)} | ent
        Sk.close()
        del Sk

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "per_step_ms": head["per_step_ms"],
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": describe(w) | {"parallelism": f"shard group x{world}: one all-gather of 8 B per rank per step "
                                                    f"({dist.get_backend()}, {torch.cuda.device_count()} GPUs)"
                                     if world > 1 else "single GPU",
                                     "mode": "CUDA-graph replay of one step" if args.graph
                                     else "soma_opt_step per step", "plan": plan},
            "effective_hbm_gbs": head["effective_hbm_gbs"],
            "effective_hbm_frac_of_peak": head["effective_hbm_frac_of_peak"],
            "effective_hbm_frac_of_8tbs": head["effective_hbm_frac_of_8tbs"],
            "algorithmic_hbm_gbs": head["algorithmic_hbm_gbs"],
            "algorithmic_hbm_frac_of_8tbs": head["algorithmic_hbm_frac_of_8tbs"],
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            # multi-rank steps add the finish kernel (rank-ordered sum of the ranks' square-sums)
            "gpu_launches": (plan["launches_per_step"] + (1 if world > 1 else 0)) * args.steps,
            "clocks": head["clocks"],
            "last_norm": head["last_norm"], "last_clip_coef": head["last_clip_coef"],
            "nonfinite": head["nonfinite"],
            "per_config": per or None,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
