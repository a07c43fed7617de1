"""Flat device layout of a workload's buffers, as a training framework holds
them: one buffer per kind (weights, gradients, first and second moments),
each tensor a view starting on a 256-byte boundary.  The gaps between views
are filled with a sentinel pattern so that a test can check nothing outside a
tensor was written.  Values are drawn on the device (see generate.py)."""
from __future__ import annotations

import torch

from .configs import Workload
from .generate import draw_grad, draw_param, torch_dtype

SENTINEL_F32 = 0x7FC0DEAD   # NaN payloads no arithmetic produces
SENTINEL_BF16 = 0x7FAD
ALIGN = 64                  # elements: 256 B of fp32, 128 B of bf16


def bytes_per_slot(grad_dtype, lowp: bool) -> int:
    """Device bytes per element slot of the flat buffers: fp32 weight, first
    and second moment, the gradient, and a 16-bit model copy if any."""
    return 12 + torch.empty((), dtype=grad_dtype).element_size() + (2 if lowp else 0)


def check_device_memory(w: Workload, device, buffer_bytes: int):
    """Refuses a list that does not fit before anything is allocated: the
    flat buffers plus one tensor's draw (its fp32 values and their cast, 8
    bytes per element of the largest tensor) against the free device memory,
    counting what torch's caching allocator holds unused (it hands that out
    again, or releases it, before an allocation fails)."""
    need = buffer_bytes + 8 * max((t.numel for t in w.tensors), default=0)
    free, _ = torch.cuda.mem_get_info(device)
    free += torch.cuda.memory_reserved(device) - torch.cuda.memory_allocated(device)
    if need > free:
        raise MemoryError(f"{w.name} needs {need / 1e9:.2f} GB on {device} for its buffers and draws; "
                          f"{free / 1e9:.2f} GB are free")


class FlatBuffers:
    def __init__(self, w: Workload, device, grad_step: int = 1, gap: int = ALIGN, shard_rank: int = 0):
        self.w = w
        self.shard_rank = shard_rank  # draws rank r's shards (see generate.draw_grad)
        self.device = torch.device(device)
        self.offsets = []
        cur = 0
        for t in w.tensors:
            self.offsets.append(cur)
            cur += (t.numel + gap + ALIGN - 1) // ALIGN * ALIGN
        total = max(cur, ALIGN)
        gdts = {torch_dtype(t.grad_dtype) for t in w.tensors}
        if len(gdts) != 1:
            raise ValueError("one gradient dtype per flat workload")
        self.grad_dtype = gdts.pop()
        lows = {t.param_lowp for t in w.tensors if t.param_lowp}
        if len(lows) > 1:
            raise ValueError("one model-copy dtype per flat workload")
        if self.device.type == "cuda":
            check_device_memory(w, self.device, total * bytes_per_slot(self.grad_dtype, bool(lows)))
        self.P = torch.empty(total, dtype=torch.float32, device=self.device)
        self.G = torch.empty(total, dtype=self.grad_dtype, device=self.device)
        self.M = torch.empty(total, dtype=torch.float32, device=self.device)
        self.V = torch.empty(total, dtype=torch.float32, device=self.device)
        for buf in (self.P, self.M, self.V):
            buf.view(torch.int32).fill_(SENTINEL_F32)
        if self.G.element_size() == 2:  # bf16 or fp16: 0x7FAD is a NaN in both
            self.G.view(torch.int16).fill_(SENTINEL_BF16)
        else:
            self.G.view(torch.int32).fill_(SENTINEL_F32)
        self.PL = None
        if lows:
            self.PL = torch.empty(total, dtype=torch_dtype(lows.pop()), device=self.device)
            self.PL.view(torch.int16).fill_(SENTINEL_BF16)
        self.p, self.g, self.m, self.v, self.plow = [], [], [], [], []
        for k, t in enumerate(w.tensors):
            sl = slice(self.offsets[k], self.offsets[k] + t.numel)
            self.p.append(self.P[sl])
            self.g.append(self.G[sl])
            self.m.append(self.M[sl])
            self.v.append(self.V[sl])
            self.plow.append(self.PL[sl] if (self.PL is not None and t.param_lowp) else None)
            self.p[-1].copy_(draw_param(w, k, self.device, shard_rank).reshape(-1))
            if self.plow[-1] is not None:
                self.plow[-1].copy_(self.p[-1].to(self.PL.dtype))
            self.m[-1].zero_()
            self.v[-1].zero_()
        self.load_grads(grad_step)

    def load_grads(self, step: int):
        for k in range(len(self.w.tensors)):
            self.g[k].copy_(draw_grad(self.w, k, step, self.device, self.shard_rank).reshape(-1))

    def gaps(self):
        """(start, end) element ranges between and after the tensor views."""
        out = []
        for k, t in enumerate(self.w.tensors):
            end = self.offsets[k + 1] if k + 1 < len(self.offsets) else self.P.numel()
            if self.offsets[k] + t.numel < end:
                out.append((self.offsets[k] + t.numel, end))
        return out

    def gaps_intact(self) -> bool:
        half = self.G.element_size() == 2
        gsent = SENTINEL_BF16 if half else SENTINEL_F32
        gi = self.G.view(torch.int16 if half else torch.int32)
        for a, b in self.gaps():
            for buf in (self.P, self.M, self.V):
                if not bool((buf.view(torch.int32)[a:b] == SENTINEL_F32).all()):
                    return False
            if not bool((gi[a:b] == gsent).all()):
                return False
            if self.PL is not None and not bool((self.PL.view(torch.int16)[a:b] == SENTINEL_BF16).all()):
                return False
        return True
