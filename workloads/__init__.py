"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle
harness.  No arithmetic of the optimizer step lives here."""
from .configs import (BF16, F16, F32, FULL, SMALL, GroupSpec, TensorSpec, Workload,
                      action_expert, cosine_lr, flat, hsdp_shard_view, many_small,
                      tiny, with_steps)
from .device import FlatBuffers
from .generate import (draw_grad, draw_grads, draw_param, draw_params, tensor_seed, torch_dtype,
                       zero_moments)

__all__ = [
    "BF16", "F16", "F32", "FlatBuffers", "FULL", "SMALL", "GroupSpec", "TensorSpec", "Workload",
    "action_expert", "cosine_lr", "flat", "hsdp_shard_view", "many_small", "tiny",
    "with_steps", "draw_grad", "draw_grads", "draw_param", "draw_params", "tensor_seed", "torch_dtype",
    "zero_moments",
]
