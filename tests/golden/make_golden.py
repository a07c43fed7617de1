"""Write tests/golden/three_tensor_steps.txt from the fp64 oracle alone.

The fixture is a worked example of the step the SomaSpeed page describes in
its two optimizer paragraphs (what a step does to each gradient, and how
the work is batched over the tensor list):
normalize by the effective-batch divisor, one global norm over owned
gradients, one clip coefficient, AdamW on every trainable tensor, frozen
tensors untouched.  Inputs are short dyadic numbers (exact in fp32 and bf16);
every expected value below is the oracle's, written as a hex float.

Run:  python tests/golden/make_golden.py
"""
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import GroupState, OracleOptimizer  # noqa: E402

OUT = os.path.join(HERE, "three_tensor_steps.txt")

# name, grad dtype, group, trainable, owned, initial weights
TENSORS = [
    ("w0", "f32", 0, 1, 1, [0.5, -0.25, 0.125, 1.0, -2.0]),
    ("w1", "bf16", 1, 1, 0, [0.75, -0.5, 0.0625]),
    ("w2", "f32", 0, 0, 1, [1.5, -1.5]),
]
GROUPS = [dict(lr=0.01, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1),
          dict(lr=0.02, beta1=0.8, beta2=0.99, eps=1e-6, weight_decay=0.0)]
DIVISOR = 2.0
MAX_NORM = 1.0
GRADS = [  # per step, per tensor
    [[3.0, -4.0, 0.5, 0.25, -1.0], [8.0, -0.5, 2.0], [100.0, -100.0]],
    [[0.0, 0.0, 0.0, 0.0, 0.0], [-1.0, 0.25, 0.5], [7.0, 7.0]],
    [[0.125, 0.0625, -0.5, 0.75, 0.03125], [0.0, 4.0, -4.0], [1.0, 2.0]],
]


def _grad(values, dtype):
    import torch
    t = torch.tensor(values, dtype=torch.float32)
    return t if dtype == "f32" else t.to(torch.bfloat16)


def compute():
    flags = [(g, t, o) for _, _, g, t, o, _ in TENSORS]
    opt = OracleOptimizer([np.array(p) for *_, p in TENSORS], flags,
                          [GroupState(**g) for g in GROUPS])
    rows = []
    for s, grads in enumerate(GRADS, start=1):
        gs = [_grad(v, TENSORS[k][1]) for k, v in enumerate(grads)]
        norm, c = opt.step(gs, DIVISOR, MAX_NORM)
        rows.append((s, norm, c, [p.copy() for p in opt.params], [m.copy() for m in opt.exp_avg],
                     [v.copy() for v in opt.exp_avg_sq]))
    return rows


def render(rows) -> str:
    out = ["# Worked example of the fused step (SomaSpeed page, optimizer paragraphs).",
           "# Inputs: dyadic values, exact in fp32/bf16.  Expected values: written by",
           "# tests/golden/make_golden.py from the fp64 oracle, as hex floats.",
           f"divisor {DIVISOR!r}", f"max_norm {MAX_NORM!r}"]
    for q, g in enumerate(GROUPS):
        out.append("group {} ".format(q) + " ".join(f"{k}={v!r}" for k, v in g.items()))
    for name, dt, grp, tr, own, p in TENSORS:
        out.append(f"tensor {name} {dt} group={grp} trainable={tr} owned={own} p0=" +
                   ",".join(repr(x) for x in p))
    for s, grads in enumerate(GRADS, start=1):
        for k, g in enumerate(grads):
            out.append(f"grad {s} {TENSORS[k][0]} " + ",".join(repr(x) for x in g))
    for s, norm, c, ps, ms, vs in rows:
        out.append(f"expect {s} norm {norm.hex()} coef {c.hex()}")
        for k in range(len(TENSORS)):
            for tag, arr in (("p", ps[k]), ("m", ms[k]), ("v", vs[k])):
                out.append(f"expect {s} {TENSORS[k][0]} {tag} " + ",".join(float(x).hex() for x in arr))
    return "\n".join(out) + "\n"


if __name__ == "__main__":
    text = render(compute())
    with open(OUT, "w") as f:
        f.write(text)
    print(f"wrote {OUT}")
