"""Reader of tests/golden/three_tensor_steps.txt (see make_golden.py there)."""
import os
from dataclasses import dataclass, field

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "three_tensor_steps.txt")


@dataclass
class Golden:
    divisor: float = 0.0
    max_norm: float = 0.0
    groups: list = field(default_factory=list)      # dicts
    tensors: list = field(default_factory=list)     # dicts: name, dtype, group, trainable, owned, p0
    grads: dict = field(default_factory=dict)       # step -> list per tensor
    expect: dict = field(default_factory=dict)      # step -> {"norm", "coef", (name, tag): [..]}


def load(path: str = PATH) -> Golden:
    g = Golden()
    names = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, *rest = line.split(" ")
            if head == "divisor":
                g.divisor = float(rest[0])
            elif head == "max_norm":
                g.max_norm = float(rest[0])
            elif head == "group":
                kv = dict(x.split("=") for x in rest[1:])
                g.groups.append({k: float(v) for k, v in kv.items()})
            elif head == "tensor":
                name, dt = rest[0], rest[1]
                kv = dict(x.split("=") for x in rest[2:])
                g.tensors.append(dict(name=name, dtype=dt, group=int(kv["group"]),
                                      trainable=bool(int(kv["trainable"])), owned=bool(int(kv["owned"])),
                                      p0=[float(x) for x in kv["p0"].split(",")]))
                names.append(name)
            elif head == "grad":
                step, name, vals = int(rest[0]), rest[1], rest[2]
                g.grads.setdefault(step, [None] * len(names))[names.index(name)] = \
                    [float(x) for x in vals.split(",")]
            elif head == "expect":
                step = int(rest[0])
                e = g.expect.setdefault(step, {})
                if rest[1] == "norm":
                    e["norm"] = float.fromhex(rest[2])
                    e["coef"] = float.fromhex(rest[4])
                else:
                    e[(rest[1], rest[2])] = [float.fromhex(x) for x in rest[3].split(",")]
    return g
