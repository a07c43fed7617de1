"""The oracle against the stored worked example (tests/golden), plus the
facts of that example that follow by hand from the SomaSpeed optimizer
paragraphs: only the owned, trainable w0 enters the norm; the frozen w2 never
moves; all-zero gradients give norm 0 and c = 1."""
import math

import numpy as np
import torch

import golden_fixture
from oracle import GroupState, OracleOptimizer


def _grad(vals, dtype):
    t = torch.tensor(vals, dtype=torch.float32)
    return t if dtype == "f32" else t.to(torch.bfloat16)


def test_fixture_by_hand():
    g = golden_fixture.load()
    w0 = np.array(g.grads[1][0]) / g.divisor
    assert g.expect[1]["norm"] == math.sqrt(float(np.sum(w0 * w0)))
    assert g.expect[1]["coef"] == g.max_norm / (g.expect[1]["norm"] + 1e-6)
    assert g.expect[2]["norm"] == 0.0 and g.expect[2]["coef"] == 1.0
    for s in g.expect:
        assert g.expect[s][("w2", "p")] == g.tensors[2]["p0"]
        assert not any(g.expect[s][("w2", "m")]) and not any(g.expect[s][("w2", "v")])


def test_oracle_reproduces_fixture_bitwise():
    g = golden_fixture.load()
    flags = [(t["group"], t["trainable"], t["owned"]) for t in g.tensors]
    opt = OracleOptimizer([np.array(t["p0"]) for t in g.tensors], flags,
                          [GroupState(**q) for q in g.groups])
    for s in sorted(g.grads):
        grads = [_grad(v, g.tensors[k]["dtype"]) for k, v in enumerate(g.grads[s])]
        norm, c = opt.step(grads, g.divisor, g.max_norm)
        assert norm == g.expect[s]["norm"] and c == g.expect[s]["coef"]
        for k, t in enumerate(g.tensors):
            assert opt.params[k].tolist() == g.expect[s][(t["name"], "p")]
            assert opt.exp_avg[k].tolist() == g.expect[s][(t["name"], "m")]
            assert opt.exp_avg_sq[k].tolist() == g.expect[s][(t["name"], "v")]
