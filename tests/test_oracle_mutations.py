"""The oracle's pins are strong enough to catch a plausible mistake in it.

Each case plants one mistake (a dropped term, a wrong sign, index or
operand, a missing clamp, ...) in a copy of oracle/oracle.c in a temporary
directory, rebuilds that copy, and runs the pin tests against it there: they
must fail.  The unmodified copy must pass.  Nothing here touches the product
library or the GPU."""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor


ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (name, [(text in oracle.c, replacement), ...])
MISTAKES = [
    ("update ignores the divisor", [("/ divisor * c;", "* c;")]),
    ("norm ignores the divisor", [("double g = grad_element(grad, dtype, i) / divisor;",
                                   "double g = grad_element(grad, dtype, i);")]),
    ("decay not scaled by lr", [("p[i] = p[i] * (1.0 - lr * weight_decay);", "p[i] = p[i] * (1.0 - weight_decay);")]),
    ("first moment with beta2", [("m[i] = beta1 * m[i] + (1.0 - beta1) * g;",
                                  "m[i] = beta2 * m[i] + (1.0 - beta2) * g;")]),
    ("second moment not squared", [("v[i] = beta2 * v[i] + (1.0 - beta2) * g * g;",
                                    "v[i] = beta2 * v[i] + (1.0 - beta2) * g;")]),
    ("bias corrections swapped", [("double m_hat = m[i] / bc1;", "double m_hat = m[i] / bc2;"),
                                  ("double v_hat = v[i] / bc2;", "double v_hat = v[i] / bc1;")]),
    ("second bias correction with beta1", [("pow(beta2, (double)step)", "pow(beta1, (double)step)")]),
    ("eps inside the square root", [("(sqrt(v_hat) + eps)", "sqrt(v_hat + eps)")]),
    ("bias correction off by one step", [("pow(beta1, (double)step)", "pow(beta1, (double)step - 1)")]),
    ("update with the wrong sign", [("p[i] = p[i] - lr * m_hat", "p[i] = p[i] + lr * m_hat")]),
    ("decay after the Adam step", [("p[i] = p[i] * (1.0 - lr * weight_decay);\n", ""),
                                   ("p[i] = p[i] - lr * m_hat / (sqrt(v_hat) + eps);",
                                    "p[i] = (p[i] - lr * m_hat / (sqrt(v_hat) + eps)) * (1.0 - lr * weight_decay);")]),
    ("bf16 widened with the wrong shift", [("<< 16;", "<< 15;")]),
    ("coefficient not clamped at 1", [("return c < 1.0 ? c : 1.0;", "return c;")]),
    ("no epsilon in the clip", [("(norm + 1e-6)", "(norm)")]),
    ("unowned tensors in the norm", [("if (!ts[k].trainable || !ts[k].owned)", "if (!ts[k].trainable)")]),
    ("step counted twice", [("groups[q].step += 1;", "groups[q].step += 2;")]),
    ("frozen-only groups step", [("present = ts[k].trainable && ts[k].group == q;", "present = ts[k].group == q;")]),
    ("group divisor ignored in the norm",
     [("double dk = groups[ts[k].group].divisor > 0.0 ? groups[ts[k].group].divisor : divisor;",
       "double dk = divisor;")]),
    ("group divisor ignored in the update", [("gp->divisor > 0.0 ? gp->divisor : divisor);", "divisor);")]),
    ("binary16 exponent bias off by one", [("ldexp((double)(1024 + f), e - 25)", "ldexp((double)(1024 + f), e - 24)")]),
    ("binary16 subnormals given the implicit bit", [("v = ldexp((double)f, -24);", "v = ldexp((double)(1024 + f), -25);")]),
    ("binary16 sign dropped", [("return sign ? -v : v;", "return v;")]),
    ("fp16 gradients decoded as bf16", [("if (dtype == ORACLE_GRAD_F16)\n", "if (0)\n")]),
    ("global norm without the square root", [("    return sqrt(total);", "    return total;")]),
    ("step norm without the square root", [("double norm = sqrt(total);", "double norm = total;")]),
    ("clip coefficient applied twice", [("/ divisor * c;", "/ divisor * c * c;")]),
    ("update with the unclipped gradient", [("/ divisor * c;", "/ divisor;")]),
    ("frozen tensors updated", [("        if (!ts[k].trainable)\n            continue;\n        const oracle_group",
                                 "        const oracle_group")]),
    ("replicated tensors not updated", [("        if (!ts[k].trainable)\n            continue;\n        const oracle_group",
                                         "        if (!ts[k].trainable || !ts[k].owned)\n            continue;\n"
                                         "        const oracle_group")]),
    ("first bias correction multiplied", [("double m_hat = m[i] / bc1;", "double m_hat = m[i] * bc1;")]),
    ("NaN norm clamped to 1", [("    if (isnan(c))\n        return c;\n", "")]),
]

PINS = ["tests/test_oracle_pins.py", "tests/test_oracle_golden.py"]


def _run_pins(tmp, name, edits):
    d = os.path.join(tmp, name.replace(" ", "_"))
    for sub in ("oracle", "tests", "workloads"):
        shutil.copytree(os.path.join(ROOT, sub), os.path.join(d, sub),
                        ignore=shutil.ignore_patterns("_build", "__pycache__", "*.so"))
    src_path = os.path.join(d, "oracle", "oracle.c")
    with open(src_path) as f:
        src = f.read()
    for old, new in edits:
        assert old in src, f"{name}: {old!r} is no longer in oracle.c"
        src = src.replace(old, new)
    with open(src_path, "w") as f:
        f.write(src)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu"] + PINS,
                       cwd=d, capture_output=True, text=True, timeout=600)
    return r.returncode, r.stdout[-2000:]


def test_planted_mistakes_fail_the_pins(tmp_path):
    cases = [("unmodified", [])] + MISTAKES
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        results = list(ex.map(lambda c: (c[0],) + _run_pins(str(tmp_path), c[0], c[1]), cases))
    base = results[0]
    assert base[1] == 0, "the pins fail on the unmodified oracle:\n" + base[2]
    survived = [name for name, rc, _ in results[1:] if rc == 0]
    assert not survived, f"planted mistakes the pins did not catch: {survived}"
