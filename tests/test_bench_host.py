"""bench.py's host side, without a GPU: the reference arm's JSON line, the
code-only kernel hash that keys the ncu traffic record, and that record."""
import json
import os
import subprocess
import sys

import bench
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e")


def test_reference_arm_prints_one_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny", "--steps", "1",
                          "--warmup", "1"], cwd=ROOT, capture_output=True, text=True, timeout=300, check=True)
    lines = [x for x in out.stdout.splitlines() if x.strip().startswith("{")]
    assert len(lines) == 1, out.stdout
    line = json.loads(lines[0])
    for key in REQUIRED:
        assert key in line, key
    assert line["impl"] == "reference" and line["value"] > 0 and line["n_gpus"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": line["unit"], "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    assert "workload" in line["config"]


def test_code_only_hash_ignores_comments_and_layout():
    a = 'int f(int x) { // the sum\n    return x + 1; /* one more */ }\nconst char* s = "// kept";\n'
    b = 'int f(int x)\n{\n  return x + 1;\n}\nconst char* s = "// kept";  // a note\n'
    c = 'int f(int x) { return x + 2; }\nconst char* s = "// kept";\n'
    d = 'int f(int x) { return x + 1; }\nconst char* s = "// changed";\n'
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)  # code changed
    assert bench._code_only(a) != bench._code_only(d)  # a string literal is code


def test_traffic_is_reported_only_for_the_code_and_list_it_was_measured_on():
    with open(bench.profile_json("action_expert")) as f:
        rec = json.load(f)
    got = bench.ncu_traffic("action_expert", W.FULL["action_expert"]().name)
    if rec["kernel_sha"] == bench.kernel_source_hash():
        assert got == rec["dram_bytes_per_launch"]
    else:  # the kernels changed since the capture: no traffic figure
        assert got is None
    # a record names its list: another list's name finds nothing
    assert bench.ncu_traffic("action_expert", W.FULL["flat"]().name) is None
    assert bench.ncu_traffic("no_such_list", W.FULL["flat"]().name) is None


def test_default_line_is_the_largest_single_gpu_list():
    # the 7B shard view is the largest list that fits one GPU; the others
    # are measured in the same run under per_config
    assert bench.DEFAULT_WORKLOAD == "hsdp_shard"
    sizes = {k: f().trainable_numel for k, f in W.FULL.items()}
    assert max(sizes, key=sizes.get) == "hsdp_shard"
    names = bench.DEFAULT_PER_CONFIG.split(",")
    assert {x.partition(":")[0] for x in names} == set(W.FULL) - {"hsdp_shard"}
    assert {x.partition(":")[2] for x in names} <= {"", "master", "graph"}
