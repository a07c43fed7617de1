"""The boundary is a C ABI: a plain C99 program (tests/c_abi/abi_check.c)
includes include/soma_opt.h, links the library and drives its host-side
calls without Python or CUDA work."""
import os
import shutil
import subprocess

import pytest

from tensor_grad_clip_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c99_program_uses_the_library(tmp_path):
    lib = build.build()
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(HERE, "c_abi", "abi_check.c"), "-o", str(exe), lib,
                    "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs g++")
def test_header_links_from_cpp(tmp_path):
    # the same program built as C++17: the header's extern "C" block gives the
    # library's unmangled names
    lib = build.build()
    exe = tmp_path / "abi_check_cpp"
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    "-x", "c++", os.path.join(HERE, "c_abi", "abi_check.c"), "-x", "none", "-o", str(exe), lib,
                    "-Wl,-rpath," + os.path.dirname(lib)], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "c abi ok" in out.stdout


@pytest.mark.gpu
@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c99_program_runs_a_step(tmp_path):
    # No Python on the path: CUDA runtime buffers, one step, the closed form,
    # and the allocation-free norm of the same gradients.
    lib = build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    exe = tmp_path / "step_check"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), os.path.join(HERE, "c_abi", "step_check.c"),
                    "-o", str(exe), lib, "-L", os.path.join(cuda, "lib64"), "-lcudart", "-lm",
                    "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(cuda, "lib64")], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert "c step ok" in out.stdout
