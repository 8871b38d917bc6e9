"""The C ABI used from a plain C program (no Python in the loop): it compiles against
include/slope.h and libslope.so on the CPU, and on a GPU its prefill and single-launch
attention agree."""
import os
import subprocess

import pytest

import ring_attention_slope_gb300 as slope

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_client", "cp_prefill_client.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    lib = slope.build()
    exe = tmp_path / "cp_prefill_client"
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                           "-I", os.path.join(CUDA, "include"), SRC, "-o", str(exe), "-L", os.path.dirname(lib),
                           "-l:" + os.path.basename(lib), "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
                           "-Wl,-rpath," + os.path.dirname(lib) + ":" + os.path.join(CUDA, "lib64")])
    return exe


def test_c_client_builds(tmp_path):
    assert _build(tmp_path).exists()


@pytest.mark.gpu
def test_c_client_runs_on_the_gpu(tmp_path):
    exe = _build(tmp_path)
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stdout + out.stderr
    assert out.stdout.startswith("ok ")
