"""tests/c_api_example.c, a plain-C user of include/cb_moe.h and libcbmoe.so: it
compiles and links against the library with gcc on any machine, and runs a
layer end to end on a GB300."""
import os
import shutil
import subprocess

import pytest

import mixture_experts_router_gb300 as cb
from mixture_experts_router_gb300 import build as cbuild

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    cbuild.build()
    libdir = os.path.dirname(cb.LIB_PATH)
    cudalib = os.path.join(CUDA, "lib64")
    exe = str(tmp_path / "c_api_example")
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", os.path.join(HERE, "c_api_example.c"), "-o", exe,
           f"-I{os.path.join(ROOT, 'include')}", f"-I{os.path.join(CUDA, 'include')}",
           f"-L{libdir}", "-lcbmoe", f"-Wl,-rpath,{libdir}", f"-L{cudalib}", "-lcudart", f"-Wl,-rpath,{cudalib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_example_builds_and_runs_without_a_gpu_path(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "workspace" in r.stdout or r.stdout.strip().endswith("ok")


@pytest.mark.gpu
def test_c_example_runs_a_layer(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ok"), r.stdout
