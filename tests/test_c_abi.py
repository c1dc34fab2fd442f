"""The C ABI used from a plain C program (tests/c/abi_demo.c), compiled with gcc against
include/smoe.h and libsmoe.so: host-side checks without a GPU, one layer with a GPU."""
import os
import shutil
import subprocess

import pytest

from routing_token_shuffle_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def demo(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    lib = build_mod.build()
    out = str(tmp_path_factory.mktemp("c_abi") / "abi_demo")
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", os.path.join(ROOT, "tests", "c", "abi_demo.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", libdir, "-lsmoe", f"-Wl,-rpath,{libdir}",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}",
           "-lm", "-o", out]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return out


def test_c_program_host_checks(demo):
    r = subprocess.run([demo], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "host checks ok" in r.stdout


@pytest.mark.gpu
def test_c_program_runs_a_layer(demo):
    r = subprocess.run([demo, "gpu"], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "ok" in r.stdout
