"""The C ABI from a plain C program (tests/c_abi/abi_demo.c): compiled with gcc against include/moe.h and linked
to libmoe.so and the CUDA runtime, with no Python in the call path.  On the CPU it runs the host-side queries and
validation; on a GB300 it routes, runs the forward and the backward on cudaMalloc buffers and checks the status."""
import os
import shutil
import subprocess

import pytest

from fine_grained_mixture_gb300 import build as b

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_demo.c")


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(os.path.realpath(nvcc)))


def _cudart_dir(cuda):
    """The directory holding libcudart.so (lib64 on x86_64; targets/<arch>/lib on other hosts)."""
    import glob
    for cand in [os.path.join(cuda, "lib64")] + sorted(glob.glob(os.path.join(cuda, "targets", "*", "lib"))):
        if os.path.exists(os.path.join(cand, "libcudart.so")):
            return cand
    pytest.skip("libcudart.so not found")


@pytest.fixture(scope="module")
def demo(tmp_path_factory):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    b.build()
    cuda = _cuda_home()
    out = str(tmp_path_factory.mktemp("c_abi") / "abi_demo")
    libdir = os.path.dirname(b.LIB)
    rt = _cudart_dir(cuda)
    cmd = ["gcc", "-O2", "-std=c11", "-o", out, SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), "-L", libdir, "-lmoe", "-L", rt, "-lcudart", "-lm",
           f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{rt}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return out


def test_c_program_host_checks(demo):
    res = subprocess.run([demo, "host"], capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    assert "host checks ok" in res.stdout


@pytest.mark.gpu
def test_c_program_runs_the_layer(demo):
    res = subprocess.run([demo, "run"], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "run ok: P = 1024" in res.stdout
