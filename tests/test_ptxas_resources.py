"""Register and spill budget of the tensor-core kernels, read from ptxas (-Xptxas -v) on the CPU.

A spill in a GEMM's main loop or epilogue costs local-memory traffic on every tile, and a register count above
what the launch's threads can share stops the launch; both are caught here, before a GPU run.  The thread counts
are the launch shapes of the kernels: the grouped GEMMs run 320 threads (448 for the weight gradients with
256-row blocks), one CTA per SM; the router GEMM runs 192 threads, two CTAs per SM.
"""
import os
import re
import subprocess
from concurrent.futures import ThreadPoolExecutor

import pytest

from fine_grained_mixture_gb300 import build as b

REGISTERS_PER_SM = 65536
UNITS = ["gemm_fwd.cu", "gemm_bwd.cu", "router.cu"]


def _ptxas_report():
    out_dir = os.path.join(b.BUILD, "ptxas_check")
    os.makedirs(out_dir, exist_ok=True)

    def one(src):
        cmd = [b._nvcc()] + b.ARCH + ["-O3", "-std=c++17", "-Xptxas", "-v", "-I", b.INCLUDE, "-I", b.CSRC, "-c",
                                      os.path.join(b.CSRC, src), "-o", os.path.join(out_dir, src + ".o")]
        r = subprocess.run(cmd, capture_output=True, text=True, timeout=900)
        assert r.returncode == 0, r.stderr[-2000:]
        return r.stderr

    with ThreadPoolExecutor(len(UNITS)) as pool:
        text = "\n".join(pool.map(one, UNITS))
    kernels, cur = {}, None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '(\w+)'", line)
        if m:
            cur = m.group(1)
            kernels[cur] = {}
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            kernels[cur]["spill"] = int(m.group(1)) + int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            kernels[cur]["regs"] = int(m.group(1))
    return kernels


def _threads(name):
    """Launch threads and resident CTAs per SM of a GEMM entry, from its mangled template arguments."""
    m = re.search(r"moe_gemm_kernelILi(\d+)ELi\d+ELi\d+ELi(\d+)E", name)
    if m:
        mode, mb = int(m.group(1)), int(m.group(2))
        # 448 threads: the weight gradients on 256-row blocks (eight epilogue warps beside the gatherers) and the
        # down-projection that recomputes A from H (eight epilogue warps beside the A producers)
        return (448 if (mode in (4, 5, 6) and mb == 2) or mode == 7 else 320), 1
    if "router_gemm_kernel" in name:
        return 192, 2
    return None


@pytest.fixture(scope="module")
def report():
    return _ptxas_report()


def test_every_tensor_core_kernel_is_reported(report):
    gemms = [k for k in report if _threads(k)]
    assert sum("moe_gemm_kernel" in k for k in gemms) >= 8 and sum("router_gemm_kernel" in k for k in gemms) == 3


def test_tensor_core_kernels_do_not_spill(report):
    spills = {k: v["spill"] for k, v in report.items() if _threads(k) and v.get("spill", 0)}
    assert not spills, spills


def test_registers_fit_the_launch(report):
    over = {}
    for k, v in report.items():
        shape = _threads(k)
        if shape and v["regs"] * shape[0] * shape[1] > REGISTERS_PER_SM:
            over[k] = (v["regs"], shape)
    assert not over, over
