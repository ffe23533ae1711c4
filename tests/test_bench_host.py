"""bench.py's roofline bookkeeping on the CPU.

The algorithmic work of the GEMM launches adds up to the layer's FLOPs; an ncu --csv log of DRAM bytes is averaged
per launch and kernel into the traffic table; the table's figures are used only while the CUDA sources are the ones
they were captured on.
"""
import json

import pytest

import bench
from fine_grained_mixture_gb300 import synth
from oracle import moe_oracle as orc

HEADER = ('"ID","Process ID","Process Name","Host Name","Kernel Name","Context","Stream","Block Size","Grid Size",'
          '"Device","CC","Section Name","Metric Name","Metric Unit","Metric Value"\n')


def _row(launch, kernel, metric, unit, value):
    return (f'"{launch}","1","python3.12","127.0.0.1","{kernel}","1","7","(448, 1, 1)","(152, 1, 1)","0","10.3",'
            f'"Command line profiler metrics","{metric}","{unit}","{value}"\n')


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_gemm_work_adds_up_to_the_layer(name):
    w = synth.WORKLOADS[name]
    P = w.T * w.K
    fwd, bwd = orc.layer_flops(P, w.n, w.d)
    work = {k: bench.kernel_flops_bytes(k, w, P) for k in bench.GEMM_NAMES}
    assert all(bound == "tensor" for bound, _ in work.values())
    step = sum(work[k][1] for k in ("gemm_up", "gemm_down", "gemm_dh", "gemm_dx", "gemm_dw"))
    assert step == fwd + bwd == 18 * w.T * w.n * w.K * w.d
    assert work["gemm_dw1"][1] + work["gemm_dw2"][1] == work["gemm_dw"][1]


def test_kernel_names_from_ncu():
    assert bench.bench_kernel_name("void moe_gemm_kernel<6, 256, 3, 2, 0>(TensorMaps, GemmArgs)") == "gemm_dw"
    assert bench.bench_kernel_name("moe_gemm_kernel<(int)0, 256, 4, 1, 0>") == "gemm_up"
    # the last template argument is the number of CTAs per MMA (2: the CTA-pair scatter-add GEMMs)
    assert bench.bench_kernel_name("void moe_gemm_kernel<3, 256, 4, 1, 0, 2>(TensorMaps, GemmArgs)") == "gemm_dx"
    assert bench.bench_kernel_name("void moe_gemm_kernel<1, 256, 4, 1, 1, 2>(TensorMaps, GemmArgs)") == "gemm_down"
    assert bench.bench_kernel_name("void route_topk_kernel<4, 0>(const float *, int)") == "route_topk"
    assert bench.bench_kernel_name("void some_library_kernel()") is None


def test_ingest_averages_per_launch_and_goes_stale_with_the_source(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    dw = "void moe_gemm_kernel<6, 256, 3, 2, 0>(TensorMaps, GemmArgs)"
    csv = tmp_path / "traffic.csv"
    csv.write_text("==PROF== Connected to process 1\n" + HEADER
                   + _row(0, dw, "dram__bytes_read.sum", "Gbyte", "1.5")
                   + _row(0, dw, "dram__bytes_write.sum", "Mbyte", "500")
                   + _row(0, dw, "gpu__time_duration.sum", "us", "350")
                   + _row(1, dw, "dram__bytes_read.sum", "byte", "500,000,000")
                   + _row(1, dw, "dram__bytes_write.sum", "byte", "0")
                   + _row(1, dw, "gpu__time_duration.sum", "ns", "250000")
                   + _row(2, "void some_library_kernel()", "dram__bytes_read.sum", "byte", "7"))
    monkeypatch.setattr(bench, "source_sha", lambda kernel=None: "digest-a")
    assert bench.ingest_ncu(str(csv), "fine7b") == 0
    table = json.loads((tmp_path / "profiles" / "dram_traffic.json").read_text())
    ent = table["gemm_dw"]["fine7b"]
    assert ent["launches"] == 2 and ent["source_sha"] == "digest-a"
    assert ent["read"] == pytest.approx(1.0e9) and ent["write"] == pytest.approx(2.5e8)
    assert ent["bytes_per_launch"] == pytest.approx(1.25e9) and ent["ncu_time_us"] == pytest.approx(300.0)
    assert set(table) == {"gemm_dw"}
    assert bench.load_traffic("gemm_dw", "fine7b") == pytest.approx(1.25e9)
    assert bench.load_traffic("gemm_dw", "sparse") is None
    monkeypatch.setattr(bench, "source_sha", lambda kernel=None: "digest-b")   # the kernels changed since the capture
    assert bench.load_traffic("gemm_dw", "fine7b") is None


def test_traffic_digest_follows_the_kernel_family_sources():
    # a GEMM's captured traffic depends on the GEMM sources, not on the host-side api.cu or the routing kernels
    assert "api.cu" not in bench.KERNEL_SOURCES["gemm"] and "route.cu" not in bench.KERNEL_SOURCES["gemm"]
    assert bench.kernel_family("gemm_dw") == "gemm" and bench.kernel_family("route_topk") == "route"
    assert bench.kernel_family("router_dz_rows") == "router" and bench.kernel_family("cast_f32_bf16") == "cast"
    assert bench.source_sha("gemm_dw") == bench.source_sha("gemm_up") != bench.source_sha("route_topk")



FAKE_SMI = r'''#!/usr/bin/env python3
import sys, time
# stand-in for the query loop: index, SM clock, max SM clock, power, active mask, then four throttle reasons
for i in range(40):
    now = time.time()
    stamp = time.strftime("%Y/%m/%d %H:%M:%S", time.localtime(now)) + ".%03d" % int((now % 1) * 1000)
    cap = "Active" if i == 3 else "Not Active"
    print(f"{stamp}, 0, {2070 - 10 * (i % 2)}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {cap}",
          flush=True)
    time.sleep(0.05)
'''


def test_clock_sampler_reads_median_clock_and_throttle_reasons(tmp_path, monkeypatch):
    smi = tmp_path / "nvidia-smi"
    smi.write_text(FAKE_SMI)
    smi.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}:{bench.os.environ['PATH']}")
    monkeypatch.setattr(bench.tempfile, "tempdir", str(tmp_path))   # the sample file stays in the test's folder
    sampler = bench.ClockSampler(0)
    sampler.start()
    t0 = bench.time.time()
    bench.time.sleep(0.5)
    t1 = bench.time.time()
    out = sampler.stop(t0, t1)
    assert out["samples"] >= 3 and out["samples_in_timed_region"] >= 3
    assert out["sm_max_mhz"] == 2070.0
    assert out["sm_mhz"] in (2060.0, 2065.0, 2070.0)
    assert out["reasons"] == ["sw_power_cap"]
    assert not list(tmp_path.glob("*.csv"))


def test_clock_sampler_without_nvidia_smi(tmp_path, monkeypatch):
    monkeypatch.setenv("PATH", str(tmp_path))
    monkeypatch.setattr(bench.tempfile, "tempdir", str(tmp_path))
    sampler = bench.ClockSampler(0)
    sampler.start()
    out = sampler.stop(0.0, 1.0)
    assert out["sm_mhz"] is None and out["reasons"] == ["nvidia-smi unavailable"]
    assert not list(tmp_path.glob("*.csv"))                          # the sample file is removed


def test_every_timed_step_includes_the_data_parallel_exchange(monkeypatch):
    """The split timing pass calls route, forward and backward apart; the all-reduce of the weight gradients must
    still run in every timed step (and the plain step must run it too)."""
    calls = []

    class FakeEvent:
        def __init__(self, **kw):
            pass

        def record(self, *a):
            calls.append("ev")

        def elapsed_time(self, other):
            return 1.0

    class FakeLayer:
        allreduce = True

        def route(self):
            calls.append("route")

        def forward(self):
            calls.append("forward")

        def backward(self):
            calls.append("backward")

        def exchange(self):
            calls.append("exchange")

        def step(self):
            for f in (self.route, self.forward, self.backward, self.exchange):
                f()

    monkeypatch.setattr(bench.torch.cuda, "Event", FakeEvent)
    monkeypatch.setattr(bench.torch.cuda, "synchronize", lambda *a: None)
    for split in (True, False):
        calls.clear()
        bench.time_steps(FakeLayer(), 3, split=split)
        assert calls.count("exchange") == 3 and calls.count("backward") == 3
        # each step's exchange follows its backward
        seq = [c for c in calls if c != "ev"]
        assert seq == ["route", "forward", "backward", "exchange"] * 3
