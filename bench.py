#!/usr/bin/env python
"""Throughput benchmark of the fine-grained MoE expert layer (routing + forward + backward) on GB300.

One step = routing (token choice by default) + forward + backward of one MoE layer over one batch of
seeded synthetic inputs already resident in HBM.  The metric is the layer's nominal FLOPs
18*T*n*K*d per second (forward 6TnKd, backward 12TnKd), reported in TFLOPS and as a fraction of the
measured dense BF16 peak.  Default workload: the fine-grained 7B-class layer T=24576, d=1536, n=256,
E=128, K=8.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload fine7b] [--mode tc|tr]
  python bench.py --impl reference ...      # the CPU oracle on the host cores, bounded sample per step

Multi-GPU: data parallelism, one rank per GPU (launch with torchrun; rank 0 prints the line).  Every rank holds
a replica of W1/W2 (broadcast from rank 0) and its own T tokens, runs route + forward + backward on them, and the
step ends with the all-reduce of dW1 and dW2 over NCCL (weak scaling: the global batch is N*T tokens).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import re
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from fine_grained_mixture_gb300 import synth  # noqa: E402

METRIC = "MoE layer fwd+bwd TFLOPS (18·T·n·K·d/s) on 1 GB300; % of BF16 dense peak"
UNIT = "TFLOPS"
L2_BYTES = 126 * 2**20
DATA = "synthetic: seeded torch CPU generator; logits ~N(0,1), X/dO ~N(0,1), W1 ~N(0,1/d), W2 ~N(0,1/n), bf16"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="fine7b", choices=list(synth.WORKLOADS))
    p.add_argument("--mode", default="tc", choices=["tc", "tr", "tr_up", "tr_down", "tr_stoch", "ec"])
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the CPU-oracle baseline sample")
    p.add_argument("--no-extras", action="store_true", help="skip the TR-vs-TC and e2e side measurements")
    p.add_argument("--router", action="store_true",
                   help="time only the router either side of the layer (logits, gate backward) and print its JSON")
    p.add_argument("--ingest-ncu", metavar="CSV", help="record per-launch DRAM bytes from an ncu --csv log "
                   "(dram__bytes_read.sum, dram__bytes_write.sum) in profiles/dram_traffic.json and exit")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            m = json.load(f)
        return dict(hbm=m["hbm_gbs"], bf16=m["bf16_tflops"], bf16_sus=m.get("bf16_tflops_sustained", m["bf16_tflops"]),
                    src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


def reduce_max(x: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the slowest replica sets the step time)."""
    if world <= 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_tflops(flops_per_rank: float, ms_max: float, world: int) -> float:
    """Whole-job throughput of N independent replicas: all ranks' FLOPs over the slowest rank's time."""
    return world * flops_per_rank / (ms_max * 1e-3) / 1e12


def layer_flops(w, P=None):
    rows = w.T * w.K if P is None else P
    return 6.0 * rows * w.n * w.d, 12.0 * rows * w.n * w.d


# ------------------------------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi sampling (200 ms) around the timed region; reads clocks and throttle reasons only."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.out = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        self.out = os.fdopen(fd, "w")
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self, t0, t1):
        self.out.close()
        if self.proc is None:
            os.unlink(self.path)
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            lines = f.readlines()
        for line in lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except Exception:
                continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        use = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median([r[1] for r in use]) if use else None,
                "sm_max_mhz": max([r[2] for r in use]) if use else None,
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside)}


# --------------------------------------------------------------------------------------- CPU oracle


def oracle_sample(w, inp, ref, experts):
    """Oracle forward+backward on the rows of `experts` (exact for those experts' rows)."""
    from oracle import moe_oracle as orc

    rows = np.concatenate([np.arange(ref["offsets"][e], ref["offsets"][e + 1]) for e in experts])
    ex_list = np.array(sorted(set(int(e) for e in experts)))
    remap = {e: i for i, e in enumerate(ex_list)}
    tok = ref["row_token"][rows]
    ex = np.array([remap[int(e)] for e in ref["row_expert"][rows]], dtype=np.int64)
    sc = ref["row_score"][rows]
    W1 = inp["W1_64"][ex_list]
    W2 = inp["W2_64"][ex_list]
    fwd = orc.forward(inp["X_64"], W1, W2, tok, ex, sc)
    orc.backward(inp["dO_64"], inp["X_64"], W1, W2, tok, ex, sc, fwd)
    return len(rows)


def cpu_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


def prepare_oracle_inputs(w, inp, mode):
    from oracle import moe_oracle as orc

    ref = orc.route(inp["logits"].numpy(), w.K, mode, u=synth.make_uniforms(w.E, 0).numpy())
    ref_inp = {"X_64": inp["X"].double().numpy(), "dO_64": inp["dO"].double().numpy(),
               "W1_64": inp["W1"].double().numpy(), "W2_64": inp["W2"].double().numpy()}
    return ref, ref_inp


# Both CPU timings of the oracle (the GPU arm's cpu_baseline and the --impl reference arm) use one sampling
# rule: each oracle call takes the rows of this many experts (cycled from expert 0), because every call also
# allocates and sums the T x d outputs O and dX, a fixed cost that a single expert's rows do not amortise.
ORACLE_EXPERTS_PER_CALL = 4


def oracle_call_experts(i, E):
    return [(i * ORACLE_EXPERTS_PER_CALL + j) % E for j in range(ORACLE_EXPERTS_PER_CALL)]


def oracle_timing(workload, mode, budget_s=None, steps=None, warmup=1):
    """Times the fp64 oracle's forward+backward on the host cores, one call of ORACLE_EXPERTS_PER_CALL experts'
    rows per step: `steps` timed steps after `warmup`, or as many as fit in `budget_s` seconds.  Returns the
    timed rows, seconds and calls.  Runs in a process without a CUDA context (see cpu_baseline)."""
    w = synth.WORKLOADS[workload]
    inp = synth.make_inputs(w, seed=0)
    ref, ref_inp = prepare_oracle_inputs(w, inp, mode)
    for i in range(warmup):  # warms the BLAS threads and the allocator
        oracle_sample(w, ref_inp, ref, oracle_call_experts(i, w.E))
    rows, t_timed, calls = 0, 0.0, 0
    while True:
        t0 = time.perf_counter()
        rows += oracle_sample(w, ref_inp, ref, oracle_call_experts(warmup + calls, w.E))
        t_timed += time.perf_counter() - t0
        calls += 1
        if (steps is not None and calls >= steps) or (budget_s is not None and t_timed > budget_s):
            break
    return {"rows": rows, "seconds": t_timed, "calls": calls, "P": int(ref["P"]), "cores": cpu_threads()}


def cpu_baseline(w, mode, budget_s):
    """The oracle timed on the host cores beside the GPU arm.  It runs in a spawned child process: a process
    that holds a CUDA context pays more for its large host allocations and unmaps (the oracle allocates the
    T x d outputs on every call), which measured the same oracle 1.7x slower than the reference arm's
    CUDA-free process."""
    import multiprocessing as mp

    with mp.get_context("spawn").Pool(1) as pool:
        r = pool.apply(oracle_timing, (w.name, mode), {"budget_s": budget_s})
    flops = 18.0 * r["rows"] * w.n * w.d
    return {"value": flops / r["seconds"] / 1e12, "unit": UNIT, "cores": r["cores"], "kind": "oracle",
            "sample": f"fp64 NumPy oracle forward+backward, {r['calls']} calls of {ORACLE_EXPERTS_PER_CALL} experts' "
                      f"rows each (experts cycled from 0; {r['rows']} of {r['P']} routed rows, {r['seconds']:.1f} s) "
                      f"of the {w.name} layer, in a CUDA-free child process; routing untimed"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = synth.WORKLOADS[args.workload]
    per_step = ORACLE_EXPERTS_PER_CALL
    r = oracle_timing(w.name, args.mode, steps=args.steps, warmup=args.warmup)
    rows_timed, t_timed = r["rows"], r["seconds"]
    flops = 18.0 * rows_timed * w.n * w.d
    value = flops / t_timed / 1e12
    sample = (f"fp64 NumPy oracle forward+backward on the rows of {per_step} experts per step "
              f"(experts cycled) of the {w.name} layer; routing untimed")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t_timed / max(args.steps, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA, "impl": "reference",
            "config": {"workload": f"{w.name}: T={w.T}, d={w.d}, n={w.n}, E={w.E}, K={w.K}, routing={args.mode}",
                       "sample_per_step": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------------- GPU arm


class Layer:
    """Resident device buffers for one workload and the step = route + forward + backward."""

    def __init__(self, w, inp, mode, dev, det=False, a_from_h=False, allreduce=False):
        import fine_grained_mixture_gb300 as moe

        self.moe, self.w, self.mode, self.det, self.a_from_h = moe, w, mode, det, a_from_h
        self.allreduce = allreduce  # data parallel: sum dW1/dW2 over the ranks at the end of each step
        flags = moe.MOE_FLAG_DETERMINISTIC if det else 0
        self.g = {k: v.to(dev) for k, v in inp.items()}
        self.u = synth.make_uniforms(w.E, 0).to(dev)  # per-expert draws of stochastic rounding
        self.rt = moe.Routing(w.T, w.E, w.K, mode, dev)
        p = self.rt.p_cap
        bf = torch.bfloat16
        self.O = torch.empty((w.T, w.d), dtype=bf, device=dev)
        self.H = torch.empty((p, 2 * w.n), dtype=bf, device=dev)
        self.dX = torch.empty((w.T, w.d), dtype=bf, device=dev)
        self.dW1 = torch.empty((w.E, w.d, 2 * w.n), dtype=bf, device=dev)
        self.dW2 = torch.empty((w.E, w.n, w.d), dtype=bf, device=dev)
        self.dS = torch.empty(p, dtype=torch.float32, device=dev)
        fflags = flags | (moe.MOE_FLAG_A_FROM_H if a_from_h else 0)
        self.wsf = torch.empty(moe.moe_forward_workspace_size(w.T, w.d, w.n, w.E, w.K, p, fflags), dtype=torch.uint8,
                               device=dev)
        self.wsb = torch.empty(moe.moe_backward_workspace_size(w.T, w.d, w.n, w.E, w.K, p, flags), dtype=torch.uint8,
                               device=dev)

    def route(self):
        self.moe.moe_route(self.g["logits"], self.w.K, self.mode, routing=self.rt, uniforms=self.u)

    def forward(self):
        self.moe.moe_forward(self.g["X"], self.g["W1"], self.g["W2"], self.rt, O=self.O, H=self.H, ws=self.wsf,
                             deterministic=self.det, a_from_h=self.a_from_h)

    def backward(self):
        self.moe.moe_backward(self.g["dO"], self.g["X"], self.g["W1"], self.g["W2"], self.H, self.rt, dX=self.dX,
                              dW1=self.dW1, dW2=self.dW2, dS=self.dS, ws=self.wsb, deterministic=self.det)

    def exchange(self):
        """Data parallel: the weight gradients summed over the ranks (nothing with a single rank)."""
        if self.allreduce:
            from fine_grained_mixture_gb300 import dp
            dp.allreduce_weight_grads(self.dW1, self.dW2)

    def step(self):
        self.route()
        self.forward()
        self.backward()
        self.exchange()

    def cached_bytes(self):
        """Bytes that live from forward to backward: X, H (P rows) and the routing metadata."""
        code, P = self.rt.device_status()
        meta = sum(t.numel() * t.element_size() for t in (
            self.rt.topk_idx, self.rt.topk_score, self.rt.tc_counts, self.rt.counts, self.rt.offsets,
            self.rt.tile_offsets, self.rt.row_token, self.rt.row_slot, self.rt.row_score, self.rt.status))
        return dict(X=self.g["X"].numel() * 2, H_rows=P * 2 * self.w.n * 2, H_alloc=self.H.numel() * 2, meta=meta, P=P)


def time_steps(layer, steps, split=False):
    """Times `steps` back-to-back steps with CUDA events on the current stream (split: also route, forward and
    backward apart; the data-parallel all-reduce is part of every step and of the total, not of the three parts)."""
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    marks = []
    ev[0].record()
    for _ in range(steps):
        if split:
            e = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            e[0].record()
            layer.route()
            e[1].record()
            layer.forward()
            e[2].record()
            layer.backward()
            e[3].record()
            layer.exchange()
            marks.append(e)
        else:
            layer.step()
    ev[1].record()
    torch.cuda.synchronize()
    total = ev[0].elapsed_time(ev[1])
    parts = None
    if split:
        parts = [sum(m[i].elapsed_time(m[i + 1]) for m in marks) for i in range(3)]
    return total, parts


def kernel_flops_bytes(name, w, P):
    """Algorithmic FLOPs (GEMM kernels) or bytes (memory-bound kernels) of one launch."""
    n, d, T, E, K = w.n, w.d, w.T, w.E, w.K
    flops = {"gemm_up": 4.0 * P * n * d, "gemm_down": 2.0 * P * n * d, "gemm_dh": 2.0 * P * n * d,
             "gemm_dx": 4.0 * P * n * d, "gemm_dw1": 4.0 * P * n * d, "gemm_dw2": 2.0 * P * n * d,
             "gemm_dw": 6.0 * P * n * d}
    if name in flops:
        return "tensor", flops[name]
    nbytes = {"cast_f32_bf16": T * d * 6.0, "route_topk": T * E * 4.0 + T * K * 8.0 + T * 8.0,
              "route_fill_tc": T * K * 8.0 + P * 12.0, "route_fill_tr": T * E * 4.0 + P * 12.0,
              "route_scan": 0.0}
    return "hbm", nbytes.get(name, 0.0)


def load_traffic(kernel, workload):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, if taken on the current source."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except Exception:
        return None
    ent = table.get(kernel, {}).get(workload)
    if not ent:
        return None
    if ent.get("source_sha") != source_sha(kernel):
        return None
    return ent.get("bytes_per_launch")


GEMM_NAMES = ["gemm_up", "gemm_down", "gemm_dh", "gemm_dx", "gemm_dw1", "gemm_dw2", "gemm_dw"]
NCU_NAMES = [("route_topk_kernel", "route_topk"), ("route_scan_kernel", "route_scan"),
             ("route_fill_tc_kernel", "route_fill_tc"), ("route_fill_tr_kernel", "route_fill_tr"),
             ("f32_to_bf16_kernel", "cast_f32_bf16"), ("fixed_to_bf16_kernel", "cast_fixed_bf16"),
             ("ds_sum_kernel", "ds_sum"), ("router_dz_rows_kernel", "router_dz_rows"),
             ("router_dz_tokens_kernel", "router_dz_tokens")]
UNIT_SCALE = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12, "ns": 1e-3, "us": 1.0, "ms": 1e3,
              "nsecond": 1e-3, "usecond": 1.0, "msecond": 1e3, "second": 1e6}


def bench_kernel_name(ncu_name):
    m = re.search(r"moe_gemm_kernel<\(?(?:int\))?(\d+)", ncu_name)
    if m:
        return GEMM_NAMES[int(m.group(1))]
    for key, name in NCU_NAMES:
        if key in ncu_name:
            return name
    return None


def ingest_ncu(csv_path, workload):
    """Average per-launch DRAM bytes per kernel from an ncu --csv log into profiles/dram_traffic.json."""
    import csv
    rows = []
    with open(csv_path) as f:
        lines = [ln for ln in f if ln.startswith('"')]
    per = {}  # launch id -> {name, metrics}
    for r in csv.DictReader(lines):
        name = bench_kernel_name(r["Kernel Name"])
        if name is None:
            continue
        ent = per.setdefault(r["ID"], {"name": name})
        ent[r["Metric Name"]] = float(r["Metric Value"].replace(",", "")) * UNIT_SCALE.get(r["Metric Unit"], 1.0)
    agg = {}
    for ent in per.values():
        if "dram__bytes_read.sum" not in ent:
            continue
        a = agg.setdefault(ent["name"], {"read": 0.0, "write": 0.0, "us": 0.0, "n": 0})
        a["read"] += ent["dram__bytes_read.sum"]
        a["write"] += ent.get("dram__bytes_write.sum", 0.0)
        a["us"] += ent.get("gpu__time_duration.sum", 0.0)
        a["n"] += 1
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            table = json.load(f)
    except Exception:
        table = {}
    for name, a in sorted(agg.items()):
        n = a["n"]
        table.setdefault(name, {})[workload] = {
            "bytes_per_launch": (a["read"] + a["write"]) / n, "read": a["read"] / n, "write": a["write"] / n,
            "launches": n, "ncu_time_us": a["us"] / n, "source_sha": source_sha(name)}
    with open(path, "w") as f:
        json.dump(table, f, indent=1, sort_keys=True)
        f.write("\n")
    print(json.dumps({k: round(v[workload]["bytes_per_launch"] / 1e6, 1) for k, v in table.items() if workload in v}))
    return 0


# The sources that define each kernel family: a captured traffic figure stays valid while these are unchanged.
KERNEL_SOURCES = {
    "gemm": ("gemm.cuh", "gemm_fwd.cu", "gemm_bwd.cu", "common.cuh", "internal.h"),
    "route": ("route.cu", "common.cuh", "internal.h"),
    "router": ("router.cu", "common.cuh", "internal.h"),
    "cast": ("elementwise.cu", "common.cuh", "internal.h"),
}


def kernel_family(kernel):
    if kernel and kernel.startswith("gemm_"):
        return "gemm"
    if kernel and kernel.startswith("router_"):
        return "router"
    if kernel and kernel.startswith("route_"):
        return "route"
    return "cast"


def source_sha(kernel=None):
    """Digest of the sources of `kernel`'s family (all of csrc/ when kernel is None)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "fine_grained_mixture_gb300", "csrc")
    files = sorted(os.listdir(csrc)) if kernel is None else KERNEL_SOURCES[kernel_family(kernel)]
    for f in files:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def main():
    args = parse()
    if args.ingest_ncu:
        return ingest_ncu(args.ingest_ncu, args.workload)
    if args.impl == "reference":
        return run_reference(args)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        from fine_grained_mixture_gb300 import dp
        dp.nccl_environment()
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from fine_grained_mixture_gb300 import build as _b
    _b.build()
    import fine_grained_mixture_gb300 as moe

    if args.router:
        if rank == 0:
            print(json.dumps({"router": router_timing(args, dev)}), flush=True)
        return 0
    w = synth.WORKLOADS[args.workload]
    pk = peaks()
    inp = synth.make_inputs(w, seed=rank)  # each rank's own tokens; the weights are made equal below
    layer = Layer(w, inp, args.mode, dev, allreduce=world > 1)
    if world > 1:
        from fine_grained_mixture_gb300 import dp
        dp.broadcast_weights(layer.g["W1"], layer.g["W2"])
    for _ in range(max(args.warmup, 3)):
        layer.step()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    launches0 = moe.kernel_launch_count()
    t0 = time.time()
    total_ms, parts = time_steps(layer, args.steps, split=True)
    t1 = time.time()
    launches = moe.kernel_launch_count() - launches0
    if world > 1:
        torch.distributed.barrier()
    # per-kernel CUDA events on the launch stream, over the same number of steps: a second pass, because
    # events between kernels would serialise the programmatic overlap of consecutive kernels
    torch.cuda.synchronize()
    moe.profile_enable(True)
    time_steps(layer, args.steps)
    moe.profile_enable(False)
    clocks = sampler.stop(t0, t1)
    prof = moe.profile_summary()

    ms = reduce_max(total_ms / args.steps, world, dev)
    ff, fb = layer_flops(w)
    value = weak_scaling_tflops(ff + fb, ms, world)
    cache = layer.cached_bytes()
    P = cache["P"]

    # roofline of the dominant kernel (largest share of the timed region)
    kern = {}
    for name, (n_launch, tot) in prof.items():
        bound, work = kernel_flops_bytes(name, w, P)
        avg = tot / n_launch
        kern[name] = {"launches_per_step": n_launch / args.steps, "ms_per_launch": avg,
                      "share": tot / sum(v[1] for v in prof.values()),
                      ("tflops" if bound == "tensor" else "gbs"): (work / (avg * 1e-3) / (1e12 if bound == "tensor" else 1e9))}
    top = max(prof.items(), key=lambda kv: kv[1][1])[0]
    bound, work = kernel_flops_bytes(top, w, P)
    avg_ms = prof[top][1] / prof[top][0]
    if bound == "tensor":
        achieved = work / (avg_ms * 1e-3) / 1e12
        # the burst peak: the kernel runs a few hundred microseconds inside a step of about a millisecond and a
        # timed loop of tens of milliseconds, far shorter than the seconds-long loop of the sustained figure
        peak = pk["bf16"]
        roof = {"bound": "tensor", "kernel": top, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "frac_of_sustained": achieved / pk["bf16_sus"],
                "traffic": load_traffic(top, w.name), "algorithmic_per_launch": work,
                "peak_kind": f"{pk['src']} burst bf16 (cuBLAS, timed alone)"}
    else:
        achieved = work / (avg_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "kernel": top, "achieved": achieved, "peak": pk["hbm"], "unit": "GB/s",
                "frac": achieved / pk["hbm"], "traffic": load_traffic(top, w.name), "algorithmic_per_launch": work,
                "peak_kind": f"{pk['src']} HBM copy bandwidth"}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": DATA,
        "config": {"workload": f"{w.name}: T={w.T}, d={w.d}, n={w.n}, E={w.E}, K={w.K}, routing={args.mode}, "
                               f"M_tile=128",
                   "parallelism": (f"data parallel x{world}: T tokens per rank, W1/W2 replicas, dW1/dW2 all-reduce "
                                   f"(NCCL, NVLS off) in every step") if world > 1 else "single GPU",
                   "l2": f"inputs larger than L2: one step touches ~{(2*w.T*w.d*3 + 6*w.E*w.d*w.n*2 + 12*P*w.n)/2**30:.1f} GiB"
                         f" vs {L2_BYTES/2**20:.0f} MiB L2; no flush"},
        "frac_of_peak": {"burst": value / world / pk["bf16"], "sustained": value / world / pk["bf16_sus"],
                         "peak_source": pk["src"]},
        "fwd_tflops": ff / ((parts[0] + parts[1]) / args.steps * 1e-3) / 1e12,
        "bwd_tflops": fb / (parts[2] / args.steps * 1e-3) / 1e12,
        "split_ms_per_step": {"route": parts[0] / args.steps, "forward": parts[1] / args.steps,
                              "backward": parts[2] / args.steps},
        "activation_bytes": {"cached_X_H_meta": cache["X"] + cache["H_rows"] + cache["meta"],
                             "bound_2Td_4TKn_plus_meta": 2 * w.T * w.d + 4 * w.T * w.K * w.n + cache["meta"],
                             "metadata": cache["meta"]},
        "roofline": roof,
        "kernels": kern,
        "clocks": clocks,
        "gpu_launches": launches,
    }

    if not args.no_extras:
        line["e2e"] = e2e_measure(layer, inp, args, world, dev)
        if rank == 0 and world == 1:
            line["tr_vs_tc"] = tr_vs_tc(args, dev)
            line["router"] = router_timing(args, dev)
            line["deterministic"] = deterministic_timing(args, w, inp, line["ms_per_step"], dev)
            line["a_from_h"] = a_from_h_timing(args, dev)
    if rank == 0 and world == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.mode, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def e2e_measure(layer, inp, args, world, dev):
    """Same metric through the public API with host buffers: every step copies its activations (logits, X,
    dO) host->device from pinned memory, runs the layer, and copies its results (O, dX) device->host.  As in
    a training loop that prefetches, the copies run on a copy stream into double-buffered device tensors, so
    step i+1's inputs and step i-1's outputs move while step i computes; every step's copies are inside the
    timed region."""
    w = layer.w
    names_in, names_out = ("logits", "X", "dO"), ("O", "dX")
    host_in = {k: inp[k].pin_memory() for k in names_in}
    host_out = [{k: torch.empty((w.T, w.d), dtype=torch.bfloat16).pin_memory() for k in names_out} for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out[0].values())
    dev_in = [{k: layer.g[k] for k in names_in}, {k: torch.empty_like(layer.g[k]) for k in names_in}]
    dev_out = [{"O": layer.O, "dX": layer.dX}, {k: torch.empty_like(getattr(layer, k)) for k in names_out}]
    main = torch.cuda.current_stream()
    copy_in, copy_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)  # one copy engine each way
    ev = lambda: torch.cuda.Event()  # noqa: E731
    in_ready = [ev(), ev()]     # inputs of buffer set b copied
    computed = [ev(), ev()]     # step on set b done (its inputs are free, its outputs final)
    out_read = [ev(), ev()]     # outputs of set b copied to the host

    def h2d_into(b):
        with torch.cuda.stream(copy_in):
            copy_in.wait_event(computed[b])  # the step that last used set b has finished with its inputs
            for k in names_in:
                dev_in[b][k].copy_(host_in[k], non_blocking=True)
            in_ready[b].record(copy_in)

    def run(n):
        for b in range(2):
            computed[b].record(main)
            out_read[b].record(main)
        h2d_into(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                h2d_into(b ^ 1)
            main.wait_event(in_ready[b])
            main.wait_event(out_read[b])  # the outputs of the step two back have reached the host
            for k in names_in:
                layer.g[k] = dev_in[b][k]
            layer.O, layer.dX = dev_out[b]["O"], dev_out[b]["dX"]
            layer.step()
            computed[b].record(main)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(computed[b])
                for k in names_out:
                    host_out[b][k].copy_(dev_out[b][k], non_blocking=True)
                out_read[b].record(copy_out)
        main.wait_stream(copy_in)
        main.wait_stream(copy_out)

    run(max(args.warmup, 3))
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    run(args.steps)
    e1.record(main)
    torch.cuda.synchronize()
    for k in names_in:
        layer.g[k] = dev_in[0][k]
    layer.O, layer.dX = dev_out[0]["O"], dev_out[0]["dX"]
    ms = reduce_max(e0.elapsed_time(e1) / args.steps, world, dev)
    ff, fb = layer_flops(w)
    return {"value": weak_scaling_tflops(ff + fb, ms, world), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "note": "weights and weight gradients stay resident in HBM; activations cross C2C each step, "
                    "copies of step i+1 (in) and i (out) overlapped with step i's compute on a copy stream"}


def tr_vs_tc(args, dev):
    """Token rounding (under each rounding rule) and expert choice vs token choice on the high-sparsity layer
    (T=16384, d=1536, n=256, E=256, K=4)."""
    w = synth.WORKLOADS["sparse"]
    inp = synth.make_inputs(w, seed=0)
    out = {}
    for mode in ("tc", "tr", "tr_up", "tr_down", "tr_stoch", "ec"):
        layer = Layer(w, inp, mode, dev)
        for _ in range(3):
            layer.step()
        torch.cuda.synchronize()
        total, _ = time_steps(layer, max(args.steps, 20))
        ms = total / max(args.steps, 20)
        code, P = layer.rt.device_status()
        ff, fb = layer_flops(w)
        fa, fba = layer_flops(w, P)
        tc_counts = layer.rt.tc_counts.cpu().numpy()
        counts = layer.rt.counts.cpu().numpy()
        tiles = int(np.sum(-(-counts // 128)))
        out[mode] = {"ms_per_step": ms, "tflops_nominal_TK": (ff + fb) / (ms * 1e-3) / 1e12,
                     "tflops_actual_P": (fa + fba) / (ms * 1e-3) / 1e12, "P": P, "m_tiles": tiles,
                     "max_abs_count_deviation": int(np.abs(counts - tc_counts).max())}
        del layer
        torch.cuda.empty_cache()
    out["speedup_tr_over_tc"] = out["tc"]["ms_per_step"] / out["tr"]["ms_per_step"]
    out["speedup_over_tc"] = {m: out["tc"]["ms_per_step"] / out[m]["ms_per_step"]
                              for m in ("tr", "tr_up", "tr_down", "tr_stoch", "ec")}
    out["workload"] = f"sparse: T={w.T}, d={w.d}, n={w.n}, E={w.E}, K={w.K}"
    return out


def deterministic_timing(args, w, inp, ms_default, dev):
    """The same step with MOE_FLAG_DETERMINISTIC (fixed-point aggregation: bitwise-reproducible O, dX and dS)."""
    layer = Layer(w, inp, args.mode, dev, det=True)
    for _ in range(3):
        layer.step()
    torch.cuda.synchronize()
    n = max(args.steps, 20)
    total, _ = time_steps(layer, n)
    ms = total / n
    ff, fb = layer_flops(w)
    del layer
    torch.cuda.empty_cache()
    return {"ms_per_step": ms, "tflops": (ff + fb) / (ms * 1e-3) / 1e12, "slowdown_vs_default": ms / ms_default}


def a_from_h_timing(args, dev):
    """Forward with A kept on chip (the down-projection recomputes A = SwiGLU(H) from the cached H, A is never
    written) against the default forward that writes A and reads it back, on the metric's workload and on the
    high-sparsity one; whole steps (route + forward + backward) and the forward alone."""
    out = {}
    for name in dict.fromkeys((args.workload, "sparse")):
        w = synth.WORKLOADS[name]
        inp = synth.make_inputs(w, seed=0)
        res = {}
        for key, flag in (("default", False), ("a_from_h", True)):
            layer = Layer(w, inp, args.mode, dev, a_from_h=flag)
            for _ in range(3):
                layer.step()
            torch.cuda.synchronize()
            n = max(args.steps, 20)
            total, parts = time_steps(layer, n, split=True)
            ff, fb = layer_flops(w)
            res[key] = {"ms_per_step": total / n, "forward_ms": parts[1] / n,
                        "tflops": (ff + fb) / (total / n * 1e-3) / 1e12,
                        "forward_workspace_bytes": layer.wsf.numel()}
            del layer
            torch.cuda.empty_cache()
        res["step_speedup"] = res["default"]["ms_per_step"] / res["a_from_h"]["ms_per_step"]
        res["forward_speedup"] = res["default"]["forward_ms"] / res["a_from_h"]["forward_ms"]
        out[name] = res
    return out


def router_timing(args, dev):
    """The router either side of the layer on the metric's workload: logits = X W_r, then the gate backward
    (dz, dX += dz W_r^T, dW_r = X^T dz) on that workload's token-choice routing."""
    import fine_grained_mixture_gb300 as moe

    w = synth.WORKLOADS[args.workload]
    gen = torch.Generator().manual_seed(0)
    X = torch.randn((w.T, w.d), generator=gen).to(torch.bfloat16).to(dev)
    Wr = synth.make_router_weights(w.d, w.E, 0).to(dev)
    z = moe.moe_router_forward(X, Wr)
    rt = moe.moe_route(z, w.K, "tc")
    dS = synth.make_row_grads(rt.p_cap, 0).to(dev)
    dX = torch.zeros((w.T, w.d), dtype=torch.bfloat16, device=dev)
    dlogits = torch.empty((w.T, w.E), dtype=torch.float32, device=dev)
    dWr = torch.empty((w.d, w.E), dtype=torch.float32, device=dev)
    n = max(args.steps, 20)
    out = {}
    for name, fn in (("forward", lambda: moe.moe_router_forward(X, Wr, logits=z)),
                     ("backward", lambda: moe.moe_router_backward(dS, rt, z, X, Wr, dX, dlogits=dlogits, dWr=dWr))):
        for _ in range(3):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / n
        flops = 2.0 * w.T * w.d * w.E * (1 if name == "forward" else 2)
        out[name] = {"us": 1e3 * ms, "tflops": flops / (ms * 1e-3) / 1e12}
    out["workload"] = f"{w.name}: T={w.T}, d={w.d}, E={w.E}, K={w.K}"
    return out


if __name__ == "__main__":
    sys.exit(main())
