"""Benchmark of the row-reduction hot path on GB300.

One step = one pass of every hot-path operation over its synthetic workload:
  block tier    8192 x 8192 fp32 sum / max / min, int32 sum
  warp tier     1,048,576 x 32 fp32 sum / max / min
  tiled tier    1,048,576 x 8 fp32 sum / max / min
  split-K tier  16 x 16,777,216 fp32 sum / max (cluster size picked by the
                library: 16 on a 152-SM GB300)
  softmax       32768 x 4096 bf16 -> fp32
  layernorm     16384 x 8192 bf16 -> mean, rstd
  combine       P = 2, 4, 8 partials of 131072 x 128 fp32 -> bf16
Every operation has its own input buffer (its own seed), so within a step no
buffer is read twice and between two reads of a buffer the step moves about
5.6 GB, far more than the 129 MB L2.

value = algorithmic HBM bytes of all ranks' steps / max-over-ranks time
(GB/s, 1e9 bytes).  Algorithmic bytes per operation: input bytes read once
plus output bytes written once.

--impl reference times the CPU oracle on a bounded sample of the same
workload (the method has no other reference implementation to run).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (fraction of GB300 peak) per reduce tier and split-K combine"
WORKLOAD = ("row reductions: block 8192x8192 f32 sum/max/min + i32 sum; warp 1Mx32 f32 "
            "sum/max/min; tiled 1Mx8 f32 sum/max/min; split-K 16x16M f32 sum/max; softmax "
            "32768x4096 bf16->f32; layernorm stats 16384x8192 bf16; split-K combine "
            "P=2,4,8 x 131072x128")
# Reductions over a non-last axis timed beside the step ([outer, axis, inner],
# fp32, 256 MiB each): a column reduce, a middle axis, a narrow inner axis, a
# single long, narrow tile that needs the split workspace, and three
# interleaved channels (the slab form).
AXIS_WORKLOADS = [(1, 8192, 8192), (256, 1024, 256), (32768, 256, 8), (1, 1 << 22, 16),
                  (21845, 1024, 3)]
# Row reductions of medium width timed beside the step (fp32, 256 MiB each).
MEDIUM_ROWS = [(1 << 20, 64), (262144, 256), (65536, 1024), (671088, 100)]
# Softmax / layernorm rows of medium width timed beside the step (bf16,
# 256 MiB each): the warp tier of the two-pass row operations; 250-element
# rows (500 bytes) are not 16-byte aligned and take its chunked form;
# 4100-element rows (8200 bytes, every other row 8 bytes past a 16-byte
# boundary) take the block tier's register form read as 8-byte vectors.
MEDIUM_ROWOPS = [(1 << 20, 128), (131072, 1024), (65536, 2048), (536870, 250), (16384, 4100),
                 (16384, 4099)]
# Long rows timed beside the step (256 MiB each): softmax / layernorm rows
# staged in shared memory (a CTA per row; clusters of 8 for 256K-element
# rows), and a few long fp32 rows per SM for the block reduce.
LONG_ROWOPS = [(4096, 32768), (608, 262144)]
LONG_REDUCE = [(200, 335544)]
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes per full-size launch from ncu captures (dram__bytes_read.sum +
# dram__bytes_write.sum of one launch of `bench.py --case <op>`, scaled by
# the units the full workload has over the captured case), keyed by
# operation name, valid only while the kernel's sources (`src`: its
# translation unit and the device header) hash to `src_sha`.
# The captures and their commands are summarised in profiles/.  Softmax's
# figure is low because half of its output was still in L2 when the single
# captured launch ended.
NCU_TRAFFIC = {
    "splitk_sum_f32": {"bytes": 1084942336, "src": ["reduce.cu", "rr_device.cuh"],
                      "src_sha": "200d80f613a727b2", "profile": "profiles/k_splitk_sum_16x4M_f32.md"},
    "combine_p8": {"bytes": 566772736, "src": ["combine.cu", "rr_device.cuh"],
                  "src_sha": "68a1353cf0e06719", "profile": "profiles/k_combine_direct_p8_32768x128.md"},
    "softmax_bf16": {"bytes": 559710208, "src": ["rowwise.cu", "rowwise.cuh", "rr_device.cuh"],
                    "src_sha": "acc28fce14c4253a", "profile": "profiles/k_softmax_reg_8192x4096_bf16.md"},
    "block_sum_f32": {"bytes": 271227904, "src": ["reduce.cu", "rr_device.cuh"],
                     "src_sha": "200d80f613a727b2", "profile": "profiles/k_block_sum_8192x8192_f32.md"},
    "layernorm_bf16": {"bytes": 271349760, "src": ["rowwise.cu", "rowwise.cuh", "rr_device.cuh"],
                      "src_sha": "acc28fce14c4253a", "profile": "profiles/k_lnstats_reg_16384x8192_bf16.md"},
    "warp_sum_f32": {"bytes": 137803776, "src": ["reduce.cu", "rr_device.cuh"],
                    "src_sha": "200d80f613a727b2", "profile": "profiles/k_warp_vec_sum_1Mx32_f32.md"},
}


def op_specs():
    """(name, tier label, builder) for each operation of one step.  A builder
    returns (inputs, run, bytes_in, bytes_out, host_run)."""
    return [
        ("block_sum_f32", "block", dict(kind="reduce", rows=8192, cols=8192, dt="f32", op="sum", cfg=1, opi=0)),
        ("block_max_f32", "block", dict(kind="reduce", rows=8192, cols=8192, dt="f32", op="max", cfg=1, opi=1)),
        ("block_min_f32", "block", dict(kind="reduce", rows=8192, cols=8192, dt="f32", op="min", cfg=1, opi=2)),
        ("block_sum_i32", "block", dict(kind="reduce", rows=8192, cols=8192, dt="i32", op="sum", cfg=1, opi=3)),
        ("warp_sum_f32", "warp", dict(kind="reduce", rows=1 << 20, cols=32, dt="f32", op="sum", cfg=1, opi=4)),
        ("warp_max_f32", "warp", dict(kind="reduce", rows=1 << 20, cols=32, dt="f32", op="max", cfg=1, opi=5)),
        ("warp_min_f32", "warp", dict(kind="reduce", rows=1 << 20, cols=32, dt="f32", op="min", cfg=1, opi=6)),
        ("tiled_sum_f32", "tiled", dict(kind="reduce", rows=1 << 20, cols=8, dt="f32", op="sum", cfg=1, opi=7)),
        ("tiled_max_f32", "tiled", dict(kind="reduce", rows=1 << 20, cols=8, dt="f32", op="max", cfg=1, opi=8)),
        ("tiled_min_f32", "tiled", dict(kind="reduce", rows=1 << 20, cols=8, dt="f32", op="min", cfg=1, opi=9)),
        ("splitk_sum_f32", "splitk", dict(kind="reduce", rows=16, cols=1 << 24, dt="f32", op="sum", cfg=2, opi=0)),
        ("splitk_max_f32", "splitk", dict(kind="reduce", rows=16, cols=1 << 24, dt="f32", op="max", cfg=2, opi=1)),
        ("softmax_bf16", "softmax", dict(kind="softmax", rows=32768, cols=4096, cfg=3, opi=0)),
        ("layernorm_bf16", "layernorm", dict(kind="lnstats", rows=16384, cols=8192, cfg=3, opi=1)),
        ("combine_p2", "combine", dict(kind="combine", P=2, rows=131072, D=128, cfg=4, opi=2)),
        ("combine_p4", "combine", dict(kind="combine", P=4, rows=131072, D=128, cfg=4, opi=4)),
        ("combine_p8", "combine", dict(kind="combine", P=8, rows=131072, D=128, cfg=4, opi=8)),
    ]


def algorithmic_bytes(spec) -> tuple:
    k = spec["kind"]
    if k == "reduce":
        return spec["rows"] * spec["cols"] * 4, spec["rows"] * 4
    if k == "softmax":
        return spec["rows"] * spec["cols"] * 2, spec["rows"] * spec["cols"] * 4
    if k == "lnstats":
        return spec["rows"] * spec["cols"] * 2, spec["rows"] * 8
    if k == "combine":
        P, R, D = spec["P"], spec["rows"], spec["D"]
        return P * R * (D * 4 + 8), R * D * 2
    raise ValueError(k)


def make_inputs(spec, device):
    import torch
    from cluster_reductions_gb300 import inputs
    seed = inputs.seed_for(spec["cfg"], spec["opi"])
    k = spec["kind"]
    if k == "reduce":
        if spec["dt"] == "i32":
            return [inputs.uniform_i32(spec["rows"], spec["cols"], seed, device)]
        return [inputs.normal_f32(spec["rows"], spec["cols"], seed, device)]
    if k == "softmax":
        return [inputs.normal_bf16(spec["rows"], spec["cols"], seed, device, 3.0)]
    if k == "lnstats":
        return [inputs.normal_bf16(spec["rows"], spec["cols"], seed, device, 1.0)]
    if k == "combine":
        O, m, l, s = inputs.combine_partials(spec["P"], spec["rows"], spec["D"], seed, device)
        return [O, m, l, torch.tensor(s)]
    raise ValueError(k)


def make_outputs(spec, ins, device):
    import torch
    k = spec["kind"]
    if k == "reduce":
        return [torch.empty(spec["rows"], dtype=ins[0].dtype, device=device)]
    if k == "softmax":
        return [torch.empty((spec["rows"], spec["cols"]), dtype=torch.float32, device=device)]
    if k == "lnstats":
        return [torch.empty(spec["rows"], dtype=torch.float32, device=device),
                torch.empty(spec["rows"], dtype=torch.float32, device=device)]
    if k == "combine":
        return [torch.empty((spec["rows"], spec["D"]), dtype=torch.bfloat16, device=device)]
    raise ValueError(k)


def run_op(rr, spec, ins, outs):
    k = spec["kind"]
    if k == "reduce":
        return rr.reduce(ins[0], spec["op"], out=outs[0])
    if k == "softmax":
        return rr.softmax(ins[0], out=outs[0])
    if k == "lnstats":
        return rr.layernorm_stats(ins[0], 1e-5, mean=outs[0], rstd=outs[1])
    if k == "combine":
        return rr.splitk_combine(ins[0], ins[1], ins[2], float(ins[3]), out=outs[0])
    raise ValueError(k)


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------- helpers

def read_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_src_sha(files=None) -> str:
    """Hash of kernel sources under cluster_reductions_gb300/csrc: the named
    files (a kernel's translation unit and the device headers it includes),
    else every file.  Comments and whitespace are left out, so editing a
    comment does not orphan a traffic figure taken from the same code."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "cluster_reductions_gb300", "csrc")
    for f in sorted(files if files else os.listdir(d)):
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        h.update(f.encode() + "".join(text.split()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(name: str):
    """The NCU_TRAFFIC entry of operation `name` while its kernel sources
    still hash to the captured `src_sha`; None when there is none or the
    kernel has changed since the counters were taken."""
    tr = NCU_TRAFFIC.get(name)
    if tr and tr.get("src_sha") == kernel_src_sha(tr.get("src")):
        return tr
    return None


def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """Largest value over all ranks (the slowest rank's time)."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(step_bytes: int, steps: int, world: int, max_ms: float) -> float:
    """Whole-job throughput: every rank runs the full step (replicas, weak
    scaling), so the job moves world * step_bytes * steps bytes in the
    slowest rank's time."""
    return world * step_bytes * steps / (max_ms / 1e3) / 1e9


# --------------------------------------------------------------------- CPU oracle timing

def oracle_sample_plan(scale: float):
    """Samples of each operation for the oracle, `scale` of its elements:
    `scale` of the rows, or, where that is under one row (the 16-row
    split-K workload), one row cut to `scale` of the elements."""
    plan = []
    for name, tier, spec in op_specs():
        s = dict(spec)
        r = spec["rows"] * scale
        if r >= 1 or spec["kind"] == "combine":
            s["rows"] = max(1, int(round(r)))
        else:
            s["rows"] = 1
            s["cols"] = max(1, int(round(spec["cols"] * r)))
        plan.append((name, tier, spec, s))
    return plan


def oracle_inputs(plan):
    """Host inputs of the sampled rows (same generators, CPU)."""
    import numpy as np
    import torch
    from cluster_reductions_gb300 import inputs
    out = []
    for name, tier, full, s in plan:
        seed = inputs.seed_for(s["cfg"], s["opi"])
        k = s["kind"]
        if k == "reduce":
            x = (inputs.uniform_i32(s["rows"], s["cols"], seed) if s["dt"] == "i32"
                 else inputs.normal_f32(s["rows"], s["cols"], seed)).numpy()
            out.append((k, s, [x]))
        elif k in ("softmax", "lnstats"):
            x = inputs.normal_bf16(s["rows"], s["cols"], seed, "cpu",
                                   3.0 if k == "softmax" else 1.0)
            out.append((k, s, [x.view(torch.int16).numpy().view(np.uint16)]))
        else:
            O, m, l, sc = inputs.combine_partials(s["P"], s["rows"], s["D"], seed)
            out.append((k, s, [O.numpy(), m.numpy(), l.numpy(), sc]))
    return out


def run_oracle_step(data, threads: int):
    """One pass of the oracle over the sampled rows, row chunks spread over
    `threads` host threads (the oracle releases the GIL inside its C code)."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    def chunks(n):
        t = max(1, min(threads, n))
        b = [n * i // t for i in range(t + 1)]
        return [(b[i], b[i + 1]) for i in range(t) if b[i + 1] > b[i]]

    jobs = []
    for k, s, arrs in data:
        if k == "reduce":
            x = arrs[0]
            jobs += [(lambda a=a, b=b, x=x, op=s["op"]: oracle.reduce_rows(x[a:b], op))
                     for a, b in chunks(x.shape[0])]
        elif k == "softmax":
            x = arrs[0]
            jobs += [(lambda a=a, b=b, x=x: oracle.softmax(x[a:b])) for a, b in chunks(x.shape[0])]
        elif k == "lnstats":
            x = arrs[0]
            jobs += [(lambda a=a, b=b, x=x: oracle.layernorm_stats(x[a:b], 1e-5))
                     for a, b in chunks(x.shape[0])]
        else:
            O, m, l, sc = arrs
            jobs += [(lambda a=a, b=b, O=O, m=m, l=l, sc=sc:
                      oracle.splitk_combine(O[:, a:b], m[:, a:b], l[:, a:b], sc))
                     for a, b in chunks(O.shape[1])]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for f in [ex.submit(j) for j in jobs]:
            f.result()


def sample_bytes(data):
    tot = 0
    for k, s, _ in data:
        bi, bo = algorithmic_bytes(s)
        tot += bi + bo
    return tot


def calibrate_oracle(target_s: float, threads: int):
    """Pick the sample fraction whose oracle pass takes about target_s."""
    import oracle
    oracle.build()
    scale = 1.0 / 8192
    for _ in range(2):
        data = oracle_inputs(oracle_sample_plan(scale))
        t0 = time.perf_counter()
        run_oracle_step(data, threads)
        dt = max(time.perf_counter() - t0, 1e-4)
        scale = min(1.0, scale * target_s / dt)
    return scale


def cpu_baseline(target_s: float):
    """Oracle throughput on a bounded sample: `scale` of every operation's
    rows, repeated until about target_s seconds of CPU work have run (one
    pass of the whole workload is faster than that on a many-core host)."""
    threads = os.cpu_count() or 1
    scale = calibrate_oracle(target_s, threads)
    plan = oracle_sample_plan(scale)
    data = oracle_inputs(plan)
    passes, dt = 0, 0.0
    t0 = time.perf_counter()
    while passes == 0 or dt < target_s:
        run_oracle_step(data, threads)
        passes += 1
        dt = time.perf_counter() - t0
    b = sample_bytes(data)
    # one pass on a single thread beside it
    t1 = time.perf_counter()
    run_oracle_step(data, 1)
    dt1 = time.perf_counter() - t1
    return {"value": round(b * passes / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"every operation of the step on {scale:.2e} of its rows "
                      f"({b / 1e6:.1f} MB algorithmic per pass), {passes} passes, fp64 C oracle, "
                      f"{threads} host threads, {dt:.2f} s",
            "single_thread_value": round(b / dt1 / 1e9, 4),
            "single_thread_sample": f"one pass of the same sample on one thread, {dt1:.2f} s",
            "cpu_model": host_cpu_model()}


def host_cpu_model() -> str:
    """The host CPU's model name as lscpu reports it, else /proc/cpuinfo's."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


# --------------------------------------------------------------------- our arm

def bench_ours(args):
    import torch
    import cluster_reductions_gb300 as rr

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", torch.cuda.current_device())
    lib = rr.load()
    specs = op_specs()
    data = []
    for name, tier, spec in specs:
        ins = make_inputs(spec, dev)
        outs = make_outputs(spec, ins, dev)
        data.append((name, tier, spec, ins, outs))
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()

    def step():
        for name, tier, spec, ins, outs in data:
            run_op(rr, spec, ins, outs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    nops = len(data)
    # Per-operation breakdown (untimed pass before the timed region): CUDA
    # events around every launch.  An event record between two launches costs
    # the stream ~2 us of front-end time, so this pass is kept out of the
    # timed region; it also picks the dominant operation.
    prof_steps = max(3, min(20, args.steps))
    pev = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(nops)] for _ in range(prof_steps)]
    for s_ in range(prof_steps):
        for i, (name, tier, spec, ins, outs) in enumerate(data):
            pev[s_][i][0].record(stream)
            run_op(rr, spec, ins, outs)
            pev[s_][i][1].record(stream)
    torch.cuda.synchronize()
    op_ms = [statistics.fmean(pev[s_][i][0].elapsed_time(pev[s_][i][1])
                              for s_ in range(prof_steps)) for i in range(nops)]
    dom = max(range(nops), key=lambda i: op_ms[i])

    # timed region: K whole steps bracketed by barrier + synchronize; events
    # only around the dominant operation's launch in every step (its live
    # average launch duration for the roofline)
    dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(dev.index) as clk:
        t_start.record(stream)
        for s_ in range(args.steps):
            for i, (name, tier, spec, ins, outs) in enumerate(data):
                if i == dom:
                    dev_ev[s_][0].record(stream)
                    run_op(rr, spec, ins, outs)
                    dev_ev[s_][1].record(stream)
                else:
                    run_op(rr, spec, ins, outs)
        t_end.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = t_start.elapsed_time(t_end)
    elapsed_ms = max_over_ranks(elapsed_ms, world)
    dom_ms = statistics.fmean(a.elapsed_time(b) for a, b in dev_ev)

    step_bytes = sum(sum(algorithmic_bytes(spec)) for _, _, spec, _, _ in data)
    value = job_gbs(step_bytes, args.steps, world, elapsed_ms)
    peak, peak_kind = read_peak()

    tiers = {}
    for i, (name, tier, spec, ins, outs) in enumerate(data):
        bi, bo = algorithmic_bytes(spec)
        gbs = (bi + bo) / (op_ms[i] / 1e3) / 1e9
        tiers[name] = {"gbs": round(gbs, 1), "ms": round(op_ms[i], 4),
                       "frac_measured": round(gbs / peak, 4),
                       "frac_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                       "rows_per_s": round(spec["rows"] / (op_ms[i] / 1e3), 1)}
    # dominant kernel: largest share of the step time, timed live
    dname, _, dspec, _, _ = data[dom]
    dbytes = sum(algorithmic_bytes(dspec))
    achieved = dbytes / (dom_ms / 1e3) / 1e9
    tr = ncu_traffic(dname)
    traffic = tr["bytes"] if tr else None
    roofline = {"bound": "hbm", "kernel": dname, "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_kind": f"{peak_kind} copy bandwidth (read+write)",
                "traffic": traffic, "algorithmic_bytes": dbytes,
                "traffic_source": tr["profile"] if traffic is not None else None}

    splitk_c, combine_v, callreduce_us, rowwise_sk, axis_r, e2e = {}, {}, {}, {}, {}, None
    medium_r, long_r = {}, {}
    tiers_b2b = {}
    step_graph = None
    if not args.no_extras:
        def timed(fn, nbytes, reps=20):
            """Average device time per call of `reps` calls captured in one
            CUDA graph and replayed, so host launch overhead does not leave the
            GPU idle between short launches.  Short calls get more reps (a
            graph of at least ~0.5 ms at the copy bandwidth), so that the
            graph's own launch and its first, unoverlapped kernel do not
            weigh on a 36 MB call."""
            reps = max(reps, min(256, -(-int(0.5e-3 * peak * 1e9) // max(1, int(nbytes)))))
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="relaxed"):
                for _ in range(reps):
                    fn()
            graph.replay()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            graph.replay()
            b.record(stream)
            torch.cuda.synchronize()
            g = nbytes / (a.elapsed_time(b) / reps / 1e3) / 1e9
            r = {"gbs": round(g, 1), "frac_measured": round(g / peak, 4)}
            if g > 1.5 * peak:  # a launch that did not happen in the graph
                r["suspect"] = "above 1.5x the measured copy bandwidth"
            return r

        # the same step captured once as a CUDA graph and replayed: the 17
        # launches back to back with no host in the loop
        try:
            gstep = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gstep, capture_error_mode="relaxed"):
                step()
            gstep.replay()
            torch.cuda.synchronize()
            greps = max(20, min(200, args.steps))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for _ in range(greps):
                gstep.replay()
            b.record(stream)
            torch.cuda.synchronize()
            gms = a.elapsed_time(b) / greps
            step_graph = {"gbs": round(step_bytes / (gms / 1e3) / 1e9, 1),
                          "ms_per_step": round(gms, 4), "steps": greps,
                          "frac_measured": round(step_bytes / (gms / 1e3) / 1e9 / peak, 4)}
            del gstep
        except Exception as e:  # graph capture unavailable: report, do not fail
            step_graph = {"unavailable": str(e)[:200]}
        # every operation of the step alone, back to back: 10 launches in one
        # CUDA graph rotating over copies of its inputs (enough copies that
        # the set exceeds L2), so the figure is the kernel's own streaming
        # rate without the launch gaps and event records of the per-operation
        # pass above
        tiers_b2b = {}
        L2_BYTES = 128 << 20
        for name, tier, spec, ins, outs in data:
            bi, bo = algorithmic_bytes(spec)
            ncopy = max(1, min(8, -(-2 * L2_BYTES // bi)))
            sets = [(ins, outs)] + [([t.clone() for t in ins], [o.clone() for o in outs])
                                    for _ in range(ncopy - 1)]
            kk = [0]

            def one():
                kk[0] = (kk[0] + 1) % len(sets)
                run_op(rr, spec, sets[kk[0]][0], sets[kk[0]][1])
            tiers_b2b[name] = timed(one, bi + bo, reps=max(10, 2 * len(sets)))
            tiers_b2b[name]["input_copies"] = len(sets)
            del sets
        # split-K tier at every cluster size (same input, outside the step)
        x_sk = next(ins[0] for name, _, _, ins, _ in data if name == "splitk_sum_f32")
        out_sk = torch.empty(16, dtype=torch.float32, device=dev)
        for C in (2, 4, 8, 16):
            try:
                splitk_c[str(C)] = timed(lambda: rr.reduce(x_sk, "sum", tier="splitk",
                                                           cluster_size=C, out=out_sk),
                                         16 * (1 << 24) * 4 + 64)
            except rr.RRError as e:
                splitk_c[str(C)] = {"unsupported": str(e)}
        # every combine variant on the step's inputs: the cluster ones (pull:
        # DSMEM loads as on the page; push: copy-engine scatter) and direct
        for name, _, spec, ins, outs in data:
            if spec["kind"] != "combine":
                continue
            nbytes = sum(algorithmic_bytes(spec))
            for mode in ("pull", "push", "direct"):
                try:
                    combine_v[f"{name}_{mode}"] = timed(
                        lambda: rr.splitk_combine(ins[0], ins[1], ins[2], float(ins[3]),
                                                  out=outs[0], mode=mode), nbytes)
                except rr.RRError as e:
                    combine_v[f"{name}_{mode}"] = {"unsupported": str(e)}
        # multi-cluster split-K on two very long rows (2 x 128M fp32, 1 GiB)
        # against one cluster of 16 per row
        x2 = torch.randn((2, 1 << 27), device=dev)
        o2 = torch.empty(2, device=dev)
        ws2 = torch.empty(2 * 1024, dtype=torch.int32, device=dev)
        nb2 = 2 * (1 << 27) * 4 + 8
        try:
            splitk_c["2x128M_one_cluster_per_row"] = timed(
                lambda: rr.reduce(x2, "sum", tier="splitk", cluster_size=16, out=o2), nb2)
            splitk_c["2x128M_multi_cluster"] = timed(
                lambda: rr.reduce_splitk_multi(x2, "sum", out=o2, workspace=ws2), nb2)
        except rr.RRError as e:
            splitk_c["2x128M"] = {"unsupported": str(e)}
        del x2
        # split-K tier of the two-pass row ops (a few very long rows); eight
        # 32 MiB inputs in rotation so that each call reads from HBM
        from cluster_reductions_gb300 import inputs as _inp
        NR = 8
        xs = [_inp.normal_bf16(16, 1 << 20, 777 + i, dev, 3.0) for i in range(NR)]
        ys = [torch.empty((16, 1 << 20), dtype=torch.float32, device=dev) for _ in range(NR)]
        kk = [0]

        def nxt():
            kk[0] = (kk[0] + 1) % NR
            return kk[0]
        rowwise_sk["softmax_16x1M_bf16"] = timed(
            lambda: (lambda i: rr.softmax(xs[i], out=ys[i]))(nxt()), 16 * (1 << 20) * 6, reps=24)
        mu, rs = torch.empty(16, device=dev), torch.empty(16, device=dev)
        rowwise_sk["layernorm_16x1M_bf16"] = timed(
            lambda: rr.layernorm_stats(xs[nxt()], 1e-5, mean=mu, rstd=rs), 16 * (1 << 20) * 2 + 128,
            reps=24)
        _t, _w = rr.last_tier()
        rowwise_sk["tier"] = "%s %s=%d %s" % (_t, "G" if rr.last_form() == "grid" else "C", _w,
                                              rr.last_form())
        g16, b16 = _inp.layernorm_params(1 << 20, 778, dev)
        del ys
        yb = [torch.empty((16, 1 << 20), dtype=torch.bfloat16, device=dev) for _ in range(NR)]
        rowwise_sk["layernorm_rewrite_16x1M_bf16"] = timed(
            lambda: (lambda i: rr.layernorm(xs[i], g16, b16, 1e-5, out=yb[i]))(nxt()),
            16 * (1 << 20) * 4 + (1 << 20) * 8, reps=24)
        del xs, yb
        # the layernorm rewrite (statistics + y = (x - mean) rstd gamma + beta,
        # bf16 out) on the layernorm workload, block tier
        xl = _inp.normal_bf16(16384, 8192, 779, dev)
        gl, bl = _inp.layernorm_params(8192, 780, dev)
        yl = torch.empty((16384, 8192), dtype=torch.bfloat16, device=dev)
        rowwise_sk["layernorm_rewrite_16384x8192_bf16"] = timed(
            lambda: rr.layernorm(xl, gl, bl, 1e-5, out=yl), 16384 * 8192 * 4 + 8192 * 8)
        del xl, yl
        # rows of medium width (33 to 4095 elements, many rows): the warp tier
        # with a warp segment per row, automatic plan, two 256 MiB inputs
        for mr, mc in MEDIUM_ROWS:
            xm = [_inp.normal_f32(mr, mc, 810 + i, dev) for i in range(2)]
            om = torch.empty(mr, device=dev)
            km = [0]

            def one_m():
                km[0] ^= 1
                rr.reduce(xm[km[0]], "sum", out=om)
            medium_r[f"{mr}x{mc}_sum_f32"] = timed(one_m, mr * mc * 4 + mr * 4)
            medium_r[f"{mr}x{mc}_sum_f32"]["tier"] = "%s C=%d" % rr.last_tier()
            del xm
        for mr, mc in MEDIUM_ROWOPS:
            xm = [_inp.normal_bf16(mr, mc, 820 + i, dev, 3.0) for i in range(2)]
            ym = torch.empty((mr, mc), device=dev)
            yb = torch.empty((mr, mc), dtype=torch.bfloat16, device=dev)
            mu, rs = torch.empty(mr, device=dev), torch.empty(mr, device=dev)
            gm, bm = _inp.layernorm_params(mc, 822, dev)
            km = [0]
            ops = {
                "softmax": (lambda x: rr.softmax(x, out=ym), mr * mc * 6),
                "lnstats": (lambda x: rr.layernorm_stats(x, 1e-5, mean=mu, rstd=rs),
                            mr * mc * 2 + mr * 8),
                "layernorm": (lambda x: rr.layernorm(x, gm, bm, 1e-5, out=yb),
                              mr * mc * 4 + mc * 8),
            }
            for name, (fn, nb) in ops.items():
                def one_r(fn=fn):
                    km[0] ^= 1
                    fn(xm[km[0]])
                key = f"{mr}x{mc}_{name}_bf16"
                medium_r[key] = timed(one_r, nb)
                t, c = rr.last_tier()
                fm = rr.last_form()
                medium_r[key]["tier"] = (f"{t} {'L' if t == 'warp' else 'C'}={c}"
                                         + ("" if fm == "direct" else " " + fm))
            del xm, ym, yb
        for mr, mc in LONG_ROWOPS:
            xm = [_inp.normal_bf16(mr, mc, 830 + i, dev, 3.0) for i in range(2)]
            ym = torch.empty((mr, mc), device=dev)
            yb = torch.empty((mr, mc), dtype=torch.bfloat16, device=dev)
            mu, rs = torch.empty(mr, device=dev), torch.empty(mr, device=dev)
            gm, bm = _inp.layernorm_params(mc, 832, dev)
            km = [0]
            ops = {
                "softmax": (lambda x: rr.softmax(x, out=ym), mr * mc * 6),
                "lnstats": (lambda x: rr.layernorm_stats(x, 1e-5, mean=mu, rstd=rs),
                            mr * mc * 2 + mr * 8),
                "layernorm": (lambda x: rr.layernorm(x, gm, bm, 1e-5, out=yb),
                              mr * mc * 4 + mc * 8),
            }
            for name, (fn, nb) in ops.items():
                def one_l(fn=fn):
                    km[0] ^= 1
                    fn(xm[km[0]])
                key = f"{mr}x{mc}_{name}_bf16"
                long_r[key] = timed(one_l, nb)
                t, c = rr.last_tier()
                fm = rr.last_form()
                long_r[key]["tier"] = f"{t} C={c}" + ("" if fm == "direct" else " " + fm)
            del xm, ym, yb
        for mr, mc in LONG_REDUCE:
            xm = [_inp.normal_f32(mr, mc, 840 + i, dev) for i in range(2)]
            om = torch.empty(mr, device=dev)
            km = [0]

            def one_lr():
                km[0] ^= 1
                rr.reduce(xm[km[0]], "sum", out=om)
            long_r[f"{mr}x{mc}_sum_f32"] = timed(one_lr, mr * mc * 4 + mr * 4)
            long_r[f"{mr}x{mc}_sum_f32"]["tier"] = "%s C=%d" % rr.last_tier()
            del xm
        # reduction over a non-last axis (automatic plan), 256 MiB inputs, two
        # rotating buffers; called straight through the C ABI so that host
        # overhead does not starve the ~40 us launches
        for shape in AXIS_WORKLOADS:
            outer, axis_n, inner = shape
            key = "x".join(map(str, shape))
            xa = [_inp.normal_f32(outer * axis_n, inner, 790 + i, dev) for i in range(2)]
            oa = torch.empty((outer, inner), device=dev)
            need = ctypes.c_size_t(0)
            rr.check(lib.rr_reduce_axis_workspace_size(outer, axis_n, inner, 16,
                                                        ctypes.byref(need)), "workspace size")
            wsa = torch.empty(max(1, need.value // 4), dtype=torch.int32, device=dev)
            opts = rr._lib.rr_axis_opts(0, 0, 0, 0, 0, wsa.data_ptr(), wsa.numel() * 4)
            nb = outer * axis_n * inner * 4 + outer * inner * 4
            for opname, opc in (("sum", 0), ("max", 1)):
                calls = [(t.data_ptr(), outer, axis_n, inner, opc, 0, oa.data_ptr()) for t in xa]
                k = [0]

                def one():
                    # the stream current at the call: the capture stream
                    # while the timing graph is being recorded
                    k[0] ^= 1
                    cur = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
                    rr.check(lib.rr_reduce_axis_ex(*calls[k[0]], cur, ctypes.byref(opts)),
                             "rr_reduce_axis_ex")
                axis_r[f"{key}_{opname}_f32"] = timed(one, nb)
            t, c = rr.last_tier()
            axis_r[f"{key}_plan"] = {"tier": t, "cluster_size": c,
                                     "workspace_bytes": need.value}
            del xa
        # the cluster all-reduce primitive alone: one cluster, 4096 back-to-back
        # combines of one fp32 per CTA, with the tail sync and with two slots
        for C in (2, 4, 8, 16):
            vals = torch.randn((4096, 1, C, 1), device=dev)
            res = torch.empty_like(vals)
            for two in (False, True):
                key = f"C{C}_{'two_slot' if two else 'tail_sync'}_us"
                try:
                    for _ in range(2):
                        rr.cluster_allreduce(vals, "sum", two_slot=two, res=res)
                    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    a.record(stream)
                    rr.cluster_allreduce(vals, "sum", two_slot=two, res=res)
                    b.record(stream)
                    torch.cuda.synchronize()
                    callreduce_us[key] = round(a.elapsed_time(b) * 1e3 / 4096, 3)
                except rr.RRError as e:
                    callreduce_us[key] = str(e)
        e2e = bench_e2e(args, rr, data, dev, stream, world)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "l2": "inputs larger than L2: every operation reads its own buffer once "
                         "per step; a step moves %.2f GB" % (step_bytes / 1e9),
                   "parallelism": f"replicas x{world}", "step_bytes": step_bytes},
        "tiers": tiers, "tiers_back_to_back": tiers_b2b, "splitk_by_cluster": splitk_c, "combine_variants": combine_v,
        "cluster_allreduce_latency": callreduce_us, "rowwise_splitk": rowwise_sk,
        "axis_reduce": axis_r, "medium_rows": medium_r, "long_rows": long_r,
        "step_graph": step_graph,
        "roofline": roofline,
        "clocks": clk.summary(), "gpu_launches": nops * args.steps, "e2e": e2e,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    # last key of the line: every measured fraction of the copy bandwidth in
    # one short object, so that a reader who keeps only the line's tail
    # still sees them all
    line["frac_summary"] = frac_summary(line)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def frac_summary(line) -> dict:
    """{section: "name=frac ..."}: the fraction of the measured copy
    bandwidth of every operation timed back to back and of the extras, in
    one short object (names shortened: "ln" = layernorm, dtype suffixes
    dropped, fractions to two decimals)."""
    out = {"step": round(line["value"] / line["roofline"]["peak"], 3)}
    for sec, short in (("tiers_back_to_back", "b2b"), ("rowwise_splitk", "rowops_split"),
                       ("long_rows", "long_rows"), ("medium_rows", "medium_rows"),
                       ("combine_variants", "combine"), ("splitk_by_cluster", "splitk_C"),
                       ("axis_reduce", "axis")):
        d = line.get(sec) or {}
        vals = []
        for k, v in d.items():
            if not (isinstance(v, dict) and "frac_measured" in v):
                continue
            if sec == "axis_reduce" and not k.endswith("_sum_f32"):
                continue
            kk = (k.replace("_bf16", "").replace("_f32", "").replace("layernorm", "ln")
                  .replace("combine_", "").replace("_sum", "") if sec != "tiers_back_to_back"
                  else k.replace("_f32", "").replace("_bf16", "").replace("layernorm", "ln"))
            vals.append(f"{kk}={v['frac_measured']:.2f}".replace("=0.", "=.").replace("=1.", "=1."))
        if vals:
            out[short] = " ".join(vals)
    return out


def bench_e2e(args, rr, data, dev, stream, world):
    """The same step through the public API with pinned host buffers: every
    call takes its inputs from host memory and writes its results to host
    memory, so each step's host -> device copies of the inputs and device ->
    host copies of the results (staged by the binding) are inside the timed
    region.  The 17 calls alternate between two CUDA streams, so one call's
    results travel back while the next call's inputs travel in."""
    import torch
    host_in, host_out, h2d, d2h = [], [], 0, 0
    for name, tier, spec, ins, outs in data:
        hi = []
        for t in ins:
            if t.dim() == 0:
                hi.append(t.cpu())
                continue
            h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
            h.copy_(t)
            hi.append(h)
            h2d += t.numel() * t.element_size()
        host_in.append(hi)
        host_out.append([torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs])
        d2h += sum(o.numel() * o.element_size() for o in outs)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]

    def step():
        for i, (name, tier, spec, ins, outs) in enumerate(data):
            with torch.cuda.stream(streams[i % 2]):
                run_op(rr, spec, host_in[i], host_out[i])

    steps = max(3, min(args.steps, args.e2e_steps))
    step()
    torch.cuda.synchronize()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for s_ in streams:
        s_.wait_event(a)
    for _ in range(steps):
        step()
    for s_ in streams:
        stream.wait_stream(s_)
    b.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms = max_over_ranks(a.elapsed_time(b), world)
    step_bytes = sum(sum(algorithmic_bytes(spec)) for _, _, spec, _, _ in data)
    return {"value": round(job_gbs(step_bytes, steps, world, ms), 2), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "ms_per_step": round(ms / steps, 3),
            "path": "public Python API with pinned host tensors in and out, two streams"}


# --------------------------------------------------------------------- reference arm

def bench_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    budget = max(0.02, min(1.0, 150.0 / max(1, args.steps + args.warmup)))
    scale = calibrate_oracle(budget, threads)
    plan = oracle_sample_plan(scale)
    data = oracle_inputs(plan)
    for _ in range(args.warmup):
        run_oracle_step(data, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run_oracle_step(data, threads)
    dt = time.perf_counter() - t0
    b = sample_bytes(data)
    value = b * args.steps / dt / 1e9
    sample = (f"every operation of the step on {scale:.2e} of its rows ({b / 1e6:.2f} MB "
              f"algorithmic per step), fp64 C oracle, {threads} host threads")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# Workloads for ncu captures: the step's operation with fewer rows (or
# columns) where the full one is large, every input still larger than L2
# except the tiled tier's, which is the full workload.  `scale` = full-size
# units / case units, to scale a captured per-launch DRAM traffic.
PROFILE_CASES = {
    "block_sum_f32": ({}, None, 1.0),
    "warp_sum_f32": ({}, None, 1.0),
    "tiled_sum_f32": ({}, None, 1.0),
    "splitk_sum_f32": ({"cols": 1 << 22}, None, 4.0),
    "softmax_bf16": ({"rows": 8192}, None, 4.0),
    "layernorm_bf16": ({}, None, 1.0),
    "combine_p8": ({"rows": 32768}, None, 4.0),
    "combine_p8_pull": ({"rows": 32768}, "pull", 4.0),
    "combine_p8_push": ({"rows": 32768}, "push", 4.0),
    # reductions over a non-last axis, [outer, axis, inner], automatic plan
    "axis_256x1024x256": ({"shape": (256, 1024, 256)}, "axis", 1.0),
    "axis_32768x256x8": ({"shape": (32768, 256, 8)}, "axis", 1.0),
    "axis_1x8192x8192": ({"shape": (1, 8192, 8192)}, "axis", 1.0),
    "axis_1x4194304x16": ({"shape": (1, 1 << 22, 16)}, "axis", 1.0),
    "axis_21845x1024x3": ({"shape": (21845, 1024, 3)}, "axis", 1.0),
    # rows of medium width (the warp-segment kernels), automatic plan
    "medium_sum_1048576x64_f32": ({"shape": (1 << 20, 64), "op": "sum"}, "medium", 1.0),
    "medium_softmax_131072x1024_bf16": ({"shape": (131072, 1024), "op": "softmax"}, "medium", 1.0),
    "medium_layernorm_131072x1024_bf16": ({"shape": (131072, 1024), "op": "layernorm"},
                                          "medium", 1.0),
    "medium_layernorm_536870x250_bf16": ({"shape": (536870, 250), "op": "layernorm"},
                                         "medium", 1.0),
    # long rows staged in shared memory, automatic plan
    "long_softmax_4096x32768_bf16": ({"shape": (4096, 32768), "op": "softmax"}, "medium", 1.0),
    "long_layernorm_2048x65536_bf16": ({"shape": (2048, 65536), "op": "layernorm"}, "medium", 1.0),
    "long_lnstats_608x262144_bf16": ({"shape": (608, 262144), "op": "lnstats"}, "medium", 1.0),
    "long_lnstats_4096x32768_bf16": ({"shape": (4096, 32768), "op": "lnstats"}, "medium", 1.0),
    # a few long rows: the row ops' split-K tier
    "rowsk_softmax_16x1048576_bf16": ({"shape": (16, 1 << 20), "op": "softmax"}, "medium", 1.0),
    "rowsk_lnstats_16x1048576_bf16": ({"shape": (16, 1 << 20), "op": "lnstats"}, "medium", 1.0),
    "rowsk_layernorm_16x1048576_bf16": ({"shape": (16, 1 << 20), "op": "layernorm"}, "medium", 1.0),
    "tiled_max_f32": ({}, None, 1.0),
    "long_softmax_608x262144_bf16": ({"shape": (608, 262144), "op": "softmax"}, "medium", 1.0),
    "long_layernorm_608x262144_bf16": ({"shape": (608, 262144), "op": "layernorm"}, "medium", 1.0),
    "ring_lnstats_8192x16392_bf16": ({"shape": (8192, 16392), "op": "lnstats"}, "medium", 1.0),
    "rowsk_lnstats_32x524288_bf16": ({"shape": (32, 1 << 19), "op": "lnstats"}, "medium", 1.0),
    # rows 8-byte but not 16-byte aligned: the register form read as 8-byte vectors
    "medium_layernorm_16384x4100_bf16": ({"shape": (16384, 4100), "op": "layernorm"}, "medium", 1.0),
    # odd widths: the chunked register form (head + vectors + tail)
    "medium_lnstats_16384x4099_bf16": ({"shape": (16384, 4099), "op": "lnstats"}, "medium", 1.0),
    "medium_layernorm_16384x4099_bf16": ({"shape": (16384, 4099), "op": "layernorm"}, "medium", 1.0),
    "medium_softmax_16384x4099_bf16": ({"shape": (16384, 4099), "op": "softmax"}, "medium", 1.0),
}


def run_case(args):
    import torch
    import cluster_reductions_gb300 as rr
    torch.cuda.set_device(0)
    rr.load()
    over, mode, scale = PROFILE_CASES[args.case]
    if mode == "axis":
        from cluster_reductions_gb300 import inputs
        outer, axis_n, inner = over["shape"]
        x = inputs.normal_f32(outer * axis_n, inner, inputs.seed_for(5, 0), "cuda")
        x = x.view(outer, axis_n, inner)
        o = torch.empty((outer, inner), device="cuda")
        torch.cuda.synchronize()
        for _ in range(args.steps):
            rr.reduce_axis(x, "sum", 1, out=o)
        torch.cuda.synchronize()
        print(json.dumps({"case": args.case, "launches": args.steps,
                          "algorithmic_bytes": (outer * axis_n * inner + outer * inner) * 4,
                          "plan": rr.last_tier(), "scale_to_full": scale,
                          "status": rr.device_status()}), flush=True)
        return
    if mode == "medium":
        from cluster_reductions_gb300 import inputs
        r, c = over["shape"]
        op = over["op"]
        if op == "sum":
            x = inputs.normal_f32(r, c, inputs.seed_for(5, 1), "cuda")
            o = torch.empty(r, device="cuda")
            fn, nb = (lambda: rr.reduce(x, "sum", out=o)), r * c * 4 + r * 4
        elif op == "softmax":
            x = inputs.normal_bf16(r, c, inputs.seed_for(5, 2), "cuda", 3.0)
            y = torch.empty((r, c), device="cuda")
            fn, nb = (lambda: rr.softmax(x, out=y)), r * c * 6
        elif op == "lnstats":
            x = inputs.normal_bf16(r, c, inputs.seed_for(5, 3), "cuda")
            mu, rs = torch.empty(r, device="cuda"), torch.empty(r, device="cuda")
            fn, nb = (lambda: rr.layernorm_stats(x, 1e-5, mean=mu, rstd=rs)), r * c * 2 + r * 8
        else:
            x = inputs.normal_bf16(r, c, inputs.seed_for(5, 3), "cuda")
            g, b = inputs.layernorm_params(c, inputs.seed_for(5, 4), "cuda")
            yb = torch.empty((r, c), dtype=torch.bfloat16, device="cuda")
            fn, nb = (lambda: rr.layernorm(x, g, b, 1e-5, out=yb)), r * c * 4 + c * 8
        torch.cuda.synchronize()
        for _ in range(args.steps):
            fn()
        torch.cuda.synchronize()
        print(json.dumps({"case": args.case, "launches": args.steps, "algorithmic_bytes": nb,
                          "plan": rr.last_tier(), "scale_to_full": scale,
                          "status": rr.device_status()}), flush=True)
        return
    base = args.case.replace("_pull", "").replace("_push", "")
    spec = dict(next(s for n, _, s in op_specs() if n == base))
    spec.update(over)
    dev = torch.device("cuda", 0)
    ins = make_inputs(spec, dev)
    outs = make_outputs(spec, ins, dev)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        if mode:
            rr.splitk_combine(ins[0], ins[1], ins[2], float(ins[3]), out=outs[0], mode=mode)
        else:
            run_op(rr, spec, ins, outs)
    torch.cuda.synchronize()
    bi, bo = algorithmic_bytes(spec)
    print(json.dumps({"case": args.case, "launches": args.steps, "algorithmic_bytes": bi + bo,
                      "scale_to_full": scale, "status": rr.device_status()}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="time only the steps (no per-cluster-size, per-variant or e2e passes), "
                         "e.g. for an ncu launch list of exactly the step's kernels")
    ap.add_argument("--case", default=None,
                    help="run one operation of the step on a workload sized for an ncu capture "
                         "(larger than L2, a few hundred MB) --steps times, and exit; one of "
                         + ", ".join(PROFILE_CASES))
    args = ap.parse_args()
    if args.case:
        if args.case not in PROFILE_CASES:
            ap.error(f"--case must be one of {', '.join(PROFILE_CASES)}")
        return run_case(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        bench_reference(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
