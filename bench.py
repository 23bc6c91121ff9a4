"""Benchmark of the W8A8 group-scaled quantized linear layer on GB300.

One step = one pass of the whole hot path over the decode-shaped dense
workload: for each token count M in {1, 8, 32} (K=8192, N=28672, BF16 out),
per-token activation quantization followed by the group-scaled INT8 GEMM, as
one library call per shape (w8a8_linear: the quantizer writes the GEMM's
operand into the workspace, then the GEMM runs).
Each GEMM of the step reads its own 235 MB weight copy, so every input is
larger than L2 and no weight bytes are reused from L2 between GEMMs.

Metric: INT8 TOPS = sum of 2*M*N*K over the step / step time (whole job over
all ranks). The dominant kernel is the GEMM (the CUDA-core batched GEMV for
M = 1, the tcgen05 narrow-tile kernel with K split for M = 8 and 32), HBM-bound at these shapes:
the roofline object reports its algorithmic bytes per launch (int8 weights,
FP32 group scales, int8 activations and scales, BF16 output) over its measured
launch duration, against the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --workload prefill|stress|moe|tiny    (other shapes, same line format)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

KERNEL_TIME_NOTE = ("per shape: its quantizer + GEMM replayed back to back K times, events "
                    "around the K launches; the GEMM overlaps the quantizer, so this includes "
                    "any part of the quantizer it does not hide")
METRIC = "INT8 TOPS & % of roofline (tensor peak or HBM GB/s) per GEMM shape, 1xGB300"
GROUP = 128


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def gemm_source_hash() -> str:
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh", "quant_math.cuh"):
        with open(os.path.join(ROOT, "moe_gemm_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per GEMM launch from an ncu capture, if it was taken on the
    current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "gemm_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload)
    if not rec or rec.get("kernel_source_hash") != gemm_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


# ------------------------------------------------------------ workloads
class Shape:
    def __init__(self, M, N, K, out, act_spec, E=1, offsets=None):
        self.M, self.N, self.K, self.out = M, N, K, out
        self.act_spec = act_spec
        self.E = E
        self.offsets = offsets

    @property
    def ops(self):
        return 2 * self.M * self.N * self.K

    def alg_bytes(self, active_experts=None):
        """Bytes the method must move per GEMM launch: weights and group
        scales (active experts only), int8 activations + scales, output."""
        G = self.K // GROUP
        e = self.E if active_experts is None else active_experts
        w = e * self.N * self.K + e * self.N * G * 4
        a = self.M * self.K + self.M * 4
        y = self.M * self.N * (2 if self.out == "bf16" else 4)
        return w + a + y


def build_workload(name):
    """Returns (description, [Shape], weight spec, kind)."""
    if name == "decode":
        shapes = [Shape(m, 28672, 8192, "bf16", workloads.DENSE[f"decode_m{m}"])
                  for m in workloads.DECODE_MS]
        desc = "decode-shaped dense: M in {1,8,32}, K=8192, N=28672, BF16 out"
        return desc, shapes, workloads.DENSE["decode_m32"], "hbm"
    if name in ("tiny", "prefill", "stress"):
        s = workloads.DENSE[name]
        desc = {"tiny": "dense tiny: M=16, K=1024, N=1024, FP32 out",
                "prefill": "prefill-shaped dense: M=4096, K=8192, N=8192, BF16 out",
                "stress": "large stress: M=8192, K=16384, N=16384, FP32 out"}[name]
        return desc, [Shape(s.M, s.N, s.K, s.out_dtype, s)], s, (
            "hbm" if name == "tiny" else "tensor")
    if name == "moe":
        spec = workloads.MOE["moe"]
        route = workloads.routing(spec)
        desc = ("MoE grouped: 64 experts, top-8 of T=512 (R=4096 rows), gate_up N=3072 K=4096 "
                "and down N=4096 K=1536, BF16 out")
        shapes = [Shape(spec.R, spec.N_up, spec.K_up, "bf16", ("up", spec, route), spec.E,
                        route.offsets),
                  Shape(spec.R, spec.N_down, spec.K_down, "bf16", ("down", spec, route), spec.E,
                        route.offsets)]
        return desc, shapes, spec, "hbm"
    raise SystemExit(f"unknown workload {name}")


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ------------------------------------------------------ cross-rank timing
def slowest_rank_ms(ms, world, device=None):
    """The largest of the ranks' times (the job ends with its slowest rank).
    Needs an initialised process group when world > 1 (nccl: a CUDA device;
    gloo: the CPU)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tops(ops_per_step, steps, world, ms):
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return ops_per_step * steps * world / (ms * 1e-3) / 1e12


# -------------------------------------------------------------- ours (GPU)
def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    import __graft_entry__
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
    import moe_gemm_gb300 as w8
    dev = torch.device("cuda", local_rank)
    peaks = load_peaks()
    desc, shapes, wspec, bound = build_workload(args.workload)

    # ---- resident inputs (weights quantized on the GPU, offline step)
    def upload_bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(
            torch.bfloat16)

    per = []
    if args.workload == "moe":
        spec = wspec
        for shp in shapes:
            which, _, route = shp.act_spec
            N, K = shp.N, shp.K
            qw = torch.empty((spec.E, N, K), dtype=torch.int8, device=dev)
            sw = torch.empty((spec.E, N, K // GROUP), dtype=torch.float32, device=dev)
            for e in range(spec.E):
                q, s = w8.quant_weight(torch.from_numpy(
                    workloads.moe_weights(spec, which, e)).to(dev))
                qw[e].copy_(q)
                sw[e].copy_(s)
            a_host = workloads.moe_activations(spec, which, route)
            per.append(dict(shape=shp, qw=qw, sw=sw, a=upload_bf16(a_host), a_host=a_host,
                            off=torch.from_numpy(route.offsets).to(dev)))
    else:
        K, N = shapes[0].K, shapes[0].N
        qw0 = torch.empty((N, K), dtype=torch.int8, device=dev)
        sw0 = torch.empty((N, K // GROUP), dtype=torch.float32, device=dev)
        for r0, wb in workloads.weight_blocks(wspec, block_rows=4096):
            q, s = w8.quant_weight(torch.from_numpy(wb).to(dev))
            qw0[r0:r0 + wb.shape[0]].copy_(q)
            sw0[r0:r0 + wb.shape[0]].copy_(s)
        for i, shp in enumerate(shapes):
            a_host = workloads.activations(shp.act_spec)
            qw = qw0 if i == 0 else qw0.clone()     # a weight copy per GEMM of the step
            sw = sw0 if i == 0 else sw0.clone()
            per.append(dict(shape=shp, qw=qw, sw=sw, a=upload_bf16(a_host), a_host=a_host,
                            off=None))
    for d in per:
        shp = d["shape"]
        odt = torch.bfloat16 if shp.out == "bf16" else torch.float32
        d["y"] = torch.empty((shp.M, shp.N), dtype=odt, device=dev)
        wsz = (w8.grouped_linear_workspace_size(shp.M, shp.E, shp.N, shp.K)
               if d["off"] is not None else w8.linear_workspace_size(shp.M, shp.N, shp.K))
        d["ws"] = torch.empty(max(wsz, 1), dtype=torch.uint8, device=dev)
        # one public call per shape: the quantizer (writing the GEMM's operand
        # into the workspace) and the GEMM; for <= 4 dense rows whose codes fit
        # beside the GEMV's stages, the GEMV quantizes them itself (one kernel)
        mr = 1 if shp.M <= 1 else (2 if shp.M <= 2 else 4)
        fused = d["off"] is None and shp.M <= 4 and shp.K * mr <= 96 * 1024
        d["launches"] = 1 if fused else 2
    torch.cuda.synchronize()

    def linear_call(d, s=None):
        s = stream if s is None else s
        if d["off"] is not None:
            w8.grouped_linear(d["a"], d["off"], d["qw"], d["sw"], out=d["y"],
                              out_dtype=d["y"].dtype, workspace=d["ws"], stream=s)
        else:
            w8.linear(d["a"], d["qw"], d["sw"], out=d["y"], out_dtype=d["y"].dtype,
                      workspace=d["ws"], stream=s)

    def shape_call(d):
        linear_call(d)

    def step():
        for d in per:
            shape_call(d)

    # The step runs as one CUDA graph (quantizer, staging/reset kernel and
    # GEMM of every shape, with their programmatic-dependent-launch edges),
    # replayed once per step: the launches a serving loop would capture.
    stream = torch.cuda.Stream(device=dev)
    graphs = not args.no_graph

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            fn()                       # eager pass on the capture stream first
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                fn()
        torch.cuda.synchronize()
        return g

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if graphs:
        g_step = capture(step)
        run_step = g_step.replay
        g_shape = [capture(lambda d=d: shape_call(d)) for d in per]
        run_shape = [g.replay for g in g_shape]
    else:
        run_step = step
        run_shape = [lambda d=d: shape_call(d) for d in per]
    with torch.cuda.stream(stream):
        for _ in range(3):
            run_step()
    torch.cuda.synchronize()

    # ---- the timed region (CUDA events on the launching stream)
    sampler = ClockSampler(local_rank) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for k in range(args.steps):
            run_step()
        t1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    elapsed_ms = t0.elapsed_time(t1)

    # ---- per-shape launch time (roofline): each shape's quantizer + GEMM
    # replayed K times back to back, timed with events around the K launches
    # (an event between two launches would cut their programmatic overlap).
    gemm_ms = []
    with torch.cuda.stream(stream):
        for i in range(len(per)):
            for _ in range(3):
                run_shape[i]()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(args.steps):
                run_shape[i]()
            s1.record(stream)
            s1.synchronize()
            gemm_ms.append(s0.elapsed_time(s1) / args.steps)

    # ---- the quantizer alone (step a1, HBM-bound: 2 B read + 1 B written per
    # element + 4 B per row), per shape, the same way
    quant_ms = []
    qbufs = [(torch.empty((d["shape"].M, d["shape"].K), dtype=torch.int8, device=dev),
              torch.empty((d["shape"].M,), dtype=torch.float32, device=dev)) for d in per]

    def quant_call(i):
        w8.quant_act(per[i]["a"], qa=qbufs[i][0], sa=qbufs[i][1], stream=stream)

    run_quant = ([capture(lambda i=i: quant_call(i)).replay for i in range(len(per))]
                 if graphs else [lambda i=i: quant_call(i) for i in range(len(per))])
    with torch.cuda.stream(stream):
        for i in range(len(per)):
            for _ in range(3):
                run_quant[i]()
            s0 = torch.cuda.Event(enable_timing=True)
            s1 = torch.cuda.Event(enable_timing=True)
            s0.record(stream)
            for _ in range(args.steps):
                run_quant[i]()
            s1.record(stream)
            s1.synchronize()
            quant_ms.append(s0.elapsed_time(s1) / args.steps)
    # Keep the same step running ~1 s more so the clock sampler sees the load
    # even when the timed region itself is shorter than its sampling period.
    if sampler:
        hold_end = time.time() + 1.0
        with torch.cuda.stream(stream):
            while time.time() < hold_end:
                for _ in range(50):
                    run_step()
                stream.synchronize()
        clocks = sampler.stop()
        clocks["note"] = "sampled every 50 ms over the timed region and a 1 s hold of the same step"
    elapsed_ms = slowest_rank_ms(elapsed_ms, world, dev)

    ops_step = sum(d["shape"].ops for d in per)
    value = job_tops(ops_step, args.steps, world, elapsed_ms)

    # ---- end to end through the public API with host buffers (rank-local)
    e2e = None
    if not args.no_e2e:
        host_in = [torch.from_numpy(np.ascontiguousarray(d["a_host"]).view(np.int16)).view(
            torch.bfloat16).pin_memory() for d in per]
        host_out = [torch.empty(d["y"].shape, dtype=d["y"].dtype).pin_memory() for d in per]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = sum(t.numel() * t.element_size() for t in host_out)

        cur = torch.cuda.current_stream()

        def e2e_step():
            for d, hi, ho in zip(per, host_in, host_out):
                d["a"].copy_(hi, non_blocking=True)
                linear_call(d, cur)
                ho.copy_(d["y"], non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(args.steps):
            e2e_step()
        e1.record(cur)
        torch.cuda.synchronize()
        ems = slowest_rank_ms(e0.elapsed_time(e1), world, dev)
        e2e = {"value": job_tops(ops_step, args.steps, world, ems), "unit": "TOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": ems / args.steps}

    # ---- roofline of the dominant kernel (the GEMM)
    if bound == "hbm":
        active = None
        if args.workload == "moe":
            cnt = np.diff(workloads.routing(wspec).offsets)
            active = int((cnt > 0).sum())
        alg = [d["shape"].alg_bytes(active) for d in per]
        achieved = sum(alg) / (sum(gemm_ms) * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(args.workload),
                "alg_bytes_per_launch": alg,
                "kernel_ms_per_launch": [round(x, 5) for x in gemm_ms],
                "kernel_time": KERNEL_TIME_NOTE,
                "quantizer_ms_per_launch": [round(x, 5) for x in quant_ms],
                "peak_source": f"{peaks['source']} HBM copy bandwidth"}
    else:
        flops = [d["shape"].ops for d in per]
        achieved = sum(flops) / (sum(gemm_ms) * 1e-3) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peak,
                "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic(args.workload),
                "ops_per_launch": flops,
                "kernel_ms_per_launch": [round(x, 5) for x in gemm_ms],
                "kernel_time": KERNEL_TIME_NOTE,
                "quantizer_ms_per_launch": [round(x, 5) for x in quant_ms],
                "peak_source": (f"{peaks['source']} dense bf16 burst (the integer path runs "
                                "on fp16 tensor cores, same rate as bf16)")}

    out = {
        "metric": METRIC, "value": round(value, 3), "unit": "TOPS", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded numpy PCG64, distributions of the workload)",
        "config": {"workload": desc, "shapes": [[d["shape"].M, d["shape"].N, d["shape"].K]
                                                 for d in per],
                   "l2": "inputs larger than L2: each GEMM reads its own weight copy "
                         f"({per[0]['shape'].N * per[0]['shape'].K * per[0]['shape'].E / 1e6:.0f} MB)",
                   "parallelism": f"replicas x{world}",
                   "launch": ("one CUDA graph per step (all shapes' kernels with their "
                              "programmatic-dependent-launch edges), replayed" if graphs
                              else "stream launches")},
        "roofline": roof,
        "gpu_launches": sum(d["launches"] for d in per) * args.steps,
    }
    if e2e:
        out["e2e"] = e2e
    if sampler:
        out["clocks"] = clocks
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(args.workload, shapes, wspec)
    if rank == 0:
        print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()


# ----------------------------------------------------- oracle (CPU) timing
def oracle_sample(workload, shapes, wspec, n_cols):
    """Inputs for the oracle on a column slice [0, n_cols) of every GEMM."""
    import oracle
    items = []
    if workload == "moe":
        spec = wspec
        for shp in shapes:
            which, _, route = shp.act_spec
            a = workloads.moe_activations(spec, which, route)
            per_e = []
            for e in range(spec.E):
                per_e.append(oracle.quant_weight(
                    workloads.moe_weights(spec, which, e, rows=np.arange(n_cols))))
            qw = np.stack([p[0] for p in per_e])
            sw = np.stack([p[1] for p in per_e])
            items.append((a, qw, sw, route.offsets))
    else:
        qw, sw = oracle.quant_weight(workloads.weights(wspec, rows=np.arange(n_cols)))
        for shp in shapes:
            items.append((workloads.activations(shp.act_spec), qw, sw, None))
    return items


def oracle_step(items):
    import oracle
    for a, qw, sw, off in items:
        qa, sa = oracle.quant_act(a)
        if off is None:
            oracle.gemm(qa, sa, qw, sw, want_T=False)
        else:
            oracle.grouped_gemm(qa, sa, off, qw, sw)


def cpu_baseline(workload, shapes, wspec, target_s=10.0):
    import oracle
    cores = oracle.max_threads()
    n_full = shapes[0].N
    n0 = min(128, n_full)
    items = oracle_sample(workload, shapes, wspec, n0)
    t = time.perf_counter()
    oracle_step(items)
    t_small = time.perf_counter() - t
    n_cols = int(min(n_full, max(n0, n0 * target_s / max(t_small, 1e-6))) // 128 * 128) or n0
    items = oracle_sample(workload, shapes, wspec, n_cols)
    reps, dt = 0, 0.0
    t = time.perf_counter()
    while reps == 0 or dt < target_s:          # whole passes until ~target_s of CPU work
        oracle_step(items)
        reps += 1
        dt = time.perf_counter() - t
    ops = reps * sum(2 * s.M * n_cols * s.K for s in shapes)
    return {"value": round(ops / dt / 1e12, 6), "unit": "TOPS", "cores": cores, "kind": "oracle",
            "sample": f"{reps} pass(es) over all rows of every GEMM of the step, output columns "
                      f"[0, {n_cols}) of {n_full}; {dt:.1f} s", "seconds": round(dt, 2)}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    desc, shapes, wspec, _ = build_workload(args.workload)
    n_cols = min(shapes[0].N, 4096)
    items = oracle_sample(args.workload, shapes, wspec, n_cols)
    for _ in range(args.warmup):
        oracle_step(items)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(items)
    dt = time.perf_counter() - t
    ops = sum(2 * s.M * n_cols * s.K for s in shapes)
    value = ops * args.steps / dt / 1e12
    cores = oracle.max_threads()
    sample = (f"every GEMM of the step with output columns [0, {n_cols}) of {shapes[0].N} "
              f"(all rows, full K)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": desc, "parallelism": "oracle on host cores (rank 0)"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TOPS", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "TOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "tiny", "prefill", "stress", "moe"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels on a stream instead of replaying a graph")
    ap.add_argument("--no-clocks", action="store_true",
                    help="skip nvidia-smi clock sampling and its 1 s hold (profiler runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
