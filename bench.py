"""Benchmark of the W8A8 group-scaled quantized linear layer on GB300.

Metric: INT8 TOPS (2*M*N*K per GEMM, 2*R*N*K grouped) and the fraction of the
roofline that binds each GEMM shape (tensor peak for large M, HBM bandwidth
for decode and MoE), on one GPU.

A default run measures every workload and prints one JSON line:
  * the headline ("value", "roofline", "e2e", "cpu_baseline", "config") is the
    large stress workload, M=8192, K=16384, N=16384, FP32 out: the largest
    single-GPU configuration;
  * "per_config" holds the same measurement for each workload: dense tiny
    16x1024x1024, decode M in {1, 8, 32} x 8192 x 28672, prefill
    4096x8192x8192, MoE grouped (64 experts, top-8 of 512 tokens; gate_up
    3072x4096 and down 4096x1536), the whole MoE expert FFN of those 512
    tokens (routing, both grouped GEMMs, SwiGLU, un-permute), decode attention
    over an INT8 KV cache (32 sequences x 4096 positions, 64 query heads on 8
    kv heads, head dim 128; the step's cache write included) and stress, each
    with its throughput, the
    roofline of its dominant kernel, the quantizer's time, the end-to-end
    number through the public API with host buffers, and the CPU oracle timed
    on the host cores on a fixed slice of the same workload.
One step of a workload = one pass of the whole hot path over it: for each of
its GEMM shapes, one fused library call (per-token quantization of the BF16
activations, then the group-scaled GEMM; w8a8_linear / w8a8_grouped_linear),
the step's calls replayed as one CUDA graph.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
  python bench.py --workload tiny|decode|prefill|moe|moe_ffn|attn_int8kv|stress   (one workload)
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

METRIC = "INT8 TOPS & % of roofline (tensor peak or HBM GB/s) per GEMM shape, 1xGB300"
GROUP = 128
WORKLOADS = ("tiny", "decode", "prefill", "moe", "moe_ffn", "attn_int8kv", "norm_quant",
             "stress")
HEADLINE = "stress"
# Workloads whose inputs fit in L2 (129 MB) get an L2 flush (a 256 MB write and a 256 MB read,
# outside the timed events) before every timed step; the others read more
# than L2 holds every step.
FLUSH_L2 = ("tiny", "prefill")
L2_FLUSH_BYTES = 256 << 20
# The CPU oracle's sample of each workload (cpu_baseline and --impl
# reference time the same slice): every row and all of K, output columns
# [0, ORACLE_COLS) of every GEMM of the step (of every expert for MoE).
ORACLE_COLS = {"tiny": 1024, "decode": 2048, "prefill": 512, "moe": 256, "stress": 512}
# The MoE expert FFN's oracle sample: its first FFN_ORACLE_TOKENS tokens, whole.
FFN_ORACLE_TOKENS = 64
# The decode attention's oracle sample: its first ATTN_ORACLE_SEQS sequences.
ATTN_ORACLE_SEQS = 2
# The RMSNorm + quantizer's oracle sample: its first NORM_ORACLE_ROWS rows.
NORM_ORACLE_ROWS = 256
NORM_EPS = 1e-6


def unit_of(name):
    """Unit of a workload's value and its scale: GEMM-bearing workloads in
    TOPS, the HBM-bound RMSNorm + quantizer in GB/s of algorithmic bytes."""
    return ("GB/s", 1e9) if name == "norm_quant" else ("TOPS", 1e12)
# Calls of one shape captured back to back in one graph for its per-launch
# time (one graph launch per call would add the host's graph-launch gaps).
SHAPE_CHAIN = 8
KERNEL_TIME_NOTE = ("per shape: its quantizer + GEMM (one library call), %d calls back to back "
                    "in one graph replayed K times, events around the K replays, median of 3 "
                    "such batches, divided by %d K; the GEMM overlaps the quantizer, so this "
                    "includes any part of the quantizer it does not hide"
                    % (SHAPE_CHAIN, SHAPE_CHAIN))


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


def kernel_source_hash() -> str:
    """Hash of every CUDA source of the library (a recorded ncu traffic figure
    is used only while the kernels it was taken on are unchanged)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "moe_gemm_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), "rb") as fh:
                h.update(f.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the workload's dominant kernel from an ncu
    capture, if it was taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    rec = d.get(workload)
    if not rec or rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    # the step's launches of the dominant kernel, summed (one launch for most
    # workloads); the per-launch figures beside it
    return rec.get("dram_bytes_per_step"), rec.get("dram_bytes_per_launch")


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


class FfnShape:
    """The MoE expert FFN of T tokens (top-k of E experts, hidden H,
    intermediate I): its two grouped GEMMs' ops, and its algorithmic bytes
    (weights and group scales of the active experts of both GEMMs, the BF16
    tokens in and out, the routing)."""

    def __init__(self, spec):
        self.spec = spec
        self.M, self.N, self.K = spec.T, spec.K_up, spec.K_up   # tokens in, tokens out
        self.out = "bf16"
        self.E = spec.E

    @property
    def ops(self):
        s = self.spec
        return 2 * s.R * (s.N_up * s.K_up + s.N_down * s.K_down)

    def alg_bytes(self, active_experts=None):
        s = self.spec
        e = s.E if active_experts is None else active_experts
        w = e * (s.N_up * s.K_up + s.N_down * s.K_down)
        sc = e * 4 * (s.N_up * s.K_up // GROUP + s.N_down * s.K_down // GROUP)
        return w + sc + 2 * s.T * s.K_up * 2 + s.T * s.topk * 8


class AttnShape:
    """Decode attention over one layer's INT8 KV cache plus the cache write of
    the step's new token: ops of the score and output products; algorithmic
    bytes = the cache (codes and per-vector scales), the new K/V vectors
    (read as BF16, written as codes + scales), q and the output."""

    def __init__(self, spec):
        self.spec = spec
        self.M, self.N, self.K = spec.B * spec.Hq, spec.S, spec.D
        self.out = "bf16"
        self.E = 1

    @property
    def ops(self):
        s = self.spec
        return 4 * s.B * s.Hq * s.S * s.D

    def alg_bytes(self, active_experts=None):
        s = self.spec
        cache = 2 * s.B * s.Hkv * s.S * (s.D + 4)
        new = 2 * s.B * s.Hkv * (2 * s.D + s.D + 4)
        return cache + new + 2 * s.B * s.Hq * s.D * 2


class NormShape:
    """RMSNorm fused with the per-token quantizer over M rows of K: its
    algorithmic bytes (BF16 rows and weight read, int8 codes and FP32 scales
    written); `ops` counts those bytes, the unit of this workload's value."""

    def __init__(self, M, K):
        self.M, self.N, self.K = M, K, K
        self.out = "int8"
        self.E = 1

    def alg_bytes(self, active_experts=None):
        return 2 * self.M * self.K + 2 * self.K + self.M * self.K + 4 * self.M

    @property
    def ops(self):
        return self.alg_bytes()


def build_workload(name):
    """Returns (description, [Shape], weight spec, roofline bound)."""
    if name == "norm_quant":
        spec = workloads.DENSE["prefill"]
        desc = ("RMSNorm fused with per-token INT8 quantization: M=4096 rows of K=8192 (the "
                "prefill activations), BF16 in, int8 codes + FP32 scales out")
        return desc, [NormShape(spec.M, spec.K)], spec, "hbm"
    if name == "attn_int8kv":
        spec = workloads.ATTN["decode"]
        desc = ("decode attention over an INT8 KV cache with per-vector scales: B=32 sequences "
                "at 4096 positions, 64 query heads on 8 kv heads, head dim 128 (the step's "
                "new K/V written into the cache, then attention), BF16 out")
        return desc, [Shape(spec.B * spec.Hq, spec.S, spec.D, "bf16", None)], spec, "hbm"
    if name == "moe_ffn":
        spec = workloads.MOE["moe"]
        desc = ("MoE expert FFN: 64 experts, top-8 of T=512 tokens, H=4096, I=1536 (routing, "
                "transfer + quantization, gate_up GEMM, SwiGLU + requantization, down GEMM, "
                "weighted un-permute), BF16 out")
        return desc, [Shape(spec.R, spec.N_up, spec.K_up, "fp32", None),
                      Shape(spec.R, spec.N_down, spec.K_down, "fp32", None)], spec, "hbm"
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


def workload_config(name):
    """The `config` object of a workload's line (identical in both arms)."""
    desc, shapes, _, _ = build_workload(name)
    return {"workload": desc, "shapes": [[s.M, s.N, s.K] for s in shapes],
            "oracle_sample": oracle_sample_desc(name, shapes)}


def oracle_sample_desc(name, shapes):
    if name == "norm_quant":
        return (f"the first {NORM_ORACLE_ROWS} rows: FP64 RMSNorm, BF16 rounding, per-token "
                "quantization")
    if name == "attn_int8kv":
        return (f"the first {ATTN_ORACLE_SEQS} sequences: their K/V cache quantized, "
                "dequantized and attended by every query head")
    if name == "moe_ffn":
        return (f"the whole FFN of the first {FFN_ORACLE_TOKENS} tokens (all their routed rows, "
                "every column of both GEMMs)")
    n = min(ORACLE_COLS[name], shapes[0].N)
    per = "of every expert, " if name == "moe" else ""
    return (f"all rows and all of K of every GEMM of the step, output columns [0, {n}) "
            f"{per}of N")


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
        pw = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(rows)}


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
class GpuContext:
    def __init__(self, args):
        import torch
        import torch.distributed as dist
        self.torch = torch
        self.dist = dist
        self.args = args
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(self.local_rank)
        if self.world > 1:
            dist.init_process_group("nccl", device_id=torch.device("cuda", self.local_rank))
        import __graft_entry__
        if self.rank == 0 or self.world == 1:
            __graft_entry__.build()
        if self.world > 1:
            dist.barrier()
        import moe_gemm_gb300 as w8
        self.w8 = w8
        self.dev = torch.device("cuda", self.local_rank)
        self.stream = torch.cuda.Stream(device=self.dev)
        self.peaks = load_peaks()
        self.flush_buf = None

    def barrier(self):
        if self.world > 1:
            self.dist.barrier()

    def moe_weights(self, spec):
        """The quantized expert weights of the MoE workload, [(qw, sw) of
        gate_up, (qw, sw) of down], made once and shared by the grouped-GEMM
        and FFN workloads (quantized on the GPU, an offline step)."""
        if getattr(self, "_moe_w", None) is None:
            torch, w8, dev = self.torch, self.w8, self.dev
            out = []
            for which, N, K in (("up", spec.N_up, spec.K_up), ("down", spec.N_down, spec.K_down)):
                qw = torch.empty((spec.E, N, K), dtype=torch.int8, device=dev)
                sw = torch.empty((spec.E, N, K // GROUP), dtype=torch.float32, device=dev)
                for e in range(spec.E):
                    q, sc = w8.quant_weight(torch.from_numpy(
                        workloads.moe_weights(spec, which, e)).to(dev))
                    qw[e].copy_(q)
                    sw[e].copy_(sc)
                out.append((qw, sw))
            self._moe_w = out
        return self._moe_w

    def flush_l2(self):
        """Write a buffer larger than L2, then read another one: the write
        evicts the step's inputs, the read evicts the write's dirty lines
        (their write-back then happens here, outside the timed events, not
        inside the next timed kernel)."""
        torch = self.torch
        if self.flush_buf is None:
            self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.dev)
            self.flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=self.dev)
            self.flush_sink = torch.empty((), dtype=torch.int64, device=self.dev)
        with torch.cuda.stream(self.stream):
            self.flush_buf.fill_(1)
            torch.sum(self.flush_read, dim=0, out=self.flush_sink)

    def capture(self, fn):
        torch = self.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(self.stream):
            fn()                       # eager pass on the capture stream first
            self.stream.synchronize()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
        torch.cuda.synchronize()
        return g

    def batch_ms(self, run, reps, batches=3):
        """Median over `batches` of the mean time of `reps` back-to-back
        calls of run() on the stream (events around each batch)."""
        torch = self.torch
        out = []
        with torch.cuda.stream(self.stream):
            for _ in range(3):
                run()
            for _ in range(batches):
                s0 = torch.cuda.Event(enable_timing=True)
                s1 = torch.cuda.Event(enable_timing=True)
                s0.record(self.stream)
                for _ in range(reps):
                    run()
                s1.record(self.stream)
                s1.synchronize()
                out.append(s0.elapsed_time(s1) / reps)
        return statistics.median(out)


def upload_bf16(torch, dev, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)


def setup_workload(ctx, name):
    """Resident inputs of a workload: per shape the BF16 activations, the
    quantized weights (quantized on the GPU by the library, an offline step),
    the output and the workspace of its fused call."""
    torch, w8, dev = ctx.torch, ctx.w8, ctx.dev
    desc, shapes, wspec, bound = build_workload(name)
    per = []
    if name == "attn_int8kv":
        spec = wspec
        q_h, k_h, v_h = workloads.attn_inputs(spec)
        B, Hkv, S, D = spec.B, spec.Hkv, spec.S, spec.D
        d = dict(shape=AttnShape(spec), attn=True, off=None, a_host=q_h,
                 a=upload_bf16(torch, dev, q_h), qw=torch.empty(0, dtype=torch.int8))
        d["kc"] = torch.empty((B, Hkv, S, D), dtype=torch.int8, device=dev)
        d["vc"] = torch.empty_like(d["kc"])
        d["ks"] = torch.empty((B, Hkv, S), dtype=torch.float32, device=dev)
        d["vs"] = torch.empty_like(d["ks"])
        kb = upload_bf16(torch, dev, k_h)
        vb = upload_bf16(torch, dev, v_h)
        w8.kv_quant(kb.view(-1, D), d["kc"], d["ks"])
        w8.kv_quant(vb.view(-1, D), d["vc"], d["vs"])
        d["kb"], d["vb"] = kb, vb                   # the BF16 cache (baseline)
        # the step's new token: position S - 1 of every (sequence, kv head)
        d["k_new"] = kb[:, :, S - 1].contiguous().view(-1, D)
        d["v_new"] = vb[:, :, S - 1].contiguous().view(-1, D)
        d["rows_new"] = (torch.arange(B * Hkv, device=dev, dtype=torch.int32) * S + (S - 1))
        d["lens"] = torch.full((B,), S, dtype=torch.int32, device=dev)
        d["scale"] = 1.0 / float(np.sqrt(D))
        d["y"] = torch.empty((B, spec.Hq, D), dtype=torch.bfloat16, device=dev)
        d["ws"] = torch.empty(max(w8.attention_decode_workspace_size(B, spec.Hq, S), 1),
                              dtype=torch.uint8, device=dev)
        d["launches"] = 4
        torch.cuda.synchronize()
        return desc, shapes, wspec, bound, [d]
    if name == "moe_ffn":
        spec = wspec
        route = workloads.routing(spec)
        up, dn = ctx.moe_weights(spec)
        x_host = workloads.moe_tokens(spec)
        d = dict(shape=FfnShape(spec), a=upload_bf16(torch, dev, x_host), a_host=x_host,
                 off=None, ffn=True, qw=up[0], sw=up[1], qw_dn=dn[0], sw_dn=dn[1],
                 ids=torch.from_numpy(route.choice).to(dev),
                 w=torch.from_numpy(workloads.moe_gate_weights(spec)).to(dev))
        d["y"] = torch.empty((spec.T, spec.K_up), dtype=torch.bfloat16, device=dev)
        d["ws"] = torch.empty(max(w8.moe_ffn_workspace_size(spec.T, spec.topk, spec.K_up,
                                                            spec.K_down, spec.E), 1),
                              dtype=torch.uint8, device=dev)
        d["launches"] = 6
        torch.cuda.synchronize()
        return desc, shapes, wspec, bound, [d]
    if name == "moe":
        spec = wspec
        cached = ctx.moe_weights(spec)
        for shp, (qw, sw) in zip(shapes, cached):
            which, _, route = shp.act_spec
            a_host = workloads.moe_activations(spec, which, route)
            per.append(dict(shape=shp, qw=qw, sw=sw, a=upload_bf16(torch, dev, a_host),
                            a_host=a_host, off=torch.from_numpy(route.offsets).to(dev)))
    else:
        K, N = shapes[0].K, shapes[0].N
        qw0 = torch.empty((N, K), dtype=torch.int8, device=dev)
        sw0 = torch.empty((N, K // GROUP), dtype=torch.float32, device=dev)
        for r0, wb in workloads.weight_blocks(wspec, block_rows=4096):
            q, s = w8.quant_weight(torch.from_numpy(wb).to(dev))
            qw0[r0:r0 + wb.shape[0]].copy_(q)
            sw0[r0:r0 + wb.shape[0]].copy_(s)
            del q, s
        for i, shp in enumerate(shapes):
            a_host = workloads.activations(shp.act_spec)
            qw = qw0 if i == 0 else qw0.clone()     # a weight copy per GEMM of the step
            sw = sw0 if i == 0 else sw0.clone()
            per.append(dict(shape=shp, qw=qw, sw=sw, a=upload_bf16(torch, dev, a_host),
                            a_host=a_host, off=None))
    for d in per:
        shp = d["shape"]
        odt = torch.bfloat16 if shp.out == "bf16" else torch.float32
        d["y"] = torch.empty((shp.M, shp.N), dtype=odt, device=dev)
        wsz = (w8.grouped_linear_workspace_size(shp.M, shp.E, shp.N, shp.K)
               if d["off"] is not None else w8.linear_workspace_size(shp.M, shp.N, shp.K))
        d["ws"] = torch.empty(max(wsz, 1), dtype=torch.uint8, device=dev)
        # one fused call per shape: the quantizer (writing the GEMM's operand
        # into the workspace) and the GEMM; for <= 4 dense rows whose codes fit
        # beside the GEMV's stages, the GEMV quantizes them itself (one kernel)
        mr = 1 if shp.M <= 1 else (2 if shp.M <= 2 else 4)
        fused = d["off"] is None and shp.M <= 4 and shp.K * mr <= 96 * 1024
        d["launches"] = 1 if fused else 2
    torch.cuda.synchronize()
    return desc, shapes, wspec, bound, per


def linear_call(ctx, d, s):
    w8 = ctx.w8
    if d.get("attn"):
        w8.kv_quant(d["k_new"], d["kc"], d["ks"], dst_rows=d["rows_new"], stream=s)
        w8.kv_quant(d["v_new"], d["vc"], d["vs"], dst_rows=d["rows_new"], stream=s)
        w8.attention_decode(d["a"], d["kc"], d["vc"], d["lens"], d["scale"], k_scale=d["ks"],
                            v_scale=d["vs"], out=d["y"], workspace=d["ws"], stream=s)
    elif d.get("ffn"):
        w8.moe_ffn(d["a"], d["ids"], d["w"], d["qw"], d["sw"], d["qw_dn"], d["sw_dn"], out=d["y"],
                   out_dtype=d["y"].dtype, workspace=d["ws"], stream=s)
    elif d["off"] is not None:
        w8.grouped_linear(d["a"], d["off"], d["qw"], d["sw"], out=d["y"],
                          out_dtype=d["y"].dtype, workspace=d["ws"], stream=s)
    else:
        w8.linear(d["a"], d["qw"], d["sw"], out=d["y"], out_dtype=d["y"].dtype,
                  workspace=d["ws"], stream=s)


def measure_workload(ctx, name, headline):
    """One workload: throughput over K timed steps, per-shape kernel times,
    the quantizer alone, the roofline of the dominant kernel, the end-to-end
    number with host buffers and (rank 0, one rank) the CPU oracle."""
    torch, w8, args = ctx.torch, ctx.w8, ctx.args
    stream = ctx.stream
    desc, shapes, wspec, bound, per = setup_workload(ctx, name)

    def step():
        for d in per:
            linear_call(ctx, d, stream)

    graphs = not args.no_graph
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    torch.cuda.synchronize()
    if graphs:
        run_step = ctx.capture(step).replay
        run_shape = [ctx.capture(lambda d=d: [linear_call(ctx, d, stream)
                                              for _ in range(SHAPE_CHAIN)]).replay for d in per]
    else:
        run_step = step
        run_shape = [lambda d=d: [linear_call(ctx, d, stream) for _ in range(SHAPE_CHAIN)]
                     for d in per]
    with torch.cuda.stream(stream):
        for _ in range(3):
            run_step()
    torch.cuda.synchronize()

    # ---- the timed region: K steps, CUDA events on the launching stream
    sampler = None
    if headline and ctx.rank == 0 and not args.no_clocks:
        sampler = ClockSampler(ctx.local_rank)
        sampler.start()
    flush = name in FLUSH_L2
    ctx.barrier()
    torch.cuda.synchronize()
    if flush:
        # inputs fit in L2: flush it before every step, time each step alone
        step_ms = []
        with torch.cuda.stream(stream):
            for _ in range(args.steps):
                ctx.flush_l2()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run_step()
                e1.record(stream)
                e1.synchronize()
                step_ms.append(e0.elapsed_time(e1))
        elapsed_ms = sum(step_ms)
    else:
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            t0.record(stream)
            for _ in range(args.steps):
                run_step()
            t1.record(stream)
        torch.cuda.synchronize()
        elapsed_ms = t0.elapsed_time(t1)
    torch.cuda.synchronize()
    ctx.barrier()

    # ---- per-shape time of the fused call (the GEMM dominates it)
    gemm_ms = [ctx.batch_ms(r, args.steps) / SHAPE_CHAIN for r in run_shape]
    # ---- the quantizer alone (step a1; HBM-bound: 2 B read + 1 B written
    # per element + 4 B per row), per shape
    qbufs = [(torch.empty((d["shape"].M, d["shape"].K), dtype=torch.int8, device=ctx.dev),
              torch.empty((d["shape"].M,), dtype=torch.float32, device=ctx.dev)) for d in per]

    def quant_call(i):
        if per[i].get("attn"):   # the step's quantizer is its cache write
            d = per[i]
            w8.kv_quant(d["k_new"], d["kc"], d["ks"], dst_rows=d["rows_new"], stream=stream)
            w8.kv_quant(d["v_new"], d["vc"], d["vs"], dst_rows=d["rows_new"], stream=stream)
            return
        w8.quant_act(per[i]["a"], qa=qbufs[i][0], sa=qbufs[i][1], stream=stream)

    run_quant = ([ctx.capture(lambda i=i: [quant_call(i) for _ in range(SHAPE_CHAIN)]).replay
                  for i in range(len(per))]
                 if graphs else [lambda i=i: [quant_call(i) for _ in range(SHAPE_CHAIN)]
                                 for i in range(len(per))])
    quant_ms = [ctx.batch_ms(r, args.steps) / SHAPE_CHAIN for r in run_quant]
    del qbufs

    clocks = None
    if sampler:
        # the same step ~1 s more, so the sampler sees the load even when the
        # timed region is shorter than its sampling period
        hold_end = time.time() + 1.0
        with torch.cuda.stream(stream):
            while time.time() < hold_end:
                for _ in range(10):
                    run_step()
                stream.synchronize()
        clocks = sampler.stop()
        clocks["note"] = "sampled every 50 ms over the timed region and a 1 s hold of the same step"
    elapsed_ms = slowest_rank_ms(elapsed_ms, ctx.world, ctx.dev)
    ops_step = sum(d["shape"].ops for d in per)
    value = job_tops(ops_step, args.steps, ctx.world, elapsed_ms)

    # ---- end to end through the public API with host buffers
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
                linear_call(ctx, d, cur)
                ho.copy_(d["y"], non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        ctx.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(args.steps):
            e2e_step()
        e1.record(cur)
        torch.cuda.synchronize()
        ems = slowest_rank_ms(e0.elapsed_time(e1), ctx.world, ctx.dev)
        e2e = {"value": round(job_tops(ops_step, args.steps, ctx.world, ems), 3), "unit": "TOPS",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(ems / args.steps, 5),
               "how": "per GEMM of the step: pinned host activations -> device, the fused "
                      "library call, output -> pinned host; stream launches"}
        del host_in, host_out

    # ---- roofline of the dominant kernel (the GEMM)
    peaks = ctx.peaks
    if bound == "hbm":
        active = None
        if name in ("moe", "moe_ffn"):
            cnt = np.diff(workloads.routing(wspec).offsets)
            active = int((cnt > 0).sum())
        alg = [d["shape"].alg_bytes(active) for d in per]
        achieved = sum(alg) / (sum(gemm_ms) * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                "traffic": (recorded_traffic(name) or (None, None))[0],
                "traffic_per_launch": (recorded_traffic(name) or (None, None))[1],
                "alg_bytes_per_launch": alg,
                "peak_source": f"{peaks['source']} HBM copy bandwidth"}
    else:
        flops = [d["shape"].ops for d in per]
        achieved = sum(flops) / (sum(gemm_ms) * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": (recorded_traffic(name) or (None, None))[0],
                "traffic_per_launch": (recorded_traffic(name) or (None, None))[1],
                "ops_per_launch": flops,
                "peak_source": (f"{peaks['source']} dense bf16 burst (the integer-exact path "
                                "runs on the fp16 tensor cores, whose dense rate equals bf16's)")}
    if name == "attn_int8kv":
        # the same attention over the BF16 cache: the cost of not quantizing
        d = per[0]

        def bf16_call():
            w8.attention_decode(d["a"], d["kb"], d["vb"], d["lens"], d["scale"], out=d["y"],
                                workspace=d["ws"], stream=stream)

        run_b = (ctx.capture(lambda: [bf16_call() for _ in range(SHAPE_CHAIN)]).replay if graphs
                 else lambda: [bf16_call() for _ in range(SHAPE_CHAIN)])
        bms = ctx.batch_ms(run_b, args.steps) / SHAPE_CHAIN
        roof["bf16_cache_attention_ms"] = round(bms, 5)
        roof["int8_cache_step_over_bf16_attention"] = round(gemm_ms[0] / bms, 4)
    roof["kernel_ms_per_launch"] = [round(x, 5) for x in gemm_ms]
    roof["kernel_time"] = KERNEL_TIME_NOTE
    roof["quantizer_ms_per_launch"] = [round(x, 5) for x in quant_ms]

    entry = {
        "workload": desc,
        "shapes": [[sh.M, sh.N, sh.K] for sh in shapes],
        "value": round(value, 3), "unit": "TOPS",
        "ms_per_step": round(elapsed_ms / args.steps, 5),
        "l2": ("flushed before every timed step (256 MB write, then 256 MB read, outside "
               "the events); inputs fit in L2" if flush else
               (f"inputs larger than L2: each step streams the "
                f"{per[0]['shape'].alg_bytes() / 1e6:.0f} MB KV cache" if name == "attn_int8kv" else
                "inputs larger than L2: each step streams "
                f"{sum(d['qw'].numel() + d.get('qw_dn', d['qw'][:0]).numel() for d in per) / 1e6:.0f} MB of weights"
                + (" (a weight copy per GEMM)" if len(per) > 1 and name != "moe" else ""))),
        "roofline": roof,
        "gpu_launches_per_step": sum(d["launches"] for d in per),
    }
    if e2e:
        entry["e2e"] = e2e
    if clocks:
        entry["clocks"] = clocks
    if ctx.rank == 0 and ctx.world == 1 and not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_baseline(name, 8.0 if headline else 3.0)
    del per
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def measure_norm(ctx, headline):
    """The RMSNorm + quantizer workload: the fused kernel over the prefill
    activations (inputs fit in L2: flushed before every timed step), the
    unfused pair (rmsnorm, then quant_act) timed the same way, and the fused
    RMSNorm + linear call against rmsnorm followed by linear."""
    torch, w8, args = ctx.torch, ctx.w8, ctx.args
    stream = ctx.stream
    desc, shapes, spec, _ = build_workload("norm_quant")
    shp = shapes[0]
    M, K = shp.M, shp.K
    x_host = workloads.activations(spec)
    g_host = workloads.norm_weight(spec)
    x = upload_bf16(torch, ctx.dev, x_host)
    g = upload_bf16(torch, ctx.dev, g_host)
    qa = torch.empty((M, K), dtype=torch.int8, device=ctx.dev)
    sa = torch.empty((M,), dtype=torch.float32, device=ctx.dev)
    ybuf = torch.empty((M, K), dtype=torch.bfloat16, device=ctx.dev)
    graphs = not args.no_graph

    def fused():
        w8.rmsnorm_quant(x, g, NORM_EPS, qa=qa, sa=sa, stream=stream)

    def unfused():
        w8.rmsnorm(x, g, NORM_EPS, out=ybuf, stream=stream)
        w8.quant_act(ybuf, qa=qa, sa=sa, stream=stream)

    def flushed_ms(run, steps):
        out = []
        with torch.cuda.stream(stream):
            for _ in range(steps):
                ctx.flush_l2()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                run()
                e1.record(stream)
                e1.synchronize()
                out.append(e0.elapsed_time(e1))
        return out

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            fused()
            unfused()
    torch.cuda.synchronize()
    run_f = ctx.capture(fused).replay if graphs else fused
    run_u = ctx.capture(unfused).replay if graphs else unfused
    ctx.barrier()
    torch.cuda.synchronize()
    step_ms = flushed_ms(run_f, args.steps)
    elapsed_ms = slowest_rank_ms(sum(step_ms), ctx.world, ctx.dev)
    ctx.barrier()
    unf_ms = statistics.median(flushed_ms(run_u, args.steps))
    fused_ms = statistics.median(step_ms)
    alg = shp.alg_bytes()
    value = alg * args.steps * ctx.world / (elapsed_ms * 1e-3) / 1e9
    achieved = alg / (fused_ms * 1e-3) / 1e9
    peaks = ctx.peaks
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": (recorded_traffic("norm_quant") or (None, None))[0],
            "traffic_per_launch": (recorded_traffic("norm_quant") or (None, None))[1],
            "alg_bytes_per_launch": [alg],
            "peak_source": f"{peaks['source']} HBM copy bandwidth",
            "kernel_ms_per_launch": [round(fused_ms, 5)],
            "kernel_time": "median over the timed steps, L2 flushed before each",
            "unfused_ms": round(unf_ms, 5),
            "unfused": "rmsnorm (BF16 rows to HBM) then quant_act, L2 flushed before each pair",
            "fused_over_unfused": round(fused_ms / unf_ms, 4)}

    # RMSNorm + linear on the prefill GEMM: fused call against the two calls
    N = spec.N
    qw = torch.empty((N, K), dtype=torch.int8, device=ctx.dev)
    sw = torch.empty((N, K // GROUP), dtype=torch.float32, device=ctx.dev)
    for r0, wb in workloads.weight_blocks(spec, block_rows=4096):
        q, sc = w8.quant_weight(torch.from_numpy(wb).to(ctx.dev))
        qw[r0:r0 + wb.shape[0]].copy_(q)
        sw[r0:r0 + wb.shape[0]].copy_(sc)
        del q, sc
    y = torch.empty((M, N), dtype=torch.bfloat16, device=ctx.dev)
    ws = torch.empty(w8.linear_workspace_size(M, N, K), dtype=torch.uint8, device=ctx.dev)

    def norm_linear():
        w8.rmsnorm_linear(x, g, NORM_EPS, qw, sw, out=y, workspace=ws, stream=stream)

    def norm_then_linear():
        w8.rmsnorm(x, g, NORM_EPS, out=ybuf, stream=stream)
        w8.linear(ybuf, qw, sw, out=y, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            norm_linear()
            norm_then_linear()
    torch.cuda.synchronize()
    run_nl = ctx.capture(norm_linear).replay if graphs else norm_linear
    run_ntl = ctx.capture(norm_then_linear).replay if graphs else norm_then_linear
    nsteps = max(3, min(args.steps, 10))
    roof["rmsnorm_linear_ms"] = round(statistics.median(flushed_ms(run_nl, nsteps)), 5)
    roof["rmsnorm_then_linear_ms"] = round(statistics.median(flushed_ms(run_ntl, nsteps)), 5)
    del qw, sw, y, ws

    entry = {"workload": desc, "shapes": [[M, K]], "value": round(value, 1), "unit": "GB/s",
             "ms_per_step": round(elapsed_ms / args.steps, 5),
             "l2": "flushed before every timed step (256 MB write, then 256 MB read, outside "
                   "the events); inputs fit in L2",
             "roofline": roof, "gpu_launches_per_step": 1}
    if not args.no_e2e:
        host_in = torch.from_numpy(np.ascontiguousarray(x_host).view(np.int16)).view(
            torch.bfloat16).pin_memory()
        host_q = torch.empty((M, K), dtype=torch.int8).pin_memory()
        host_s = torch.empty((M,), dtype=torch.float32).pin_memory()
        cur = torch.cuda.current_stream()

        def e2e_step():
            x.copy_(host_in, non_blocking=True)
            w8.rmsnorm_quant(x, g, NORM_EPS, qa=qa, sa=sa, stream=cur)
            host_q.copy_(qa, non_blocking=True)
            host_s.copy_(sa, non_blocking=True)

        for _ in range(args.warmup):
            e2e_step()
        torch.cuda.synchronize()
        ctx.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(cur)
        for _ in range(args.steps):
            e2e_step()
        e1.record(cur)
        torch.cuda.synchronize()
        ems = slowest_rank_ms(e0.elapsed_time(e1), ctx.world, ctx.dev)
        entry["e2e"] = {"value": round(alg * args.steps * ctx.world / (ems * 1e-3) / 1e9, 1),
                        "unit": "GB/s", "h2d_bytes_per_step": int(2 * M * K),
                        "d2h_bytes_per_step": int(M * K + 4 * M),
                        "ms_per_step": round(ems / args.steps, 5),
                        "how": "pinned host rows -> device, the fused call, codes and scales "
                               "-> pinned host; stream launches"}
        del host_in, host_q, host_s
    if ctx.rank == 0 and ctx.world == 1 and not args.no_cpu_baseline:
        entry["cpu_baseline"] = cpu_baseline("norm_quant", 8.0 if headline else 3.0)
    del x, g, qa, sa, ybuf
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def measure_int_path_peak(ctx):
    """Rate of the integer-exact arithmetic the GEMMs run: tcgen05.mma
    kind::f16 on exact int8 integers at the instruction shapes the GEMMs
    issue, and dp4a (the CUDA-core GEMV). Timed with CUDA events."""
    torch, w8 = ctx.torch, ctx.w8
    out = {}
    # the GEMMs' instruction streams: N=256 (large dense tiles), N=128 and N=32
    # (wide and narrow tiles), each instruction on operands of its own
    for n, chains, steps in ((256, 1, 4000), (128, 1, 4000), (32, 1, 8000), (128, 2, 4000)):
        macs = [0]

        def run(n=n, chains=chains, steps=steps):
            macs[0] = w8.probe_tc_rate(n, chains, steps, distinct=True, stream=ctx.stream)

        ms = ctx.batch_ms(run, 1, batches=3)
        out[f"tcgen05_f16_m128_n{n}_x{chains}_tflops"] = round(2 * macs[0] / (ms * 1e-3) / 1e12, 1)
    macs = [0]

    def run_dp4a():
        macs[0] = w8.probe_dp4a_rate(20000, stream=ctx.stream)

    ms = ctx.batch_ms(run_dp4a, 1, batches=3)
    out["dp4a_tops"] = round(2 * macs[0] / (ms * 1e-3) / 1e12, 1)
    out["how"] = ("w8a8_probe_tc_rate / w8a8_probe_dp4a_rate: one CTA per SM issuing the "
                  "instruction back to back (zero operands), CUDA events, median of 3; "
                  "tensor-core entries are M=128 x N x K=16 with `x` accumulators taking turns, "
                  "each instruction on its own A and B operands")
    if w8.device_error(clear=True) != 0:
        out["error"] = "a probe's bounded wait gave up"
    return out


def run_ours(args):
    ctx = GpuContext(args)
    names = WORKLOADS if args.workload == "all" else (args.workload,)
    head = HEADLINE if args.workload == "all" else args.workload
    int_peak = None
    if not args.no_probe:
        int_peak = measure_int_path_peak(ctx)
    entries = {}
    for name in names:
        entries[name] = (measure_norm(ctx, name == head) if name == "norm_quant"
                         else measure_workload(ctx, name, name == head))
    h = entries[head]
    roof = dict(h["roofline"])
    if int_peak and roof["bound"] == "tensor":
        ip = int_peak["tcgen05_f16_m128_n256_x1_tflops"]
        roof["int_path_peak"] = ip
        roof["frac_of_int_path_peak"] = round(roof["achieved"] / ip, 4)
    out = {
        "metric": METRIC, "value": h["value"], "unit": "TOPS", "n_gpus": ctx.world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": h["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
        "data": "synthetic (seeded numpy PCG64, distributions of the workload)",
        "config": workload_config(head),
        "timing": {"l2": h["l2"], "parallelism": f"replicas x{ctx.world}",
                   "launch": ("one CUDA graph per step (all shapes' kernels with their "
                              "programmatic-dependent-launch edges), replayed"
                              if not args.no_graph else "stream launches")},
        "roofline": roof,
        "gpu_launches": h["gpu_launches_per_step"] * args.steps,
    }
    for k in ("e2e", "clocks", "cpu_baseline"):
        if k in h:
            out[k] = h[k]
    if int_peak:
        out["int_path_peak"] = int_peak
    if len(entries) > 1:
        out["per_config"] = entries
    if ctx.rank == 0:
        print(json.dumps(out))
    if ctx.world > 1:
        ctx.dist.destroy_process_group()


# ----------------------------------------------------- oracle (CPU) timing
def oracle_items(name):
    """Inputs of the oracle's sample of a workload (ORACLE_COLS)."""
    import oracle
    _, shapes, wspec, _ = build_workload(name)
    if name == "norm_quant":
        rows = np.arange(NORM_ORACLE_ROWS)
        item = ("norm", workloads.activations(wspec, rows=rows), workloads.norm_weight(wspec))
        return [item], NormShape(NORM_ORACLE_ROWS, wspec.K).alg_bytes()
    if name == "attn_int8kv":
        spec = wspec
        q_h, k_h, v_h = workloads.attn_inputs(spec)
        ns = ATTN_ORACLE_SEQS
        item = ("attn", q_h[:ns], k_h[:ns], v_h[:ns], np.full(ns, spec.S, np.int32),
                1.0 / np.sqrt(spec.D))
        return [item], 4 * ns * spec.Hq * spec.S * spec.D
    if name == "moe_ffn":
        # the whole FFN of the first FFN_ORACLE_TOKENS tokens, with the
        # weights of the experts they use (ids renumbered over those experts)
        spec = wspec
        nt = FFN_ORACLE_TOKENS
        ids = workloads.routing(spec).choice[:nt]
        used = np.unique(ids)
        local = np.searchsorted(used, ids).astype(np.int32)
        W = []
        for which in ("up", "down"):
            qs = [oracle.quant_weight(workloads.moe_weights(spec, which, int(e))) for e in used]
            W += [np.stack([q for q, _ in qs]), np.stack([s for _, s in qs])]
        item = ("ffn", workloads.moe_tokens(spec)[:nt], local,
                workloads.moe_gate_weights(spec)[:nt], W)
        ops = 2 * nt * spec.topk * (spec.N_up * spec.K_up + spec.N_down * spec.K_down)
        return [item], ops
    n_cols = min(ORACLE_COLS[name], shapes[0].N)
    items = []
    if name == "moe":
        spec = wspec
        for shp in shapes:
            which, _, route = shp.act_spec
            a = workloads.moe_activations(spec, which, route)
            per_e = [oracle.quant_weight(workloads.moe_weights(spec, which, e,
                                                               rows=np.arange(n_cols)))
                     for e in range(spec.E)]
            qw = np.stack([p[0] for p in per_e])
            sw = np.stack([p[1] for p in per_e])
            items.append((a, qw, sw, route.offsets))
    else:
        qw, sw = oracle.quant_weight(workloads.weights(wspec, rows=np.arange(n_cols)))
        for shp in shapes:
            items.append((workloads.activations(shp.act_spec), qw, sw, None))
    ops = sum(2 * s.M * n_cols * s.K for s in shapes)
    return items, ops


def oracle_step(items):
    import oracle
    for it in items:
        if isinstance(it[0], str) and it[0] == "norm":
            _, x, g = it
            oracle.quant_act(oracle.bf16_round(oracle.rmsnorm(x, g, float(np.float32(NORM_EPS)))))
            continue
        if isinstance(it[0], str) and it[0] == "attn":
            _, q, k, v, lens, scale = it
            qk, sk = oracle.kv_quant(k)
            qv, sv = oracle.kv_quant(v)
            oracle.attention_decode(q, oracle.kv_dequant(qk, sk), oracle.kv_dequant(qv, sv), lens,
                                    scale)
            continue
        if isinstance(it[0], str) and it[0] == "ffn":
            _, x, ids, w, W = it
            oracle.moe_ffn(x, ids, w, *W)
            continue
        a, qw, sw, off = it
        qa, sa = oracle.quant_act(a)
        if off is None:
            oracle.gemm(qa, sa, qw, sw, want_T=False)
        else:
            oracle.grouped_gemm(qa, sa, off, qw, sw)


def cpu_baseline(name, target_s):
    """The oracle as it stands, on the host cores, over whole passes of the
    workload's fixed sample until about target_s seconds have passed."""
    import oracle
    _, shapes, _, _ = build_workload(name)
    items, ops = oracle_items(name)
    reps, dt = 0, 0.0
    t = time.perf_counter()
    while reps == 0 or dt < target_s:
        oracle_step(items)
        reps += 1
        dt = time.perf_counter() - t
    unit, scale = unit_of(name)
    return {"value": round(ops * reps / dt / scale, 6), "unit": unit,
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": oracle_sample_desc(name, shapes), "passes": reps, "seconds": round(dt, 2)}


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    name = HEADLINE if args.workload == "all" else args.workload
    _, shapes, _, _ = build_workload(name)
    items, ops = oracle_items(name)
    for _ in range(args.warmup):
        oracle_step(items)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(items)
    dt = time.perf_counter() - t
    unit, scale = unit_of(name)
    value = ops * args.steps / dt / scale
    cores = oracle.max_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": workload_config(name),
        "timing": {"parallelism": "the CPU oracle on the host cores (rank 0)"},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cores,
                         "kind": "oracle", "sample": oracle_sample_desc(name, shapes)},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all", choices=("all",) + WORKLOADS)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-probe", action="store_true",
                    help="skip the integer-path rate probes")
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
