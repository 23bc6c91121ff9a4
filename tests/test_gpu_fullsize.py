"""GPU parity at the full workload sizes, on sampled outputs.

The CUDA path runs the whole problem (weights quantized on the GPU from the
seeded FP32 weights, activations quantized on the GPU, one GEMM call), and
again exactly as bench.py launches it (one fused quantizer + GEMM call,
w8a8_linear / w8a8_grouped_linear), which must give the same output bits. The oracle recomputes sampled output
rows/columns from its own quantization of the same seeded inputs; the
sampled weight rows and activation rows are also compared bit-exactly.
"""
import zlib

import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import moe_gemm_gb300 as w8  # noqa: E402
from tests.test_gpu_parity import DEV, bf16_bits_of, check_bf16, check_fp32, to_dev_bf16  # noqa: E402

G = 128


def gpu_quant_weights(gen_blocks, N, K):
    qw = torch.empty((N, K), dtype=torch.int8, device=DEV)
    sw = torch.empty((N, K // G), dtype=torch.float32, device=DEV)
    for r0, wb in gen_blocks:
        q, s = w8.quant_weight(torch.from_numpy(wb).to(DEV))
        qw[r0:r0 + wb.shape[0]].copy_(q)
        sw[r0:r0 + wb.shape[0]].copy_(s)
    return qw, sw


@pytest.mark.parametrize("name,n_rows,n_cols", [
    ("decode_m1", None, 96), ("decode_m8", None, 96), ("decode_m32", None, 96),
    ("prefill", 48, 48), ("stress", 32, 32),
])
def test_dense_full_size_sampled(name, n_rows, n_cols):
    spec = workloads.DENSE[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    qw, sw = gpu_quant_weights(workloads.weight_blocks(spec), spec.N, spec.K)
    a_bits = workloads.activations(spec)
    a_dev = to_dev_bf16(a_bits)
    qa, sa = w8.quant_act(a_dev)
    dt = torch.bfloat16 if spec.out_dtype == "bf16" else torch.float32
    y = torch.full((spec.M, spec.N), float("nan"), dtype=dt, device=DEV)
    w8.gemm(qa, sa, qw, sw, out_dtype=dt, out=y)
    y_lin = torch.full((spec.M, spec.N), float("nan"), dtype=dt, device=DEV)
    w8.linear(a_dev, qw, sw, out_dtype=dt, out=y_lin)
    torch.cuda.synchronize()
    assert torch.equal(y_lin, y)
    del y_lin

    rows = np.arange(spec.M) if n_rows is None else np.sort(
        rng.choice(spec.M, n_rows, replace=False))
    cols = np.sort(np.concatenate([[0, spec.N - 1], rng.choice(spec.N, n_cols, replace=False)]))
    qa_o, sa_o = oracle.quant_act(a_bits[rows])
    qw_o, sw_o = oracle.quant_weight(workloads.weights(spec, rows=cols))
    rows_t = torch.from_numpy(rows).to(DEV)
    cols_t = torch.from_numpy(cols).to(DEV)
    np.testing.assert_array_equal(qa.index_select(0, rows_t).cpu().numpy(), qa_o)
    np.testing.assert_array_equal(sa.index_select(0, rows_t).cpu().numpy().view(np.uint32),
                                  sa_o.view(np.uint32))
    np.testing.assert_array_equal(qw.index_select(0, cols_t).cpu().numpy(), qw_o)
    np.testing.assert_array_equal(sw.index_select(0, cols_t).cpu().numpy().view(np.uint32),
                                  sw_o.view(np.uint32))
    y_ref, T = oracle.gemm(qa_o, sa_o, qw_o, sw_o)
    y_s = y.index_select(0, rows_t).index_select(1, cols_t)
    if dt == torch.float32:
        check_fp32(y_s.cpu().numpy(), y_ref, T, spec.K)
    else:
        check_bf16(bf16_bits_of(y_s), y_ref, T)
    # nothing left unwritten anywhere in the output
    assert not torch.isnan(y.float()).any().item()


@pytest.mark.parametrize("which", ["up", "down"])
def test_moe_full_size_sampled(which):
    spec = workloads.MOE["moe"]
    route = workloads.routing(spec)
    N, K = (spec.N_up, spec.K_up) if which == "up" else (spec.N_down, spec.K_down)
    E, R = spec.E, spec.R
    qw = torch.empty((E, N, K), dtype=torch.int8, device=DEV)
    sw = torch.empty((E, N, K // G), dtype=torch.float32, device=DEV)
    for e in range(E):
        q, s = w8.quant_weight(torch.from_numpy(workloads.moe_weights(spec, which, e)).to(DEV))
        qw[e].copy_(q)
        sw[e].copy_(s)
    a_bits = workloads.moe_activations(spec, which, route)
    a_dev = to_dev_bf16(a_bits)
    qa, sa = w8.quant_act(a_dev)
    off = route.offsets
    off_t = torch.from_numpy(off).to(DEV)
    y = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    w8.grouped_gemm(qa, sa, off_t, qw, sw, out=y)
    y_lin = torch.full((R, N), float("nan"), dtype=torch.bfloat16, device=DEV)
    w8.grouped_linear(a_dev, off_t, qw, sw, out=y_lin)
    torch.cuda.synchronize()
    assert not torch.isnan(y.float()).any().item()          # every routed row written
    assert torch.equal(y_lin, y)

    counts = np.diff(off)
    rng = np.random.default_rng(7 if which == "up" else 8)
    experts = sorted({int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 10 ** 9)))}
                     | set(rng.choice(np.nonzero(counts)[0], 3, replace=False).tolist()))
    cols = np.sort(rng.choice(N, 24, replace=False))
    cols_t = torch.from_numpy(cols).to(DEV)
    for e in experts:
        lo, hi = int(off[e]), int(off[e + 1])
        qa_o, sa_o = oracle.quant_act(a_bits[lo:hi])
        qw_o, sw_o = oracle.quant_weight(workloads.moe_weights(spec, which, e, rows=cols))
        np.testing.assert_array_equal(qa[lo:hi].cpu().numpy(), qa_o)
        np.testing.assert_array_equal(qw[e].index_select(0, cols_t).cpu().numpy(), qw_o)
        y_ref, T = oracle.gemm(qa_o, sa_o, qw_o, sw_o)
        check_bf16(bf16_bits_of(y[lo:hi].index_select(1, cols_t)), y_ref, T)
