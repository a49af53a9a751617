"""Parity of the block-scaled MXFP8 grouped GEMMs (tcgen05 kind::mxf8f6f4) with
the CPU oracle, through the C ABI.

The operands are quantised on the GPU (bit-exact with the oracle's quantiser,
see test_gpu_kernels.py); the references quantise the same bf16 inputs with
the oracle's own MXFP8 rule and multiply in float64. Both sides therefore use
identical operand values, and the GEMM results must agree to fp32
accumulation plus one bf16 rounding: rel-Frobenius <= 5e-3.
Quantised outputs of the fused epilogues are computed from fp32 accumulators
whose summation order differs from the oracle's, so those are compared after
dequantisation against the oracle's quantisation of its own values, within
the MXFP8 tolerance rel-Frobenius <= 1e-2.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.helpers import f64, u8, scales_tiled_to_rowmajor, rel_fro, max_abs_rel

pytestmark = pytest.mark.gpu
DEV = "cuda"


def B():
    from mixture_experts_expert_sort_b300 import binding
    return binding


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _offsets(sizes):
    return torch.tensor(np.concatenate([[0], np.cumsum(sizes)]), dtype=torch.int32)


def _deq(q, s, mn, kdim):
    """Dequantise a GPU MXFP8 tensor [mn, kdim] (test-side decode of the layout)."""
    sc = scales_tiled_to_rowmajor(u8(s), mn, kdim)
    return O.mx_dequantize(u8(q), sc, axis=1)


@pytest.mark.parametrize("sizes,K,N", [([128, 256], 128, 256), ([256, 0, 384, 128], 512, 512),
                                       ([128, 128], 256, 384)])
def test_mx_fprop_colwise_weights(sizes, K, N):
    """B_e = W[e] with W [E, K, N]; the weight copy is column-wise [N, E*K]."""
    E = len(sizes)
    rows = int(sum(sizes))
    A = _bf16((rows, K), 11)
    W = _bf16((E, K, N), 12, 0.05)
    off = _offsets(sizes)
    qa = B().mxfp8_quantize(A.to(DEV), dirs=B().QUANT_ROWWISE)
    qw = B().mxfp8_quantize(W.reshape(E * K, N).to(DEV), dirs=B().QUANT_COLWISE)
    C = B().moe_grouped_gemm_mxfp8(B().GEMM_FPROP, qa["q_row"], qa["s_row"], qw["q_col"],
                                   qw["s_col"], off.to(DEV), b_row_stride=0, b_k_stride=K, N=N,
                                   K=K)
    Aq = O.mx_qdq(f64(A), axis=1)
    Wq = np.stack([O.mx_qdq(f64(W[e]), axis=0) for e in range(E)])
    ref = O.grouped_gemm_fprop(Aq, Wq, off.numpy())
    assert rel_fro(f64(C), ref) <= 5e-3, rel_fro(f64(C), ref)
    assert B().device_error() == 0


@pytest.mark.parametrize("sizes,K,N", [([128, 256], 128, 256), ([256, 0, 128], 256, 384)])
def test_mx_fprop_rowwise_weights(sizes, K, N):
    """B_e = W[e] with W [E, N, K] used as [N, K]; the copy is row-wise [E*N, K]."""
    E = len(sizes)
    rows = int(sum(sizes))
    A = _bf16((rows, K), 13)
    W = _bf16((E, N, K), 14, 0.05)
    off = _offsets(sizes)
    qa = B().mxfp8_quantize(A.to(DEV), dirs=B().QUANT_ROWWISE)
    qw = B().mxfp8_quantize(W.reshape(E * N, K).to(DEV), dirs=B().QUANT_ROWWISE)
    C = B().moe_grouped_gemm_mxfp8(B().GEMM_FPROP, qa["q_row"], qa["s_row"], qw["q_row"],
                                   qw["s_row"], off.to(DEV), b_row_stride=N, b_k_stride=0, N=N,
                                   K=K)
    Aq = O.mx_qdq(f64(A), axis=1)
    Wq = np.stack([O.mx_qdq(f64(W[e]), axis=1) for e in range(E)])
    ref = O.grouped_gemm_fprop(Aq, Wq, off.numpy(), b_layout=1)
    assert rel_fro(f64(C), ref) <= 5e-3, rel_fro(f64(C), ref)
    assert B().device_error() == 0


@pytest.mark.parametrize("sizes,M,N", [([128, 256], 128, 256), ([256, 0, 384, 128], 256, 512)])
def test_mx_wgrad(sizes, M, N):
    E = len(sizes)
    rows = int(sum(sizes))
    A = _bf16((rows, M), 15)
    Y = _bf16((rows, N), 16)
    off = _offsets(sizes)
    qa = B().mxfp8_quantize(A.to(DEV), dirs=B().QUANT_COLWISE)
    qy = B().mxfp8_quantize(Y.to(DEV), dirs=B().QUANT_COLWISE)
    C = B().moe_grouped_gemm_mxfp8(B().GEMM_WGRAD, qa["q_col"], qa["s_col"], qy["q_col"],
                                   qy["s_col"], off.to(DEV), M=M, N=N)
    ref = O.grouped_gemm_wgrad(O.mx_qdq(f64(A), axis=0), O.mx_qdq(f64(Y), axis=0), off.numpy())
    assert rel_fro(f64(C), ref) <= 5e-3, rel_fro(f64(C), ref)
    assert np.all(f64(C)[[i for i, s in enumerate(sizes) if s == 0]] == 0)
    assert B().device_error() == 0


@pytest.mark.parametrize("sizes,H,F", [([128, 256], 128, 256), ([256, 0, 128], 256, 384)])
def test_mx_fc1_swiglu(sizes, H, F):
    E = len(sizes)
    rows = int(sum(sizes))
    x = _bf16((rows, H), 17)
    W1 = _bf16((E, H, 2 * F), 18, 0.05)
    p = torch.rand(rows, generator=torch.Generator().manual_seed(19))
    off = _offsets(sizes)
    qx = B().mxfp8_quantize(x.to(DEV), dirs=B().QUANT_ROWWISE)
    qw = B().mxfp8_quantize(W1.reshape(E * H, 2 * F).to(DEV), dirs=B().QUANT_COLWISE)
    o = B().moe_fc1_swiglu_mxfp8(qx["q_row"], qx["s_row"], qw["q_col"], qw["s_col"], off.to(DEV),
                                 p.to(DEV), F)
    xq = O.mx_qdq(f64(x), axis=1)
    wq = np.stack([O.mx_qdq(f64(W1[e]), axis=0) for e in range(E)])
    y1 = O.grouped_gemm_fprop(xq, wq, off.numpy())
    assert rel_fro(f64(o["gu"]), y1) <= 5e-3
    g, u = y1[:, :F], y1[:, F:]
    h32 = O.to_f32(O.silu(g) * u * f64(p)[:, None])
    h_row = _deq(o["q_row"], o["s_row"], rows, F)
    h_col = _deq(o["q_col"], o["s_col"], F, rows).T
    assert rel_fro(h_row, O.mx_qdq(h32, axis=1)) <= 1e-2
    assert rel_fro(h_col, O.mx_qdq(h32, axis=0)) <= 1e-2
    # the two quantisations differ only in block direction
    assert rel_fro(h_row, h32) <= 0.06 and rel_fro(h_col, h32) <= 0.06


@pytest.mark.parametrize("sizes,H,F", [([128, 256], 128, 256), ([256, 0, 128], 256, 384)])
def test_mx_fc2_dgrad_swiglu_bwd(sizes, H, F):
    E = len(sizes)
    rows = int(sum(sizes))
    dy2 = _bf16((rows, H), 20)
    W2 = _bf16((E, F, H), 21, 0.05)
    gu = _bf16((rows, 2 * F), 22)
    p = torch.rand(rows, generator=torch.Generator().manual_seed(23))
    off = _offsets(sizes)
    qd = B().mxfp8_quantize(dy2.to(DEV), dirs=B().QUANT_ROWWISE)
    qw = B().mxfp8_quantize(W2.reshape(E * F, H).to(DEV), dirs=B().QUANT_ROWWISE)
    o = B().moe_fc2_dgrad_swiglu_bwd_mxfp8(qd["q_row"], qd["s_row"], qw["q_row"], qw["s_row"],
                                           off.to(DEV), p.to(DEV), gu.to(DEV), F)
    dq = O.mx_qdq(f64(dy2), axis=1)
    wq = np.stack([O.mx_qdq(f64(W2[e]), axis=1) for e in range(E)])
    dh = O.grouped_gemm_fprop(dq, wq, off.numpy(), b_layout=1)
    g, u = f64(gu)[:, :F], f64(gu)[:, F:]
    pp = f64(p)[:, None]
    dA = dh * pp
    dy1 = O.to_f32(np.concatenate([dA * u * O.dsilu(g), dA * O.silu(g)], axis=1))
    r_row = _deq(o["q_row"], o["s_row"], rows, 2 * F)
    r_col = _deq(o["q_col"], o["s_col"], 2 * F, rows).T
    assert rel_fro(r_row, O.mx_qdq(dy1, axis=1)) <= 1e-2
    assert rel_fro(r_col, O.mx_qdq(dy1, axis=0)) <= 1e-2
    dp = f64(o["dp"]).sum(1)
    ref_dp = (dh * O.silu(g) * u).sum(1)
    assert rel_fro(dp, ref_dp) <= 1e-4
    assert B().device_error() == 0
