"""Parity of the tcgen05 grouped GEMMs and the fused SwiGLU epilogues with the
CPU oracle, through the C ABI (BF16 inputs, fp32 accumulation, bf16 outputs).

Tolerances: relative Frobenius error <= 5e-3 and max-abs error <= 1e-2 of
max|ref| (one bf16 rounding of each output is <= 2^-9 relative).
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.helpers import f64, i32, rel_fro, max_abs_rel

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


def _close(got, ref, tol=5e-3):
    assert rel_fro(got, ref) <= tol, rel_fro(got, ref)
    assert max_abs_rel(got, ref) <= 1e-2, max_abs_rel(got, ref)


FPROP_CASES = [
    # group sizes, K, N, b_layout
    ([128, 256], 128, 256, 0),
    ([128, 256], 128, 256, 1),
    ([256, 0, 384, 128], 512, 512, 0),
    ([256, 0, 384, 128], 512, 512, 1),
    ([128, 128], 192, 384, 0),   # N not a multiple of 256 -> 128-wide tiles
    ([128, 128], 192, 384, 1),
    ([100, 37, 300], 256, 256, 0),  # ragged groups (rows masked in the epilogue)
    ([100, 37, 300], 256, 256, 1),
]


@pytest.mark.parametrize("sizes,K,N,b_layout", FPROP_CASES)
def test_grouped_gemm_fprop(sizes, K, N, b_layout):
    E = len(sizes)
    rows = int(sum(sizes))
    A = _bf16((rows, K), 1 + K)
    Bw = _bf16((E, K, N) if b_layout == 0 else (E, N, K), 2 + N, 0.1)
    off = _offsets(sizes)
    C = B().moe_grouped_gemm_bf16(B().GEMM_FPROP, A.to(DEV), Bw.to(DEV), off.to(DEV),
                                  b_layout=b_layout)
    ref = O.grouped_gemm_fprop(f64(A), f64(Bw), i32(off), b_layout)
    _close(f64(C), ref)
    assert B().device_error() == 0


WGRAD_CASES = [
    ([128, 256], 128, 256),
    ([256, 0, 384, 128], 256, 512),
    ([128, 128], 384, 384),
    ([64, 192], 128, 128),
]


@pytest.mark.parametrize("sizes,M,N", WGRAD_CASES)
def test_grouped_gemm_wgrad(sizes, M, N):
    E = len(sizes)
    rows = int(sum(sizes))
    A = _bf16((rows, M), 3 + M)
    Y = _bf16((rows, N), 4 + N)
    off = _offsets(sizes)
    C = B().moe_grouped_gemm_bf16(B().GEMM_WGRAD, A.to(DEV), Y.to(DEV), off.to(DEV))
    ref = O.grouped_gemm_wgrad(f64(A), f64(Y), i32(off))
    _close(f64(C), ref)
    assert B().device_error() == 0


@pytest.mark.parametrize("sizes,H,F", [([128, 256], 128, 256), ([256, 0, 128], 256, 384),
                                       ([128, 128], 128, 192)])
def test_fc1_swiglu(sizes, H, F):
    E = len(sizes)
    rows = int(sum(sizes))
    xp = _bf16((rows, H), 5)
    w1 = _bf16((E, H, 2 * F), 6, 0.05)
    p = torch.rand(rows, generator=torch.Generator().manual_seed(7))
    off = _offsets(sizes)
    gu, h = B().moe_fc1_swiglu_bf16(xp.to(DEV), w1.to(DEV), off.to(DEV), p.to(DEV))
    y1 = O.grouped_gemm_fprop(f64(xp), f64(w1), i32(off))
    g, u = y1[:, :F], y1[:, F:]
    href = O.silu(g) * u * f64(p)[:, None]
    _close(f64(gu), y1)
    _close(f64(h), href)


@pytest.mark.parametrize("sizes,H,F", [([128, 256], 128, 256), ([256, 0, 128], 256, 384)])
def test_fc2_dgrad_swiglu_bwd(sizes, H, F):
    E = len(sizes)
    rows = int(sum(sizes))
    dy2 = _bf16((rows, H), 8)
    w2 = _bf16((E, F, H), 9, 0.05)
    gu = _bf16((rows, 2 * F), 10)
    p = torch.rand(rows, generator=torch.Generator().manual_seed(11))
    off = _offsets(sizes)
    dy1, dp_part = B().moe_fc2_dgrad_swiglu_bwd_bf16(dy2.to(DEV), w2.to(DEV), off.to(DEV),
                                                     p.to(DEV), gu.to(DEV))
    dh = O.grouped_gemm_fprop(f64(dy2), f64(w2), i32(off), b_layout=1)
    g, u = f64(gu)[:, :F], f64(gu)[:, F:]
    pp = f64(p)[:, None]
    a = O.silu(g) * u
    dA = dh * pp
    ref_dy1 = np.concatenate([dA * u * O.dsilu(g), dA * O.silu(g)], axis=1)
    _close(f64(dy1), ref_dy1)
    dp = f64(dp_part).sum(1)
    ref_dp = (dh * a).sum(1)
    assert rel_fro(dp, ref_dp) <= 1e-4
