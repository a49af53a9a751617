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


# ------------------------------------------------------------- row gathers
# The gathered operand is the un-permuted [T, .] source: permuted row r is
# source row src[r] // k of an expert-sort plan, zero where src[r] = -1. The
# oracle builds the permuted copy explicitly and multiplies that.

def _plan(T, E, k, align, seed):
    g = np.random.default_rng(seed)
    idx = np.stack([g.permutation(E - 1)[:k] for _ in range(T)])  # expert E-1 gets no rows
    counts, off, dest, src = O.permute_plan(idx, E, align)
    return torch.from_numpy(off), torch.from_numpy(dest), torch.from_numpy(src)


GATHER_FPROP_CASES = [
    # T, E, k, align, K, N, b_layout
    (300, 4, 2, 128, 256, 256, 0),   # 256-wide tiles (CTA pairs), pad rows in every group
    (300, 4, 2, 128, 256, 256, 1),
    (37, 3, 1, 64, 192, 384, 0),     # 128-wide tiles, one partial tile per group
    (37, 3, 1, 64, 192, 384, 1),
]


@pytest.mark.parametrize("T,E,k,align,K,N,b_layout", GATHER_FPROP_CASES)
def test_grouped_gemm_fprop_gathered(T, E, k, align, K, N, b_layout):
    off, dest, src = _plan(T, E, k, align, 20 + T)
    x = _bf16((T, K), 21)
    Bw = _bf16((E, K, N) if b_layout == 0 else (E, N, K), 22, 0.1)
    C = B().moe_grouped_gemm_bf16(B().GEMM_FPROP, x.to(DEV), Bw.to(DEV), off.to(DEV),
                                  b_layout=b_layout, gather_a=(src.to(DEV), k))
    xp = O.permute(f64(x), i32(dest), k, int(off[-1]))
    ref = O.grouped_gemm_fprop(xp, f64(Bw), i32(off), b_layout)
    assert C.shape[0] == xp.shape[0]
    _close(f64(C), ref)
    assert B().device_error() == 0


@pytest.mark.parametrize("T,E,k,M,N,which", [
    (300, 4, 2, 256, 512, "a"),   # CTA pairs (M % 256 == 0)
    (300, 4, 2, 256, 512, "b"),
    (200, 3, 2, 128, 256, "a"),   # one CTA per tile
    (200, 3, 2, 384, 384, "b"),   # 128-wide tiles
])
def test_grouped_gemm_wgrad_gathered(T, E, k, M, N, which):
    off, dest, src = _plan(T, E, k, 128, 30 + T)
    rows = int(off[-1])
    if which == "a":  # dW = X_e^T Y_e with X gathered from [T, M]
        X, Y = _bf16((T, M), 31), _bf16((rows, N), 32)
        C = B().moe_grouped_gemm_bf16(B().GEMM_WGRAD, X.to(DEV), Y.to(DEV), off.to(DEV),
                                      gather_a=(src.to(DEV), k))
        A_ref, Y_ref = O.permute(f64(X), i32(dest), k, rows), f64(Y)
    else:  # dW = H_e^T D_e with D gathered from [T, N]
        X, Y = _bf16((rows, M), 33), _bf16((T, N), 34)
        C = B().moe_grouped_gemm_bf16(B().GEMM_WGRAD, X.to(DEV), Y.to(DEV), off.to(DEV),
                                      gather_b=(src.to(DEV), k))
        A_ref, Y_ref = f64(X), O.permute(f64(Y), i32(dest), k, rows)
    ref = O.grouped_gemm_wgrad(A_ref, Y_ref, i32(off))
    _close(f64(C), ref)
    assert np.all(f64(C)[E - 1] == 0)  # the expert with no rows
    assert B().device_error() == 0


@pytest.mark.parametrize("T,E,k,H,F", [(300, 4, 2, 128, 256), (200, 3, 2, 256, 192)])
def test_fc1_swiglu_gathered(T, E, k, H, F):
    off, dest, src = _plan(T, E, k, 128, 40 + T)
    rows = int(off[-1])
    x = _bf16((T, H), 41)
    w1 = _bf16((E, H, 2 * F), 42, 0.05)
    p = torch.rand(rows, generator=torch.Generator().manual_seed(43))
    gu, h = B().moe_fc1_swiglu_bf16(x.to(DEV), w1.to(DEV), off.to(DEV), p.to(DEV),
                                    gather_x=(src.to(DEV), k))
    xp = O.permute(f64(x), i32(dest), k, rows)
    y1 = O.grouped_gemm_fprop(xp, f64(w1), i32(off))
    href = O.silu(y1[:, :F]) * y1[:, F:] * f64(p)[:, None]
    _close(f64(gu), y1)
    _close(f64(h), href)
    assert B().device_error() == 0


@pytest.mark.parametrize("T,E,k,H,F", [(300, 4, 2, 128, 256), (200, 3, 2, 256, 384)])
def test_fc2_dgrad_swiglu_bwd_gathered(T, E, k, H, F):
    off, dest, src = _plan(T, E, k, 128, 50 + T)
    rows = int(off[-1])
    dout = _bf16((T, H), 51)
    w2 = _bf16((E, F, H), 52, 0.05)
    gu = _bf16((rows, 2 * F), 53)
    p = torch.rand(rows, generator=torch.Generator().manual_seed(54))
    dy1, dp_part = B().moe_fc2_dgrad_swiglu_bwd_bf16(dout.to(DEV), w2.to(DEV), off.to(DEV),
                                                     p.to(DEV), gu.to(DEV),
                                                     gather_dy=(src.to(DEV), k))
    dy2 = O.permute(f64(dout), i32(dest), k, rows)
    dh = O.grouped_gemm_fprop(dy2, f64(w2), i32(off), b_layout=1)
    g, u = f64(gu)[:, :F], f64(gu)[:, F:]
    dA = dh * f64(p)[:, None]
    ref_dy1 = np.concatenate([dA * u * O.dsilu(g), dA * O.silu(g)], axis=1)
    _close(f64(dy1), ref_dy1)
    assert rel_fro(f64(dp_part).sum(1), (dh * O.silu(g) * u).sum(1)) <= 1e-4
    assert B().device_error() == 0


def test_gather_source_row_out_of_range_is_flagged_and_zero():
    """A src entry naming a row past the source tensor is read as a zero row
    and sets MOE_DEVERR_BAD_INDEX (the kernel checks it before the copy)."""
    T, E, k, K, N = 300, 4, 2, 256, 256
    off, dest, src = _plan(T, E, k, 128, 60)
    bad = src.clone()
    r_bad = int(dest[5])            # the permuted row of token 2, slot 1
    bad[r_bad] = (T + 3) * k        # source row T + 3 >= T
    x = _bf16((T, K), 61)
    Bw = _bf16((E, K, N), 62, 0.1)
    C = B().moe_grouped_gemm_bf16(B().GEMM_FPROP, x.to(DEV), Bw.to(DEV), off.to(DEV),
                                  gather_a=(bad.to(DEV), k))
    assert B().device_error() & B().MOE_DEVERR_BAD_INDEX
    xp = O.permute(f64(x), i32(dest), k, int(off[-1]))
    xp[r_bad] = 0.0
    _close(f64(C), O.grouped_gemm_fprop(xp, f64(Bw), i32(off), 0))
    assert B().device_error() == 0
