"""MXFP4 conversions on the GPU against the oracle, byte for byte: direct
FP8 -> FP4, FP4 -> FP8, and the scale-aware row -> column conversion (to FP4
and to the FP8 wgrad operand). Inputs are made by the oracle from seeded
values whose magnitude varies by block (so every scale byte range is used),
with zero, -0 and NaN blocks."""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import mxfp4_oracle as Q
from tests.helpers import scales_rowmajor_to_tiled, scales_tiled_to_rowmajor, u8

pytestmark = pytest.mark.gpu
DEV = "cuda"
SHAPES = [(128, 128), (256, 384), (384, 256), (1024, 2048)]


def B():
    from mixture_experts_expert_sort_b300 import binding
    return binding


def _values(rows, cols, seed):
    rng = np.random.default_rng(seed)
    v = rng.normal(size=(rows, cols))
    # a magnitude per row block, spanning about 2^-60 .. 2^60
    v *= np.repeat(np.ldexp(1.0, rng.integers(-60, 60, (rows, cols // 32))), 32, axis=1)
    v[1, 32:64] = 0.0                       # an all-zero block
    v[2, 64:96] = 0.0
    v[2, 70] = -0.0                         # -0 keeps its sign
    v[3, :32] = rng.normal(size=32) * 2.0 ** -130  # subnormal magnitudes
    v[4, 96:128] = rng.choice([6.0, -6.0, 0.25, 0.75, 1.25, 2.5, 5.0], 32)  # ties, top binade
    v[5, 0:32] = np.nan                     # a NaN block
    return v


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_mxfp4_from_mxfp8(rows, cols):
    c8, s8 = O.mx_quantize(_values(rows, cols, rows + cols), axis=1)
    out = B().mxfp4_from_mxfp8(_up(c8), _up(scales_rowmajor_to_tiled(s8, rows, cols)))
    c4, s4 = Q.mxfp4_from_mxfp8(c8, s8)
    np.testing.assert_array_equal(u8(out["q4"]), Q.pack_e2m1(c4))
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(out["s4"]), rows, cols), s4)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_mxfp8_from_mxfp4(rows, cols):
    c4, s4 = Q.mx4_quantize(_values(rows, cols, 7 + rows), axis=1)
    out = B().mxfp8_from_mxfp4(_up(Q.pack_e2m1(c4)), _up(scales_rowmajor_to_tiled(s4, rows, cols)))
    c8, s8 = Q.mxfp8_from_mxfp4(c4, s4)
    np.testing.assert_array_equal(u8(out["q8"]), c8)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(out["s8"]), rows, cols), s8)


@pytest.mark.parametrize("rows,cols", SHAPES)
def test_mxfp4_rowwise_to_colwise(rows, cols):
    c4, s4 = Q.mx4_quantize(_values(rows, cols, 11 + cols), axis=1)
    q4, s4t = _up(Q.pack_e2m1(c4)), _up(scales_rowmajor_to_tiled(s4, rows, cols))
    cc, sc = Q.mxfp4_row_to_col(c4, s4)
    out = B().mxfp4_rowwise_to_colwise(q4, s4t)
    np.testing.assert_array_equal(u8(out["q4c"]), Q.pack_e2m1(cc))
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(out["s4c"]), cols, rows), sc)
    c8c, s8c = Q.mxfp8_col_from_mxfp4_row(c4, s4)
    out8 = B().mxfp8_colwise_from_mxfp4_rowwise(q4, s4t)
    np.testing.assert_array_equal(u8(out8["q8c"]), c8c)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(out8["s8c"]), cols, rows), s8c)


def test_mxfp4_chain_fp8_to_fp4_to_fp8():
    """FP8 -> FP4 -> FP8 equals the oracle's chain (the second step is lossless)."""
    rows, cols = 256, 512
    c8, s8 = O.mx_quantize(_values(rows, cols, 99), axis=1)
    o4 = B().mxfp4_from_mxfp8(_up(c8), _up(scales_rowmajor_to_tiled(s8, rows, cols)))
    o8 = B().mxfp8_from_mxfp4(o4["q4"], o4["s4"])
    c4, s4 = Q.mxfp4_from_mxfp8(c8, s8)
    r8, rs8 = Q.mxfp8_from_mxfp4(c4, s4)
    np.testing.assert_array_equal(u8(o8["q8"]), r8)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(o8["s8"]), rows, cols), rs8)
