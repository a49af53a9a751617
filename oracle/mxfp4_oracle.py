"""CPU oracle for MXFP4 activation compression: direct FP8 <-> FP4 conversion
and the scale-aware FP4 row-wise -> column-wise conversion.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
the CPU legs of ``bench.py`` may import it; the product path never calls it.

Sources:

[MXFP4-HOPPER]  the hgpu.org abstract on MXFP4 training of MoE models on
                Hopper: activations (and expert-parallel traffic) are kept in
                MXFP4 while the MoE GEMMs run in FP8; FP8 values are quantised
                to FP4 and de-quantised back directly, without a BF16 round
                trip, and the column-wise FP4 copy is produced from the
                row-wise one by a conversion that recomputes the block scales.
[OCPMX]         OCP Microscaling Formats (MX) v1.0: 32-element blocks share
                an E8M0 scale X = 2^(floor(log2 max|V|) - emax_elem); FP4 is
                E2M1 (1 sign, 2 exponent bits with bias 1, 1 mantissa bit; no
                Inf or NaN; values 0, 0.5, 1, 1.5, 2, 3, 4, 6; emax_elem = 2);
                elements round to nearest, ties to even, and saturate.

Readings where the sources are silent (each is repeated in the design notes):

* every conversion is defined on exact values: decode the input (exact in
  float64), then quantise with the [OCPMX] rule of the output format. FP8 ->
  FP4 and the row -> column conversion therefore equal quantising the decoded
  values; FP4 -> FP8 is lossless (every E2M1 value times its block scale is an
  E4M3 value times the MXFP8 scale the rule picks);
* "scale-aware" row -> column conversion: the column blocks get their own
  scales, computed from the decoded values of the 32 rows they span;
* an all-zero block gets scale byte 0 and zero elements that keep their sign
  (as for MXFP8); a block holding Inf or NaN gets scale byte 0xFF (NaN) and
  element codes 0 (E2M1 has no NaN code; the NaN scale makes the block NaN);
* two E2M1 codes per byte, element 2i in the low nibble, element 2i + 1 in the
  high nibble; scales use the same 512-byte tiled layout as MXFP8.
"""
from __future__ import annotations

import numpy as np

from oracle.moe_oracle import MX_BLOCK, _blocks, mx_dequantize, mx_quantize

f64 = np.float64

E2M1_EMAX = 2  # exponent of the largest E2M1 binade [OCPMX]
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])  # magnitude of codes 0..7


def e2m1_code(a):
    """Magnitude code (0..7) of the E2M1 value nearest to a >= 0.

    Nearest by absolute distance over the eight magnitudes; at a tie the even
    code (mantissa bit 0) wins. Values above 6 are nearest to 6: saturation,
    applied first by clipping (at very large a the float64 distances to the
    eight magnitudes would all be equal).
    """
    a = np.minimum(np.asarray(a, dtype=f64), 6.0)
    d = np.abs(a[..., None] - E2M1_VALUES)
    dmin = d.min(axis=-1, keepdims=True)
    cand = d == dmin
    even = cand & (np.arange(8) % 2 == 0)
    pick = np.where(even.any(axis=-1, keepdims=True), even, cand)
    return np.argmax(pick, axis=-1).astype(np.uint8)


def e2m1_decode(code):
    c = np.asarray(code, dtype=np.int64)
    return np.where(c & 8, -1.0, 1.0) * E2M1_VALUES[c & 7]


def e8m0_value(s):
    s = np.asarray(s, dtype=np.int64)
    return np.where(s == 255, np.nan, np.ldexp(1.0, s - 127))


def mx4_quantize(a, axis=-1):
    """MXFP4 (E2M1 elements, E8M0 scales) with 32-blocks along ``axis``.

    Per block: amax = max |v|; e = clamp(floor(log2 amax) - 2, -127, 127)
    (amax = 0 -> -127); element code = sign | e2m1_code(|v| * 2^-e).
    Returns (codes uint8 0..15 shaped like a, scales uint8 with the axis / 32).
    """
    shape = np.shape(a)
    axis = axis % len(shape)
    blk = _blocks(a, axis)  # [outer, n/32, 32, inner]
    amax = np.abs(blk).max(axis=2)
    finite = np.isfinite(amax)
    _, ex = np.frexp(np.where(finite, amax, 0.0))  # amax = m 2^ex, m in [0.5, 1)
    e = np.clip(np.where(finite & (amax > 0), ex - 1 - E2M1_EMAX, -127), -127, 127)
    scaled = np.abs(np.where(finite[:, :, None, :], blk, 0.0)) * np.ldexp(1.0, -e)[:, :, None, :]
    codes = e2m1_code(scaled) | (np.signbit(blk).astype(np.uint8) << 3)
    codes = np.where(finite[:, :, None, :], codes, 0).astype(np.uint8)
    scales = np.where(finite, e + 127, 255).astype(np.uint8)
    sshape = shape[:axis] + (shape[axis] // MX_BLOCK,) + shape[axis + 1:]
    return codes.reshape(shape), scales.reshape(sshape)


def mx4_dequantize(codes, scales, axis=-1):
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1)
    v = e2m1_decode(c).reshape(c.shape[:-1] + (c.shape[-1] // MX_BLOCK, MX_BLOCK))
    v = v * e8m0_value(s)[..., None]
    return np.moveaxis(v.reshape(c.shape), -1, axis)


def pack_e2m1(codes):
    """Bytes of codes [..., n] (n even): element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed):
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# ---------------------------------------------------------------------------
# The conversions [MXFP4-HOPPER], on [rows, cols] matrices whose row-wise
# blocks run along cols.
# ---------------------------------------------------------------------------

def mxfp4_from_mxfp8(c8, s8):
    """Direct FP8 -> FP4: row-wise MXFP8 (codes [rows, cols], scales
    [rows, cols/32]) to row-wise MXFP4 over the same blocks."""
    return mx4_quantize(mx_dequantize(c8, s8, axis=1), axis=1)


def mxfp8_from_mxfp4(c4, s4):
    """FP4 -> FP8 de-quantisation: row-wise MXFP4 to row-wise MXFP8 by the
    MXFP8 rule on the decoded values (lossless)."""
    return mx_quantize(mx4_dequantize(c4, s4, axis=1), axis=1)


def mxfp4_row_to_col(c4, s4):
    """Row-wise MXFP4 [rows, cols] to column-wise MXFP4 stored transposed:
    codes [cols, rows] and scales [cols, rows/32], blocks of 32 rows with
    scales recomputed from the decoded values."""
    v = mx4_dequantize(c4, s4, axis=1)
    c, s = mx4_quantize(v, axis=0)
    return c.T.copy(), s.T.copy()


def mxfp8_col_from_mxfp4_row(c4, s4):
    """Row-wise MXFP4 to the column-wise MXFP8 operand of a weight-gradient
    GEMM: the row -> column conversion, then FP4 -> FP8 (stored transposed,
    codes [cols, rows], scales [cols, rows/32])."""
    cc, sc = mxfp4_row_to_col(c4, s4)
    return mx_quantize(mx4_dequantize(cc, sc, axis=1), axis=1)
