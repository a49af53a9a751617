"""Pins of the MXFP4 oracle (oracle/mxfp4_oracle.py) to values fixed by the
OCP MX v1.0 E2M1 format and by the mathematics, not by the oracle itself:
hand-worked roundings at every tie and saturation point, hand-worked blocks,
the byte packing, and exactness properties (lossless FP4 -> FP8, lossless
conversions of values that are exactly representable)."""
import numpy as np
import pytest

from oracle import moe_oracle as O
from oracle import mxfp4_oracle as Q


# value -> E2M1 magnitude code; ties between neighbours go to the even code
E2M1_TABLE = [
    (0.0, 0), (0.1, 0), (0.25, 0), (0.2500001, 1), (0.5, 1), (0.7499999, 1), (0.75, 2),
    (1.0, 2), (1.25, 2), (1.2500001, 3), (1.5, 3), (1.75, 4), (2.0, 4), (2.5, 4),
    (2.5000001, 5), (3.0, 5), (3.5, 6), (4.0, 6), (5.0, 6), (5.0000001, 7), (6.0, 7),
    (7.0, 7), (1e30, 7),
]


@pytest.mark.parametrize("v,code", E2M1_TABLE)
def test_e2m1_rounding_table(v, code):
    assert int(Q.e2m1_code(np.array(v))) == code


def test_e2m1_decode_all_codes():
    expect = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = Q.e2m1_decode(np.arange(16))
    np.testing.assert_array_equal(got[:8], expect)
    np.testing.assert_array_equal(got[8:], -np.array(expect))
    assert np.signbit(got[8])  # code 8 is -0


def test_pack_nibbles():
    np.testing.assert_array_equal(Q.pack_e2m1(np.array([1, 2, 15, 0], np.uint8)), [0x21, 0x0F])
    c = np.random.default_rng(0).integers(0, 16, (4, 64)).astype(np.uint8)
    np.testing.assert_array_equal(Q.unpack_e2m1(Q.pack_e2m1(c)), c)


def _block(vals):
    b = np.zeros(32)
    b[:len(vals)] = vals
    return b[None, :]


def test_hand_worked_blocks():
    # a single 48 = 6 * 2^3: floor(log2 48) = 5, e = 5 - 2 = 3, 48 / 8 = 6 -> code 7
    c, s = Q.mx4_quantize(_block([48.0]), axis=1)
    assert s[0, 0] == 127 + 3 and c[0, 0] == 7 and not c[0, 1:].any()
    # all ones: e = 0 - 2 = -2, 1 * 4 = 4 -> code 6, value 4 * 2^-2 = 1
    c, s = Q.mx4_quantize(np.ones((1, 32)), axis=1)
    assert s[0, 0] == 125 and (c == 6).all()
    # one outlier: 100 -> e = 6 - 2 = 4; 100 / 16 = 6.25 saturates to 6 (96);
    # 1 / 16 = 0.0625 rounds to 0
    c, s = Q.mx4_quantize(_block([100.0] + [1.0] * 31), axis=1)
    assert s[0, 0] == 131 and c[0, 0] == 7 and (c[0, 1:] == 0).all()
    v = Q.mx4_dequantize(c, s, axis=1)
    assert v[0, 0] == 96.0
    # negative values keep the sign bit
    c, s = Q.mx4_quantize(_block([-3.0, 1.5]), axis=1)  # e = 1 - 2 = -1: -6 -> 0xF, 3 -> 5
    assert s[0, 0] == 126 and c[0, 0] == 0xF and c[0, 1] == 5


def test_zero_nan_and_tiny_blocks():
    z = np.zeros((1, 32))
    z[0, 3] = -0.0
    c, s = Q.mx4_quantize(z, axis=1)
    assert s[0, 0] == 0 and c[0, 3] == 8 and (np.delete(c[0], 3) == 0).all()
    for bad in (np.nan, np.inf, -np.inf):
        c, s = Q.mx4_quantize(_block([1.0, bad]), axis=1)
        assert s[0, 0] == 255 and not c.any()
        assert np.isnan(Q.mx4_dequantize(c, s, axis=1)).all()
    # amax 2^-140: the exponent clamps to -127 and 2^-140 * 2^127 = 2^-13 rounds to 0
    c, s = Q.mx4_quantize(_block([2.0 ** -140]), axis=1)
    assert s[0, 0] == 0 and c[0, 0] == 0


def _exact_fp4_values(rng, rows, cols):
    """Values m * 2^s, m on the E2M1 grid, with every row block's largest
    magnitude 4 or 6 times its 2^s (so the block scale is exactly 2^s)."""
    m = rng.choice(Q.E2M1_VALUES, (rows, cols)) * rng.choice([-1.0, 1.0], (rows, cols))
    m[:, ::32] = rng.choice([4.0, 6.0, -6.0], (rows, cols // 32))
    s = rng.integers(-20, 20, (rows, cols // 32))
    return m * np.repeat(np.ldexp(1.0, s), 32, axis=1)


def test_exact_values_round_trip():
    v = _exact_fp4_values(np.random.default_rng(1), 8, 128)
    c, s = Q.mx4_quantize(v, axis=1)
    np.testing.assert_array_equal(Q.mx4_dequantize(c, s, axis=1), v)


def test_fp4_to_fp8_is_lossless():
    rng = np.random.default_rng(2)
    c4 = rng.integers(0, 16, (4, 256)).astype(np.uint8)
    s4 = rng.integers(0, 255, (4, 8)).astype(np.uint8)  # every finite scale byte range
    s4[0, 0], s4[1, 1] = 0, 254
    c8, s8 = Q.mxfp8_from_mxfp4(c4, s4)
    np.testing.assert_array_equal(O.mx_dequantize(c8, s8, axis=1), Q.mx4_dequantize(c4, s4, axis=1))


def test_fp8_to_fp4_exact_on_fp4_values():
    v = _exact_fp4_values(np.random.default_rng(3), 8, 256)
    c8, s8 = O.mx_quantize(v, axis=1)
    assert np.array_equal(O.mx_dequantize(c8, s8, axis=1), v)  # E2M1 values are E4M3 values
    c4, s4 = Q.mxfp4_from_mxfp8(c8, s8)
    np.testing.assert_array_equal(Q.mx4_dequantize(c4, s4, axis=1), v)


def test_fp8_to_fp4_hand_worked():
    # an MXFP8 block holding 7 and 1 (scale 2^0): FP4 e = floor(log2 7) - 2 = 0,
    # 7 saturates to 6 and 1 stays 1 -> codes 7 and 2
    c8, s8 = O.mx_quantize(_block([7.0, 1.0]), axis=1)
    c4, s4 = Q.mxfp4_from_mxfp8(c8, s8)
    assert s4[0, 0] == 127 and c4[0, 0] == 7 and c4[0, 1] == 2


def test_row_to_col_exact_on_powers_of_two():
    """X[r, c] = +-2^(a_r + b_c) with exponents spanning 3 binades: every row
    block and every column block is exactly representable, so the column-wise
    copy decodes to X itself (transposed) whatever the scales."""
    rng = np.random.default_rng(4)
    a = rng.integers(0, 2, 64)
    b = rng.integers(0, 2, 128)
    x = np.ldexp(1.0, a[:, None] + b[None, :] + 5) * rng.choice([-1.0, 1.0], (64, 128))
    c4, s4 = Q.mx4_quantize(x, axis=1)
    cc, sc = Q.mxfp4_row_to_col(c4, s4)
    assert cc.shape == (128, 64) and sc.shape == (128, 2)
    np.testing.assert_array_equal(Q.mx4_dequantize(cc, sc, axis=1), x.T)


def test_row_to_col_recomputes_scales():
    """Hand-worked: rows 0..31 of column 0 hold 6 (in a row block with scale
    2^0) and 1 * 2^-3 = 0.125 in the others (row blocks scaled 2^-5). The
    column block's amax is 6, so its scale is 2^0 and 0.125 rounds to 0; the
    row scale of the small rows (2^-5) would have kept it."""
    x = np.zeros((32, 32))
    x[0, 0] = 6.0
    x[1:, 0] = 0.125
    x[1:, 1] = 0.125  # amax of rows 1..31 is 0.125: e = -3 - 2 = -5
    c4, s4 = Q.mx4_quantize(x, axis=1)
    assert s4[0, 0] == 127 and (s4[1:, 0] == 122).all()
    cc, sc = Q.mxfp4_row_to_col(c4, s4)
    assert sc[0, 0] == 127 and cc[0, 0] == 7 and (cc[0, 1:] == 0).all()
    # column 1: amax 0.125 -> scale 2^-5, 0.125 * 32 = 4 -> code 6
    assert sc[1, 0] == 122 and (cc[1, 1:] == 6).all()


def test_fp8_col_from_fp4_row_is_lossless_fp4_col():
    rng = np.random.default_rng(5)
    x = rng.normal(size=(64, 96)) * np.exp(rng.normal(size=(64, 1)))
    c4, s4 = Q.mx4_quantize(x, axis=1)
    c8c, s8c = Q.mxfp8_col_from_mxfp4_row(c4, s4)
    cc, sc = Q.mxfp4_row_to_col(c4, s4)
    np.testing.assert_array_equal(O.mx_dequantize(c8c, s8c, axis=1),
                                  Q.mx4_dequantize(cc, sc, axis=1))


def test_act4_chain_exact_on_powers_of_two():
    """The wgrad operand chain of the MXFP4 activation mode (row-wise MXFP8 ->
    row-wise MXFP4 -> column-wise MXFP4, groups padded to 32 rows) returns
    values that every step represents exactly: +-2^(a_r + b_c) spanning three
    binades in every row block and every column block. 50 rows: the last
    column block is padded with zero rows."""
    rng = np.random.default_rng(6)
    a = rng.integers(0, 2, 50)
    b = rng.integers(0, 2, 64)
    x = np.ldexp(1.0, a[:, None] + b[None, :] - 3) * rng.choice([-1.0, 1.0], (50, 64))
    np.testing.assert_array_equal(O.act4_cols_in_groups(x), x)


def test_act4_chain_is_coarser_than_mxfp8():
    """On random data the chain loses more than column-wise MXFP8 alone (E2M1
    keeps one mantissa bit against E4M3's three: about 5x the mean error
    here), and stays within the E2M1 rounding of its two FP4 steps (the
    row-wise FP8 step is finer than both)."""
    rng = np.random.default_rng(7)
    x = rng.normal(size=(96, 64))
    m8 = np.abs(O.mx_qdq_cols_in_groups(x) - x).mean()
    m4 = np.abs(O.act4_cols_in_groups(x) - x).mean()
    assert 3 * m8 < m4 < 8 * m8
    # per column block: |err| <= 2 * (half the largest E2M1 spacing, 1.0, times the
    # block scale 2^(floor(log2 amax) - 2)) plus the FP8 step
    amax = np.abs(x).reshape(3, 32, 64).max(axis=1)
    scale = np.ldexp(1.0, np.floor(np.log2(amax)).astype(int) - 2)
    err = np.abs(O.act4_cols_in_groups(x) - x).reshape(3, 32, 64)
    assert np.all(err <= 2.0 * scale[:, None, :] + 2.0 ** -4 * amax[:, None, :])


def test_planted_mxfp4_mistakes_are_caught(monkeypatch):
    """Plausible slips in the MXFP4 oracle fail the pins above: the E4M3
    exponent offset (8) in place of E2M1's (2); ties rounded away from zero;
    row -> column reusing the row scales."""
    # wrong emax: the all-ones block would get scale 2^-8 and saturate
    with monkeypatch.context() as m:
        m.setattr(Q, "E2M1_EMAX", 8)
        c, s = Q.mx4_quantize(np.ones((1, 32)), axis=1)
        assert not (s[0, 0] == 125 and (c == 6).all())
    # ties away from zero: 0.25 -> 0.5 and 2.5 -> 3 instead of 0 and 2
    def away(a):
        a = np.minimum(np.asarray(a, dtype=float), 6.0)
        d = np.abs(a[..., None] - Q.E2M1_VALUES)
        # the larger of two equidistant candidates
        return (7 - np.argmin(d[..., ::-1], axis=-1)).astype(np.uint8)
    assert int(away(np.array(0.25))) != 0 and int(away(np.array(2.5))) != 4
    # reusing row scales for the column blocks keeps 0.125 instead of rounding it to 0
    x = np.zeros((32, 32))
    x[0, 0] = 6.0
    x[1:, 0] = 0.125
    x[1:, 1] = 0.125
    c4, s4 = Q.mx4_quantize(x, axis=1)
    v = Q.mx4_dequantize(c4, s4, axis=1)  # row scales applied: 0.125 survives
    assert v[5, 0] == 0.125
    cc, sc = Q.mxfp4_row_to_col(c4, s4)
    assert Q.mx4_dequantize(cc, sc, axis=1)[0, 5] == 0.0  # the real conversion drops it
