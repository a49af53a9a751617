"""The grouped GEMMs' tile order, run on the host through moe_selftest_tile_order
(the same band_order function the kernels call per tile). No GPU needed.

Every expert's grid must be visited exactly once in any configuration; the
Mixtral-shape experts must keep the plain orders (m-tiles fastest, or n-tiles
fastest for a weight gradient whose A is the larger operand); the experts of
the T=65536 workload must run in the bands the design states.
"""
import random

import pytest

from mixture_experts_expert_sort_b300 import binding as B

WAVE2 = 148  # two waves of the 74 CTA pairs of a B300
SHARE = 32 << 20  # the L2 share of the resident band, bytes


def order(mtiles, ntiles, band_rows, prefer_m=True, min_band=WAVE2, tile_m=256, tile_n=256):
    mt, nt = B.selftest_tile_order(mtiles, ntiles, tile_m, tile_n, band_rows, prefer_m, min_band)
    return list(zip(mt.tolist(), nt.tolist()))


def rows(K, elt):
    return SHARE // elt // K


def test_every_tile_once_on_random_grids():
    rng = random.Random(5)
    for _ in range(400):
        mtiles, ntiles = rng.randint(1, 90), rng.randint(1, 130)
        band_rows = rng.choice([0, 1, 255, 256, 700, 1116, 5000, 11718, 1 << 40])
        o = order(mtiles, ntiles, band_rows, rng.random() < 0.5, rng.choice([0, 1, 148, 300]),
                  rng.choice([128, 256]), rng.choice([128, 256]))
        assert sorted(o) == [(m, n) for m in range(mtiles) for n in range(ntiles)]


@pytest.mark.parametrize("name,mtiles,ntiles,K,elt,prefer_m", [
    ("BF16 FC1, 2,176 rows per expert", 9, 112, 4096, 2, True),
    ("BF16 FC1 dgrad", 9, 16, 28672, 2, True),
    ("BF16 FC2", 9, 16, 14336, 2, True),
    ("MXFP8 FC1, 4,224 rows per expert", 17, 112, 4096, 1, True),
    ("MXFP8 FC1 dgrad", 17, 16, 28672, 1, True),
    ("MXFP8 FC2", 17, 16, 14336, 1, True),
    ("MXFP8 FC1 wgrad (M = H)", 16, 112, 4224, 1, True),
    ("MXFP8 FC2 wgrad (M = F > N = H)", 56, 16, 4224, 1, False),
])
def test_mixtral_shapes_keep_the_plain_order(name, mtiles, ntiles, K, elt, prefer_m):
    o = order(mtiles, ntiles, rows(K, elt), prefer_m)
    if prefer_m:
        assert o == [(m, n) for n in range(ntiles) for m in range(mtiles)], name
    else:
        assert o == [(m, n) for m in range(mtiles) for n in range(ntiles)], name


def _bands(o, along_m, g, other):
    """Check that o runs in bands of g tiles of the banded index, each band
    visiting all `other` tiles with the banded index fastest."""
    per = g * other
    for b in range(0, len(o), per):
        band = o[b:b + per]
        idx = [m if along_m else n for m, n in band]
        assert set(idx) == set(range(b // per * g, b // per * g + len(set(idx))))
        first = idx[:len(set(idx))]
        assert first == sorted(first)  # banded index fastest


def test_long_workload_runs_in_bands():
    # 16,384 rows per expert (T = 65536, top-2, E = 8), MXFP8 (one-byte elements)
    fc1 = order(64, 112, rows(4096, 1))
    _bands(fc1, True, 32, 112)
    assert fc1[:3] == [(0, 0), (1, 0), (2, 0)] and fc1[32] == (0, 1)
    dgrad = order(64, 16, rows(28672, 1))
    _bands(dgrad, False, 4, 64)
    assert dgrad[:5] == [(0, 0), (0, 1), (0, 2), (0, 3), (1, 0)]
    wgrad = order(16, 112, rows(16384, 1))  # FC1 wgrad: M = H, K = the expert's rows
    _bands(wgrad, True, 8, 112)


def test_short_bands_fall_back_to_the_plain_order():
    # a band of 2 n-tiles x 9 m-tiles would hold 18 tiles, under two waves
    o = order(9, 16, rows(28672, 2))
    assert o == [(m, n) for n in range(16) for m in range(9)]
    o = order(9, 16, rows(28672, 2), min_band=0)  # allowed: bands of 2 n-tiles
    assert o[:4] == [(0, 0), (0, 1), (1, 0), (1, 1)]


def test_bad_arguments():
    with pytest.raises(B.MoeError):
        B.selftest_tile_order(0, 4, 256, 256, 100, True, 0)
    with pytest.raises(B.MoeError):
        B.selftest_tile_order(4, 4, 256, 256, -1, True, 0)
