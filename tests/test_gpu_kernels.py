"""Parity of the memory-bound kernels (route, expert sort, permute, unpermute,
MXFP8 quantise, route backward) with the CPU oracle, through the C ABI.

Integer and byte outputs must match bit-exactly; fp32/bf16 sums within the
rounding of one fp32 accumulation and one bf16 rounding.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.helpers import f64, i32, u8, scales_tiled_to_rowmajor, bf16_round

pytestmark = pytest.mark.gpu

DEV = "cuda"


def B():
    from mixture_experts_expert_sort_b300 import binding
    return binding


def _logits(T, E, seed, ties=False):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn((T, E), generator=g)
    if ties:
        lg[::3] = torch.round(lg[::3])
        lg[1::5, 0] = 0.0
        if E > 1:
            lg[1::5, 1] = -0.0
    return lg


@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (257, 4, 2), (4096, 8, 2), (3001, 64, 6),
                                   (1000, 256, 8), (513, 37, 5), (100, 8, 8)])
@pytest.mark.parametrize("ties", [False, True])
def test_route(T, E, k, ties):
    lg = _logits(T, E, T + E + k, ties)
    idx, w = B().moe_route(lg.to(DEV), k)
    ridx, rw = O.route(lg.numpy(), k)
    np.testing.assert_array_equal(i32(idx), ridx)
    assert np.max(np.abs(f64(w) - rw)) <= 2e-6


def test_route_empty():
    idx, w = B().moe_route(torch.zeros((0, 8), device=DEV), 2)
    assert idx.shape == (0, 2)


@pytest.mark.parametrize("align", [1, 32, 128])
@pytest.mark.parametrize("T,E,k,skew", [(256, 4, 2, 0), (8192, 8, 2, 0), (16384, 64, 6, 1),
                                        (1000, 3, 3, 0), (2049, 16, 1, 2), (7, 64, 6, 1)])
def test_permute_plan(T, E, k, skew, align):
    lg = _logits(T, E, 10 * T + E, ties=True)
    if skew == 1:
        lg[:, E - 4:] -= 1e4  # experts with no tokens
        lg[:, 0] += 3.0  # one hot expert
    if skew == 2:
        lg[:, 5] += 1e4  # every token on one expert
    idx, _ = B().moe_route(lg.to(DEV), k)
    plan = B().moe_permute_plan(idx, E, align)
    counts, offsets, dest, src = O.permute_plan(i32(idx), E, align)
    np.testing.assert_array_equal(i32(plan["counts"]), counts)
    np.testing.assert_array_equal(i32(plan["offsets"]), offsets)
    np.testing.assert_array_equal(i32(plan["dest"])[:T * k], dest)
    gsrc = i32(plan["src"])
    np.testing.assert_array_equal(gsrc[:len(src)], src)
    assert np.all(gsrc[len(src):] == -1)
    assert B().device_error() == 0


def test_permute_plan_bad_index_sets_error_flag():
    idx = torch.tensor([[0, 1], [2, 9], [1, 0]], dtype=torch.int32, device=DEV)
    plan = B().moe_permute_plan(idx, 4, 1)
    flags = B().device_error()
    assert flags & B().MOE_DEVERR_BAD_INDEX
    d = i32(plan["dest"])
    assert d[3] == -1
    assert list(i32(plan["counts"])) == [2, 2, 1, 0]


@pytest.mark.parametrize("T,H,E,k", [(256, 128, 4, 2), (1500, 1024, 8, 2), (777, 2048, 64, 6)])
def test_permute_unpermute(T, H, E, k):
    g = torch.Generator().manual_seed(T + H)
    x = torch.randn((T, H), generator=g).to(torch.bfloat16)
    lg = _logits(T, E, T * 7)
    idx, w = B().moe_route(lg.to(DEV), k)
    plan = B().moe_permute_plan(idx, E, 128)
    rows = int(plan["offsets"][-1].item())
    xp, p_rows = B().moe_permute(x.to(DEV), plan["dest"], plan["offsets"], plan["counts"], k,
                                 rows, w=w)
    ref = O.permute(f64(x), i32(plan["dest"])[:T * k], k, rows)
    np.testing.assert_array_equal(f64(xp), ref)
    pref = np.zeros(rows)
    pref[i32(plan["dest"])[:T * k]] = f64(w).reshape(-1)
    np.testing.assert_array_equal(f64(p_rows), pref)
    # unpermute with weights: fp32 accumulation, one bf16 rounding
    y = torch.randn((rows, H), generator=g).to(torch.bfloat16)
    out = B().moe_unpermute(y.to(DEV), plan["dest"], T, k, w=w)
    oref = O.unpermute(f64(y), i32(plan["dest"])[:T * k], k, f64(w))
    # one bf16 rounding of the result (half an ulp, <= 2^-8 relative) plus the
    # fp32 accumulation error of k products (<= k * 2^-24 * sum |w y|)
    mag = O.unpermute(np.abs(f64(y)), i32(plan["dest"])[:T * k], k, np.abs(f64(w)))
    bound = np.abs(oref) * 2.0 ** -8 + (k + 1) * 2.0 ** -24 * mag + 1e-30
    assert np.all(np.abs(f64(out) - oref) <= bound)
    # without weights (the backward of the permute): identity experts sum back to k*x
    back = B().moe_unpermute(xp, plan["dest"], T, k)
    np.testing.assert_array_equal(f64(back), bf16_round(k * f64(x)))


def _quant_input(rows, cols, seed, special=True):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((rows, cols), generator=g) * torch.exp2(torch.randint(-20, 20, (rows, 1),
                                                                          generator=g).float())
    if special:
        x[3, :64] = 0.0  # zero blocks
        x[5, 32:64] = -0.0
        x[7, 0] = 500.0  # saturating element
        x[9, 5] = 1e-41  # tiny
        x[rows // 2] *= 100.0  # outlier row
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 256), (1024, 2048)])
def test_mxfp8_quantize_both_directions(rows, cols):
    x = _quant_input(rows, cols, rows + cols)
    q = B().mxfp8_quantize(x.to(DEV))
    xr = f64(x)
    c_row, s_row = O.mx_quantize(xr, axis=1)
    c_col, s_col = O.mx_quantize(xr, axis=0)
    np.testing.assert_array_equal(u8(q["q_row"]), c_row)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(q["s_row"]), rows, cols), s_row)
    np.testing.assert_array_equal(u8(q["q_col"]), c_col.T)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(q["s_col"]), cols, rows), s_col.T)


@pytest.mark.parametrize("rows,cols", [(128, 128), (384, 640)])
def test_mxfp8_scales_to_canonical(rows, cols):
    """The device conversion of both scale copies to row-major bytes equals
    the oracle's scales (row-wise [rows, cols/32]; column-wise [cols, rows/32])."""
    x = _quant_input(rows, cols, 11 * rows + cols)
    q = B().mxfp8_quantize(x.to(DEV))
    _, s_row = O.mx_quantize(f64(x), axis=1)
    _, s_col = O.mx_quantize(f64(x), axis=0)
    np.testing.assert_array_equal(u8(B().mxfp8_scales_to_canonical(q["s_row"], rows, cols)), s_row)
    np.testing.assert_array_equal(u8(B().mxfp8_scales_to_canonical(q["s_col"], cols, rows)),
                                  s_col.T)


def test_mxfp8_quantize_large_ragged_work_items():
    """A matrix large enough that every CTA takes work items of several row
    tiles (85,376 x 4,224: items of 3 row tiles, the last item of each strip
    one tile short, and a last strip 128 columns wide), bit-exact against both
    oracles' quantisers on sampled rows and 32-row blocks, the last ones included."""
    from oracle import cpp_oracle as CO
    rows, cols = 85376, 4224
    g = torch.Generator(device=DEV).manual_seed(21)
    x = (torch.randn((rows, cols), generator=g, device=DEV) *
         torch.exp2(torch.randint(-12, 12, (rows, 1), generator=g, device=DEV).float()))
    x = x.to(torch.bfloat16)
    q = B().mxfp8_quantize(x)
    rng = np.random.default_rng(21)
    pick_rows = np.unique(np.concatenate([[0, 1, rows - 1, rows - 32, rows - 96],
                                          rng.choice(rows, 40, replace=False)]))
    xr = f64(x[torch.as_tensor(pick_rows, device=DEV)])
    s_row = scales_tiled_to_rowmajor(u8(q["s_row"]), rows, cols)
    s_col = scales_tiled_to_rowmajor(u8(q["s_col"]), cols, rows)
    for quantize in (O.mx_quantize, CO.mx_quantize):
        c, s = quantize(xr, axis=1)
        np.testing.assert_array_equal(u8(q["q_row"][torch.as_tensor(pick_rows, device=DEV)]), c)
        np.testing.assert_array_equal(s_row[pick_rows], s)
    blocks = np.unique(np.concatenate([[0, rows // 32 - 1, rows // 32 - 3],
                                       rng.choice(rows // 32, 12, replace=False)]))
    for b in blocks:
        xb = f64(x[32 * b:32 * b + 32])
        for quantize in (O.mx_quantize, CO.mx_quantize):
            c, s = quantize(xb, axis=0)
            np.testing.assert_array_equal(u8(q["q_col"][:, 32 * b:32 * b + 32]).T, c)
            np.testing.assert_array_equal(s_col[:, b], s[0])


def test_mxfp8_quantize_nonfinite_block():
    x = _quant_input(128, 128, 3, special=False)
    x[2, 40] = float("inf")
    x[6, 100] = float("nan")
    q = B().mxfp8_quantize(x.to(DEV), dirs=B().QUANT_ROWWISE)
    c, s = O.mx_quantize(f64(x), axis=1)
    np.testing.assert_array_equal(u8(q["q_row"]), c)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(q["s_row"]), 128, 128), s)


def test_mxfp8_quantize_fused_permute():
    T, H, E, k = 300, 256, 8, 2
    x = _quant_input(T, H, 77)
    idx, w = B().moe_route(_logits(T, E, 5).to(DEV), k)
    plan = B().moe_permute_plan(idx, E, 128)
    rows = int(plan["offsets"][-1].item())
    q = B().mxfp8_quantize(x.to(DEV), rows=rows, src=plan["src"], src_div=k)
    xp = O.permute(f64(x), i32(plan["dest"])[:T * k], k, rows)
    c_row, s_row = O.mx_quantize(xp, axis=1)
    c_col, s_col = O.mx_quantize(xp, axis=0)
    np.testing.assert_array_equal(u8(q["q_row"]), c_row)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(q["s_row"]), rows, H), s_row)
    np.testing.assert_array_equal(u8(q["q_col"]), c_col.T)
    np.testing.assert_array_equal(scales_tiled_to_rowmajor(u8(q["s_col"]), H, rows), s_col.T)


@pytest.mark.parametrize("use_dest", [False, True])
def test_route_backward(use_dest):
    T, E, k, n_part = 1000, 64, 6, 5
    idx, w = B().moe_route(_logits(T, E, 9).to(DEV), k)
    g = torch.Generator().manual_seed(4)
    if use_dest:
        plan = B().moe_permute_plan(idx, E, 128)
        rows = int(plan["offsets"][-1].item())
        dp = torch.randn((rows, n_part), generator=g)
        dl = B().moe_route_backward(dp.to(DEV), w, idx, E, dest=plan["dest"])
        dsum = f64(dp)[i32(plan["dest"])[:T * k]].sum(1).reshape(T, k)
    else:
        dp = torch.randn((T * k, n_part), generator=g)
        dl = B().moe_route_backward(dp.to(DEV), w, idx, E)
        dsum = f64(dp).sum(1).reshape(T, k)
    ref = O.route_backward(dsum, f64(w), i32(idx), E)
    assert np.max(np.abs(f64(dl) - ref)) <= 1e-5 * max(1.0, np.max(np.abs(ref)))
