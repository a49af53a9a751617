"""Pins for the C++ oracle (oracle/moe_oracle.cpp), independent of the CUDA path.

The C++ oracle is the plain per-expert loop written a second time, in a
different language and without library primitives. It is pinned the same way
as the numpy oracle, against what the pages and the mathematics fix:

* brute force for top-k (exact ties, +0/-0) and for the expert-sort plan;
* the closed form of the k = 2 routing weights;
* the hand-worked MXFP8 blocks of tests/golden/mxfp8_blocks.txt, every E4M3
  byte, the library's float8 conversion, exact round trips on representable
  blocks, and hand-worked E2M1 codes;
* E = 1, k = 1 reducing to a dense SwiGLU MLP, central differences of the
  exact backward, and invariance under a permutation of the tokens;
* for the router: written-out dot products, an aux loss of exactly 1 under
  balanced routing, its one-expert closed form, and central differences of
  the aux loss through the projection;
* the MXFP8 and MXFP4-activation layers equal to the block-scaled reference
  of tests/test_oracle_mx_directions.py, whose only quantised product is a
  GEMM blocked along its own reduction index;
* and agreement with the numpy oracle on random layers.

Planted mistakes are compiled into copies of the C++ source (one textual
change each, in a temporary directory) and must trip one of these pins.
"""
import ctypes
import itertools
import os
import subprocess

import numpy as np
import pytest
import torch

from oracle import cpp_oracle as CO
from oracle import moe_oracle as O
from oracle import mxfp4_oracle as Q
from tests.test_oracle_mx_directions import CASES, _layer, _rel, reference_layer
from tests.test_oracle_pins import _brute_plan, _brute_topk, _dense_swiglu_mlp, _golden_blocks


def _layer_cpp(x, lg, W1, W2, dout, k, mode="bf16", save_bf16=True):
    r = CO.layer(x, lg, W1, W2, dout, k, mode, save_bf16)
    return {n: r[n] for n in ("out", "dX", "dW1", "dW2", "dlogits")}


# --------------------------------------------------------------------- routing

@pytest.mark.parametrize("E,k", [(4, 2), (8, 2), (64, 6), (5, 5), (1, 1)])
def test_cpp_route_matches_brute_force(E, k):
    rng = np.random.default_rng(E * 100 + k + 1)
    lg = rng.standard_normal((300, E))
    lg[::3] = np.round(lg[::3])  # many exact ties
    lg[1::7, 0] = 0.0
    if E > 1:
        lg[1::7, 1] = -0.0  # +0 and -0 tie
    idx, w = CO.route(lg, k)
    for t in range(lg.shape[0]):
        assert list(idx[t]) == _brute_topk(list(lg[t]), k)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-15)


def test_cpp_route_weights_closed_form_k2():
    rng = np.random.default_rng(8)
    lg = rng.standard_normal((500, 8)) * 3
    idx, w = CO.route(lg, 2)
    l0 = lg[np.arange(500), idx[:, 0]]
    l1 = lg[np.arange(500), idx[:, 1]]
    np.testing.assert_allclose(w[:, 0], 1.0 / (1.0 + np.exp(l1 - l0)), rtol=1e-14)


def test_cpp_route_backward_is_softmax_jacobian():
    # dl_j = sum_i dp_i dw_i/dl_j with dw_i/dl_j = w_i (delta_ij - w_j), written out
    rng = np.random.default_rng(9)
    T, E, k = 50, 6, 3
    lg = rng.standard_normal((T, E))
    idx, w = CO.route(lg, k)
    dp = rng.standard_normal((T, k))
    dl = CO.route_backward(dp, w, idx, E)
    for t in range(T):
        ref = np.zeros(E)
        for j in range(k):
            ref[idx[t, j]] = sum(dp[t, i] * w[t, i] * ((i == j) - w[t, j]) for i in range(k))
        np.testing.assert_allclose(dl[t], ref, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- permute plan

@pytest.mark.parametrize("align", [1, 32, 128])
@pytest.mark.parametrize("E,k,T", [(4, 2, 37), (8, 2, 100), (64, 6, 50), (3, 3, 20), (1, 1, 9)])
def test_cpp_plan_matches_brute_force(E, k, T, align):
    rng = np.random.default_rng(E + k + T + align + 1)
    idx, _ = CO.route(rng.standard_normal((T, E)), k)
    counts, offsets, dest, src = CO.permute_plan(idx, E, align)
    bc, bo, bd = _brute_plan(idx, E, align)
    assert list(counts) == bc and list(offsets) == bo and list(dest) == bd
    assert len(src) == offsets[-1]
    for i, r in enumerate(dest):
        assert src[r] == i
    assert (src == -1).sum() == offsets[-1] - T * k


def test_cpp_plan_empty_experts_and_identity_experts():
    counts, offsets, dest, _ = CO.permute_plan(np.full((10, 1), 2, dtype=np.int32), 4, 32)
    assert list(counts) == [0, 0, 10, 0] and list(offsets) == [0, 0, 0, 32, 32]
    assert list(dest) == list(range(10))
    rng = np.random.default_rng(4)
    T, H, E, k = 40, 16, 5, 3
    x = rng.standard_normal((T, H))
    idx, w = CO.route(rng.standard_normal((T, E)), k)
    _, offsets, dest, _ = CO.permute_plan(idx, E, 8)
    xp = CO.permute(x, dest, k, int(offsets[-1]))
    np.testing.assert_allclose(CO.unpermute(xp, dest, k, w), x, rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(CO.unpermute(xp, dest, k), k * x)
    used = np.zeros(int(offsets[-1]), bool)
    used[dest] = True
    assert np.all(xp[~used] == 0)


# ------------------------------------------------------------------ MX formats

@pytest.mark.parametrize("case", _golden_blocks(), ids=lambda c: c[0])
def test_cpp_mxfp8_hand_worked_blocks(case):
    name, vals, scale, codes = case
    c, s = CO.mx_quantize(np.array([vals]), axis=1)
    assert int(s[0, 0]) == scale
    assert [int(v) for v in c[0]] == codes
    c0, s0 = CO.mx_quantize(np.array([vals]).T, axis=0)  # the same block down a column
    assert int(s0[0, 0]) == scale and [int(v) for v in c0[:, 0]] == codes


def _lib_e4m3(codes):
    return torch.from_numpy(np.asarray(codes, dtype=np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def test_cpp_every_e4m3_byte_round_trips():
    # Each finite byte's value (from the library's float8 table), placed in a
    # block whose largest element is 256 (scale byte 127, e = 0), quantises
    # back to the same byte.
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = _lib_e4m3(codes)
    n = len(codes)
    flat = np.zeros((n + 30) // 31 * 31)
    flat[:n] = vals
    blocks = np.zeros((flat.size // 31, 32))
    blocks[:, 0] = 256.0
    blocks[:, 1:] = flat.reshape(-1, 31)
    c, s = CO.mx_quantize(blocks, axis=1)
    assert np.all(s == 127)
    np.testing.assert_array_equal(c[:, 1:].reshape(-1)[:n], codes)


def test_cpp_e4m3_rounding_matches_library_conversion():
    rng = np.random.default_rng(21)
    grid = _lib_e4m3(np.arange(0, 127))
    v = np.concatenate([rng.uniform(0, 448, 60000), np.exp2(rng.uniform(-12, 8.8, 60000)),
                        (grid[:-1] + grid[1:]) / 2])  # exact midpoints
    v = v.astype(np.float32).astype(np.float64)
    v = v[v <= 448]
    v = np.concatenate([v, np.zeros((-len(v)) % 31)])
    blocks = np.zeros((len(v) // 31, 32))
    blocks[:, 0] = 256.0  # scale 2^0: the block's values are rounded as they are
    blocks[:, 1:] = v.reshape(-1, 31)
    c, s = CO.mx_quantize(blocks, axis=1)
    assert np.all(s == 127)
    lib = torch.from_numpy(blocks[:, 1:].copy()).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    np.testing.assert_array_equal(c[:, 1:], lib)


def test_cpp_mxfp8_round_trip_and_saturation():
    rng = np.random.default_rng(22)
    grid = _lib_e4m3(np.arange(0, 127))
    for s in [-20, -3, 0, 7, 40]:
        vals = rng.choice(grid, size=(64, 32))
        vals[:, 0] = rng.choice(grid[grid >= 256], size=64)  # the top binade sets the scale
        vals *= np.where(rng.random((64, 32)) < 0.5, -1, 1) * 2.0 ** s
        c, sc = CO.mx_quantize(vals, axis=1)
        assert np.all(sc == s + 127)
        back = _lib_e4m3(c) * 2.0 ** s
        np.testing.assert_array_equal(back, vals)
    blk = np.ones((1, 32))
    blk[0, :4] = [500.0, 470.0, 448.0, -460.0]  # amax 500 -> e = 0, three saturate
    c, s = CO.mx_quantize(blk, axis=1)
    assert s[0, 0] == 127 and list(c[0, :4]) == [0x7E, 0x7E, 0x7E, 0xFE]
    blk[0, 7] = np.nan
    c, s = CO.mx_quantize(blk, axis=1)
    assert s[0, 0] == 255 and np.all(c == 0x7F)


def test_cpp_e2m1_hand_worked_codes():
    # amax 6 -> floor(log2 6) - 2 = 0 -> scale byte 127; E2M1 magnitudes
    # 0, .5, 1, 1.5, 2, 3, 4, 6 are codes 0..7, sign in bit 3; ties to the even code:
    # .25 -> 0, .75 -> 1 (2 is even: 1.0), 1.25 -> 1.0 (2), 1.75 -> 2.0 (4),
    # 2.5 -> 2.0 (4), 3.5 -> 4.0 (6), 5 -> 4.0 (6), 7 saturates to 6 (7), -3 -> 8|5.
    vals = [6.0, 0.0, 0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 1.75, 2.0, 2.5, 3.0, 3.5, 4.0, 5.0, -3.0,
            -0.0] + [0.0] * 15
    want = [7, 0, 0, 1, 2, 2, 2, 3, 4, 4, 4, 5, 6, 6, 6, 13, 8] + [0] * 15
    c, s = CO.mx_quantize(np.array([vals]), axis=1, fmt=4)
    assert s[0, 0] == 127 and [int(v) for v in c[0]] == want
    blk = np.array([vals]) * 2.0 ** -5  # the same block at another scale
    blk[0, 0] = 6.0 * 2.0 ** -5 * 1.2  # amax 7.2 * 2^-5 -> still binade 2^2 * 2^-5
    c, s = CO.mx_quantize(blk, axis=1, fmt=4)
    assert s[0, 0] == 127 - 5 and [int(v) for v in c[0, 1:]] == want[1:]


def test_cpp_mx_quantize_agrees_with_numpy_oracle():
    rng = np.random.default_rng(23)
    a = rng.standard_normal((64, 96)) * np.exp2(rng.integers(-140, 140, (64, 1)))
    a[0, :32] = 0.0
    a[1, :32] = -0.0
    a[2, 5] = 1e4
    a[3, 7] = np.inf
    for axis in (0, 1):
        c, s = CO.mx_quantize(a, axis=axis)
        rc, rs = O.mx_quantize(a, axis=axis)
        np.testing.assert_array_equal(c, rc)
        np.testing.assert_array_equal(s, rs)
        b = np.where(np.isfinite(a), a, 1.0)
        c4, s4 = CO.mx_quantize(b, axis=axis, fmt=4)
        rc4, rs4 = Q.mx4_quantize(b, axis=axis)
        np.testing.assert_array_equal(c4, rc4)
        np.testing.assert_array_equal(s4, rs4)


# ------------------------------------------------------------------- the layer

def test_cpp_single_expert_top1_is_dense_swiglu_mlp():
    rng = np.random.default_rng(24)
    T, H, F = 5, 6, 4
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((1, H, 2 * F))
    W2 = rng.standard_normal((1, F, H))
    r = CO.layer(x, rng.standard_normal((T, 1)), W1, W2, np.zeros((T, H)), 1)
    np.testing.assert_allclose(r["out"], _dense_swiglu_mlp(x, W1[0], W2[0]), rtol=1e-12,
                               atol=1e-12)


def _tiny(seed, T=7, H=5, F=4, E=3):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((T, H)), rng.standard_normal((T, E)),
            rng.standard_normal((E, H, 2 * F)) * 0.5, rng.standard_normal((E, F, H)) * 0.5,
            rng.standard_normal((T, H)))


def test_cpp_gradients_central_differences():
    x, lg, W1, W2, dout = _tiny(31)
    k = 2
    assert np.min(np.abs(np.diff(np.sort(lg, axis=1), axis=1))) > 1e-3
    g = CO.layer(x, lg, W1, W2, dout, k, save_bf16=False)

    def loss():
        return float((CO.layer(x, lg, W1, W2, dout, k)["out"] * dout).sum())

    eps = 1e-6
    for name, arr, grad in [("x", x, g["dX"]), ("W1", W1, g["dW1"]), ("W2", W2, g["dW2"]),
                            ("logits", lg, g["dlogits"])]:
        num = np.zeros_like(arr)
        for pos in itertools.product(*[range(s) for s in arr.shape]):
            old = arr[pos]
            arr[pos] = old + eps
            lp = loss()
            arr[pos] = old - eps
            lm = loss()
            arr[pos] = old
            num[pos] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(num - grad) / np.linalg.norm(num)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("mode", ["bf16", "mxfp8"])
def test_cpp_token_permutation_invariance(mode):
    rng = np.random.default_rng(25)
    T, H, F, E, k = 96, 64, 64, 4, 2
    x, lg = rng.standard_normal((T, H)), rng.standard_normal((T, E))
    W1 = rng.standard_normal((E, H, 2 * F)) * 0.1
    W2 = rng.standard_normal((E, F, H)) * 0.1
    dout = rng.standard_normal((T, H))
    a = _layer_cpp(x, lg, W1, W2, dout, k, mode)
    perm = rng.permutation(T)
    b = _layer_cpp(x[perm], lg[perm], W1, W2, dout[perm], k, mode)
    for n in ("out", "dX", "dlogits"):  # row-local in both modes
        np.testing.assert_allclose(b[n], a[n][perm], rtol=1e-12, atol=1e-12)
    if mode == "bf16":  # the MXFP8 wgrads block their tokens in token order
        for n in ("dW1", "dW2"):
            np.testing.assert_allclose(b[n], a[n], rtol=1e-10, atol=1e-12)


TOL = 1e-10  # relative Frobenius error: summation order only


@pytest.mark.parametrize("T,H,F,E,k,gs", CASES)
@pytest.mark.parametrize("mode", ["mxfp8", "mxfp8_act4"])
def test_cpp_mx_layer_equals_block_scaled_reference(T, H, F, E, k, gs, mode):
    x, lg, W1, W2, dout = _layer(41 + T, T, H, F, E, k, gs)
    ref = reference_layer(x, lg, W1, W2, dout, k, act4=mode == "mxfp8_act4")
    got = _layer_cpp(x, lg, W1, W2, dout, k, mode)
    for n in ref:
        assert _rel(got[n], ref[n]) < TOL, (n, _rel(got[n], ref[n]))


@pytest.mark.parametrize("save_bf16", [True, False])
def test_cpp_bf16_layer_equals_reference(save_bf16):
    T, H, F, E, k, gs = CASES[1]
    x, lg, W1, W2, dout = _layer(45, T, H, F, E, k, gs)
    ref = reference_layer(x, lg, W1, W2, dout, k, mx=False, save_bf16=save_bf16)
    got = _layer_cpp(x, lg, W1, W2, dout, k, "bf16", save_bf16)
    for n in ref:
        assert _rel(got[n], ref[n]) < TOL, (n, _rel(got[n], ref[n]))


@pytest.mark.parametrize("mode,mx", [("bf16", False), ("mxfp8", True), ("mxfp8_act4", "act4")])
def test_cpp_layer_agrees_with_numpy_oracle(mode, mx):
    rng = np.random.default_rng(26)
    T, H, F, E, k = 150, 64, 96, 5, 2
    x, lg = rng.standard_normal((T, H)), rng.standard_normal((T, E))
    lg[:, 4] -= 1e4  # an expert with no tokens
    W1 = rng.standard_normal((E, H, 2 * F)) * 0.1
    W2 = rng.standard_normal((E, F, H)) * 0.1
    dout = rng.standard_normal((T, H))
    r = CO.layer(x, lg, W1, W2, dout, k, mode)
    f = O.layer_forward(x, lg, W1, W2, k, mx=mx)
    b = O.layer_backward(f, x, W1, W2, dout)
    np.testing.assert_array_equal(r["idx"], f["idx"])
    for n, ref in [("out", f["out"]), ("dX", b["dX"]), ("dW1", b["dW1"]), ("dW2", b["dW2"]),
                   ("dlogits", b["dlogits"]), ("dp", b["dp"])]:
        assert _rel(r[n], ref) < TOL, (n, _rel(r[n], ref))
    assert np.all(r["dW1"][4] == 0) and np.all(r["dW2"][4] == 0)


# ------------------------------------------------------- router and aux loss

def test_cpp_router_logits_brute_force():
    rng = np.random.default_rng(41)
    x, Wr = rng.standard_normal((5, 7)), rng.standard_normal((7, 3))
    ref = np.zeros((5, 3))
    for t in range(5):
        for e in range(3):
            for h in range(7):
                ref[t, e] += x[t, h] * Wr[h, e]
    r = CO.router_forward(x, Wr, 2)
    np.testing.assert_allclose(r["logits"], ref, rtol=1e-13)
    idx, w = CO.route(ref, 2)
    np.testing.assert_array_equal(r["idx"], idx)


def test_cpp_aux_loss_is_one_when_balanced():
    # every expert selected by every token (k = E) with equal logits: f = P = 1/E
    E, T = 4, 16
    r = CO.router_forward(np.ones((T, 3)), np.zeros((3, E)), E)
    assert r["aux"] == 1.0
    np.testing.assert_array_equal(r["f"], np.full(E, 1 / E))
    np.testing.assert_array_equal(r["P"], np.full(E, 1 / E))


def test_cpp_aux_loss_all_on_one_expert_closed_form():
    # every token picks expert 0 (k = 1) with logit a against 0: L = E * P_0
    E, T, a = 5, 10, 2.0
    Wr = np.zeros((1, E))
    Wr[0, 0] = a
    r = CO.router_forward(np.ones((T, 1)), Wr, 1)
    assert abs(r["aux"] - E * np.exp(a) / (np.exp(a) + E - 1)) < 1e-14


def test_cpp_router_backward_brute_force():
    rng = np.random.default_rng(43)
    T, H, E = 4, 6, 3
    x, Wr, dl = rng.standard_normal((T, H)), rng.standard_normal((H, E)), rng.standard_normal((T, E))
    r = CO.router_forward(x, Wr, 2)
    dlo, dx, dW = CO.router_backward(x, Wr, r["logits"], r["f"], dl, 0.0)
    np.testing.assert_array_equal(dlo, dl)
    for t in range(T):
        for h in range(H):
            assert abs(dx[t, h] - sum(dl[t, e] * Wr[h, e] for e in range(E))) < 1e-12
    for h in range(H):
        for e in range(E):
            assert abs(dW[h, e] - sum(x[t, h] * dl[t, e] for t in range(T))) < 1e-12


def test_cpp_aux_gradient_central_differences():
    # d aux / d Wr and d aux / d x through the logits; no routing decision is
    # near a tie, so the routed fractions stay fixed under the steps
    rng = np.random.default_rng(44)
    T, H, E, k = 6, 4, 5, 2
    x, Wr = rng.standard_normal((T, H)), rng.standard_normal((H, E))
    r = CO.router_forward(x, Wr, k)
    assert np.min(np.abs(np.diff(np.sort(r["logits"], axis=1), axis=1))) > 1e-3
    dl, dx, dW = CO.router_backward(x, Wr, r["logits"], r["f"], np.zeros((T, E)), 1.0)
    np.testing.assert_allclose(dl.sum(axis=1), 0.0, atol=1e-15)
    eps = 1e-6
    for arr, grad in ((Wr, dW), (x, dx)):
        num = np.zeros_like(arr)
        for pos in itertools.product(*[range(n) for n in arr.shape]):
            old = arr[pos]
            arr[pos] = old + eps
            lp = CO.router_forward(x, Wr, k)["aux"]
            arr[pos] = old - eps
            lm = CO.router_forward(x, Wr, k)["aux"]
            arr[pos] = old
            num[pos] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=1e-6, atol=1e-10)


def test_cpp_router_agrees_with_numpy_oracle():
    rng = np.random.default_rng(45)
    T, H, E, k = 200, 48, 16, 4
    x, Wr, dr = rng.standard_normal((T, H)), rng.standard_normal((H, E)), rng.standard_normal((T, E))
    r = CO.router_forward(x, Wr, k)
    lg = O.router_logits(x, Wr)
    idx, _ = O.route(lg, k)
    L, f, P = O.aux_load_balance(lg, idx, E)
    np.testing.assert_array_equal(r["idx"], idx)
    np.testing.assert_allclose([r["aux"]], [L], rtol=1e-13)
    np.testing.assert_allclose(r["f"], f, rtol=1e-15)
    np.testing.assert_allclose(r["P"], P, rtol=1e-13)
    dl, dx, dW = CO.router_backward(x, Wr, r["logits"], r["f"], dr, 0.03)
    dl_ref = dr + 0.03 * O.aux_load_balance_grad(lg, f)
    dx_ref, dW_ref = O.router_backward(x, Wr, dl_ref)
    for got, ref in ((dl, dl_ref), (dx, dx_ref), (dW, dW_ref)):
        assert _rel(got, ref) < TOL


# ------------------------------------------- planted mistakes must trip a pin

PLANTS = {
    # name: (original text, planted text, the pin that must fail)
    "top-k ties to the higher index": ("lg[e] > lg[best]", "lg[e] >= lg[best]", "route"),
    "router gradient sign": ("(dp[(size_t)t * k + j] - s)", "(dp[(size_t)t * k + j] + s)",
                             "fd"),
    "groups not padded to align": ("offsets[e] + (counts[e] + align - 1) / align * align",
                                   "offsets[e] + counts[e]", "plan"),
    "E4M3 ties away from zero": ("std::nearbyint(a / q)", "std::round(a / q)", "golden"),
    "scale exponent off by one": ("int e = ex - 1 - f.emax;", "int e = ex - f.emax;", "golden"),
    "SwiGLU derivative drops a term": ("dA * uv * dsilu(gv)", "dA * uv * sigmoid(gv)", "fd"),
    "gate and up swapped": ("Mat g = cols(y1, 0, F), u = cols(y1, F, F)",
                            "Mat g = cols(y1, F, F), u = cols(y1, 0, F)", "dense"),
    "W1 fprop blocked along 2F": ("qdq(W1e, 0, kE4M3) : W1e;  // blocks along H",
                                  "qdq(W1e, 1, kE4M3) : W1e;  // blocks along H", "mx"),
    "W2 dgrad blocked along F": ("qdq(W2e, 1, kE4M3) : W2e;  // blocks along H",
                                 "qdq(W2e, 0, kE4M3) : W2e;  // blocks along H", "mx"),
    "dY1 row-wise along tokens": ("dy1_row = qdq(dy1_32, 1, kE4M3);",
                                  "dy1_row = qdq_cols_in_group(dy1_32);", "mx"),
    "wgrad x blocked along H": ("x_col = qdq_cols_in_group(xe);", "x_col = qdq(xe, 1, kE4M3);",
                                "mx"),
    "act4 chain skips FP4": ("Mat row4 = qdq(row8, 1, kE2M1);", "Mat row4 = row8;", "act4"),
    "gate/up read unrounded": ("if (save_bf16) {", "if (false) {", "bf16"),
    "aux softmax not normalised": ("P[e] += s[(size_t)e] / z / T;", "P[e] += s[(size_t)e] / T;",
                                   "aux"),
    "aux gradient sign flipped": ("(f[e] - c)", "(c - f[e])", "aux_fd"),
}


def _planted_lib(tmp_path, name):
    orig, planted, _ = PLANTS[name]
    src = open(CO.SRC).read()
    assert src.count(orig) == 1, name
    path = tmp_path / "planted.cpp"
    path.write_text(src.replace(orig, planted))
    so = tmp_path / "planted.so"
    subprocess.run([os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-ffp-contract=off",
                    "-shared", "-fPIC", "-o", str(so), str(path)], check=True)
    return ctypes.CDLL(str(so))


def _pin_fails(pin):
    """Run the pin; True when it fails (AssertionError)."""
    try:
        if pin == "route":
            test_cpp_route_matches_brute_force(8, 2)
        elif pin == "plan":
            test_cpp_plan_matches_brute_force(4, 2, 37, 32)
        elif pin == "golden":
            for case in _golden_blocks():
                test_cpp_mxfp8_hand_worked_blocks(case)
        elif pin == "fd":
            test_cpp_gradients_central_differences()
        elif pin == "dense":
            test_cpp_single_expert_top1_is_dense_swiglu_mlp()
        elif pin == "mx":
            test_cpp_mx_layer_equals_block_scaled_reference(*CASES[0], "mxfp8")
        elif pin == "act4":
            test_cpp_mx_layer_equals_block_scaled_reference(*CASES[0], "mxfp8_act4")
        elif pin == "bf16":
            test_cpp_bf16_layer_equals_reference(True)
        elif pin == "aux":
            test_cpp_aux_loss_is_one_when_balanced()
        elif pin == "aux_fd":
            test_cpp_aux_gradient_central_differences()
    except AssertionError:
        return True
    return False


@pytest.mark.parametrize("name", sorted(PLANTS))
def test_cpp_planted_mistake_is_caught(name, tmp_path, monkeypatch):
    assert not _pin_fails(PLANTS[name][2])  # the real oracle passes the pin
    monkeypatch.setattr(CO, "_lib", _planted_lib(tmp_path, name))
    assert _pin_fails(PLANTS[name][2]), name
