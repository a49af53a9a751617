"""Pins for the CPU oracle: checks against facts that do not come from the oracle.

Each test ties one oracle function to something independent of it: brute
force on tiny inputs, a closed form, a library routine the oracle does not
use, a hand-worked example from the OCP MX rules, an invariant of the
mathematics, or central finite differences.
"""
import itertools
import os

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------- routing

def _brute_topk(row, k):
    """Rank of expert e = number of experts that beat it (higher logit, or equal and lower index)."""
    E = len(row)
    ranks = []
    for e in range(E):
        r = sum(1 for f in range(E) if row[f] > row[e] or (row[f] == row[e] and f < e))
        ranks.append(r)
    sel = [None] * k
    for e, r in enumerate(ranks):
        if r < k:
            sel[r] = e
    return sel


@pytest.mark.parametrize("E,k", [(4, 2), (8, 2), (64, 6), (5, 5), (1, 1)])
def test_route_matches_brute_force(E, k):
    rng = np.random.default_rng(E * 100 + k)
    lg = rng.standard_normal((300, E))
    lg[::3] = np.round(lg[::3])  # many exact ties
    lg[1::7, 0] = 0.0
    if E > 1:
        lg[1::7, 1] = -0.0  # +0 and -0 tie
    idx, w = O.route(lg, k)
    for t in range(lg.shape[0]):
        assert list(idx[t]) == _brute_topk(list(lg[t]), k)


def test_route_weights_closed_form_k2():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((500, 8)) * 3
    idx, w = O.route(lg, 2)
    l0 = lg[np.arange(500), idx[:, 0]]
    l1 = lg[np.arange(500), idx[:, 1]]
    w0 = 1.0 / (1.0 + np.exp(l1 - l0))  # logistic of the logit gap
    np.testing.assert_allclose(w[:, 0], w0, rtol=1e-14)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=1e-15)


def test_route_weights_equal_full_softmax_renormalised():
    rng = np.random.default_rng(8)
    lg = rng.standard_normal((200, 64))
    idx, w = O.route(lg, 6)
    full = np.exp(lg - lg.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    sel = np.take_along_axis(full, idx, 1)
    np.testing.assert_allclose(w, sel / sel.sum(1, keepdims=True), rtol=1e-13)


# ---------------------------------------------------------------- permute plan

def _brute_plan(idx, E, align):
    T, k = idx.shape
    counts = [0] * E
    dest = [None] * (T * k)
    offsets = [0]
    for e in range(E):
        row = offsets[-1]
        for t in range(T):
            for j in range(k):
                if idx[t, j] == e:
                    dest[t * k + j] = row
                    row += 1
                    counts[e] += 1
        n = counts[e]
        offsets.append(offsets[-1] + (n + align - 1) // align * align)
    return counts, offsets, dest


@pytest.mark.parametrize("align", [1, 32, 128])
@pytest.mark.parametrize("E,k,T", [(4, 2, 37), (8, 2, 100), (64, 6, 50), (3, 3, 20), (1, 1, 9)])
def test_plan_matches_brute_force(E, k, T, align):
    rng = np.random.default_rng(E + k + T + align)
    idx, _ = O.route(rng.standard_normal((T, E)), k)
    counts, offsets, dest, src = O.permute_plan(idx, E, align)
    bc, bo, bd = _brute_plan(idx, E, align)
    assert list(counts) == bc
    assert list(offsets) == bo
    assert list(dest) == bd
    # src is the inverse of dest, -1 on padding rows
    assert len(src) == offsets[-1]
    for i, r in enumerate(dest):
        assert src[r] == i
    assert (src == -1).sum() == offsets[-1] - T * k


def test_plan_empty_experts_and_single_expert():
    idx = np.full((10, 1), 2, dtype=np.int32)
    counts, offsets, dest, src = O.permute_plan(idx, 4, 32)
    assert list(counts) == [0, 0, 10, 0]
    assert list(offsets) == [0, 0, 0, 32, 32]
    assert list(dest) == list(range(10))


def test_identity_experts_permute_unpermute():
    rng = np.random.default_rng(3)
    T, H, E, k = 40, 16, 5, 3
    x = rng.standard_normal((T, H))
    idx, w = O.route(rng.standard_normal((T, E)), k)
    _, offsets, dest, _ = O.permute_plan(idx, E, 8)
    xp = O.permute(x, dest, k, offsets[-1])
    back = O.unpermute(xp, dest, k, w)
    np.testing.assert_allclose(back, x, rtol=1e-14, atol=1e-14)
    # padding rows are zero
    used = np.zeros(offsets[-1], bool)
    used[dest] = True
    assert np.all(xp[~used] == 0)


# ----------------------------------------------------------------------- MXFP8

def _parse_list(s, conv):
    out = []
    for tok in s.split(","):
        n, v = tok.strip().split("*")
        out += [conv(v)] * int(n)
    return out


def _golden_blocks():
    rows = []
    with open(os.path.join(GOLDEN, "mxfp8_blocks.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            name, vals, scale, codes = [p.strip() for p in line.split(";")]
            rows.append((name, _parse_list(vals, float), int(scale),
                         _parse_list(codes, lambda h: int(h, 16))))
    return rows


@pytest.mark.parametrize("case", _golden_blocks(), ids=lambda c: c[0])
def test_mxfp8_hand_worked_blocks(case):
    name, vals, scale, codes = case
    assert len(vals) == 32 and len(codes) == 32
    c, s = O.mx_quantize(np.array([vals]), axis=1)
    assert int(s[0, 0]) == scale
    assert [int(v) for v in c[0]] == codes


def test_e4m3_decode_encode_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = O.e4m3_decode(codes)
    # the grid point itself must round to itself and encode back to its byte
    r = O.e4m3_round(np.abs(vals))
    np.testing.assert_array_equal(r, np.abs(vals))
    back = O.e4m3_encode(np.signbit(vals), r)
    np.testing.assert_array_equal(back, codes)
    # decode agrees with the library's float8 type on every finite byte
    lib = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(vals, lib)


def test_e4m3_round_matches_library_conversion():
    # In range (|v| <= 448) the library cast is round-to-nearest-even too;
    # the oracle does not use it, so agreement pins the rounding.
    rng = np.random.default_rng(11)
    v = np.concatenate([
        rng.uniform(0, 448, 200000),
        np.exp2(rng.uniform(-12, 8.8, 200000)),
        # exact midpoints between neighbouring grid points
        (O.e4m3_decode(np.arange(0, 126)) + O.e4m3_decode(np.arange(1, 127))) / 2,
    ]).astype(np.float32).astype(np.float64)
    v = v[v <= 448]
    ours = O.e4m3_round(v)
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, lib)


def test_bf16_round_matches_library_conversion():
    # torch's float32 -> bfloat16 cast rounds to nearest even; the oracle's
    # bit-level rounding does not call it, so agreement pins to_bf16.
    rng = np.random.default_rng(12)
    v = np.concatenate([
        rng.standard_normal(100000) * np.exp2(rng.uniform(-60, 60, 100000)),
        # exact midpoints between neighbouring bf16 values, both parities
        (np.arange(1, 20001, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        -(np.arange(1, 20001, dtype=np.uint32) << 16 | 0x8000).view(np.float32),
        [0.0, -0.0, np.inf, -np.inf, 3.3895313892515355e38, 1e-45, -1e-40],
    ]).astype(np.float32)
    ours = O.to_bf16(v)
    lib = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(ours, lib)
    assert np.signbit(O.to_bf16(np.array([-0.0])))[0]
    assert np.isnan(O.to_bf16(np.array([np.nan])))[0]


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_mx_qdq_equals_decoded_codes(axis):
    # mx_qdq skips the byte encoding; it must equal decoding the codes and
    # scales that mx_quantize writes (the decode is pinned by the library
    # E4M3 table above), on random and special blocks.
    rng = np.random.default_rng(13)
    a = rng.standard_normal((64, 96, 64)) * np.exp2(rng.integers(-140, 140, (64, 1, 1)))
    a[0, :32] = 0.0
    a[1, :32] = -0.0
    a[2, 5] = 1e4  # saturating
    a[3, 7] = np.inf
    a[4, 9, 3] = np.nan
    codes, scales = O.mx_quantize(a, axis=axis)
    ref = O.mx_dequantize(codes, scales, axis=axis)
    got = O.mx_qdq(a, axis=axis)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    np.testing.assert_array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_mxfp8_roundtrip_exact_on_representable_blocks():
    rng = np.random.default_rng(5)
    grid = O.e4m3_decode(np.arange(0, 127))  # non-negative finite grid
    for s in [-20, -3, 0, 7, 40]:
        vals = rng.choice(grid, size=(64, 32))
        vals[:, 0] = rng.choice(grid[grid >= 256], size=64)  # top binade sets the scale
        vals *= np.where(rng.random((64, 32)) < 0.5, -1, 1)
        vals *= 2.0 ** s
        c, sc = O.mx_quantize(vals, axis=1)
        assert np.all(sc == s + 127)
        np.testing.assert_array_equal(O.mx_dequantize(c, sc, axis=1), vals)


def test_mxfp8_error_bound_random():
    # RNE error is at most half a grid step: |v - q| <= 2^(floor(log2|v|) - 4)
    # in the normal range, <= 2^-10 * scale below it.
    rng = np.random.default_rng(6)
    v = rng.standard_normal((100, 256)) * np.exp2(rng.integers(-30, 30, (100, 1)))
    c, s = O.mx_quantize(v, axis=1)
    q = O.mx_dequantize(c, s, axis=1)
    scale = np.repeat(O.e8m0_decode(s), 32, axis=1)
    mag = np.abs(v) / scale
    step = np.where(mag >= 2 ** -6, np.exp2(np.floor(np.log2(np.maximum(mag, 1e-300))) - 3), 2.0 ** -9)
    sat = mag > 448
    err = np.abs(v - q) / scale
    assert np.all(err[~sat] <= step[~sat] / 2 * (1 + 1e-12))
    assert np.all(np.abs(q[sat]) / scale[sat] == 448)


def test_mxfp8_axis_and_nonfinite():
    rng = np.random.default_rng(9)
    a = rng.standard_normal((64, 96))
    c0, s0 = O.mx_quantize(a, axis=0)
    c1, s1 = O.mx_quantize(a.T.copy(), axis=1)
    np.testing.assert_array_equal(c0, c1.T)
    np.testing.assert_array_equal(s0, s1.T)
    a[3, 40] = np.inf
    c, s = O.mx_quantize(a, axis=1)
    assert s[3, 1] == 255 and np.all(c[3, 32:64] == 0x7F)
    assert s[3, 0] != 255


# ------------------------------------------------------------------- the layer

def _dense_swiglu_mlp(x, W1, W2):
    """Textbook loops: out[t,h] = sum_f silu(sum_i x W1[:,f]) * (sum_i x W1[:,F+f]) * W2[f,h]."""
    T, H = x.shape
    F = W2.shape[0]
    out = np.zeros((T, W2.shape[1]))
    for t in range(T):
        for f in range(F):
            g = sum(x[t, i] * W1[i, f] for i in range(H))
            u = sum(x[t, i] * W1[i, F + f] for i in range(H))
            a = g / (1.0 + np.exp(-g)) * u
            for h in range(W2.shape[1]):
                out[t, h] += a * W2[f, h]
    return out


def test_single_expert_top1_is_dense_swiglu_mlp():
    rng = np.random.default_rng(12)
    T, H, F = 5, 6, 4
    x = rng.standard_normal((T, H))
    W1 = rng.standard_normal((1, H, 2 * F))
    W2 = rng.standard_normal((1, F, H))
    fwd = O.layer_forward(x, rng.standard_normal((T, 1)), W1, W2, k=1)
    np.testing.assert_allclose(fwd["out"], _dense_swiglu_mlp(x, W1[0], W2[0]), rtol=1e-12, atol=1e-12)


def _tiny_layer(seed, T=7, H=5, F=4, E=3, k=2):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    lg = rng.standard_normal((T, E))
    W1 = rng.standard_normal((E, H, 2 * F)) * 0.5
    W2 = rng.standard_normal((E, F, H)) * 0.5
    dout = rng.standard_normal((T, H))
    return x, lg, W1, W2, dout


def _loss(x, lg, W1, W2, dout, k):
    return float((O.layer_forward(x, lg, W1, W2, k)["out"] * dout).sum())


def test_gradients_central_differences():
    # The exact chain rule (gate/up not rounded to their saved bf16 copies).
    x, lg, W1, W2, dout = _tiny_layer(13)
    k = 2
    srt = np.sort(lg, axis=1)
    assert np.min(np.abs(np.diff(srt, axis=1))) > 1e-3  # no near-ties in the selection
    fwd = O.layer_forward(x, lg, W1, W2, k, save_bf16=False)
    g = O.layer_backward(fwd, x, W1, W2, dout)
    eps = 1e-6
    for name, arr, grad in [("x", x, g["dX"]), ("W1", W1, g["dW1"]),
                            ("W2", W2, g["dW2"]), ("logits", lg, g["dlogits"])]:
        num = np.zeros_like(arr)
        for pos in itertools.product(*[range(s) for s in arr.shape]):
            old = arr[pos]
            arr[pos] = old + eps
            lp = _loss(x, lg, W1, W2, dout, k)
            arr[pos] = old - eps
            lm = _loss(x, lg, W1, W2, dout, k)
            arr[pos] = old
            num[pos] = (lp - lm) / (2 * eps)
        err = np.linalg.norm(num - grad) / np.linalg.norm(num)
        assert err < 1e-6, (name, err)


@pytest.mark.parametrize("mx", [False, True])
def test_token_permutation_invariance(mx):
    rng = np.random.default_rng(14)
    T, H, F, E, k = 96, 64, 64, 4, 2
    x = rng.standard_normal((T, H))
    lg = rng.standard_normal((T, E))
    W1 = rng.standard_normal((E, H, 2 * F)) * 0.1
    W2 = rng.standard_normal((E, F, H)) * 0.1
    dout = rng.standard_normal((T, H))
    f = O.layer_forward(x, lg, W1, W2, k, mx=mx)
    b = O.layer_backward(f, x, W1, W2, dout)
    # out, dX and dlogits use only row-wise blocks, so they are invariant in
    # MXFP8 too; dW uses column blocks (rows in token order) and is checked in BF16.
    perm = rng.permutation(T)
    f2 = O.layer_forward(x[perm], lg[perm], W1, W2, k, mx=mx)
    b2 = O.layer_backward(f2, x[perm], W1, W2, dout[perm])
    np.testing.assert_allclose(f2["out"], f["out"][perm], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b2["dX"], b["dX"][perm], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(b2["dlogits"], b["dlogits"][perm], rtol=1e-12, atol=1e-12)
    if not mx:
        np.testing.assert_allclose(b2["dW1"], b["dW1"], rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(b2["dW2"], b["dW2"], rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("mx", [False, True, "act4"])
def test_sampled_mode_equals_full_mode(mx):
    rng = np.random.default_rng(15)
    T, H, F, E, k = 200, 64, 96, 5, 2
    x = rng.standard_normal((T, H))
    lg = rng.standard_normal((T, E))
    lg[:, 4] -= 1e4  # one expert with no tokens
    W1 = rng.standard_normal((E, H, 2 * F)) * 0.1
    W2 = rng.standard_normal((E, F, H)) * 0.1
    dout = rng.standard_normal((T, H))
    f = O.layer_forward(x, lg, W1, W2, k, mx=mx)
    b = O.layer_backward(f, x, W1, W2, dout)
    toks = np.array([0, 5, 17, 199, 100])
    s = O.sampled_token_outputs(x, lg, W1, W2, dout, k, toks, mx=mx)
    np.testing.assert_allclose(s["out"], f["out"][toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s["dX"], b["dX"][toks], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s["dlogits"], b["dlogits"][toks], rtol=1e-12, atol=1e-13)
    cols = np.arange(32, 64)
    w = O.sampled_weight_grads(x, lg, W1, W2, dout, k, cols, mx=mx)
    np.testing.assert_allclose(w["dW1g"], b["dW1"][:, :, cols], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(w["dW1u"], b["dW1"][:, :, F + cols], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(w["dW2"], b["dW2"][:, cols, :], rtol=1e-12, atol=1e-13)
    assert np.all(b["dW1"][4] == 0) and np.all(b["dW2"][4] == 0)


def test_stream_matches_full_loop():
    x, lg, W1, W2, dout = _tiny_layer(16, T=30, E=4)
    f = O.layer_forward(x, lg, W1, W2, 2)
    b = O.layer_backward(f, x, W1, W2, dout)
    out = np.zeros_like(x)
    for e, tok, slot, y2, dxp, dp, dW1e, dW2e in O.layer_fwd_bwd_expert_stream(x, lg, W1, W2, dout, 2):
        np.add.at(out, tok, y2)
        np.testing.assert_allclose(dW1e, b["dW1"][e], rtol=1e-14)
        np.testing.assert_allclose(dW2e, b["dW2"][e], rtol=1e-14)
    np.testing.assert_allclose(out, f["out"], rtol=1e-14)


# ------------------------------------------- planted mistakes must trip a pin

def test_planted_mistakes_are_caught(monkeypatch):
    """A wrong SwiGLU derivative or a swapped gate/up fails the pins above."""
    x, lg, W1, W2, dout = _tiny_layer(17)
    fwd = O.layer_forward(x, lg, W1, W2, 2)
    good = O.layer_backward(fwd, x, W1, W2, dout)

    with monkeypatch.context() as m:
        m.setattr(O, "dsilu", lambda z: O.sigmoid(z))  # drops the z*s*(1-s) term
        bad = O.layer_backward(fwd, x, W1, W2, dout)
    assert np.linalg.norm(bad["dX"] - good["dX"]) > 1e-3 * np.linalg.norm(good["dX"])

    rng = np.random.default_rng(18)
    xs, W1s, W2s = rng.standard_normal((3, 4)), rng.standard_normal((1, 4, 6)), rng.standard_normal((1, 3, 4))
    with monkeypatch.context() as m:
        m.setattr(O, "silu", lambda z: z)  # plain GLU instead of SwiGLU
        out = O.layer_forward(xs, np.zeros((3, 1)), W1s, W2s, 1)["out"]
    assert not np.allclose(out, _dense_swiglu_mlp(xs, W1s[0], W2s[0]))


def test_grouped_gemm_brute_force():
    rng = np.random.default_rng(19)
    offsets = np.array([0, 3, 3, 7])
    A = rng.standard_normal((8, 4))
    B = rng.standard_normal((3, 4, 5))
    C = O.grouped_gemm_fprop(A, B, offsets)
    Ct = O.grouped_gemm_fprop(A, np.transpose(B, (0, 2, 1)).copy(), offsets, b_layout=1)
    for r in range(8):
        e = 0 if r < 3 else (2 if r < 7 else None)
        for n in range(5):
            want = 0.0 if e is None else sum(A[r, i] * B[e, i, n] for i in range(4))
            assert abs(C[r, n] - want) < 1e-12 and abs(Ct[r, n] - want) < 1e-12
    Y = rng.standard_normal((8, 6))
    W = O.grouped_gemm_wgrad(A, Y, offsets)
    assert np.all(W[1] == 0)
    for e, (r0, r1) in enumerate([(0, 3), (3, 3), (3, 7)]):
        for m in range(4):
            for n in range(6):
                want = sum(A[r, m] * Y[r, n] for r in range(r0, r1))
                assert abs(W[e, m, n] - want) < 1e-12


# ------------------------------------------------------- router and aux loss

def test_router_logits_brute_force():
    rng = np.random.default_rng(31)
    x, Wr = rng.standard_normal((5, 7)), rng.standard_normal((7, 3))
    ref = np.zeros((5, 3))
    for t in range(5):
        for e in range(3):
            for h in range(7):
                ref[t, e] += x[t, h] * Wr[h, e]
    np.testing.assert_allclose(O.router_logits(x, Wr), ref, rtol=1e-13)


def test_aux_loss_is_one_when_balanced():
    # uniform probabilities (equal logits) and round-robin routing: f = P = 1/E
    E, k, T = 8, 2, 64
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    L, f, P = O.aux_load_balance(np.zeros((T, E)), idx, E)
    assert L == 1.0
    np.testing.assert_array_equal(f, np.full(E, 1 / E))


def test_aux_loss_all_on_one_expert_closed_form():
    # every token picks expert 0 (k=1) with logit a against 0: L = E * P_0
    E, T, a = 5, 10, 2.0
    lg = np.zeros((T, E))
    lg[:, 0] = a
    L, f, P = O.aux_load_balance(lg, np.zeros((T, 1), dtype=int), E)
    assert abs(L - E * np.exp(a) / (np.exp(a) + E - 1)) < 1e-14


def test_aux_grad_finite_differences_and_row_sums():
    rng = np.random.default_rng(32)
    T, E, k = 6, 5, 2
    lg = rng.standard_normal((T, E))
    idx, _ = O.route(lg, k)
    _, f, _ = O.aux_load_balance(lg, idx, E)
    g = O.aux_load_balance_grad(lg, f)

    def loss(l):  # f held fixed: the routing decision carries no gradient
        return E * np.sum(f * O.softmax_all(l).mean(axis=0))
    num = np.zeros_like(lg)
    eps = 1e-6
    for t in range(T):
        for e in range(E):
            lp, lm = lg.copy(), lg.copy()
            lp[t, e] += eps
            lm[t, e] -= eps
            num[t, e] = (loss(lp) - loss(lm)) / (2 * eps)
    np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-10)
    np.testing.assert_allclose(g.sum(axis=1), 0.0, atol=1e-15)


def test_router_backward_brute_force():
    rng = np.random.default_rng(33)
    T, H, E = 4, 6, 3
    x, Wr, dl = rng.standard_normal((T, H)), rng.standard_normal((H, E)), rng.standard_normal((T, E))
    dx, dW = O.router_backward(x, Wr, dl)
    for t in range(T):
        for h in range(H):
            assert abs(dx[t, h] - sum(dl[t, e] * Wr[h, e] for e in range(E))) < 1e-12
    for h in range(H):
        for e in range(E):
            assert abs(dW[h, e] - sum(x[t, h] * dl[t, e] for t in range(T))) < 1e-12


def test_planted_aux_mistakes_are_caught(monkeypatch):
    """An unnormalised softmax or a flipped sign in the aux gradient trips the
    pins above (the balanced-loss value and the finite differences)."""
    E, k, T = 4, 2, 8
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(T)])
    real_softmax = O.softmax_all
    with monkeypatch.context() as m:
        m.setattr(O, "softmax_all", lambda l: np.exp(np.asarray(l, dtype=float)))
        L, _, _ = O.aux_load_balance(np.zeros((T, E)), idx, E)
    assert L != 1.0
    rng = np.random.default_rng(35)
    lg = rng.standard_normal((T, E))
    f = np.full(E, 1.0 / E) + np.linspace(-0.1, 0.1, E)
    good = O.aux_load_balance_grad(lg, f)
    s = real_softmax(lg)
    flipped = (E / T) * s * ((s * f).sum(axis=1, keepdims=True) - f)
    assert np.linalg.norm(flipped - good) > 0.5 * np.linalg.norm(good)
