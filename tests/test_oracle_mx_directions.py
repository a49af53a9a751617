"""Pins for the oracle's MXFP8 operand directions.

"Efficient MoE Training for Biological Foundation Models", §Challenge 2 gives
MXFP8 one scale per block of 32 consecutive values, and §Challenge 3
quantises the operands of every low-precision GEMM. A block-scaled tensor-core
product can only apply one scale per operand per step of its reduction, so the
blocks of both operands must run along the GEMM's contraction index K. The
oracle encodes this as a fixed axis per operand (x, H, dOut and dY1 row-wise,
the weights along H or F, the wgrad operands along tokens inside an expert
group). Nothing else in the pins says that each of those axes is the K of its
GEMM.

This file rebuilds the MXFP8 layer independently of those per-operand
choices. Its only quantised product is `block_scaled_gemm(A, B)`: it
quantises A [M, K] in blocks along K and B [K, N] in blocks along K (zero
padding K to a multiple of 32, which is how a group's last column block is
padded) and sums, one K block at a time, code times 2^scale on both sides,
with the scales indexed by the K block. Codes are decoded with the library's
float8 type; bf16 rounding is the library's cast. The reference layer then
calls it with each GEMM's operands written as the chain rule gives them, so
the direction of every block follows from which index is contracted.

The oracle's forward and backward must agree with it to fp64 summation-order
precision, and planted mistakes (one operand blocked along its other axis)
must not.
"""
import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from oracle import mxfp4_oracle as Q

TOL = 1e-10  # relative Frobenius error: summation order only


# ------------------------------------------------------- independent reference

def _decode_e4m3(codes):
    t = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _pad_rows(a, mult=32):
    a = np.asarray(a, dtype=np.float64)
    n = a.shape[0]
    out = np.zeros(((n + mult - 1) // mult * mult,) + a.shape[1:])
    out[:n] = a
    return out


def block_scaled_gemm(A, B):
    """C[m, n] = sum_kb sum_i qa[m, 32kb+i] 2^sa[m, kb] * qb[32kb+i, n] 2^sb[kb, n].

    A [M, K] is quantised in 32-blocks along K (axis 1), B [K, N] along K
    (axis 0); K is zero-padded to a multiple of 32 first.
    """
    A = _pad_rows(np.asarray(A, dtype=np.float64).T).T
    B = _pad_rows(B)
    qa, sa = O.mx_quantize(A, axis=1)
    qb, sb = O.mx_quantize(B, axis=0)
    va, vb = _decode_e4m3(qa), _decode_e4m3(qb)
    M, K = A.shape
    C = np.zeros((M, B.shape[1]))
    for kb in range(K // 32):
        fa = np.ldexp(1.0, sa[:, kb].astype(np.int64) - 127)  # scale of A's block kb, per row m
        fb = np.ldexp(1.0, sb[kb, :].astype(np.int64) - 127)  # scale of B's block kb, per column n
        for i in range(32):
            kk = 32 * kb + i
            C += np.outer(va[:, kk] * fa, vb[kk, :] * fb)
    return C


def act4_operand(A, k_axis):
    """Values of an activation operand in the MXFP4-activation mode: MXFP8 in
    blocks along the operand's non-K axis (its row-wise copy), then FP4 over
    the same blocks, then FP4 in blocks along K (tokens), then FP8 (lossless).
    K is zero-padded to a multiple of 32 first."""
    A = np.asarray(A, dtype=np.float64)
    A = _pad_rows(A) if k_axis == 0 else _pad_rows(A.T).T
    other = 1 - k_axis
    v = O.mx_dequantize(*O.mx_quantize(A, axis=other), axis=other)
    v = Q.mx4_dequantize(*Q.mx4_quantize(v, axis=other), axis=other)
    v = Q.mx4_dequantize(*Q.mx4_quantize(v, axis=k_axis), axis=k_axis)
    return v


def _bf16(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64)).to(torch.float32).to(
        torch.bfloat16).to(torch.float64).numpy()


def _f32(a):
    return np.asarray(a, dtype=np.float32).astype(np.float64)


def _sig(z):
    return 1.0 / (1.0 + np.exp(-z))


def reference_layer(x, lg, W1, W2, dout, k, act4=False, mx=True, save_bf16=True):
    """The MXFP8 layer with every quantised product a block_scaled_gemm (or,
    with mx=False, the BF16-mode layer with plain products).

    Readings shared with the oracle (stated in its header): activations are
    rounded to fp32 before they are quantised; the SwiGLU backward reads the
    gate/up values saved in bf16 (unless save_bf16 is False); the elementwise
    backward is straight-through.
    """
    gemm = block_scaled_gemm if mx else (lambda A, B: np.asarray(A) @ np.asarray(B))
    rnd = _f32 if mx else (lambda a: a)
    T, H = x.shape
    E, _, F2 = W1.shape
    F = F2 // 2
    idx, w = O.route(lg, k)  # routing is pinned on its own
    out = np.zeros((T, H))
    dX = np.zeros((T, H))
    dp = np.zeros((T, k))
    dW1 = np.zeros(W1.shape)
    dW2 = np.zeros(W2.shape)
    for e in range(E):
        rows = [(t, j) for t in range(T) for j in range(k) if idx[t, j] == e]
        if not rows:
            continue
        tok = np.array([t for t, _ in rows])
        slot = np.array([j for _, j in rows])
        p = w[tok, slot][:, None]
        xe, dye = x[tok], dout[tok]
        # forward: FC1 contracts H, FC2 contracts F
        y1 = gemm(xe, W1[e])
        g, u = y1[:, :F], y1[:, F:]
        h = rnd(g * _sig(g) * u * p)
        y2 = gemm(h, W2[e])
        # backward: FC2 dgrad contracts H, FC1 dgrad contracts 2F, wgrads contract tokens
        gb, ub = (_bf16(g), _bf16(u)) if save_bf16 else (g, u)
        dh = gemm(dye, W2[e].T)
        sg = _sig(gb)
        dA = dh * p
        dpe = (dh * gb * sg * ub).sum(axis=1)
        dy1 = rnd(np.concatenate([dA * ub * sg * (1.0 + gb * (1.0 - sg)), dA * gb * sg], axis=1))
        dxp = gemm(dy1, W1[e].T)
        n = len(rows)
        if act4:
            hT = act4_operand(h.T, k_axis=1)  # [F, n_pad]
            xT = act4_operand(xe.T, k_axis=1)  # [H, n_pad]
            dW2[e] = block_scaled_gemm(hT, _pad_rows(dye))
            dW1[e] = block_scaled_gemm(xT, _pad_rows(dy1))
        else:
            dW2[e] = gemm(h.T, dye)
            dW1[e] = gemm(xe.T, dy1)
        for i in range(n):
            out[tok[i]] += y2[i]
            dX[tok[i]] += dxp[i]
            dp[tok[i], slot[i]] = dpe[i]
    dl = np.zeros(lg.shape)
    for t in range(T):
        s = sum(w[t, i] * dp[t, i] for i in range(k))
        for j in range(k):
            dl[t, idx[t, j]] = w[t, j] * (dp[t, j] - s)
    return {"out": out, "dX": dX, "dW1": dW1, "dW2": dW2, "dlogits": dl}


# ------------------------------------------------------------------ the layers

def _layer(seed, T, H, F, E, k, group_sizes=None):
    """A small layer whose operands carry one x30 outlier in every 32-block
    along their GEMM's K (so that blocking along the wrong axis moves the
    result far beyond rounding). group_sizes (k = 1) fixes each expert's
    token count through the logits."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H))
    x[:, ::32] *= 30.0  # one per row-wise block of x (along H)
    W1 = rng.standard_normal((E, H, 2 * F)) * 0.05
    W1[:, ::32, :] *= 30.0  # one per block of W1 along H (FC1's K)
    W2 = rng.standard_normal((E, F, H)) * 0.05
    W2[:, :, 5::32] *= 30.0  # one per block of W2 along H (FC2 dgrad's K)
    dout = rng.standard_normal((T, H))
    dout[3::32, :] *= 30.0  # one per token block of dOut (FC2 wgrad's K)
    lg = rng.standard_normal((T, E))
    if group_sizes is not None:
        assert k == 1 and sum(group_sizes) == T
        owner = np.repeat(np.arange(E), group_sizes)
        rng.shuffle(owner)
        lg[np.arange(T), owner] += 100.0
    return x, lg, W1, W2, dout


def _rel(a, b):
    """Relative Frobenius error (absolute when b is zero, as dlogits is at k = 1)."""
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / (nb if nb > 0 else 1.0))


def _oracle(x, lg, W1, W2, dout, k, mx, save_bf16=True):
    f = O.layer_forward(x, lg, W1, W2, k, mx=mx, save_bf16=save_bf16)
    b = O.layer_backward(f, x, W1, W2, dout)
    return {"out": f["out"], **{n: b[n] for n in ("dX", "dW1", "dW2", "dlogits")}}


CASES = [
    # T, H, F, E, k, group sizes (k = 1)
    (96, 64, 96, 2, 1, (32, 64)),   # groups of whole 32-row blocks
    (70, 64, 64, 3, 2, None),       # ragged groups: padded last column blocks
]


@pytest.mark.parametrize("T,H,F,E,k,gs", CASES)
def test_oracle_mxfp8_layer_equals_block_scaled_reference(T, H, F, E, k, gs):
    x, lg, W1, W2, dout = _layer(41 + T, T, H, F, E, k, gs)
    ref = reference_layer(x, lg, W1, W2, dout, k)
    got = _oracle(x, lg, W1, W2, dout, k, True)
    for n in ref:
        assert _rel(got[n], ref[n]) < TOL, (n, _rel(got[n], ref[n]))
    # and the quantisation matters: the BF16-mode oracle is far from it
    plain = _oracle(x, lg, W1, W2, dout, k, False)
    assert _rel(plain["out"], ref["out"]) > 1e-3


@pytest.mark.parametrize("T,H,F,E,k,gs", CASES)
def test_oracle_act4_weight_grads_equal_block_scaled_reference(T, H, F, E, k, gs):
    x, lg, W1, W2, dout = _layer(43 + T, T, H, F, E, k, gs)
    ref = reference_layer(x, lg, W1, W2, dout, k, act4=True)
    got = _oracle(x, lg, W1, W2, dout, k, "act4")
    for n in ref:
        assert _rel(got[n], ref[n]) < TOL, (n, _rel(got[n], ref[n]))
    # the MXFP4 chain changes the weight gradients, and only them
    mx8 = _oracle(x, lg, W1, W2, dout, k, True)
    assert _rel(mx8["dW1"], ref["dW1"]) > 1e-3 and _rel(mx8["dW2"], ref["dW2"]) > 1e-3
    assert _rel(mx8["dX"], ref["dX"]) < TOL


@pytest.mark.parametrize("save_bf16", [True, False])
def test_oracle_bf16_layer_equals_reference(save_bf16):
    """The BF16 mode: plain products, and the backward reads gate/up through
    their bf16 copies (the library's cast) unless save_bf16 is False."""
    T, H, F, E, k, gs = CASES[1]
    x, lg, W1, W2, dout = _layer(45, T, H, F, E, k, gs)
    ref = reference_layer(x, lg, W1, W2, dout, k, mx=False, save_bf16=save_bf16)
    got = _oracle(x, lg, W1, W2, dout, k, False, save_bf16)
    for n in ref:
        assert _rel(got[n], ref[n]) < TOL, (n, _rel(got[n], ref[n]))
    other = reference_layer(x, lg, W1, W2, dout, k, mx=False, save_bf16=not save_bf16)
    assert _rel(got["dW1"], other["dW1"]) > 1e-4  # the rounding is visible


# ------------------------------------------- planted wrong axes must be caught

def _plants():
    """Each plant blocks one operand along its other axis (shapes T=96,
    H=64, F=96: x and dOut are [n, 64], H is [n, 96], dY1 is [n, 192])."""
    real = O.mx_qdq

    def along_tokens(ncols):
        def f(a, axis=-1):
            a = np.asarray(a)
            if a.ndim == 2 and axis in (1, -1) and a.shape[1] == ncols and a.shape[0] % 32 == 0:
                axis = 0
            return real(a, axis)
        return f

    def weights_right():  # the weights keep their own axes while mx_qdq is patched
        return [("_w1_fprop", lambda W, mx: real(np.asarray(W, float), 0)),
                ("_w2_fprop", lambda W, mx: real(np.asarray(W, float), 0)),
                ("_w1_dgrad", lambda W, mx: real(np.asarray(W, float), 1)),
                ("_w2_dgrad", lambda W, mx: real(np.asarray(W, float), 1))]

    return {
        "W1 fprop along 2F": [("_w1_fprop", lambda W, mx: real(np.asarray(W, float), 1))],
        "W2 fprop along H": [("_w2_fprop", lambda W, mx: real(np.asarray(W, float), 1))],
        "W1 dgrad along H": [("_w1_dgrad", lambda W, mx: real(np.asarray(W, float), 0))],
        "W2 dgrad along F": [("_w2_dgrad", lambda W, mx: real(np.asarray(W, float), 0))],
        "wgrad operands along features": [
            ("mx_qdq_cols_in_groups", lambda a: real(np.asarray(a, float), 1))],
        "H row-wise along tokens": [("mx_qdq", along_tokens(96))] + weights_right(),
        "dY1 row-wise along tokens": [("mx_qdq", along_tokens(192))] + weights_right(),
        "x and dOut row-wise along tokens": [("mx_qdq", along_tokens(64))] + weights_right(),
    }


@pytest.mark.parametrize("plant", sorted(_plants()))
def test_planted_wrong_axis_is_caught(plant, monkeypatch):
    T, H, F, E, k, gs = CASES[0]
    x, lg, W1, W2, dout = _layer(41 + T, T, H, F, E, k, gs)
    ref = reference_layer(x, lg, W1, W2, dout, k)
    with monkeypatch.context() as m:
        for name, fn in _plants()[plant]:
            m.setattr(O, name, fn)
        got = _oracle(x, lg, W1, W2, dout, k, True)
    worst = max(_rel(got[n], ref[n]) for n in ref)
    assert worst > 1e-3, (plant, worst)


def test_planted_act4_chain_along_tokens_first_is_caught(monkeypatch):
    T, H, F, E, k, gs = CASES[0]
    x, lg, W1, W2, dout = _layer(47, T, H, F, E, k, gs)
    ref = reference_layer(x, lg, W1, W2, dout, k, act4=True)

    def swapped(a):  # the FP8/FP4 row-wise steps blocked along tokens instead
        n = np.shape(a)[0]
        v = _pad_rows(a)
        v = O.mx_dequantize(*O.mx_quantize(v, axis=0), axis=0)
        v = Q.mx4_dequantize(*Q.mx4_quantize(v, axis=0), axis=0)
        return Q.mx4_dequantize(*Q.mx4_quantize(v, axis=0), axis=0)[:n]

    with monkeypatch.context() as m:
        m.setattr(O, "act4_cols_in_groups", swapped)
        got = _oracle(x, lg, W1, W2, dout, k, "act4")
    assert max(_rel(got["dW1"], ref["dW1"]), _rel(got["dW2"], ref["dW2"])) > 1e-3
