"""CPU oracle for the Mixtral-style MoE expert layer (forward and backward).

TEST INFRASTRUCTURE ONLY. This module exists to check the CUDA path. Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline/reference legs of
``bench.py`` may import it. The product path never calls it and has no CPU
fallback.

It is written as the per-expert loop that the sources describe, in float64,
with no blocking or fusion: for every expert, take the (token, slot) pairs
routed to it, run the expert's SwiGLU MLP on those tokens, scale by the
routing weight and add the result back into the token rows.

Sources (cited by short tag in the docstrings below):

[EMT]     "Efficient MoE Training for Biological Foundation Models"
          (NVIDIA Developer Blog tutorial): §Challenge 1 (per-expert loop with
          ``expert_mask``, ``routing_weights`` and ``index_add_``;
          GroupedLinear with ``split_sizes`` and ``out_features =
          2*intermediate_size``), §Challenge 2 (MXFP8: one scale per block of
          32 consecutive values), §Challenge 3 (``gate_up`` ->
          ``ScaledSwiGLU`` -> ``down``; the SwiGLU is multiplied by the
          routing probabilities).
[MOEBIO]  "How MoE Architecture Cuts Costs and Boosts Efficiency: Efficient
          Training of Biological Foundation Models", the paragraph on the
          Router (Top-K routing: keep the K highest-scoring experts).
[OCPMX]   OCP Microscaling Formats (MX) v1.0: shared E8M0 scale
          X = 2^(floor(log2 max|V|) - emax_elem), elements rounded to
          nearest-even and saturated; E4M3 emax_elem = 8, max normal 448.

Readings where the sources are silent (each is repeated in the design notes):

* top-k ties go to the lower expert index; +0 and -0 tie;
* routing weights are the softmax over the k selected logits (equal to a
  softmax over all E renormalised by the top-k sum);
* SwiGLU is silu(gate) * up, gate = FC1 columns [0, F), up = [F, 2F);
* within one expert the routed rows are ordered by token, then slot;
* the router receives a gradient through the k selected softmax weights;
  the selection itself has none;
* MXFP8 quantisation follows [OCPMX]: an all-zero block gets scale byte 0
  (exponent clamped to -127) and zero elements that keep their sign; a block
  holding Inf or NaN gets scale byte 0xFF and element bytes 0x7F;
* in MXFP8 mode every GEMM consumes operands whose 32-blocks run along its
  reduction dimension (row-wise for forward and dgrad, column-wise, i.e.
  along tokens inside an expert group, for wgrad); intermediate activations
  are rounded to float32 before they are quantised; the elementwise
  backward is straight-through;
* the SwiGLU backward works from the gate/up values that the forward saved
  in BF16 (save_bf16=True, the default, in every precision): [EMT §Challenge
  3] trains with 16-bit activations and converts each low-precision GEMM's
  result back to the 16-bit format. Two results depend on that rounding far
  more than the tolerance: in MXFP8 mode the values this step produces decide
  quantised codes, and dlogits = w (dp - sum w dp) cancels when a token's dp
  values are close (for a single token the rounding alone moves it by 6%).
  The forward SwiGLU consumes the GEMM result unrounded (the fused path folds
  the conversion into the epilogue). save_bf16=False gives the exact
  chain-rule gradient that the finite-difference pin checks;
* in the MXFP8 mode with MXFP4 activations (mx == "act4") the wgrad operands
  X and H are the FP8 -> FP4 -> column-wise FP4 chain of their row-wise MXFP8
  copies (act4_cols_in_groups; the MXFP4 readings are in mxfp4_oracle.py);
  everything else is as in MXFP8 mode.
"""
from __future__ import annotations

import numpy as np

MX_BLOCK = 32
E4M3_EMAX = 8  # exponent of the largest E4M3 binade [OCPMX]
E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6  # 2^-6 is the smallest normal E4M3 value
E4M3_MANT_BITS = 3

f64 = np.float64


# ---------------------------------------------------------------------------
# Routing [MOEBIO Router paragraph; EMT §Challenge 1 ``routing_weights``]
# ---------------------------------------------------------------------------

def route(logits, k):
    """Top-k experts per token and their renormalised softmax weights.

    Experts are ordered by (logit descending, expert index ascending) with a
    stable sort of the negated logits; slot j holds the j-th best expert.
    w[t, j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k selected.
    Returns idx int32 [T, k] and w float64 [T, k].
    """
    lg = np.asarray(logits, dtype=f64)
    order = np.argsort(-lg, axis=1, kind="stable")[:, :k]
    sel = np.take_along_axis(lg, order, axis=1)
    z = np.exp(sel - sel[:, :1])
    w = z / z.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w


def route_backward(dp, w, idx, E):
    """Gradient of the loss w.r.t. the logits from dL/dw (dp [T, k]).

    Softmax over the selected logits: dl_j = w_j * (dp_j - sum_i w_i dp_i);
    experts that were not selected get 0.
    """
    dp = np.asarray(dp, dtype=f64)
    T, k = dp.shape
    s = (w * dp).sum(axis=1, keepdims=True)
    dsel = w * (dp - s)
    dl = np.zeros((T, E), dtype=f64)
    rows = np.repeat(np.arange(T), k)
    dl[rows, idx.reshape(-1)] = dsel.reshape(-1)
    return dl


# ---------------------------------------------------------------------------
# Router projection and auxiliary load-balancing loss
# [MOEBIO Router paragraph: a score for every expert per token; MOEBIO
#  "Engineering Challenges of Efficient Training": an auxiliary loss that
#  penalises uneven expert load]
# ---------------------------------------------------------------------------

def router_logits(x, Wr):
    """logits[t, e] = sum_h x[t, h] * Wr[h, e] (x [T, H], Wr [H, E])."""
    return np.asarray(x, dtype=f64) @ np.asarray(Wr, dtype=f64)


def softmax_all(logits):
    """Softmax of every token's logits over all E experts."""
    lg = np.asarray(logits, dtype=f64)
    z = np.exp(lg - lg.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def aux_load_balance(logits, idx, E):
    """Load-balancing loss L = E * sum_e f_e * P_e.

    f_e = fraction of the routed (token, slot) pairs that go to expert e;
    P_e = mean over tokens of the softmax probability of expert e. The loss is
    1 for perfectly balanced routing and grows as load concentrates.
    Returns (L, f [E], P [E]).
    """
    idx = np.asarray(idx)
    T, k = idx.shape
    f = np.bincount(idx.reshape(-1), minlength=E).astype(f64) / (T * k)
    P = softmax_all(logits).mean(axis=0)
    return float(E * np.sum(f * P)), f, P


def aux_load_balance_grad(logits, f):
    """dL/dlogits with f held fixed (the selection has no gradient):
    dL/dl[t, e] = (E / T) * s[t, e] * (f_e - sum_i f_i * s[t, i])."""
    s = softmax_all(logits)
    T, E = s.shape
    c = (s * np.asarray(f, dtype=f64)[None, :]).sum(axis=1, keepdims=True)
    return (E / T) * s * (np.asarray(f, dtype=f64)[None, :] - c)


def router_backward(x, Wr, dlogits):
    """Gradients of the projection: dx = dlogits @ Wr^T, dWr = x^T @ dlogits."""
    dl = np.asarray(dlogits, dtype=f64)
    return dl @ np.asarray(Wr, dtype=f64).T, np.asarray(x, dtype=f64).T @ dl


# ---------------------------------------------------------------------------
# Permutation into contiguous per-expert groups
# [EMT §Challenge 1: per-expert token lists and ``split_sizes``]
# ---------------------------------------------------------------------------

def roundup(n, a):
    return (n + a - 1) // a * a


def permute_plan(idx, E, align):
    """Counting-sort plan of the routed rows by expert.

    counts[e]  = number of (t, j) with idx[t, j] == e  (the split sizes);
    offsets    = exclusive prefix sum of roundup(counts, align), E + 1 long;
    dest[t*k+j] = row of Xp that receives token t for slot j; rows inside a
                 group are in flat-index (token, then slot) order;
    src[r]     = flat index t*k+j held by Xp row r, -1 for padding rows.
    """
    flat = np.asarray(idx).reshape(-1).astype(np.int64)
    counts = np.bincount(flat, minlength=E).astype(np.int64)
    padded = roundup(counts, align)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(padded)
    order = np.argsort(flat, kind="stable")  # grouped by expert, flat order kept
    first = np.zeros(E, dtype=np.int64)
    first[1:] = np.cumsum(counts)[:-1]
    rank = np.empty_like(flat)
    rank[order] = np.arange(flat.size) - first[flat[order]]
    dest = offsets[flat] + rank
    src = np.full(int(offsets[-1]), -1, dtype=np.int64)
    src[dest] = np.arange(flat.size)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            dest.astype(np.int32), src.astype(np.int32))


def permute(x, dest, k, rows_total):
    """Xp[dest[t*k+j]] = x[t]; padding rows are zero."""
    x = np.asarray(x, dtype=f64)
    xp = np.zeros((rows_total, x.shape[1]), dtype=f64)
    xp[np.asarray(dest)] = np.repeat(x, k, axis=0)
    return xp


def unpermute(y, dest, k, w=None):
    """out[t] = sum_j w[t, j] * y[dest[t*k+j]] (w = 1 when None).

    The sum over slots is the ``index_add_`` of [EMT §Challenge 1].
    """
    y = np.asarray(y, dtype=f64)
    rows = y[np.asarray(dest)]
    T = rows.shape[0] // k
    rows = rows.reshape(T, k, -1)
    if w is not None:
        rows = rows * np.asarray(w, dtype=f64)[:, :, None]
    return rows.sum(axis=1)


# ---------------------------------------------------------------------------
# MXFP8: E4M3 elements, E8M0 scale per 32 consecutive values
# [EMT §Challenge 2; OCPMX]
# ---------------------------------------------------------------------------

def e4m3_round(a):
    """Round magnitudes a >= 0 to the E4M3 grid, ties to even, saturating.

    In the binade [2^b, 2^(b+1)) the grid spacing is 2^(b-3); below the
    smallest normal (2^-6) the subnormal spacing 2^-9 applies. Dividing by
    the spacing is exact (a power of two), so rounding the quotient to the
    nearest integer with ties to even is exact round-to-nearest-even.
    """
    a = np.asarray(a, dtype=f64)
    _, ex = np.frexp(a)  # a = m * 2^ex, m in [0.5, 1)  =>  floor(log2 a) = ex - 1
    b = np.maximum(ex - 1, E4M3_MIN_NORMAL_EXP)
    q = np.ldexp(1.0, b - E4M3_MANT_BITS)
    r = np.rint(a / q) * q
    return np.minimum(r, E4M3_MAX)


def e4m3_encode(neg, r):
    """Byte of an E4M3 value: sign | exponent field (bias 7) | 3 mantissa bits."""
    r = np.asarray(r, dtype=f64)
    _, ex = np.frexp(r)
    normal = r >= 2.0 ** E4M3_MIN_NORMAL_EXP
    efield = np.where(normal, ex - 1 + 7, 0)
    mant = np.where(normal, r / np.ldexp(1.0, ex - 1) * 8 - 8, r / 2.0 ** -9)
    code = (efield.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    code = np.where(r == 0, 0, code)
    return (code | (np.asarray(neg, dtype=np.int64) << 7)).astype(np.uint8)


def e4m3_decode(code):
    """Value of E4M3 bytes (the encoding has no infinities; 0x7F/0xFF are NaN)."""
    c = np.asarray(code, dtype=np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return s * mag


def e8m0_decode(s):
    s = np.asarray(s, dtype=np.int64)
    return np.where(s == 255, np.nan, np.ldexp(1.0, s - 127))


def _blocks(a, axis):
    """View of ``a`` as [outer, n/32, 32, inner]: the 32-blocks along ``axis``."""
    a = np.asarray(a, dtype=f64)
    axis = axis % a.ndim
    n = a.shape[axis]
    if n % MX_BLOCK:
        raise ValueError("blocked axis must be a multiple of 32")
    outer = int(np.prod(a.shape[:axis], dtype=np.int64))
    inner = int(np.prod(a.shape[axis + 1:], dtype=np.int64))
    return a.reshape(outer, n // MX_BLOCK, MX_BLOCK, inner)


def _block_exponent(blk):
    """Per block: whether it is finite, and the shared scale exponent
    e = clamp(floor(log2 amax) - 8, -127, 127), -127 for an all-zero block."""
    amax = np.abs(blk).max(axis=2)  # NaN propagates; Inf stays Inf
    finite = np.isfinite(amax)
    _, ex = np.frexp(np.where(finite, amax, 0.0))  # amax = m * 2^ex, m in [0.5, 1)
    e = np.where(finite & (amax > 0), ex - 1 - E4M3_EMAX, -127)
    return finite, np.clip(e, -127, 127)


def _scaled_magnitudes(blk, finite, e):
    """RNE_E4M3(|v| * 2^-e) of every element (0 inside non-finite blocks)."""
    scaled = np.abs(blk) * np.ldexp(1.0, -e)[:, :, None, :]  # exact: a power of two
    if not finite.all():
        scaled = np.where(finite[:, :, None, :], scaled, 0.0)
    return e4m3_round(scaled)


def mx_quantize(a, axis=-1):
    """MXFP8 (E4M3 elements, E8M0 scales) with 32-blocks along ``axis``.

    For each block: amax = max |v|; scale exponent
    e = clamp(floor(log2 amax) - 8, -127, 127) (amax = 0 -> -127);
    element = RNE_E4M3(v * 2^-e), saturated to +-448.
    Returns (codes uint8 shaped like a, scales uint8 with the axis divided by 32).
    """
    shape = np.shape(a)
    axis = axis % len(shape)
    blk = _blocks(a, axis)
    finite, e = _block_exponent(blk)
    mag = _scaled_magnitudes(blk, finite, e)
    codes = e4m3_encode(np.signbit(blk), mag)
    codes = np.where(finite[:, :, None, :], codes, np.uint8(0x7F)).astype(np.uint8)
    scales = np.where(finite, e + 127, 255).astype(np.uint8)
    sshape = shape[:axis] + (shape[axis] // MX_BLOCK,) + shape[axis + 1:]
    return codes.reshape(shape), scales.reshape(sshape)


def mx_dequantize(codes, scales, axis=-1):
    c = np.moveaxis(np.asarray(codes), axis, -1)
    s = np.moveaxis(np.asarray(scales), axis, -1)
    v = e4m3_decode(c).reshape(c.shape[:-1] + (c.shape[-1] // MX_BLOCK, MX_BLOCK))
    v = v * e8m0_decode(s)[..., None]
    return np.moveaxis(v.reshape(c.shape), -1, axis)


MX_SLAB = 1 << 21  # elements per slab of blocks handled at once by mx_qdq


def mx_qdq(a, axis=-1):
    """The values an MXFP8 GEMM operand carries: each element's quantised
    value times its block's scale, sign(v) * RNE_E4M3(|v| * 2^-e) * 2^e
    (NaN in a block holding Inf or NaN). This is mx_dequantize(mx_quantize(a))
    without the round trip through the byte encoding. Blocks are independent,
    so they are handled a slab of about MX_SLAB elements at a time, which
    bounds the temporary memory of very large operands."""
    b4 = _blocks(a, axis)
    inner = b4.shape[3]
    blk = b4.reshape(-1, 1, MX_BLOCK, inner)  # one row per 32-block (times inner)
    out = np.empty(blk.shape)
    step = max(1, MX_SLAB // (MX_BLOCK * inner))
    for i in range(0, blk.shape[0], step):
        b = blk[i:i + step]
        finite, e = _block_exponent(b)
        v = _scaled_magnitudes(b, finite, e) * np.ldexp(1.0, e)[:, :, None, :]
        v = np.copysign(v, b)
        if not finite.all():
            v = np.where(finite[:, :, None, :], v, np.nan)
        out[i:i + step] = v
    return out.reshape(np.shape(a))


def mx_qdq_cols_in_groups(a):
    """Column-wise (along rows) MXFP8 of one expert group's rows.

    The group is padded with zero rows to a multiple of 32, so the blocks are
    rows [32b, 32b+32) of the group, as in a 32-aligned permuted buffer.
    Returns the dequantised values of the real rows only.
    """
    a = np.asarray(a, dtype=f64)
    n = a.shape[0]
    pad = np.zeros((roundup(n, MX_BLOCK), a.shape[1]), dtype=f64)
    pad[:n] = a
    return mx_qdq(pad, axis=0)[:n]


def act4_cols_in_groups(a):
    """Column-wise operand values of one expert group's rows in the MXFP4
    activation mode [MXFP4-HOPPER]: the rows are quantised row-wise to MXFP8,
    converted directly to row-wise MXFP4, then to column-wise MXFP4 (blocks
    of 32 rows, scales recomputed) and to column-wise MXFP8 (lossless). The
    group is padded with zero rows to a multiple of 32, as in a 32-aligned
    permuted buffer. Returns the values of the real rows only."""
    from oracle import mxfp4_oracle as Q  # that module builds on this one
    a = np.asarray(a, dtype=f64)
    n = a.shape[0]
    pad = np.zeros((roundup(n, MX_BLOCK), a.shape[1]), dtype=f64)
    pad[:n] = a
    c4, s4 = Q.mxfp4_from_mxfp8(*mx_quantize(pad, axis=1))
    cc, sc = Q.mx4_quantize(Q.mx4_dequantize(c4, s4, axis=1), axis=0)
    return Q.mx4_dequantize(cc, sc, axis=0)[:n]


def wgrad_act_cols(a, mx):
    """The column-wise (wgrad) operand values of an activation: MXFP8
    column-wise, or the MXFP4 chain when mx == "act4"."""
    return act4_cols_in_groups(a) if mx == "act4" else mx_qdq_cols_in_groups(a)


def to_f32(a):
    return np.asarray(a, dtype=np.float32).astype(f64)


def to_bf16(a):
    """Round to float32, then to bfloat16 (8 exponent, 7 fraction bits) with
    round-to-nearest-even on the 16 discarded bits, returned as float64.

    Adding 0x7FFF plus the lowest kept bit to the float32 bit pattern and
    clearing the low 16 bits rounds the magnitude to nearest, ties to even;
    a carry into the exponent field is the correct rounding up to the next
    binade (and to infinity past the largest finite value). NaN stays NaN.
    """
    x = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    r = np.where(np.isnan(x), u | 0x00400000, r).astype(np.uint32)
    return r.view(np.float32).astype(f64)


def saved_gate_up(g, u, save_bf16):
    """Gate and up values the backward reads: their BF16 copies when the
    forward saves them in BF16, else the exact values."""
    return (to_bf16(g), to_bf16(u)) if save_bf16 else (g, u)


# ---------------------------------------------------------------------------
# Expert MLP [EMT §Challenge 1 GroupedLinear gate_up; §Challenge 3 ScaledSwiGLU, down]
# ---------------------------------------------------------------------------

def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def dsilu(z):
    s = sigmoid(z)
    return s * (1.0 + z * (1.0 - s))


def expert_rows(idx, e):
    """(tokens, slots) routed to expert e, ordered by token then slot."""
    return np.nonzero(np.asarray(idx) == e)


def _w1_fprop(W1e, mx):
    W = np.asarray(W1e, dtype=f64)
    return mx_qdq(W, axis=0) if mx else W  # blocks along H (the reduction dim)


def _w2_fprop(W2e, mx):
    W = np.asarray(W2e, dtype=f64)
    return mx_qdq(W, axis=0) if mx else W  # blocks along F


def _w1_dgrad(W1e, mx):
    W = np.asarray(W1e, dtype=f64)
    return mx_qdq(W, axis=1) if mx else W  # blocks along 2F


def _w2_dgrad(W2e, mx):
    W = np.asarray(W2e, dtype=f64)
    return mx_qdq(W, axis=1) if mx else W  # blocks along H


def expert_forward(xe, p, W1e, W2e, mx=False):
    """One expert on its routed rows: Y2 = (silu(g) * u * p) @ W2, [g|u] = xe @ W1.

    xe [n, H], p [n] routing weights, W1e [H, 2F], W2e [F, H].
    Returns (y2 [n, H], saved) where saved holds g, u and the FC2 input.
    """
    F = np.asarray(W2e).shape[0]
    xin = np.asarray(xe, dtype=f64)
    if mx:
        xin = mx_qdq(xin, axis=1)
    y1 = xin @ _w1_fprop(W1e, mx)
    g, u = y1[:, :F], y1[:, F:]
    h = silu(g) * u * np.asarray(p, dtype=f64)[:, None]
    hin = mx_qdq(to_f32(h), axis=1) if mx else h
    y2 = hin @ _w2_fprop(W2e, mx)
    return y2, {"g": g, "u": u, "h": h}


def expert_backward(xe, p, W1e, W2e, dy2, saved, mx=False, save_bf16=True):
    """Chain rule through one expert.

    dH = dY2 @ W2^T; a = silu(g)*u; dA = dH*p; dp = sum_f dH*a;
    dg = dA*u*silu'(g); du = dA*silu(g); dY1 = [dg | du];
    dW2 = H^T @ dY2; dXp = dY1 @ W1^T; dW1 = Xp^T @ dY1.
    Returns (dxp [n, H], dp [n], dW1e [H, 2F], dW2e [F, H]).
    """
    g, u = saved_gate_up(saved["g"], saved["u"], save_bf16)
    h = saved["h"]
    p = np.asarray(p, dtype=f64)[:, None]
    dy2 = np.asarray(dy2, dtype=f64)
    xe = np.asarray(xe, dtype=f64)
    dy2_row = mx_qdq(dy2, axis=1) if mx else dy2
    dh = dy2_row @ _w2_dgrad(W2e, mx).T
    a = silu(g) * u
    dA = dh * p
    dp = (dh * a).sum(axis=1)
    dg = dA * u * dsilu(g)
    du = dA * silu(g)
    dy1 = np.concatenate([dg, du], axis=1)
    if mx:
        dy1_32 = to_f32(dy1)
        dy1_row = mx_qdq(dy1_32, axis=1)
        dy1_col = mx_qdq_cols_in_groups(dy1_32)
        h_col = wgrad_act_cols(to_f32(h), mx)
        dy2_col = mx_qdq_cols_in_groups(dy2)
        x_col = wgrad_act_cols(xe, mx)
    else:
        dy1_row = dy1_col = dy1
        h_col, dy2_col, x_col = h, dy2, xe
    dW2e = h_col.T @ dy2_col
    dxp = dy1_row @ _w1_dgrad(W1e, mx).T
    dW1e = x_col.T @ dy1_col
    return dxp, dp, dW1e, dW2e


# ---------------------------------------------------------------------------
# The whole layer, written as the per-expert loop of [EMT §Challenge 1]
# ---------------------------------------------------------------------------

def layer_forward(x, logits, W1, W2, k, mx=False, save_bf16=True):
    """out[t] = sum over the experts e chosen by t of the weighted expert MLP.

    Returns a dict with out [T, H], idx, w and the per-expert saved state
    (the backward reads gate/up through their BF16 copies when save_bf16).
    """
    x = np.asarray(x, dtype=f64)
    idx, w = route(logits, k)
    T, H = x.shape
    E = np.asarray(W1).shape[0]
    out = np.zeros((T, H), dtype=f64)
    saved = []
    for e in range(E):
        tok, slot = expert_rows(idx, e)
        p = w[tok, slot]
        y2, s = expert_forward(x[tok], p, W1[e], W2[e], mx)
        np.add.at(out, tok, y2)
        saved.append((tok, slot, s))
    return {"out": out, "idx": idx, "w": w, "saved": saved, "k": k, "mx": mx,
            "save_bf16": save_bf16}


def layer_backward(fwd, x, W1, W2, dout):
    """Gradients of L = sum(out * dout): dX, dW1, dW2, dlogits (and dp [T, k])."""
    x = np.asarray(x, dtype=f64)
    dout = np.asarray(dout, dtype=f64)
    idx, w, k, mx = fwd["idx"], fwd["w"], fwd["k"], fwd["mx"]
    T, H = x.shape
    E = np.asarray(W1).shape[0]
    dX = np.zeros((T, H), dtype=f64)
    dp = np.zeros((T, k), dtype=f64)
    dW1 = np.zeros(np.asarray(W1).shape, dtype=f64)
    dW2 = np.zeros(np.asarray(W2).shape, dtype=f64)
    for e in range(E):
        tok, slot, s = fwd["saved"][e]
        dxp, dpe, dW1[e], dW2[e] = expert_backward(
            x[tok], w[tok, slot], W1[e], W2[e], dout[tok], s, mx, fwd["save_bf16"])
        np.add.at(dX, tok, dxp)
        dp[tok, slot] = dpe
    dlogits = route_backward(dp, w, idx, E)
    return {"dX": dX, "dW1": dW1, "dW2": dW2, "dlogits": dlogits, "dp": dp}


def layer_fwd_bwd_expert_stream(x, logits, W1, W2, dout, k, mx=False, save_bf16=True):
    """The same per-expert loop, yielding each expert's results in turn.

    Yields (e, tok, slot, y2, dxp, dp, dW1e, dW2e) and holds only one
    expert's gradients at a time, so very wide layers fit in host memory.
    """
    x = np.asarray(x, dtype=f64)
    dout = np.asarray(dout, dtype=f64)
    idx, w = route(logits, k)
    E = np.asarray(W1).shape[0]
    for e in range(E):
        tok, slot = expert_rows(idx, e)
        p = w[tok, slot]
        y2, s = expert_forward(x[tok], p, W1[e], W2[e], mx)
        dxp, dpe, dW1e, dW2e = expert_backward(x[tok], p, W1[e], W2[e], dout[tok], s, mx,
                                               save_bf16)
        yield e, tok, slot, y2, dxp, dpe, dW1e, dW2e


# ---------------------------------------------------------------------------
# Sampled mode: exact values at chosen positions of very large layers
# ---------------------------------------------------------------------------

SAMPLED_THREADS = 4


def map_experts(fn, E):
    """[fn(e) for e in range(E)]. Experts share no state, so a few host
    threads run them at once (numpy releases the interpreter lock inside its
    array operations); every expert's arithmetic is unchanged."""
    from concurrent.futures import ThreadPoolExecutor
    workers = max(1, min(E, SAMPLED_THREADS))
    if workers == 1:
        return [fn(e) for e in range(E)]
    with ThreadPoolExecutor(max_workers=workers) as ex:
        return list(ex.map(fn, range(E)))

def sampled_token_outputs(x, logits, W1, W2, dout, k, tokens, mx=False, save_bf16=True):
    """out, dX and dlogits for the given tokens only.

    Each of these depends only on the token's own k routed rows (every
    quantisation block used here lies inside one row), so they are computed
    exactly, row by row, with the same expert functions as the full loop.
    """
    x = np.asarray(x)
    dout = np.asarray(dout)
    tokens = np.asarray(tokens)
    idx_all, w_all = route(np.asarray(logits)[tokens], k)
    E = np.asarray(W1).shape[0]
    H = x.shape[1]
    nt = tokens.size
    out = np.zeros((nt, H))
    dX = np.zeros((nt, H))
    dp = np.zeros((nt, k))

    def one(e):
        ti, sj = expert_rows(idx_all, e)
        if ti.size == 0:
            return None
        xe = x[tokens[ti]].astype(f64)
        p = w_all[ti, sj]
        y2, s = expert_forward(xe, p, W1[e], W2[e], mx)
        # Row-local backward: dY1 row quantisation and the dgrads need only
        # the row itself; the wgrad outputs of expert_backward are discarded.
        dy2 = dout[tokens[ti]].astype(f64)
        g, u = saved_gate_up(s["g"], s["u"], save_bf16)
        dy2_row = mx_qdq(dy2, axis=1) if mx else dy2
        dh = dy2_row @ _w2_dgrad(W2[e], mx).T
        a = silu(g) * u
        dA = dh * p[:, None]
        dpe = (dh * a).sum(axis=1)
        dy1 = np.concatenate([dA * u * dsilu(g), dA * silu(g)], axis=1)
        dy1_row = mx_qdq(to_f32(dy1), axis=1) if mx else dy1
        dxp = dy1_row @ _w1_dgrad(W1[e], mx).T
        return ti, sj, y2, dxp, dpe

    for r in map_experts(one, E):  # combined in expert order
        if r is None:
            continue
        ti, sj, y2, dxp, dpe = r
        np.add.at(out, ti, y2)
        np.add.at(dX, ti, dxp)
        dp[ti, sj] = dpe
    dlogits = route_backward(dp, w_all, idx_all, E)
    return {"out": out, "dX": dX, "dlogits": dlogits, "idx": idx_all, "w": w_all}


def sampled_weight_grads(x, logits, W1, W2, dout, k, fcols, mx=False, save_bf16=True):
    """dW1[:, :, c], dW1[:, :, F+c] and dW2[:, c, :] for the FFN columns c in fcols.

    fcols must be whole 32-aligned blocks of [0, F), so every row-wise block
    of H and every column-wise block of dY1 that they touch is complete.
    Exact over all routed rows of every expert.
    Returns dW1g [E, H, nc], dW1u [E, H, nc], dW2s [E, nc, H].
    """
    x = np.asarray(x)
    dout = np.asarray(dout)
    fcols = np.asarray(fcols)
    if fcols.size % MX_BLOCK or np.any(fcols.reshape(-1, MX_BLOCK)[:, 0] % MX_BLOCK) \
            or np.any(np.diff(fcols.reshape(-1, MX_BLOCK), axis=1) != 1):
        raise ValueError("fcols must be whole 32-aligned blocks")
    idx, w = route(logits, k)
    E, H, F2 = np.asarray(W1).shape
    F = F2 // 2
    nc = fcols.size
    dW1g = np.zeros((E, H, nc))
    dW1u = np.zeros((E, H, nc))
    dW2s = np.zeros((E, nc, H))

    def one(e):
        tok, slot = expert_rows(idx, e)
        if tok.size == 0:
            return
        xe = x[tok].astype(f64)
        p = w[tok, slot][:, None]
        W1e = np.asarray(W1[e], dtype=f64)
        W2e = np.asarray(W2[e], dtype=f64)
        xin = mx_qdq(xe, axis=1) if mx else xe
        # FC1 columns c and F+c (W1 quantised along H: each column is whole).
        W1f = mx_qdq(W1e[:, np.concatenate([fcols, F + fcols])], axis=0) if mx else \
            W1e[:, np.concatenate([fcols, F + fcols])]
        y1 = xin @ W1f
        g, u = y1[:, :nc], y1[:, nc:]
        h = silu(g) * u * p
        g, u = saved_gate_up(g, u, save_bf16)
        # dH columns c: dY2 (row-quantised along H) times W2 rows c (quantised along H).
        dy2 = dout[tok].astype(f64)
        dy2_row = mx_qdq(dy2, axis=1) if mx else dy2
        W2d = mx_qdq(W2e[fcols], axis=1) if mx else W2e[fcols]
        dh = dy2_row @ W2d.T
        dA = dh * p
        dg = dA * u * dsilu(g)
        du = dA * silu(g)
        if mx:
            h_col = wgrad_act_cols(to_f32(h), mx)
            dy2_col = mx_qdq_cols_in_groups(dy2)
            x_col = wgrad_act_cols(xe, mx)
            dg_col = mx_qdq_cols_in_groups(to_f32(dg))
            du_col = mx_qdq_cols_in_groups(to_f32(du))
        else:
            h_col, dy2_col, x_col, dg_col, du_col = h, dy2, xe, dg, du
        dW2s[e] = h_col.T @ dy2_col
        dW1g[e] = x_col.T @ dg_col
        dW1u[e] = x_col.T @ du_col

    map_experts(one, E)
    return {"dW1g": dW1g, "dW1u": dW1u, "dW2": dW2s}


# ---------------------------------------------------------------------------
# Grouped GEMM [EMT §Challenge 1: GroupedLinear over per-expert row groups]
# ---------------------------------------------------------------------------

def grouped_gemm_fprop(A, B, offsets, b_layout=0):
    """C[r] = A[r] @ B_e for the rows r of group e (offsets[e] <= r < offsets[e+1]).

    b_layout 0: B[e] is [K, N]; 1: B[e] is [N, K] (used transposed).
    Rows outside every group are left zero.
    """
    A = np.asarray(A, dtype=f64)
    B = np.asarray(B, dtype=f64)
    offsets = np.asarray(offsets)
    N = B.shape[2] if b_layout == 0 else B.shape[1]
    C = np.zeros((A.shape[0], N))
    for e in range(len(offsets) - 1):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        Be = B[e] if b_layout == 0 else B[e].T
        C[r0:r1] = A[r0:r1] @ Be
    return C


def grouped_gemm_wgrad(A, B, offsets):
    """C[e] = A[rows_e]^T @ B[rows_e]: the reduction runs over group e's rows."""
    A = np.asarray(A, dtype=f64)
    B = np.asarray(B, dtype=f64)
    offsets = np.asarray(offsets)
    E = len(offsets) - 1
    C = np.zeros((E, A.shape[1], B.shape[1]))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        C[e] = A[r0:r1].T @ B[r0:r1]
    return C
