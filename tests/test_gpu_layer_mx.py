"""Whole-layer parity (MXFP8): the library's forward + backward against the CPU
oracles' per-expert loop with MXFP8 emulation (numpy, and at full parity the
C++ oracle too), on the seeded workloads.

Bit-exact: routing indices, the expert-sort plan, and every MXFP8 byte and
scale the layer computes from inputs that both sides hold identically (x and
dOut gathered into expert order, W1 and W2, each row- and column-wise).
Float results (out, dX, dW1, dW2, dlogits) must have relative Frobenius error
<= 1e-2 against the oracle emulating the same quantisation (the MXFP8
tolerance the layer is held to). Quantised intermediates (H, dY1) come from
fp32 accumulators whose summation order differs from the oracle's, so they
are covered by that tolerance rather than compared byte for byte.
"""
import numpy as np
import pytest
import torch

from mixture_experts_expert_sort_b300 import inputs as I
from oracle import cpp_oracle as CO
from oracle import moe_oracle as O
from tests.helpers import f64, i32, u8, rel_fro, max_abs_rel, scales_tiled_to_rowmajor

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_MX = 1e-2


def _run(wl, inp, precision="mxfp8", after_forward=None):
    """Forward and backward; after_forward(L) inspects the workspace between
    the two (in the MXFP4-activation mode the backward reuses the bytes of
    the forward's row-wise FP8 copies of x and H)."""
    from mixture_experts_expert_sort_b300 import binding
    from mixture_experts_expert_sort_b300.layer import MoELayer
    L = MoELayer(wl.T, wl.H, wl.F, wl.E, wl.k, precision=precision, align=wl.align)
    d = {k: v.to(DEV) for k, v in inp.items()}
    out = L.forward(d["logits"], d["x"], d["w1"], d["w2"])
    if after_forward is not None:
        torch.cuda.synchronize()
        after_forward(L)
    dx, dw1, dw2, dl = L.backward(d["dout"], d["w1"], d["w2"])
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return L, {"out": out, "dX": dx, "dW1": dw1, "dW2": dw2, "dlogits": dl}


def _check(name, got, ref):
    e = rel_fro(got, ref)
    assert e <= TOL_MX, (name, e, max_abs_rel(got, ref))


def _rows_of(L, wl):
    """Rows of the permuted buffer: src (flat routed index or -1) and R_max."""
    src = i32(L.part("src"))
    return src, src.size


def _gathered(x, src, k, rows):
    """The permuted copy of x for the given permuted rows (zero rows where src < 0)."""
    s = src[rows]
    out = np.zeros((rows.size, x.shape[1]))
    ok = s >= 0
    out[ok] = x[s[ok] // k]
    return out


def _check_rowwise(L, name, mn, kd, rows, ref_vals):
    """GPU row-wise copy [mn, kd] at `rows` == the oracle's quantisation of ref_vals."""
    sel = torch.as_tensor(rows, device=DEV)
    q = u8(L.part(f"{name}_q_row").view(mn, kd)[sel])
    s = scales_tiled_to_rowmajor(u8(L.part(f"{name}_s_row")), mn, kd)[rows]
    for quantize in (O.mx_quantize, CO.mx_quantize):  # both oracles
        rq, rs = quantize(ref_vals, axis=1)
        np.testing.assert_array_equal(q, rq, err_msg=f"{name} row-wise codes")
        np.testing.assert_array_equal(s, rs, err_msg=f"{name} row-wise scales")


def _check_colwise(L, name, mn, kd, blocks, block_vals):
    """GPU column-wise copy (data [kd, mn], blocks of 32 rows of the [mn, kd]
    operand) at 32-row blocks `blocks` == the oracle's quantisation along rows."""
    qd = L.part(f"{name}_q_col").view(kd, mn)
    s = scales_tiled_to_rowmajor(u8(L.part(f"{name}_s_col")), kd, mn)
    for b, vals in zip(blocks, block_vals):
        for quantize in (O.mx_quantize, CO.mx_quantize):  # both oracles
            rq, rs = quantize(vals, axis=0)  # [32, kd], [1, kd]
            np.testing.assert_array_equal(u8(qd[:, 32 * b:32 * b + 32]).T, rq,
                                          err_msg=f"{name} column-wise codes, block {b}")
            np.testing.assert_array_equal(s[:, b], rs[0],
                                          err_msg=f"{name} column-wise scales, {b}")


def _check_input_quantisation(L, wl, inp, n_rows=None, n_blocks=None, seed=0, act4=False):
    """Bit-exact MXFP8 of the gathered x and dOut and of both weights (in the
    MXFP4 activation mode x is checked by _check_act4_x_forward and
    _check_act4_x instead)."""
    rng = np.random.default_rng(seed)
    src, R = _rows_of(L, wl)
    k = wl.k

    def pick(n, m):
        return np.arange(n) if m is None or m >= n else np.sort(rng.choice(n, m, replace=False))

    for name, t in (("x", inp["x"]), ("dy2", inp["dout"])):
        if act4 and name == "x":
            continue
        x = t.float().numpy()
        rows = pick(R, n_rows)
        _check_rowwise(L, name, R, wl.H, rows, _gathered(x, src, k, rows))
        blocks = pick(R // 32, n_blocks)
        _check_colwise(L, name, R, wl.H, blocks,
                       [_gathered(x, src, k, np.arange(32 * b, 32 * b + 32)) for b in blocks])
    for name, w in (("w1", inp["w1"]), ("w2", inp["w2"])):
        wv = w.float().numpy().reshape(-1, w.shape[2])  # [E*H, 2F] or [E*F, H]
        mn, kd = wv.shape
        rows = pick(mn, n_rows)
        _check_rowwise(L, name, mn, kd, rows, wv[rows].astype(np.float64))
        blocks = pick(mn // 32, n_blocks)
        _check_colwise(L, name, mn, kd, blocks,
                       [wv[32 * b:32 * b + 32].astype(np.float64) for b in blocks])


def _check_cpp_oracle(L, wl, inp, g, mode):
    """The same results against the C++ oracle: its routing and plan bit for
    bit, the float outputs at the same tolerance."""
    r = CO.layer(f64(inp["x"]), f64(inp["logits"]), f64(inp["w1"]), f64(inp["w2"]),
                 f64(inp["dout"]), wl.k, mode)
    np.testing.assert_array_equal(i32(L.part("idx")).reshape(wl.T, wl.k), r["idx"])
    counts, offsets, dest, src = CO.permute_plan(r["idx"], wl.E, wl.align)
    np.testing.assert_array_equal(i32(L.part("counts")), counts)
    np.testing.assert_array_equal(i32(L.part("offsets")), offsets)
    np.testing.assert_array_equal(i32(L.part("dest")), dest)
    np.testing.assert_array_equal(i32(L.part("src"))[:len(src)], src)
    for n in ("out", "dX", "dW1", "dW2", "dlogits"):
        _check(n + " (C++ oracle)", f64(g[n]), r[n])


def _check_plan(L, wl, idx_ref):
    np.testing.assert_array_equal(i32(L.part("idx")).reshape(wl.T, wl.k), idx_ref)
    counts, offsets, dest, src = O.permute_plan(idx_ref, wl.E, wl.align)
    np.testing.assert_array_equal(i32(L.part("counts")), counts)
    np.testing.assert_array_equal(i32(L.part("offsets")), offsets)
    np.testing.assert_array_equal(i32(L.part("dest")), dest)
    gsrc = i32(L.part("src"))
    np.testing.assert_array_equal(gsrc[:len(src)], src)
    assert np.all(gsrc[len(src):] == -1)


EDGE = [
    # T, H, F, E, k, zipf_s, zero_experts, outlier_frac
    (256, 256, 256, 4, 2, 0.0, 0, 0.0),     # a tiny Mixtral-like layer
    (300, 256, 384, 8, 2, 0.0, 0, 0.0),     # ragged T; F not a multiple of 256
    (500, 256, 256, 16, 3, 1.2, 4, 0.0),    # skewed routing with empty experts
    (600, 512, 128, 8, 2, 0.0, 0, 0.02),    # outlier rows x100 stress the block scales
    (77, 256, 128, 1, 1, 0.0, 0, 0.0),      # single expert, top-1: a dense SwiGLU MLP
    (1, 256, 128, 4, 2, 0.0, 0, 0.0),       # a single token
]


@pytest.mark.parametrize("T,H,F,E,k,zs,ze,of", EDGE)
def test_mx_layer_full_parity(T, H, F, E, k, zs, ze, of):
    wl = I.Workload("edge_mx", T, H, F, E, k, "mxfp8", 3000 + T + E, zipf_s=zs,
                    zero_experts=ze, outlier_frac=of)
    inp = I.make_all(wl)
    L, g = _run(wl, inp)
    x, lg = f64(inp["x"]), f64(inp["logits"])
    w1, w2, dout = f64(inp["w1"]), f64(inp["w2"]), f64(inp["dout"])
    fwd = O.layer_forward(x, lg, w1, w2, wl.k, mx=True)
    bwd = O.layer_backward(fwd, x, w1, w2, dout)
    _check_plan(L, wl, fwd["idx"])
    _check_input_quantisation(L, wl, inp)
    np.testing.assert_allclose(f64(L.part("w")).reshape(wl.T, wl.k), fwd["w"], atol=2e-6)
    _check("out", f64(g["out"]), fwd["out"])
    _check("dX", f64(g["dX"]), bwd["dX"])
    _check("dW1", f64(g["dW1"]), bwd["dW1"])
    _check("dW2", f64(g["dW2"]), bwd["dW2"])
    _check("dlogits", f64(g["dlogits"]), bwd["dlogits"])
    _check_cpp_oracle(L, wl, inp, g, "mxfp8")


def test_mx_layer_deterministic():
    wl = I.Workload("edge_mx", 300, 256, 384, 8, 2, "mxfp8", 3308)
    inp = I.make_all(wl)
    _, a = _run(wl, inp)
    _, b = _run(wl, inp)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def _sampled_parity(wl, n_tokens=256):
    """Full-size workload: out, dX and dlogits at n_tokens seeded tokens, two
    32-column FFN blocks of dW1 (gate and up) and dW2 exact over every routed
    row, bit-exact plan and input-side MXFP8 on sampled rows and blocks."""
    inp = I.make_all(wl)
    L, g = _run(wl, inp)
    x = inp["x"].float().numpy()
    lg = inp["logits"].numpy()
    w1 = inp["w1"].float().numpy()
    w2 = inp["w2"].float().numpy()
    dout = inp["dout"].float().numpy()
    idx_ref, _ = O.route(lg, wl.k)
    _check_plan(L, wl, idx_ref)
    _check_input_quantisation(L, wl, inp, n_rows=256, n_blocks=8, seed=wl.seed)
    rng = np.random.default_rng(wl.seed)
    toks = np.sort(rng.choice(wl.T, n_tokens, replace=False))
    s = O.sampled_token_outputs(x, lg, w1, w2, dout, wl.k, toks, mx=True)
    _check("out", f64(g["out"])[toks], s["out"])
    _check("dX", f64(g["dX"])[toks], s["dX"])
    _check("dlogits", f64(g["dlogits"])[toks], s["dlogits"])
    fb = np.sort(rng.choice(wl.F // 32, 2, replace=False))
    cols = np.concatenate([np.arange(32 * b, 32 * b + 32) for b in fb])
    wg = O.sampled_weight_grads(x, lg, w1, w2, dout, wl.k, cols, mx=True)
    tc = torch.as_tensor(cols, device=DEV)
    _check("dW1 gate", f64(g["dW1"][:, :, tc]), wg["dW1g"])
    _check("dW1 up", f64(g["dW1"][:, :, wl.F + tc]), wg["dW1u"])
    _check("dW2", f64(g["dW2"][:, tc, :]), wg["dW2"])
    # experts that received no token get exactly zero weight gradients
    empty = np.nonzero(i32(L.part("counts")) == 0)[0]
    for e in empty:
        assert not torch.any(g["dW1"][int(e)]) and not torch.any(g["dW2"][int(e)])


def _check_act4_x_forward(L, wl, inp):
    """MXFP4 activation mode after the forward, bit-exact: the row-wise MXFP8
    of the gathered x that FC1 read, and the MXFP4 copy made from it."""
    from oracle import mxfp4_oracle as Q
    src, R = _rows_of(L, wl)
    xg = _gathered(inp["x"].float().numpy(), src, wl.k, np.arange(R))
    _check_rowwise(L, "x", R, wl.H, np.arange(R), xg)
    c4, s4 = Q.mxfp4_from_mxfp8(*O.mx_quantize(xg, axis=1))
    np.testing.assert_array_equal(u8(L.part("x4_q_row")).reshape(R, wl.H // 2), Q.pack_e2m1(c4))
    np.testing.assert_array_equal(
        scales_tiled_to_rowmajor(u8(L.part("x4_s_row")), R, wl.H), s4)


def _check_act4_x(L, wl, inp):
    """MXFP4 activation mode after the backward, bit-exact: the column-wise
    MXFP8 operand of FC1's wgrad that the backward rebuilt from the MXFP4
    copy of x (in the bytes of the forward's row-wise FP8 copy)."""
    from oracle import mxfp4_oracle as Q
    src, R = _rows_of(L, wl)
    xg = _gathered(inp["x"].float().numpy(), src, wl.k, np.arange(R))
    c4, s4 = Q.mxfp4_from_mxfp8(*O.mx_quantize(xg, axis=1))
    np.testing.assert_array_equal(u8(L.part("x4_q_row")).reshape(R, wl.H // 2), Q.pack_e2m1(c4))
    c8c, s8c = Q.mxfp8_col_from_mxfp4_row(c4, s4)
    np.testing.assert_array_equal(u8(L.part("x_q_col")).reshape(wl.H, R), c8c)
    np.testing.assert_array_equal(
        scales_tiled_to_rowmajor(u8(L.part("x_s_col")), wl.H, R), s8c)


@pytest.mark.parametrize("T,H,F,E,k,zs,ze,of", EDGE[:4] + EDGE[5:])
def test_act4_layer_full_parity(T, H, F, E, k, zs, ze, of):
    """MXFP8 compute with X and H carried to the backward as MXFP4: every
    output against the oracle emulating the same FP8 -> FP4 -> column-wise
    chain, and the x side byte for byte."""
    wl = I.Workload("edge_mx4", T, H, F, E, k, "mxfp8", 3100 + T + E, zipf_s=zs,
                    zero_experts=ze, outlier_frac=of)
    inp = I.make_all(wl)
    L, g = _run(wl, inp, precision="mxfp8_act4",
                after_forward=lambda L: _check_act4_x_forward(L, wl, inp))
    x, lg = f64(inp["x"]), f64(inp["logits"])
    w1, w2, dout = f64(inp["w1"]), f64(inp["w2"]), f64(inp["dout"])
    fwd = O.layer_forward(x, lg, w1, w2, wl.k, mx="act4")
    bwd = O.layer_backward(fwd, x, w1, w2, dout)
    _check_plan(L, wl, fwd["idx"])
    _check_input_quantisation(L, wl, inp, act4=True)
    _check_act4_x(L, wl, inp)
    _check("out", f64(g["out"]), fwd["out"])
    _check("dX", f64(g["dX"]), bwd["dX"])
    _check("dW1", f64(g["dW1"]), bwd["dW1"])
    _check("dW2", f64(g["dW2"]), bwd["dW2"])
    _check("dlogits", f64(g["dlogits"]), bwd["dlogits"])
    _check_cpp_oracle(L, wl, inp, g, "mxfp8_act4")
    # the MXFP4 chain is what the weight gradients saw: the plain MXFP8
    # oracle differs from it by more than the tolerance on dW1
    ref8 = O.layer_backward(O.layer_forward(x, lg, w1, w2, wl.k, mx=True), x, w1, w2, dout)
    assert rel_fro(bwd["dW1"], ref8["dW1"]) > 2 * rel_fro(f64(g["dW1"]), bwd["dW1"])


@pytest.mark.slow
def test_mixtral_mx_workload_sampled_parity():
    """T=16384, H=4096, F=14336, E=8, top-2, MXFP8."""
    _sampled_parity(I.WORKLOADS["mixtral_mx"])


@pytest.mark.slow
def test_finegrained_workload_sampled_parity():
    """T=16384, H=2048, F=1408, E=64, top-6, MXFP8, Zipf-skewed routing with
    four experts that receive no token."""
    wl = I.WORKLOADS["finegrained"]
    _sampled_parity(wl)


@pytest.mark.slow
def test_long_workload_sampled_parity():
    """T=65536, H=4096, F=14336, E=8, top-2, MXFP8, 1% of x rows scaled x100."""
    _sampled_parity(I.WORKLOADS["long"])


@pytest.mark.slow
def test_mixtral_act4_workload_sampled_parity():
    """T=16384, H=4096, F=14336, E=8, top-2, MXFP8 compute with MXFP4-carried
    X and H: sampled tokens and weight-gradient columns against the oracle."""
    wl = I.WORKLOADS["mixtral_mx"]
    inp = I.make_all(wl)
    L, g = _run(wl, inp, precision="mxfp8_act4")
    x = inp["x"].float().numpy()
    lg = inp["logits"].numpy()
    w1 = inp["w1"].float().numpy()
    w2 = inp["w2"].float().numpy()
    dout = inp["dout"].float().numpy()
    rng = np.random.default_rng(wl.seed + 1)
    toks = np.sort(rng.choice(wl.T, 128, replace=False))
    s = O.sampled_token_outputs(x, lg, w1, w2, dout, wl.k, toks, mx="act4")
    _check("out", f64(g["out"])[toks], s["out"])
    _check("dX", f64(g["dX"])[toks], s["dX"])
    fb = np.sort(rng.choice(wl.F // 32, 1, replace=False))
    cols = np.arange(32 * fb[0], 32 * fb[0] + 32)
    wg = O.sampled_weight_grads(x, lg, w1, w2, dout, wl.k, cols, mx="act4")
    tc = torch.as_tensor(cols, device=DEV)
    _check("dW1 gate", f64(g["dW1"][:, :, tc]), wg["dW1g"])
    _check("dW1 up", f64(g["dW1"][:, :, wl.F + tc]), wg["dW1u"])
    _check("dW2", f64(g["dW2"][:, tc, :]), wg["dW2"])
