"""Whole-layer parity (BF16): the library's forward + backward against the CPU
oracles' per-expert loop (numpy, and at full parity the C++ oracle too), on the
seeded synthetic workloads.

Integer results (routing indices, counts, offsets, dest, src) must match
bit-exactly. Float results must have relative Frobenius error <= 5e-3 and
max-abs error <= 1e-2 * max|ref| (the BF16 tolerance the layer is held to),
on every shape. The oracle's backward reads gate/up through their bf16
copies, as the layer saves them; dlogits = w (dp - sum w dp) would otherwise
be dominated by that rounding wherever a token's dp values nearly cancel.
"""
import numpy as np
import pytest
import torch

from mixture_experts_expert_sort_b300 import inputs as I
from oracle import cpp_oracle as CO
from oracle import moe_oracle as O
from tests.helpers import f64, i32, rel_fro, max_abs_rel

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL_FRO, TOL_MAX = 5e-3, 1e-2


def _layer(wl, precision="bf16"):
    from mixture_experts_expert_sort_b300.layer import MoELayer
    return MoELayer(wl.T, wl.H, wl.F, wl.E, wl.k, precision=precision, align=wl.align)


def _run(wl, inp):
    L = _layer(wl)
    d = {k: v.to(DEV) for k, v in inp.items()}
    out = L.forward(d["logits"], d["x"], d["w1"], d["w2"])
    dx, dw1, dw2, dl = L.backward(d["dout"], d["w1"], d["w2"])
    torch.cuda.synchronize()
    from mixture_experts_expert_sort_b300 import binding
    assert binding.device_error() == 0
    return L, {"out": out, "dX": dx, "dW1": dw1, "dW2": dw2, "dlogits": dl}


def _check(name, got, ref):
    e1, e2 = rel_fro(got, ref), max_abs_rel(got, ref)
    assert e1 <= TOL_FRO and e2 <= TOL_MAX, (name, e1, e2)


def _full_parity(wl, inp):
    L, g = _run(wl, inp)
    x, lg = f64(inp["x"]), f64(inp["logits"])
    w1, w2, dout = f64(inp["w1"]), f64(inp["w2"]), f64(inp["dout"])
    fwd = O.layer_forward(x, lg, w1, w2, wl.k)
    bwd = O.layer_backward(fwd, x, w1, w2, dout)
    # integer parts: bit-exact
    np.testing.assert_array_equal(i32(L.part("idx")).reshape(wl.T, wl.k), fwd["idx"])
    counts, offsets, dest, src = O.permute_plan(fwd["idx"], wl.E, wl.align)
    np.testing.assert_array_equal(i32(L.part("counts")), counts)
    np.testing.assert_array_equal(i32(L.part("offsets")), offsets)
    np.testing.assert_array_equal(i32(L.part("dest")), dest)
    np.testing.assert_array_equal(i32(L.part("src"))[:len(src)], src)
    np.testing.assert_allclose(f64(L.part("w")).reshape(wl.T, wl.k), fwd["w"], atol=2e-6)
    _check("out", f64(g["out"]), fwd["out"])
    _check("dX", f64(g["dX"]), bwd["dX"])
    _check("dW1", f64(g["dW1"]), bwd["dW1"])
    _check("dW2", f64(g["dW2"]), bwd["dW2"])
    _check("dlogits", f64(g["dlogits"]), bwd["dlogits"])
    _check_cpp_oracle(L, wl, inp, g, "bf16")


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


def test_tiny_workload_full_parity():
    wl = I.WORKLOADS["tiny"]
    _full_parity(wl, I.make_all(wl))


EDGE = [
    # T, H, F, E, k, zipf_s, zero_experts
    (77, 128, 128, 1, 1, 0.0, 0),      # single expert, top-1: a dense SwiGLU MLP
    (200, 128, 128, 4, 4, 0.0, 0),     # k = E
    (300, 256, 384, 8, 2, 0.0, 0),     # F not a multiple of 256, ragged T
    (500, 128, 256, 16, 3, 1.2, 4),    # skewed routing with empty experts
    (1, 128, 128, 4, 2, 0.0, 0),       # a single token
]


@pytest.mark.parametrize("T,H,F,E,k,zs,ze", EDGE)
def test_edge_workloads_full_parity(T, H, F, E, k, zs, ze):
    wl = I.Workload("edge", T, H, F, E, k, "bf16", 2000 + T + E, zipf_s=zs, zero_experts=ze)
    _full_parity(wl, I.make_all(wl))


def test_deterministic_bytes():
    wl = I.WORKLOADS["tiny"]
    inp = I.make_all(wl)
    _, a = _run(wl, inp)
    _, b = _run(wl, inp)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.slow
def test_mixtral_workload_sampled_parity():
    """T=8192, H=4096, F=14336, E=8, k=2 (BF16), checked at 256 seeded tokens
    (out, dX, dlogits) and two 32-column FFN blocks of dW1 / dW2 (exact over
    every routed row)."""
    wl = I.WORKLOADS["mixtral"]
    inp = I.make_all(wl)
    L, g = _run(wl, inp)
    x = inp["x"].float().numpy()
    lg = inp["logits"].numpy()
    w1 = inp["w1"].float().numpy()
    w2 = inp["w2"].float().numpy()
    dout = inp["dout"].float().numpy()
    rng = np.random.default_rng(wl.seed)
    toks = np.sort(rng.choice(wl.T, 256, replace=False))
    s = O.sampled_token_outputs(x, lg, w1, w2, dout, wl.k, toks)
    np.testing.assert_array_equal(i32(L.part("idx")).reshape(wl.T, wl.k)[toks], s["idx"])
    _check("out", f64(g["out"])[toks], s["out"])
    _check("dX", f64(g["dX"])[toks], s["dX"])
    _check("dlogits", f64(g["dlogits"])[toks], s["dlogits"])
    fb = np.sort(rng.choice(wl.F // 32, 2, replace=False))
    cols = np.concatenate([np.arange(32 * b, 32 * b + 32) for b in fb])
    wg = O.sampled_weight_grads(x, lg, w1, w2, dout, wl.k, cols)
    dW1 = g["dW1"]
    tc = torch.as_tensor(cols, device=DEV)
    _check("dW1 gate", f64(dW1[:, :, tc]), wg["dW1g"])
    _check("dW1 up", f64(dW1[:, :, wl.F + tc]), wg["dW1u"])
    _check("dW2", f64(g["dW2"][:, tc, :]), wg["dW2"])
