"""Parity of the router projection and the auxiliary load-balancing loss
(moe_router_forward / moe_router_backward) with the CPU oracles (numpy and C++).

The logits are fp32 sums over H on the GPU and exact on the CPU, so they are
compared within the rounding bound of an H-term fp32 sum. The routing decision
is bit-exact for every token whose top-(k+1) logits are separated by more than
twice that bound; for the rare closer tokens the GPU's choice must be a valid
top-k of the exact logits within the bound. The aux statistics, the logit
gradient (fp32) and dx / dW_r (bf16) are compared within tolerances derived
from their arithmetic.
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

CASES = [
    # T, H, E, k
    (300, 256, 8, 2),
    (8192, 4096, 8, 2),      # Mixtral shape
    (4096, 2048, 64, 6),     # fine-grained shape
    (100, 128, 256, 8),
    (1, 64, 4, 2),
    (50, 128, 1, 1),          # a single expert: seven zero-padded expert columns
    (77, 192, 3, 2),          # E not a multiple of 4, H not a multiple of 128
]


def _inputs(T, H, E, k):
    wl = I.Workload("router", T, H, 256, E, k, "bf16", 4000 + T + E)
    return wl, I.make_x(wl), I.make_router_weights(wl), I.make_dlogits(wl)


def _bound(x, wr):
    """Rounding bound of an H-term fp32 sum: H * 2^-24 * sum_h |x_h w_h| (+ the final rounding)."""
    H = x.shape[1]
    return (H + 1) * 2.0 ** -24 * (np.abs(x) @ np.abs(wr))


@pytest.mark.parametrize("T,H,E,k", CASES)
def test_router_forward(T, H, E, k):
    from mixture_experts_expert_sort_b300 import binding as B
    wl, x, wr, _ = _inputs(T, H, E, k)
    o = B.moe_router_forward(x.to(DEV), wr.to(DEV), k)
    torch.cuda.synchronize()
    assert B.device_error() == 0
    xf, wf = f64(x), f64(wr)
    ref = O.router_logits(xf, wf)
    bound = _bound(xf, wf)
    lg = f64(o["logits"])
    assert np.all(np.abs(lg - ref) <= bound), np.max(np.abs(lg - ref) / bound)
    ridx, rw = O.route(ref, k)
    gidx = i32(o["idx"])
    # tokens whose top-(k+1) values are separated by more than twice the bound
    srt = -np.sort(-ref, axis=1)[:, :min(k + 1, E)]
    gaps = np.abs(np.diff(srt, axis=1)).min(axis=1) if srt.shape[1] > 1 else np.full(T, np.inf)
    clear = gaps > 2 * bound.max(axis=1)
    np.testing.assert_array_equal(gidx[clear], ridx[clear])
    for t in np.nonzero(~clear)[0]:  # near ties: a valid top-k of the exact logits
        kth = srt[t, k - 1]
        assert np.all(ref[t, gidx[t]] >= kth - 2 * bound[t].max()), t
    np.testing.assert_allclose(f64(o["w"])[clear], rw[clear], atol=1e-5)
    L, f, P = O.aux_load_balance(ref, ridx, E)
    aux = f64(o["aux"])
    assert abs(aux[0] - L) <= 1e-5 * L + E * (~clear).sum() / (T * k), (aux[0], L)
    np.testing.assert_allclose(aux[1 + E:], P, rtol=1e-5, atol=1e-7)
    assert np.abs(aux[1:1 + E] - f).max() <= (~clear).sum() / (T * k) + 1e-7
    # the C++ oracle: the same exact logits, routing and statistics
    c = CO.router_forward(xf, wf, k)
    assert np.all(np.abs(lg - c["logits"]) <= bound)
    np.testing.assert_array_equal(gidx[clear], c["idx"][clear])
    assert abs(aux[0] - c["aux"]) <= 1e-5 * c["aux"] + E * (~clear).sum() / (T * k)
    np.testing.assert_allclose(aux[1 + E:], c["P"], rtol=1e-5, atol=1e-7)


@pytest.mark.parametrize("T,H,E,k", CASES)
def test_router_backward(T, H, E, k):
    from mixture_experts_expert_sort_b300 import binding as B
    wl, x, wr, dl_route = _inputs(T, H, E, k)
    g = torch.Generator().manual_seed(T + H + E)
    dx_in = torch.randn((T, H), generator=g).to(torch.bfloat16)
    coeff = 0.02
    xd, wd = x.to(DEV), wr.to(DEV)
    o = B.moe_router_forward(xd, wd, k)
    dl, dx, dw = B.moe_router_backward(xd, wd, o["logits"], o["aux"], dl_route.to(DEV), coeff,
                                       dx_in=dx_in.to(DEV))
    torch.cuda.synchronize()
    assert B.device_error() == 0
    xf, wf = f64(x), f64(wr)
    ref = O.router_logits(xf, wf)
    ridx, _ = O.route(ref, k)
    _, f, _ = O.aux_load_balance(ref, ridx, E)
    dl_ref = f64(dl_route) + coeff * O.aux_load_balance_grad(ref, f)
    assert rel_fro(f64(dl), dl_ref) <= 1e-5, rel_fro(f64(dl), dl_ref)
    dx_ref, dw_ref = O.router_backward(xf, wf, dl_ref)
    dx_ref = dx_ref + f64(dx_in)
    for name, got, r in (("dx", f64(dx), dx_ref), ("dW_r", f64(dw), dw_ref)):
        assert rel_fro(got, r) <= 5e-3 and max_abs_rel(got, r) <= 1e-2, (name, rel_fro(got, r))
    # the C++ oracle, from its own forward
    c = CO.router_forward(xf, wf, k)
    dlc, dxc, dwc = CO.router_backward(xf, wf, c["logits"], c["f"], f64(dl_route), coeff)
    assert rel_fro(f64(dl), dlc) <= 1e-5, rel_fro(f64(dl), dlc)
    for name, got, r in (("dx", f64(dx), dxc + f64(dx_in)), ("dW_r", f64(dw), dwc)):
        assert rel_fro(got, r) <= 5e-3 and max_abs_rel(got, r) <= 1e-2, (name, rel_fro(got, r))


def test_router_deterministic():
    from mixture_experts_expert_sort_b300 import binding as B
    wl, x, wr, dl_route = _inputs(4096, 2048, 64, 6)
    xd, wd, dd = x.to(DEV), wr.to(DEV), dl_route.to(DEV)
    runs = []
    for _ in range(2):
        o = B.moe_router_forward(xd, wd, 6)
        dl, dx, dw = B.moe_router_backward(xd, wd, o["logits"], o["aux"], dd, 0.01)
        runs.append([o["logits"], o["idx"], o["aux"], dl, dx, dw])
    for a, b in zip(*runs):
        assert torch.equal(a, b)
