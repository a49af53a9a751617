"""The layer captured as a CUDA graph (MoELayer.capture): a replay computes
exactly what the eager calls compute, on the data the buffers hold at replay
time (BF16, MXFP8 and MXFP8 with MXFP4-carried activations)."""
import pytest
import torch

from mixture_experts_expert_sort_b300 import binding as B
from mixture_experts_expert_sort_b300 import inputs as I
from mixture_experts_expert_sort_b300.layer import MoELayer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _buffers(wl, seed):
    inp = I.make_all(I.Workload(wl.name, wl.T, wl.H, wl.F, wl.E, wl.k, wl.precision, seed))
    d = {k: v.to(DEV) for k, v in inp.items()}
    T, H, F, E = wl.T, wl.H, wl.F, wl.E
    bf = torch.bfloat16
    d.update(out=torch.empty((T, H), dtype=bf, device=DEV),
             dx=torch.empty((T, H), dtype=bf, device=DEV),
             dw1=torch.empty((E, H, 2 * F), dtype=bf, device=DEV),
             dw2=torch.empty((E, F, H), dtype=bf, device=DEV),
             dlogits=torch.empty((T, E), dtype=torch.float32, device=DEV))
    return d


def _eager(L, d):
    out = L.forward(d["logits"], d["x"], d["w1"], d["w2"])
    dx, dw1, dw2, dl = L.backward(d["dout"], d["w1"], d["w2"])
    torch.cuda.synchronize()
    return {"out": out, "dx": dx, "dw1": dw1, "dw2": dw2, "dlogits": dl}


@pytest.mark.parametrize("T,H,F,E,k,precision", [
    (256, 128, 256, 4, 2, "bf16"),
    (300, 256, 384, 8, 2, "mxfp8"),
    (256, 256, 256, 4, 2, "mxfp8_act4"),
])
def test_graph_replay_equals_eager(T, H, F, E, k, precision):
    wl = I.Workload("graph", T, H, F, E, k, precision, 5100 + T)
    L = MoELayer(T, H, F, E, k, precision=precision, align=wl.align)
    d = _buffers(wl, 5100 + T)
    g = L.capture(d["logits"], d["x"], d["w1"], d["w2"], d["dout"], d["out"], d["dx"],
                  d["dw1"], d["dw2"], d["dlogits"])
    # new data in the captured buffers: the replay must read it
    d2 = _buffers(wl, 6100 + T)
    for n in ("logits", "x", "w1", "w2", "dout"):
        d[n].copy_(d2[n])
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert B.device_error() == 0
        ref = _eager(MoELayer(T, H, F, E, k, precision=precision, align=wl.align), d2)
        for n in ref:
            assert torch.equal(d[n], ref[n]), n
