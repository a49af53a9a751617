"""MoELayer: owns the device workspace of one layer shape and calls the
library's whole-layer forward and backward (argument marshalling only)."""
from __future__ import annotations

import torch

from . import binding as B


class MoELayer:
    def __init__(self, T, H, F, E, k, precision="bf16", align=128, device="cuda"):
        self.T, self.H, self.F, self.E, self.k = T, H, F, E, k
        self.precision = precision
        self.cfg = B.layer_config(T, H, F, E, k, precision, align)
        nbytes = B.moe_layer_workspace_size(self.cfg)
        if nbytes == 0:
            raise B.MoeError(f"unsupported layer config T={T} H={H} F={F} E={E} k={k} "
                             f"precision={precision} align={align}")
        self.device = torch.device(device)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)

    def _expect(self, **named):
        """Each operand must have the shape and dtype the library's layer
        entry points take (the C ABI sees only pointers)."""
        T, H, F, E = self.T, self.H, self.F, self.E
        want = {"logits": ((T, E), torch.float32), "dlogits": ((T, E), torch.float32),
                "x": ((T, H), torch.bfloat16), "out": ((T, H), torch.bfloat16),
                "dout": ((T, H), torch.bfloat16), "dx": ((T, H), torch.bfloat16),
                "w1": ((E, H, 2 * F), torch.bfloat16), "dw1": ((E, H, 2 * F), torch.bfloat16),
                "w2": ((E, F, H), torch.bfloat16), "dw2": ((E, F, H), torch.bfloat16)}
        for name, t in named.items():
            shape, dtype = want[name]
            if tuple(t.shape) != shape or t.dtype != dtype:
                raise B.MoeError(f"{name}: expected {dtype} {list(shape)}, got {t.dtype} "
                                 f"{list(t.shape)}")

    def forward(self, logits, x, w1, w2, out=None, stream=None):
        out = out if out is not None else torch.empty((self.T, self.H), dtype=torch.bfloat16,
                                                      device=self.device)
        self._expect(logits=logits, x=x, w1=w1, w2=w2, out=out)
        return B.moe_layer_forward(self.cfg, logits, x, w1, w2, out, self.workspace, stream)

    def backward(self, dout, w1, w2, dx=None, dw1=None, dw2=None, dlogits=None, stream=None):
        dev = self.device
        dx = dx if dx is not None else torch.empty((self.T, self.H), dtype=torch.bfloat16,
                                                   device=dev)
        dw1 = dw1 if dw1 is not None else torch.empty((self.E, self.H, 2 * self.F),
                                                      dtype=torch.bfloat16, device=dev)
        dw2 = dw2 if dw2 is not None else torch.empty((self.E, self.F, self.H),
                                                      dtype=torch.bfloat16, device=dev)
        dlogits = dlogits if dlogits is not None else torch.empty((self.T, self.E),
                                                                  dtype=torch.float32, device=dev)
        self._expect(dout=dout, w1=w1, w2=w2, dx=dx, dw1=dw1, dw2=dw2, dlogits=dlogits)
        return B.moe_layer_backward(self.cfg, dout, w1, w2, dx, dw1, dw2, dlogits, self.workspace,
                                    stream)

    def capture(self, logits, x, w1, w2, dout, out, dx, dw1, dw2, dlogits):
        """Record one forward + backward over these fixed device buffers as a
        CUDA graph and return it (a torch.cuda.CUDAGraph): each replay() runs the
        layer's launches again on the current stream, reading the buffers' data
        as it is at replay time, with no host work per launch. The layer runs
        once on the capture stream first, so every kernel's one-time launch
        set-up happens outside the capture."""
        self._expect(logits=logits, x=x, w1=w1, w2=w2, out=out, dout=dout, dx=dx, dw1=dw1,
                     dw2=dw2, dlogits=dlogits)
        cs = torch.cuda.Stream(device=self.device)
        cs.wait_stream(torch.cuda.current_stream(self.device))

        def step():
            self.forward(logits, x, w1, w2, out=out, stream=cs)
            self.backward(dout, w1, w2, dx=dx, dw1=dw1, dw2=dw2, dlogits=dlogits, stream=cs)

        with torch.cuda.stream(cs):
            step()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            step()
        torch.cuda.current_stream(self.device).wait_stream(cs)
        return graph

    def part(self, name):
        """A typed view of one saved intermediate in the workspace."""
        pid, dtype = B.PARTS[name]
        off, nbytes = B.moe_layer_workspace_part(self.cfg, pid)
        esz = torch.empty((), dtype=dtype).element_size()
        return self.workspace[off:off + nbytes].view(dtype)[: nbytes // esz]
