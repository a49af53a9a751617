"""Seeded synthetic inputs for the MoE expert layer.

This module only draws random numbers and gives them the shapes and value
distributions of the five workloads; it performs none of the layer's
arithmetic. Both the CUDA path (through the tests and the benchmark) and the
CPU oracle are fed from here, so the two always see identical inputs.

Workloads (T tokens, H hidden, F FFN width, E experts, top-k):

* ``tiny``        T=256,   H=128,  F=256,   E=4,  k=2, BF16
* ``mixtral``     T=8192,  H=4096, F=14336, E=8,  k=2, BF16
* ``mixtral_mx``  T=16384, H=4096, F=14336, E=8,  k=2, MXFP8
* ``finegrained`` T=16384, H=2048, F=1408,  E=64, k=6, MXFP8, skewed routing
* ``long``        T=65536, H=4096, F=14336, E=8,  k=2, MXFP8, 1 % outlier rows

Distributions: x ~ N(0,1) rounded to bf16; W1 [E,H,2F] (gate columns
[0,F), up columns [F,2F)) and W2 [E,F,H] ~ N(0, 0.02^2) rounded to bf16;
router logits fp32 N(0,1) [T,E]; upstream gradient dOut ~ N(0,1) bf16.
``finegrained`` adds a per-expert bias b_e = -1.2*ln(r_e) to the logits, with
r a seeded permutation of 1..E (Zipf(s=1.2) log-popularity); the four experts
with the largest r get b_e = -1e4 so that they receive no token at all.
``long`` scales round(0.01*T) seeded rows of x by 100. The optional router
projection W_r [H, E] is N(0, 1/H) in bf16.

Every tensor has its own seed (workload seed * 16 + tensor id), so a tensor's
values do not depend on which other tensors were drawn.
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    F: int
    E: int
    k: int
    precision: str  # "bf16", "mxfp8" or "mxfp8_act4" (MXFP8 with MXFP4-carried X and H)
    seed: int
    zipf_s: float = 0.0  # > 0: Zipf-skewed per-expert logit bias
    zero_experts: int = 0  # experts forced to receive no token
    outlier_frac: float = 0.0  # fraction of x rows scaled by outlier_scale
    outlier_scale: float = 100.0
    align: int = 128  # rows per expert group are padded to a multiple of this

    @property
    def R(self) -> int:
        return self.T * self.k

    def with_tokens(self, T: int) -> "Workload":
        return replace(self, T=T)

    def gemm_flops_fwd_bwd(self) -> float:
        # FC1 (2*R*H*2F) + FC2 (2*R*F*H), times 3 for fprop, dgrad and wgrad.
        return 18.0 * self.T * self.k * self.H * self.F


WORKLOADS = {
    "tiny": Workload("tiny", 256, 128, 256, 4, 2, "bf16", 1001),
    "mixtral": Workload("mixtral", 8192, 4096, 14336, 8, 2, "bf16", 1002),
    "mixtral_mx": Workload("mixtral_mx", 16384, 4096, 14336, 8, 2, "mxfp8", 1003),
    "mixtral_mx4": Workload("mixtral_mx4", 16384, 4096, 14336, 8, 2, "mxfp8_act4", 1003),
    "finegrained": Workload("finegrained", 16384, 2048, 1408, 64, 6, "mxfp8", 1004,
                            zipf_s=1.2, zero_experts=4),
    "long": Workload("long", 65536, 4096, 14336, 8, 2, "mxfp8", 1005, outlier_frac=0.01),
}

_X, _W1, _W2, _LOGITS, _DOUT, _BIAS_PERM, _OUTLIER_ROWS, _WROUTER, _DLOGITS = range(9)


def _gen(wl: Workload, tensor_id: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed * 16 + tensor_id)
    return g


def _normal(shape, std, wl, tid, device, dtype):
    g = _gen(wl, tid, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(dtype)


def expert_bias(wl: Workload) -> torch.Tensor:
    """Per-expert logit bias (fp32, [E]); zeros unless the workload is skewed."""
    if wl.zipf_s <= 0:
        return torch.zeros(wl.E, dtype=torch.float32)
    g = _gen(wl, _BIAS_PERM, "cpu")
    r = torch.randperm(wl.E, generator=g).to(torch.float64) + 1.0  # ranks 1..E
    b = -wl.zipf_s * torch.log(r)
    if wl.zero_experts:
        b[r > wl.E - wl.zero_experts] = -1.0e4
    return b.to(torch.float32)


def outlier_rows(wl: Workload) -> torch.Tensor:
    n = int(round(wl.outlier_frac * wl.T))
    if n == 0:
        return torch.zeros(0, dtype=torch.int64)
    g = _gen(wl, _OUTLIER_ROWS, "cpu")
    return torch.randperm(wl.T, generator=g)[:n].sort().values


def make_x(wl: Workload, device="cpu") -> torch.Tensor:
    x = _normal((wl.T, wl.H), 1.0, wl, _X, device, torch.float32)
    rows = outlier_rows(wl)
    if rows.numel():
        x[rows.to(x.device)] *= wl.outlier_scale
    return x.to(torch.bfloat16)


def make_w1(wl: Workload, device="cpu") -> torch.Tensor:
    return _normal((wl.E, wl.H, 2 * wl.F), 0.02, wl, _W1, device, torch.bfloat16)


def make_w2(wl: Workload, device="cpu") -> torch.Tensor:
    return _normal((wl.E, wl.F, wl.H), 0.02, wl, _W2, device, torch.bfloat16)


def make_logits(wl: Workload, device="cpu") -> torch.Tensor:
    lg = _normal((wl.T, wl.E), 1.0, wl, _LOGITS, device, torch.float32)
    return lg + expert_bias(wl).to(lg.device)[None, :]


def make_dout(wl: Workload, device="cpu") -> torch.Tensor:
    return _normal((wl.T, wl.H), 1.0, wl, _DOUT, device, torch.bfloat16)


def make_router_weights(wl: Workload, device="cpu") -> torch.Tensor:
    """Router projection W_r [H, E] ~ N(0, 1/H) in bf16 (logits of order 1)."""
    return _normal((wl.H, wl.E), wl.H ** -0.5, wl, _WROUTER, device, torch.bfloat16)


def make_dlogits(wl: Workload, device="cpu") -> torch.Tensor:
    """An upstream gradient for the router logits, fp32 N(0,1) [T, E]."""
    return _normal((wl.T, wl.E), 1.0, wl, _DLOGITS, device, torch.float32)


def make_all(wl: Workload, device="cpu") -> dict:
    return {
        "x": make_x(wl, device),
        "logits": make_logits(wl, device),
        "w1": make_w1(wl, device),
        "w2": make_w2(wl, device),
        "dout": make_dout(wl, device),
    }
