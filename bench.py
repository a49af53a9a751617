"""Benchmark: MoE expert layer forward + backward on B300.

One step = one pass of the whole layer (route, expert sort, permute, FC1 +
scaled SwiGLU, FC2, combine, and the full backward) over one batch of T
tokens, through the libmoe C ABI.

Prints ONE JSON line (rank 0). Default: 1 GPU, the Mixtral-8x7B expert-layer
shape in MXFP8 (T=16384, H=4096, F=14336, E=8, top-2). The other workloads
(tiny, Mixtral BF16, MXFP8 with MXFP4-carried activations, fine-grained
skewed, long) are measured the same way in the same run and reported under
"workloads" in that line (--configs none skips them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--configs all|none|a,b]
                  [--impl ours|reference]

Timing: W untimed steps, then K steps between CUDA events on the launching
stream; per-kernel times are means over the K steps (the statistic of
ms_per_step). Roofline denominators: the measured BF16 burst rate (times 2,
the nominal dense MXFP8/BF16 ratio, for MXFP8 GEMMs) and the measured HBM
copy bandwidth.

Multi-GPU (launched with torch.distributed.run): each rank runs its own
T-token batch (the layer is data-parallel over tokens; no collective is on
the data path), so scaling is weak and `value` sums the tokens of all ranks
over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import datetime
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_experts_expert_sort_b300 import inputs as I  # noqa: E402

METRIC = "MoE-layer tokens/s (fwd+bwd) and grouped-GEMM TFLOP/s, % of B300 peak"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                "sm_max_mhz": pk.get("sm_max_mhz", 2032.0), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0,
                "sm_max_mhz": 2032.0, "source": "fallback"}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples every 50 ms while running. mark_begin()/mark_end()
    bracket the timed region on the host clock; stop() reports the median SM
    clock and the throttle reasons of the samples taken inside it (all samples
    when none fell inside)."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def mark_begin(self):
        self.t0 = datetime.datetime.now()

    def mark_end(self):
        self.t1 = datetime.datetime.now()

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 10:
                    try:
                        ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f")
                    except ValueError:
                        ts = None
                    rows.append((ts, parts[1:]))
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for ts, r in rows
                  if ts is not None and self.t0 is not None and self.t1 is not None
                  and self.t0 <= ts <= self.t1]
        use = inside or [r for _, r in rows]
        sm = [float(r[1]) for r in use if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows), "samples_in_timed_region": len(inside)}


# ------------------------------------------------------------- the step

class Step:
    """The layer pass as the sequence of C-ABI calls that moe_layer_forward /
    moe_layer_backward make, over the same workspace, with optional CUDA events
    between calls for the per-kernel breakdown."""

    def __init__(self, wl, dev, router=False, gather=False):
        from mixture_experts_expert_sort_b300 import binding as B
        from mixture_experts_expert_sort_b300.layer import MoELayer
        self.B = B
        self.wl = wl
        self.router = router
        self.mx = wl.precision in ("mxfp8", "mxfp8_act4")
        self.act4 = wl.precision == "mxfp8_act4"
        # BF16 only: read x and dOut through row gathers instead of the
        # permuted copies the layer makes (a comparison, not the layer's sequence)
        self.gather = gather and not self.mx
        self.layer = MoELayer(wl.T, wl.H, wl.F, wl.E, wl.k, precision=wl.precision,
                              align=wl.align, device=dev)
        L = self.layer
        self.P = {n: L.part(n) for n in B.PARTS}
        self.rmax = self.P["src"].numel()
        self.nparts = self.P["dp"].numel() // self.rmax
        self.plan_ws = torch.empty(B.moe_permute_plan_workspace_size(wl.T, wl.E, wl.k),
                                   dtype=torch.uint8, device=dev)
        if router:
            # Router projection W_r [H, E], its gradient, the logits it produces,
            # the aux statistics and the router workspace.
            self.w_r = I.make_router_weights(wl, device=dev)
            self.dw_r = torch.empty_like(self.w_r)
            self.logits_r = torch.empty((wl.T, wl.E), dtype=torch.float32, device=dev)
            self.aux = torch.empty(1 + 2 * wl.E, dtype=torch.float32, device=dev)
            self.router_ws = torch.empty(B.moe_router_workspace_size(wl.T, wl.H, wl.E),
                                         dtype=torch.uint8, device=dev)
        self.NAMES = [n for n, _ in self._ops(*([None] * 10))]
        # kernels per step: the plan is three launches, the router forward five
        # and its backward four, every other call one
        self.launches_per_step = len(self.NAMES) + 2 + (7 if router else 0)

    def _ops(self, logits, x, w1, w2, dout, out, dx, dw1, dw2, dlogits):
        B, wl, P = self.B, self.wl, self.P
        L = B.lib()
        s = B.stream_handle()
        T, H, F, E, k, R = wl.T, wl.H, wl.F, wl.E, wl.k, self.rmax
        # Every tensor of the step is bound once, so each address is checked
        # and taken once; the calls then pass plain integers.
        addr, keep = {}, []

        def p(t):
            if t is None:
                return None
            a = addr.get(id(t))
            if a is None:
                a = addr[id(t)] = B.ptr(t)
                keep.append(t)  # the id stays this tensor's while the step holds it
            return a
        self._bound = keep
        RC = B.QUANT_ROWWISE | B.QUANT_COLWISE
        npart = self.nparts
        if self.router:
            first = ("router_fwd", lambda: L.moe_router_forward(
                p(x), p(self.w_r), T, H, E, k, p(self.logits_r), p(P["idx"]), p(P["w"]),
                p(self.aux), p(self.router_ws), self.router_ws.numel(), s))
        else:
            first = ("route", lambda: L.moe_route(p(logits), T, E, k, p(P["idx"]), p(P["w"]), s))
        ops = [
            first,
            ("plan", lambda: L.moe_permute_plan(
                p(P["idx"]), T, E, k, wl.align, p(P["counts"]), p(P["offsets"]), p(P["dest"]),
                p(P["src"]), R, p(self.plan_ws), self.plan_ws.numel(), s)),
        ]
        if self.gather:
            import ctypes
            g = ctypes.byref(B.RowGather(p(P["src"]), k, T))
            ops += [
                ("p_rows", lambda: L.moe_permute(
                    p(x), p(P["dest"]), p(P["offsets"]), p(P["counts"]), p(P["w"]), T, H, E, k,
                    None, p(P["p_rows"]), s)),
                ("fc1_swiglu", lambda: L.moe_fc1_swiglu_bf16(
                    p(x), p(w1), p(P["offsets"]), p(P["p_rows"]), E, R, H, F, p(P["gu"]),
                    p(P["h"]), g, s)),
                ("fc2", lambda: L.moe_grouped_gemm_bf16(
                    0, p(P["h"]), p(w2), 0, p(P["offsets"]), E, R, 0, H, F, p(P["y2"]), None,
                    None, s)),
                ("unpermute", lambda: L.moe_unpermute(p(P["y2"]), p(P["dest"]), None, T, H, k,
                                                      p(out), s)),
                ("fc2_dgrad_swiglu_bwd", lambda: L.moe_fc2_dgrad_swiglu_bwd_bf16(
                    p(dout), p(w2), p(P["offsets"]), p(P["p_rows"]), p(P["gu"]), E, R, H, F,
                    p(P["dy1"]), p(P["dp"]), g, s)),
                ("fc2_wgrad", lambda: L.moe_grouped_gemm_bf16(
                    1, p(P["h"]), p(dout), 0, p(P["offsets"]), E, R, F, H, 0, p(dw2), None, g,
                    s)),
                ("fc1_dgrad", lambda: L.moe_grouped_gemm_bf16(
                    0, p(P["dy1"]), p(w1), 1, p(P["offsets"]), E, R, 0, H, 2 * F, p(P["dxp"]),
                    None, None, s)),
                ("fc1_wgrad", lambda: L.moe_grouped_gemm_bf16(
                    1, p(x), p(P["dy1"]), 0, p(P["offsets"]), E, R, H, 2 * F, 0, p(dw1), g, None,
                    s)),
            ]
        elif not self.mx:
            ops += [
                ("permute_x", lambda: L.moe_permute(
                    p(x), p(P["dest"]), p(P["offsets"]), p(P["counts"]), p(P["w"]), T, H, E, k,
                    p(P["xp"]), p(P["p_rows"]), s)),
                ("fc1_swiglu", lambda: L.moe_fc1_swiglu_bf16(
                    p(P["xp"]), p(w1), p(P["offsets"]), p(P["p_rows"]), E, R, H, F, p(P["gu"]),
                    p(P["h"]), None, s)),
                ("fc2", lambda: L.moe_grouped_gemm_bf16(
                    0, p(P["h"]), p(w2), 0, p(P["offsets"]), E, R, 0, H, F, p(P["y2"]), None,
                    None, s)),
                ("unpermute", lambda: L.moe_unpermute(p(P["y2"]), p(P["dest"]), None, T, H, k,
                                                      p(out), s)),
                ("permute_dout", lambda: L.moe_permute(
                    p(dout), p(P["dest"]), p(P["offsets"]), p(P["counts"]), None, T, H, E, k,
                    p(P["dy2"]), None, s)),
                ("fc2_dgrad_swiglu_bwd", lambda: L.moe_fc2_dgrad_swiglu_bwd_bf16(
                    p(P["dy2"]), p(w2), p(P["offsets"]), p(P["p_rows"]), p(P["gu"]), E, R, H, F,
                    p(P["dy1"]), p(P["dp"]), None, s)),
                ("fc2_wgrad", lambda: L.moe_grouped_gemm_bf16(
                    1, p(P["h"]), p(P["dy2"]), 0, p(P["offsets"]), E, R, F, H, 0, p(dw2), None,
                    None, s)),
                ("fc1_dgrad", lambda: L.moe_grouped_gemm_bf16(
                    0, p(P["dy1"]), p(w1), 1, p(P["offsets"]), E, R, 0, H, 2 * F, p(P["dxp"]),
                    None, None, s)),
                ("fc1_wgrad", lambda: L.moe_grouped_gemm_bf16(
                    1, p(P["xp"]), p(P["dy1"]), 0, p(P["offsets"]), E, R, H, 2 * F, 0, p(dw1),
                    None, None, s)),
            ]
        else:
            def q(name):
                return [p(P[f"{name}_{t}"]) for t in ("q_row", "s_row", "q_col", "s_col")]

            def to_fp4(name, cols):  # row-wise MXFP8 -> the MXFP4 copy carried to the backward
                return lambda: L.mxfp4_from_mxfp8(p(P[f"{name}_q_row"]), p(P[f"{name}_s_row"]),
                                                  R, cols, p(P[f"{name}4_q_row"]),
                                                  p(P[f"{name}4_s_row"]), s)

            def col_from_fp4(name, cols):  # the wgrad operand rebuilt from the MXFP4 copy
                return lambda: L.mxfp8_colwise_from_mxfp4_rowwise(
                    p(P[f"{name}4_q_row"]), p(P[f"{name}4_s_row"]), R, cols,
                    p(P[f"{name}_q_col"]), p(P[f"{name}_s_col"]), s)
            xdirs = B.QUANT_ROWWISE if self.act4 else RC
            ops += [
                ("p_rows", lambda: L.moe_permute(
                    p(x), p(P["dest"]), p(P["offsets"]), p(P["counts"]), p(P["w"]), T, H, E, k,
                    None, p(P["p_rows"]), s)),
                ("quant_x", lambda: L.mxfp8_quantize(p(x), R, H, H, p(P["src"]), k, xdirs,
                                                     *q("x"), s)),
                ("quant_w1", lambda: L.mxfp8_quantize(p(w1), E * H, 2 * F, 2 * F, None, 1, RC,
                                                      *q("w1"), s)),
                ("quant_w2", lambda: L.mxfp8_quantize(p(w2), E * F, H, H, None, 1, RC,
                                                      *q("w2"), s)),
                ("fc1_swiglu", lambda: L.moe_fc1_swiglu_mxfp8(
                    p(P["x_q_row"]), p(P["x_s_row"]), R, H, p(P["w1_q_col"]), p(P["w1_s_col"]),
                    p(P["offsets"]), p(P["p_rows"]), E, F, p(P["gu"]),
                    *(q("h")[:2] + ([None, None] if self.act4 else q("h")[2:])), s)),
            ]
            if self.act4:
                ops += [("x_to_fp4", to_fp4("x", H)), ("h_to_fp4", to_fp4("h", F))]
            ops += [
                ("fc2", lambda: L.moe_grouped_gemm_mxfp8(
                    0, p(P["h_q_row"]), p(P["h_s_row"]), R, F, p(P["w2_q_col"]),
                    p(P["w2_s_col"]), H, E * F, 0, F, p(P["offsets"]), E, 0, H, F, p(P["y2"]),
                    s)),
                ("unpermute", lambda: L.moe_unpermute(p(P["y2"]), p(P["dest"]), None, T, H, k,
                                                      p(out), s)),
                ("quant_dout", lambda: L.mxfp8_quantize(p(dout), R, H, H, p(P["src"]), k, RC,
                                                        *q("dy2"), s)),
                ("fc2_dgrad_swiglu_bwd", lambda: L.moe_fc2_dgrad_swiglu_bwd_mxfp8(
                    p(P["dy2_q_row"]), p(P["dy2_s_row"]), R, H, p(P["w2_q_row"]),
                    p(P["w2_s_row"]), p(P["offsets"]), p(P["p_rows"]), p(P["gu"]), E, F,
                    *q("dy1"), p(P["dp"]), s)),
            ]
            if self.act4:
                ops += [("h_col_from_fp4", col_from_fp4("h", F)),
                        ("x_col_from_fp4", col_from_fp4("x", H))]
            ops += [
                ("fc2_wgrad", lambda: L.moe_grouped_gemm_mxfp8(
                    1, p(P["h_q_col"]), p(P["h_s_col"]), F, R, p(P["dy2_q_col"]),
                    p(P["dy2_s_col"]), H, R, 0, 0, p(P["offsets"]), E, F, H, 0, p(dw2), s)),
                ("fc1_dgrad", lambda: L.moe_grouped_gemm_mxfp8(
                    0, p(P["dy1_q_row"]), p(P["dy1_s_row"]), R, 2 * F, p(P["w1_q_row"]),
                    p(P["w1_s_row"]), E * H, 2 * F, H, 0, p(P["offsets"]), E, 0, H, 2 * F,
                    p(P["dxp"]), s)),
                ("fc1_wgrad", lambda: L.moe_grouped_gemm_mxfp8(
                    1, p(P["x_q_col"]), p(P["x_s_col"]), H, R, p(P["dy1_q_col"]),
                    p(P["dy1_s_col"]), 2 * F, R, 0, 0, p(P["offsets"]), E, H, 2 * F, 0, p(dw1),
                    s)),
            ]
        ops += [
            ("unpermute_dx", lambda: L.moe_unpermute(p(P["dxp"]), p(P["dest"]), None, T, H, k,
                                                     p(dx), s)),
            ("route_bwd", lambda: L.moe_route_backward(
                p(P["dp"]), npart, npart, p(P["dest"]), p(P["w"]), p(P["idx"]), T, E, k,
                p(dlogits), s)),
        ]
        if self.router:
            # aux-loss gradient (coefficient 0.01), dX += dlogits W_r^T, dW_r
            ops.append(("router_bwd", lambda: L.moe_router_backward(
                p(x), p(self.w_r), p(self.logits_r), p(self.aux), p(dlogits), 0.01, T, H, E,
                p(dlogits), p(dx), p(dx), p(self.dw_r), p(self.router_ws),
                self.router_ws.numel(), s)))
        return ops

    def bind(self, *tensors):
        self._tensors = tensors
        self.ops = self._ops(*tensors)

    def capture(self):
        """The same calls recorded once as a CUDA graph on a capture stream
        (after one run there, so every kernel's one-time launch set-up is done);
        replay() then issues the whole step with no host work per launch."""
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(cs):
            ops = self._ops(*self._tensors)  # bound to the capture stream
            for name, fn in ops:
                self.B._check(fn(), name)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=cs):
            for name, fn in ops:
                self.B._check(fn(), name)
        torch.cuda.current_stream().wait_stream(cs)
        return graph

    def run(self, ev=None):
        chk = self.B._check
        for i, (name, fn) in enumerate(self.ops):
            if ev is not None:
                ev[i].record()
            chk(fn(), name)
        if ev is not None:
            ev[len(self.ops)].record()


def kernel_work(wl):
    """Algorithmic work per launch: flops for GEMMs, bytes for the rest."""
    T, H, F, E, k = wl.T, wl.H, wl.F, wl.E, wl.k
    R = T * k
    q2 = 2 * (1 + 1 / 32)  # bytes written per element by a two-direction MXFP8 quantisation
    q8, q4 = 1 + 1 / 32, 0.5 + 1 / 32  # bytes per element of one MXFP8 / MXFP4 copy
    act4 = wl.precision == "mxfp8_act4"
    return {
        "fc1_swiglu": ("flops", 4.0 * R * H * F),
        "fc2": ("flops", 2.0 * R * H * F),
        "fc2_dgrad_swiglu_bwd": ("flops", 2.0 * R * H * F),
        "fc2_wgrad": ("flops", 2.0 * R * H * F),
        "fc1_dgrad": ("flops", 4.0 * R * H * F),
        "fc1_wgrad": ("flops", 4.0 * R * H * F),
        "route": ("bytes", T * E * 4.0 + R * 8.0),
        "plan": ("bytes", R * 4.0 * 3),
        "permute_x": ("bytes", T * H * 2.0 + R * H * 2.0),
        "p_rows": ("bytes", R * 4.0 * 3),
        "quant_x": ("bytes", T * H * 2.0 + R * H * (q8 if act4 else q2)),
        # MXFP4 activation mode: FP8 -> FP4 copies and the rebuilt column-wise FP8
        "x_to_fp4": ("bytes", R * H * (q8 + q4)),
        "h_to_fp4": ("bytes", R * F * (q8 + q4)),
        "x_col_from_fp4": ("bytes", R * H * (q4 + q8)),
        "h_col_from_fp4": ("bytes", R * F * (q4 + q8)),
        "quant_w1": ("bytes", E * H * 2.0 * F * (2.0 + q2)),
        "quant_w2": ("bytes", E * F * H * (2.0 + q2)),
        "quant_dout": ("bytes", T * H * 2.0 + R * H * q2),
        "unpermute": ("bytes", R * H * 2.0 + T * H * 2.0),
        "permute_dout": ("bytes", T * H * 2.0 + R * H * 2.0),
        "unpermute_dx": ("bytes", R * H * 2.0 + T * H * 2.0),
        "route_bwd": ("bytes", R * 4.0 * 2 + T * E * 4.0),
        # router projection: read x and W_r, write logits (then route + aux read them)
        "router_fwd": ("bytes", T * H * 2.0 + H * E * 2.0 + T * E * 4.0 * 3 + R * 8.0),
        # aux gradient (logits, dlogits), dX read + write, x for dW_r, dW_r
        "router_bwd": ("bytes", T * E * 4.0 * 3 + T * H * 2.0 * 3 + H * E * 2.0 * 2),
    }


# ------------------------------------------------------------ CPU oracle

_ORACLE_INPUTS = {}


def _oracle_inputs(wl):
    """The workload's inputs on the host, routed once (before any clock starts)."""
    if wl.name not in _ORACLE_INPUTS:
        from oracle import moe_oracle as O
        inp = I.make_all(wl)
        lg = inp["logits"].numpy()
        idx, w = O.route(lg, wl.k)
        _ORACLE_INPUTS[wl.name] = {
            "x": inp["x"].float().numpy(), "w1": inp["w1"].float().numpy(),
            "w2": inp["w2"].float().numpy(), "dout": inp["dout"].float().numpy(), "w": w,
            "rows": [O.expert_rows(idx, e) for e in range(wl.E)]}
    return _ORACLE_INPUTS[wl.name]


def oracle_sample_time(wl, rows, e, ffn=None):
    """Time the oracle, as it stands, on a bounded sample of the workload:
    expert e's forward + backward on its first `rows` routed rows, full H,
    and the first `ffn` FFN columns (all F when None; the expert MLP is a sum
    over FFN columns, so a column slice is the same computation on a
    narrower expert; a slice of whole 32-blocks keeps every MXFP8 block
    whole). The sample's share of the expert's weight quantisation is
    included in MXFP8 modes. Inputs are drawn and routed before the clock
    starts. Returns (seconds, token equivalents = rows / k * ffn / F, rows,
    ffn)."""
    from oracle import moe_oracle as O
    d = _oracle_inputs(wl)
    tok, slot = d["rows"][e]
    tok, slot = tok[:rows], slot[:rows]
    mx = {"bf16": False, "mxfp8": True, "mxfp8_act4": "act4"}[wl.precision]
    fs = wl.F if ffn is None else min(ffn, wl.F)
    cols = np.concatenate([np.arange(fs), wl.F + np.arange(fs)])
    w1e, w2e = d["w1"][e][:, cols], d["w2"][e][:fs]
    xe, p, dy = d["x"][tok], d["w"][tok, slot], d["dout"][tok]
    t0 = time.perf_counter()
    y2, saved = O.expert_forward(xe, p, w1e, w2e, mx)
    O.expert_backward(xe, p, w1e, w2e, dy, saved, mx)
    return time.perf_counter() - t0, len(tok) / wl.k * fs / wl.F, len(tok), fs


def nonempty_experts(wl):
    return [e for e in range(wl.E) if len(_oracle_inputs(wl)["rows"][e][0]) > 0]


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _set_blas_threads():
    n = str(host_cores())
    for v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ.setdefault(v, n)


# ---------------------------------------------------------------- arms

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, wl, world, rank):
    """The oracle, as it stands, on the host cores: each step is one expert's
    forward + backward on its first args.ref_rows routed rows of the workload
    (the experts taken in turn)."""
    if rank != 0:
        return
    _set_blas_threads()
    experts = nonempty_experts(wl)
    for i in range(min(args.warmup, 1)):
        oracle_sample_time(wl, args.ref_rows, experts[i % len(experts)], args.ref_ffn)
    times, toks = [], 0.0
    for i in range(args.steps):
        dt, n, _, fs = oracle_sample_time(wl, args.ref_rows, experts[i % len(experts)],
                                          args.ref_ffn)
        times.append(dt)
        toks += n
    tot = sum(times)
    value = toks / tot
    cores = host_cores()
    sample = (f"one expert per step (experts in turn): its first {args.ref_rows} routed rows of "
              f"the {wl.name} workload, full H={wl.H}, the first {fs} of F={wl.F} FFN columns, "
              f"fwd+bwd in fp64, counted as rows/k * {fs}/{wl.F} tokens")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
    }
    print(json.dumps(line), flush=True)


def source_hash(files):
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "mixture_experts_expert_sort_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel, wl):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, or
    None when there is none for this workload or the kernel's source files
    changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f).get(f"{wl.name}/{kernel}")
    except Exception:
        return None
    if not t or t.get("source_sha256_16") != source_hash(t["sources"]):
        return None
    return t["bytes_per_launch"]


def config_of(wl):
    return {"workload": f"{wl.name}: MoE expert layer T={wl.T} H={wl.H} F={wl.F} E={wl.E} "
                        f"top-{wl.k} {wl.precision.upper()} fwd+bwd",
            "T": wl.T, "H": wl.H, "F": wl.F, "E": wl.E, "k": wl.k, "precision": wl.precision,
            "global_batch_tokens": wl.T,
            "l2": "inputs larger than L2 (weights alone 2*E*H*F*3 bytes per step)"
                  if 6 * wl.E * wl.H * wl.F > 126e6 else
                  "inputs smaller than L2 (latency-bound small case)"}


def is_mx(wl):
    return wl.precision in ("mxfp8", "mxfp8_act4")


def tensor_peak(peaks, mx):
    """Tensor roofline denominator for the GEMMs' own dtype: the measured BF16
    burst rate (the timed region is well under a second), times the nominal
    dense MXFP8/BF16 ratio 4.5/2.25 = 2 for the MXFP8 path."""
    kind = f"bf16 burst ({peaks['source']})"
    if mx:
        return 2.0 * peaks["bf16_tflops"], f"mxfp8 = 2 x {kind}"
    return peaks["bf16_tflops"], kind


def timed_steps(args, wl, world, local, dev):
    """W untimed steps, then K timed steps of workload wl with CUDA events
    between the calls on the launching stream. Returns the timing record and
    the step with its bound tensors."""
    from mixture_experts_expert_sort_b300 import binding as B
    rank = int(os.environ.get("RANK", "0"))
    # Seeded synthetic inputs generated on the device (rank-distinct seeds).
    wlr = wl if rank == 0 else I.Workload(wl.name, wl.T, wl.H, wl.F, wl.E, wl.k, wl.precision,
                                          wl.seed + 100 * rank, wl.zipf_s, wl.zero_experts,
                                          wl.outlier_frac)
    inp = I.make_all(wlr, device=dev)
    T, H, F, E = wl.T, wl.H, wl.F, wl.E
    bf = torch.bfloat16
    t = {"logits": inp["logits"], "x": inp["x"], "w1": inp["w1"], "w2": inp["w2"],
         "dout": inp["dout"], "out": torch.empty((T, H), dtype=bf, device=dev),
         "dx": torch.empty((T, H), dtype=bf, device=dev),
         "dw1": torch.empty((E, H, 2 * F), dtype=bf, device=dev),
         "dw2": torch.empty((E, F, H), dtype=bf, device=dev),
         "dlogits": torch.empty((T, E), dtype=torch.float32, device=dev)}
    step = Step(wl, dev, router=args.router, gather=args.gather_operands)
    step.bind(t["logits"], t["x"], t["w1"], t["w2"], t["dout"], t["out"], t["dx"], t["dw1"],
              t["dw2"], t["dlogits"])
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if B.device_error() != 0:
        raise RuntimeError(f"device error flag set during warm-up ({wl.name})")

    nk = len(step.NAMES)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
           for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    clocks.mark_begin()
    t0.record()
    for i in range(args.steps):
        step.run(ev=evs[i])
    t1.record()
    torch.cuda.synchronize()
    clocks.mark_end()
    barrier(world)
    clk = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), world)
    # mean over the timed steps, the statistic of ms_per_step
    per_kernel = {n: sum(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(args.steps))
                  / args.steps for j, n in enumerate(step.NAMES)}
    if B.device_error() != 0:
        raise RuntimeError(f"device error flag set during the timed region ({wl.name})")
    # Where a step is short enough for the host's per-call work to show, the
    # step is also timed as CUDA-graph replays (longer steps hide it behind
    # the GPU work, and replays timed after the per-call loop would only run
    # further into the power cap).
    graph = graph_steps(step, args, world) if ms / args.steps < GRAPH_MS else None
    return {"ms_step": ms / args.steps, "per_kernel": per_kernel, "clocks": clk,
            "launches": step.launches_per_step * args.steps, "graph": graph}, step, t


GRAPH_MS = 2.0  # steps shorter than this are also timed from a CUDA graph


def graph_steps(step, args, world):
    """The same K steps replayed from a CUDA graph of the step (no host work
    per launch), bracketed like the per-call loop by a barrier and a
    synchronisation on both sides. Returns {"ms_per_step": ...}, or
    {"error": ...} if the capture is refused, so the line still reports the
    per-call timing."""
    from mixture_experts_expert_sort_b300 import binding as B
    try:
        g = step.capture()
        g.replay()  # one untimed replay
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            g.replay()
        b.record()
        torch.cuda.synchronize()
        barrier(world)
        ms = max_over_ranks(a.elapsed_time(b), world) / args.steps
        if B.device_error() != 0:
            raise RuntimeError("device error flag set during the graph replays")
        del g
        return {"ms_per_step": ms}
    except Exception as e:  # the per-call measurement stands on its own
        return {"error": f"{type(e).__name__}: {e}"[:300]}


def summarise(wl, rec, world, peaks):
    """Throughput, GEMM rate and the dominant kernel's roofline of one workload."""
    ms_step, per_kernel, clk = rec["ms_step"], rec["per_kernel"], rec["clocks"]
    work = kernel_work(wl)
    mx = is_mx(wl)
    gemm_names = [n for n in per_kernel if work[n][0] == "flops"]
    gemm_ms = sum(per_kernel[n] for n in gemm_names)
    gemm_tflops = wl.gemm_flops_fwd_bwd() / (gemm_ms / 1000.0) / 1e12
    peak_t, peak_t_kind = tensor_peak(peaks, mx)
    dom = max(per_kernel, key=lambda n: per_kernel[n])
    kind, amount = work[dom]
    sec = per_kernel[dom] / 1000.0
    if kind == "flops":
        ach = amount / sec / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peak_t, "unit": "TFLOP/s",
                "frac": ach / peak_t, "traffic": None, "kernel": dom, "peak_kind": peak_t_kind,
                "work_per_launch": amount, "ms_per_launch": per_kernel[dom]}
    else:
        ach = amount / sec / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"], "traffic": None, "kernel": dom,
                "peak_kind": f"hbm copy ({peaks['source']})", "work_per_launch": amount,
                "ms_per_launch": per_kernel[dom]}
    if clk and clk.get("sm_mhz") and kind == "flops":
        # the same fraction against the burst peak scaled to the sampled SM clock
        roof["frac_at_sampled_clock"] = roof["frac"] * peaks["sm_max_mhz"] / clk["sm_mhz"]
    roof["traffic"] = measured_traffic(dom, wl)
    kern = {}
    for n in per_kernel:
        k_, amt = work[n]
        s = per_kernel[n] / 1000.0
        kern[n] = {"ms": round(per_kernel[n], 4),
                   ("tflops" if k_ == "flops" else "gbs"):
                       round(amt / s / (1e12 if k_ == "flops" else 1e9), 1)}
    graph = rec.get("graph")
    if graph and "ms_per_step" in graph:
        graph = {"value": world * wl.T / (graph["ms_per_step"] / 1000.0), "unit": "tokens/s",
                 "ms_per_step": graph["ms_per_step"],
                 "how": "the same step captured once as a CUDA graph, K replays timed"}
    return {
        "value": world * wl.T / (ms_step / 1000.0), "unit": "tokens/s", "ms_per_step": ms_step,
        **({"graph": graph} if graph else {}),
        "gemm_tflops": gemm_tflops, "gemm_frac_of_peak": gemm_tflops / peak_t,
        "gemm_frac_of_spec": gemm_tflops / (4500.0 if mx else 2250.0),
        "roofline": roof, "clocks": clk, "gpu_launches": rec["launches"], "kernels": kern,
        "kernels_sum_ms": round(sum(per_kernel.values()), 4),
    }


def e2e_measure(args, step, t, world):
    """End to end through the public layer API with host buffers. Every step
    copies its inputs from pinned host memory and reads its results back, as a
    training loop does; the copies of one step overlap the compute of its
    neighbours (two slots of device buffers, an input-copy stream and a
    result-copy stream ordered by events), dOut is copied in while the
    forward runs and out is read back while the backward runs, and the
    compute stays on the launching stream. dW stays resident, as in training."""
    layer = step.layer
    x, logits, dout, out, dx, dlogits = t["x"], t["logits"], t["dout"], t["out"], t["dx"], \
        t["dlogits"]
    w1, w2, dw1, dw2 = t["w1"], t["w2"], t["dw1"], t["dw2"]
    T = x.shape[0]
    h_x = x.cpu().pin_memory()
    h_lg = logits.cpu().pin_memory()
    h_do = dout.cpu().pin_memory()
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h_dx = torch.empty(dx.shape, dtype=dx.dtype).pin_memory()
    h_dl = torch.empty(dlogits.shape, dtype=dlogits.dtype).pin_memory()
    slots = [{"x": torch.empty_like(x), "lg": torch.empty_like(logits),
              "do": torch.empty_like(dout), "out": torch.empty_like(out),
              "dx": torch.empty_like(dx), "dl": torch.empty_like(dlogits)} for _ in range(2)]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = [{k: torch.cuda.Event() for k in ("in_fwd", "in", "fwd", "comp", "out")}
          for _ in range(2)]
    e2e_steps = max(2, min(args.steps, 10))

    def e2e_run(n):
        for i in range(n):
            sl, e = slots[i % 2], ev[i % 2]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(e["comp"])  # step i-2 is done with these inputs
                # the forward's inputs first; dOut's copy then overlaps the forward
                sl["lg"].copy_(h_lg, non_blocking=True)
                sl["x"].copy_(h_x, non_blocking=True)
                e["in_fwd"].record(s_in)
                sl["do"].copy_(h_do, non_blocking=True)
                e["in"].record(s_in)
            comp.wait_event(e["in_fwd"])
            if i >= 2:
                comp.wait_event(e["out"])  # step i-2's results have been read back
            layer.forward(sl["lg"], sl["x"], w1, w2, out=sl["out"])
            e["fwd"].record(comp)
            with torch.cuda.stream(s_out):
                # out is read back while the backward runs
                s_out.wait_event(e["fwd"])
                h_out.copy_(sl["out"], non_blocking=True)
            comp.wait_event(e["in"])
            layer.backward(sl["do"], w1, w2, dx=sl["dx"], dw1=dw1, dw2=dw2, dlogits=sl["dl"])
            e["comp"].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(e["comp"])
                h_dx.copy_(sl["dx"], non_blocking=True)
                h_dl.copy_(sl["dl"], non_blocking=True)
                e["out"].record(s_out)
        for e in ev:
            comp.wait_event(e["out"])

    e2e_run(2)
    torch.cuda.synchronize()
    barrier(world)
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    a0.record()
    e2e_run(e2e_steps)
    a1.record()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a0.elapsed_time(a1) / e2e_steps, world)
    h2d = h_x.numel() * 2 + h_lg.numel() * 4 + h_do.numel() * 2
    d2h = h_out.numel() * 2 + h_dx.numel() * 2 + h_dl.numel() * 4
    return {"value": world * T / (e2e_ms / 1000.0), "unit": "tokens/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "api": "moe_layer_forward + moe_layer_backward, host pinned inputs/outputs"}


def dtype_of(wl):
    return ("e4m3 (mxfp8); x, h carried as e2m1 (mxfp4)" if wl.precision == "mxfp8_act4"
            else "e4m3 (mxfp8)" if is_mx(wl) else "bf16")


def run_ours(args, wl, world, rank, local):
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from mixture_experts_expert_sort_b300 import binding as B
    B.lib()
    peaks = load_peaks()
    rec, step, t = timed_steps(args, wl, world, local, dev)
    e2e = e2e_measure(args, step, t, world)
    head = summarise(wl, rec, world, peaks)
    del step, t
    torch.cuda.empty_cache()
    # The other workloads, each measured the same way (its own warm-up and K
    # timed steps), as sub-results of the same line.
    others = {}
    names = [] if args.configs == "none" else (
        [n for n in I.WORKLOADS if n != wl.name] if args.configs == "all"
        else [n for n in args.configs.split(",") if n and n != wl.name])
    for n in names:
        w = I.WORKLOADS[n]
        r, st, tt = timed_steps(args, w, world, local, dev)
        s = summarise(w, r, world, peaks)
        s["config"] = config_of(w)
        s["dtype"] = dtype_of(w)
        others[n] = s
        del st, tt
        torch.cuda.empty_cache()
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": head["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype_of(wl), "data": "synthetic (seeded, generated on the device)",
        "config": dict(config_of(wl), router=("router projection x W_r, top-k, aux "
                                              "load-balancing loss and their backward included"
                                              if args.router else "logits given (no router)"),
                       **({"operands": "x and dOut read through row gathers (tile::gather4), "
                                       "no permuted copies; e2e still uses the layer's copies"}
                          if args.gather_operands and not is_mx(wl) else {})),
        "gemm_tflops": head["gemm_tflops"],
        "gemm_frac_of_peak": head["gemm_frac_of_peak"],
        "gemm_frac_of_spec": head["gemm_frac_of_spec"],
        "roofline": head["roofline"],
        "e2e": e2e,
        "gpu_launches": head["gpu_launches"],
        "clocks": head["clocks"],
        "kernels": head["kernels"],
        "kernels_sum_ms": head["kernels_sum_ms"],
        **({"graph": head["graph"]} if "graph" in head else {}),
        "peaks": {k: peaks[k] for k in ("bf16_tflops", "hbm_gbs", "sm_max_mhz", "source")},
        "workloads": others,
    }
    if world == 1 and not args.no_cpu_baseline:
        _set_blas_threads()
        e = nonempty_experts(wl)[0]
        dt, n, rows, _ = oracle_sample_time(wl, args.cpu_rows, e)
        line["cpu_baseline"] = {
            "value": n / dt, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"expert {e}'s forward+backward on its first {rows} routed rows of the "
                      f"workload (full H and F), fp64, counted as rows/k = {n:g} tokens; "
                      f"{dt:.1f} s"}
    print(json.dumps(line), flush=True)


def library_peaks(seconds=3.0):
    """Dense GEMM throughput of the vendor libraries on this GPU, for the tensor rooflines:
    cuBLAS BF16 (torch.mm) and cuBLASLt MXFP8 (torch._scaled_mm with 1x32 E8M0 block scales),
    each as a burst (median of 20 timed calls) and sustained (back-to-back calls for `seconds`,
    last half). Shapes: 8192^3 and the Mixtral FC1 GEMM (M = 32768 routed rows, K = 4096,
    N = 28672)."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    g = torch.Generator(device=dev).manual_seed(1)
    res = {"gpu": torch.cuda.get_device_name(dev), "shapes": {}}
    for name, (M, K, N) in {"square_8192": (8192, 8192, 8192),
                            "mixtral_fc1": (32768, 4096, 28672)}.items():
        flop = 2.0 * M * N * K
        a16 = torch.randn((M, K), device=dev, generator=g).to(torch.bfloat16)
        b16 = torch.randn((N, K), device=dev, generator=g).to(torch.bfloat16)
        a8, b8 = a16.to(torch.float8_e4m3fn), b16.to(torch.float8_e4m3fn)
        sa = torch.full((128 * -(-M // 128) * 4 * -(-K // 128),), 127, dtype=torch.uint8,
                        device=dev).view(torch.float8_e8m0fnu)
        sb = torch.full((128 * -(-N // 128) * 4 * -(-K // 128),), 127, dtype=torch.uint8,
                        device=dev).view(torch.float8_e8m0fnu)
        fns = {"bf16": lambda: torch.mm(a16, b16.t()),
               "mxfp8": lambda: torch._scaled_mm(a8, b8.t(), sa, sb, out_dtype=torch.bfloat16)}
        out = {}
        for kind, fn in fns.items():
            time.sleep(5.0)  # let clocks recover from the previous loop before the burst
            clk = ClockSampler(0)
            clk.start()
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(20):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
                fn()
                e1.record()
                e1.synchronize()
                ts.append(e0.elapsed_time(e1))
            burst = flop / (sorted(ts)[len(ts) // 2] / 1e3) / 1e12
            burst_clk = clk.stop()
            clk = ClockSampler(0)
            clk.start()
            per = sorted(ts)[len(ts) // 2] / 1e3
            n = max(4, int(seconds / per))
            marks = []
            for i in range(n):
                if i in (n // 2, n - 1):
                    ev = torch.cuda.Event(enable_timing=True)
                    ev.record()
                    marks.append(ev)
                fn()
            torch.cuda.synchronize()
            sus_ms = marks[0].elapsed_time(marks[1]) / (n - 1 - n // 2)
            out[kind] = {"burst_tflops": round(burst, 1), "burst_clocks": burst_clk,
                         "sustained_tflops": round(flop / (sus_ms / 1e3) / 1e12, 1),
                         "sustained_clocks": clk.stop()}
        res["shapes"][name] = out
        del a16, b16, a8, b8, sa, sb
        torch.cuda.empty_cache()
    print(json.dumps(res))


def main():
    if "--library-peaks" in sys.argv:
        library_peaks()
        return
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="mixtral_mx", choices=sorted(I.WORKLOADS))
    ap.add_argument("--configs", default="all",
                    help="other workloads measured as sub-results of the line: all, none, or "
                         "a comma-separated list")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-rows", type=int, default=2048,
                    help="routed rows of one expert in the CPU-baseline sample")
    ap.add_argument("--ref-rows", type=int, default=512,
                    help="routed rows of one expert per step of the reference arm")
    ap.add_argument("--ref-ffn", type=int, default=1024,
                    help="FFN columns of that expert per step of the reference arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=0, help="override T (profiling cases)")
    ap.add_argument("--experts", type=int, default=0, help="override E (profiling cases)")
    ap.add_argument("--gather-operands", action="store_true",
                    help="BF16: time the step with x and dOut read through row gathers "
                         "instead of the layer's permuted copies")
    ap.add_argument("--router", action="store_true",
                    help="compute the logits with the router projection (x W_r) and add the "
                         "aux load-balancing loss and the router backward to the step")
    args = ap.parse_args()
    wl = I.WORKLOADS[args.workload]
    if args.tokens or args.experts:
        args.configs = "none"
        # A reduced case of the same layer shape (H, F, k kept), for profiling.
        wl = I.Workload(wl.name + "_reduced", args.tokens or wl.T, wl.H, wl.F,
                        args.experts or wl.E, wl.k, wl.precision, wl.seed, wl.zipf_s,
                        wl.zero_experts, wl.outlier_frac)
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, wl, world, rank)
    else:
        run_ours(args, wl, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
