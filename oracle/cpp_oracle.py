"""ctypes front of the C++ oracle (oracle/moe_oracle.cpp).

TEST INFRASTRUCTURE ONLY. Only the test suite and ``__graft_entry__`` (its
build step and the smoke check) may import it; the product path never calls
it. The library is built with the host compiler into oracle/libmoe_oracle.so
(``build()``, also run by ``__graft_entry__.build()``), without fused
multiply-adds or fast-math, so every operation rounds as written.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "libmoe_oracle.so")
MODES = {"bf16": 0, "mxfp8": 1, "mxfp8_act4": 2}

_lib = None


def build(force: bool = False) -> str:
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        cxx = os.environ.get("CXX", "g++")
        tmp = LIB + ".tmp"
        subprocess.run([cxx, "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
                        "-shared", "-fPIC", "-o", tmp, SRC], check=True)
        os.replace(tmp, LIB)
    return LIB


def lib():
    global _lib
    if _lib is None:
        build()
        _lib = C.CDLL(LIB)
    return _lib


def _d(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _p(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None else None


def _ok(status, what):
    if status != 0:
        raise ValueError(f"{what}: bad arguments")


def route(logits, k):
    """idx int32 [T, k] (best first, ties to the lower index), w float64 [T, k]."""
    lg = _d(logits)
    T, E = lg.shape
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k))
    _ok(lib().moe_oracle_route(_p(lg), T, E, k, _p(idx), _p(w)), "route")
    return idx, w


def route_backward(dp, w, idx, E):
    dp, w = _d(dp), _d(w)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = dp.shape
    dl = np.empty((T, E))
    _ok(lib().moe_oracle_route_backward(_p(dp), _p(w), _p(idx), T, E, k, _p(dl)),
        "route_backward")
    return dl


def permute_plan(idx, E, align):
    """counts [E], offsets [E+1], dest [T*k], src [offsets[E]] (int32)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, k = idx.shape
    cap = T * k + E * (align - 1)
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E + 1, dtype=np.int32)
    dest = np.empty(T * k, dtype=np.int32)
    src = np.empty(max(cap, 1), dtype=np.int32)
    _ok(lib().moe_oracle_permute_plan(_p(idx), T, k, E, align, _p(counts), _p(offsets),
                                      _p(dest), _p(src), C.c_longlong(cap)), "permute_plan")
    return counts, offsets, dest, src[:offsets[-1]].copy()


def permute(x, dest, k, rows):
    x = _d(x)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    T, H = x.shape
    xp = np.empty((rows, H))
    _ok(lib().moe_oracle_permute(_p(x), _p(dest), T, H, k, C.c_longlong(rows), _p(xp)),
        "permute")
    return xp


def unpermute(y, dest, k, w=None):
    y = _d(y)
    dest = np.ascontiguousarray(dest, dtype=np.int32)
    T, H = dest.size // k, y.shape[1]
    out = np.empty((T, H))
    wv = _d(w) if w is not None else None
    _ok(lib().moe_oracle_unpermute(_p(y), _p(dest), _p(wv), T, H, k, _p(out)), "unpermute")
    return out


def mx_quantize(a, axis=1, fmt=8):
    """Codes [rows, cols] and E8M0 scales of a 2-D matrix, 32-blocks along
    axis (fmt 8: E4M3 bytes; fmt 4: E2M1 codes 0..15, one per byte)."""
    a = _d(a)
    rows, cols = a.shape
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty((rows, cols // 32) if axis == 1 else (rows // 32, cols), dtype=np.uint8)
    _ok(lib().moe_oracle_mx_quantize(_p(a), C.c_longlong(rows), C.c_longlong(cols), axis, fmt,
                                     _p(codes), _p(scales)), "mx_quantize")
    return codes, scales


def layer(x, logits, W1, W2, dout, k, mode="bf16", save_bf16=True):
    """Forward and backward of the layer for L = sum(out * dout).

    Returns a dict with out, dX, dW1, dW2, dlogits, dp, idx and w."""
    x, lg, W1, W2, dout = _d(x), _d(logits), _d(W1), _d(W2), _d(dout)
    T, H = x.shape
    E, _, F2 = W1.shape
    F = F2 // 2
    r = {"out": np.empty((T, H)), "dX": np.empty((T, H)), "dW1": np.empty((E, H, F2)),
         "dW2": np.empty((E, F, H)), "dlogits": np.empty((T, E)), "dp": np.empty((T, k)),
         "idx": np.empty((T, k), dtype=np.int32), "w": np.empty((T, k))}
    _ok(lib().moe_oracle_layer(_p(x), _p(lg), _p(W1), _p(W2), _p(dout), T, H, F, E, k,
                               MODES[mode], int(bool(save_bf16)), _p(r["out"]), _p(r["dX"]),
                               _p(r["dW1"]), _p(r["dW2"]), _p(r["dlogits"]), _p(r["dp"]),
                               _p(r["idx"]), _p(r["w"])), "layer")
    return r


def router_forward(x, Wr, k):
    """logits [T, E], idx, w [T, k], and (L, f [E], P [E]) of the aux loss."""
    x, Wr = _d(x), _d(Wr)
    T, H = x.shape
    E = Wr.shape[1]
    lg = np.empty((T, E))
    idx = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k))
    aux = np.empty(1 + 2 * E)
    _ok(lib().moe_oracle_router_forward(_p(x), _p(Wr), T, H, E, k, _p(lg), _p(idx), _p(w),
                                        _p(aux)), "router_forward")
    return {"logits": lg, "idx": idx, "w": w, "aux": float(aux[0]), "f": aux[1:1 + E].copy(),
            "P": aux[1 + E:].copy()}


def router_backward(x, Wr, logits, f, dlogits_route, coeff):
    """dlogits = dlogits_route + coeff * dAux/dlogits, dx = dlogits Wr^T, dWr = x^T dlogits."""
    x, Wr, lg, f, dr = _d(x), _d(Wr), _d(logits), _d(f), _d(dlogits_route)
    T, H = x.shape
    E = Wr.shape[1]
    dl, dx, dw = np.empty((T, E)), np.empty((T, H)), np.empty((H, E))
    _ok(lib().moe_oracle_router_backward(_p(x), _p(Wr), _p(lg), _p(f), _p(dr),
                                         C.c_double(coeff), T, H, E, _p(dl), _p(dx), _p(dw)),
        "router_backward")
    return dl, dx, dw
