"""Thin ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here takes torch CUDA tensors, checks that each one is dense
device memory of the element type the C declaration documents (the entry
points take plain pointers, so a host tensor would reach a kernel as an
invalid address, a strided view would be read as if it were dense and a wrong
dtype would be reinterpreted), passes raw device pointers and the current CUDA
stream to the C entry point of the same name, and raises on a non-zero status. All
computation happens in the library's kernels; if the library is missing this
module raises instead of computing anything elsewhere.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")
_lib = None

MOE_OK, MOE_ERR_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_DEVICE = range(5)
MOE_DEVERR_BAD_INDEX, MOE_DEVERR_TIMEOUT, MOE_DEVERR_CAPACITY = 1, 2, 4
QUANT_ROWWISE, QUANT_COLWISE = 1, 2
GEMM_FPROP, GEMM_WGRAD = 0, 1

_p, _i, _ll, _sz, _u = C.c_void_p, C.c_int, C.c_longlong, C.c_size_t, C.c_uint


class RowGather(C.Structure):
    """moe_row_gather: permuted row r reads source row src[r] // src_div
    (src[r] < 0: a zero row); src_rows is the source tensor's row count."""
    _fields_ = [("src", _p), ("src_div", _i), ("src_rows", _ll)]


_g = C.POINTER(RowGather)

# name -> (restype, argtypes); mirrors include/moe.h
SIGNATURES = {
    "moe_status_string": (C.c_char_p, [_i]),
    "moe_device_error": (_i, [_p, C.POINTER(_u)]),
    "moe_selftest_wait_timeout": (_i, [_p]),
    "moe_selftest_tile_order": (_i, [_i, _i, _i, _i, _ll, _i, _i, _p, _p]),
    "moe_route": (_i, [_p, _i, _i, _i, _p, _p, _p]),
    "moe_route_backward": (_i, [_p, _ll, _i, _p, _p, _p, _i, _i, _i, _p, _p]),
    "moe_rows_padded_max": (_ll, [_i, _i, _i, _i]),
    "moe_permute_plan_workspace_size": (_sz, [_i, _i, _i]),
    "moe_permute_plan": (_i, [_p, _i, _i, _i, _i, _p, _p, _p, _p, _ll, _p, _sz, _p]),
    "moe_permute_plan_static": (_i, [_p, _i, _i, _i, _i, _p, _p, _p, _p, _ll, _p]),
    "moe_permute": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _p, _p, _p]),
    "moe_unpermute": (_i, [_p, _p, _p, _i, _i, _i, _p, _p]),
    "mxfp8_quantize": (_i, [_p, _ll, _i, _ll, _p, _i, _i, _p, _p, _p, _p, _p]),
    "mxfp8_scales_to_canonical": (_i, [_p, _ll, _i, _p, _p]),
    "mxfp4_from_mxfp8": (_i, [_p, _p, _ll, _i, _p, _p, _p]),
    "mxfp8_from_mxfp4": (_i, [_p, _p, _ll, _i, _p, _p, _p]),
    "mxfp4_rowwise_to_colwise": (_i, [_p, _p, _ll, _i, _p, _p, _p]),
    "mxfp8_colwise_from_mxfp4_rowwise": (_i, [_p, _p, _ll, _i, _p, _p, _p]),
    "moe_grouped_gemm_bf16": (_i, [_i, _p, _p, _i, _p, _i, _ll, _i, _i, _i, _p, _g, _g, _p]),
    "moe_fc1_swiglu_bf16": (_i, [_p, _p, _p, _p, _i, _ll, _i, _i, _p, _p, _g, _p]),
    "moe_swiglu_bwd_parts": (_i, [_i]),
    "moe_fc2_dgrad_swiglu_bwd_bf16": (_i, [_p, _p, _p, _p, _p, _i, _ll, _i, _i, _p, _p, _g,
                                           _p]),
    "moe_grouped_gemm_mxfp8": (_i, [_i, _p, _p, _ll, _ll, _p, _p, _ll, _ll, _ll, _ll, _p, _i,
                                    _i, _i, _i, _p, _p]),
    "moe_fc1_swiglu_mxfp8": (_i, [_p, _p, _ll, _i, _p, _p, _p, _p, _i, _i, _p, _p, _p, _p, _p,
                                  _p]),
    "moe_fc2_dgrad_swiglu_bwd_mxfp8": (_i, [_p, _p, _ll, _i, _p, _p, _p, _p, _p, _i, _i, _p, _p,
                                            _p, _p, _p, _p]),
    "moe_router_workspace_size": (_sz, [_i, _i, _i]),
    "moe_router_forward": (_i, [_p, _p, _i, _i, _i, _i, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_router_backward": (_i, [_p, _p, _p, _p, _p, C.c_float, _i, _i, _i, _p, _p, _p, _p, _p,
                                 _sz, _p]),
    "moe_layer_workspace_size": (_sz, [_p]),
    "moe_layer_workspace_part": (_i, [_p, _i, C.POINTER(_sz), C.POINTER(_sz)]),
    "moe_layer_forward": (_i, [_p, _p, _p, _p, _p, _p, _p, _sz, _p]),
    "moe_layer_backward": (_i, [_p, _p, _p, _p, _p, _p, _p, _p, _p, _sz, _p]),
}


class MoeError(RuntimeError):
    pass


def lib():
    """Load libmoe.so (built in-tree by mixture_experts_expert_sort_b300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MoeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m mixture_experts_expert_sort_b300.build`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != MOE_OK:
        msg = lib().moe_status_string(status).decode()
        raise MoeError(f"{what} failed: {msg}")


BF16, F32, I32, U8 = torch.bfloat16, torch.float32, torch.int32, torch.uint8


def ptr(t, dtype=None):
    """Device address of a dense (contiguous) CUDA tensor of element type
    `dtype` (the type the C declaration documents); None stays None."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise MoeError(f"tensor of shape {tuple(t.shape)} with strides {t.stride()} is not "
                       "contiguous: the library reads every operand as a dense array")
    return _device_address(t, dtype)


def ptr_rows(t, dtype=None):
    """Device address of a CUDA matrix whose rows may be strided (the caller
    passes t.stride(0) as the leading dimension) but are dense within."""
    if t.dim() != 2 or (t.shape[1] > 1 and t.stride(1) != 1) or t.stride(0) < t.shape[1]:
        raise MoeError(f"tensor of shape {tuple(t.shape)} with strides {t.stride()} is not a "
                       "matrix of dense rows")
    return _device_address(t, dtype)


def _is_device(t):
    return t.device.type == "cuda"


def _device_address(t, dtype):
    if dtype is not None and t.dtype != dtype:
        raise MoeError(f"tensor of shape {tuple(t.shape)} has element type {t.dtype}; the "
                       f"library reads this argument as {dtype}")
    if not _is_device(t):
        raise MoeError(f"a {t.device.type} tensor was passed where the library needs device "
                       "memory")
    return t.data_ptr()


def stream_handle(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def device_error(stream=None) -> int:
    flags = C.c_uint(0)
    st = lib().moe_device_error(stream_handle(stream), C.byref(flags))
    if st not in (MOE_OK, MOE_ERR_DEVICE):
        _check(st, "moe_device_error")
    return flags.value


def selftest_wait_timeout(stream=None):
    """Run the library's bounded-wait self-test (about 2 s on the device); the
    timeout bit then shows in device_error()."""
    _check(lib().moe_selftest_wait_timeout(stream_handle(stream)), "moe_selftest_wait_timeout")


def selftest_tile_order(mtiles, ntiles, tile_m, tile_n, band_rows, prefer_m, min_band_tiles):
    """Host-side: the (m-tile, n-tile) the grouped GEMMs process as each local
    tile index of one expert's grid, as two int32 numpy arrays."""
    import numpy as np
    mt = np.empty(mtiles * ntiles, dtype=np.int32)
    nt = np.empty(mtiles * ntiles, dtype=np.int32)
    _check(lib().moe_selftest_tile_order(mtiles, ntiles, tile_m, tile_n, band_rows,
                                         int(bool(prefer_m)), min_band_tiles,
                                         mt.ctypes.data, nt.ctypes.data),
           "moe_selftest_tile_order")
    return mt, nt


# ----------------------------------------------------------------- routing

def moe_route(logits, k, idx=None, w=None, stream=None):
    T, E = logits.shape
    dev = logits.device
    idx = idx if idx is not None else torch.empty((T, k), dtype=torch.int32, device=dev)
    w = w if w is not None else torch.empty((T, k), dtype=torch.float32, device=dev)
    _check(lib().moe_route(ptr(logits, F32), T, E, k, ptr(idx, I32), ptr(w, F32),
                           stream_handle(stream)), "moe_route")
    return idx, w


def moe_route_backward(dp, w, idx, E, dest=None, dlogits=None, stream=None):
    """dp: [rows, n_part] fp32 partials (rows indexed by dest if given, else flat t*k+j)."""
    T, k = idx.shape
    dp2 = dp if dp.dim() == 2 else dp.reshape(-1, 1)
    dlogits = dlogits if dlogits is not None else torch.empty((T, E), dtype=torch.float32,
                                                              device=idx.device)
    _check(lib().moe_route_backward(ptr_rows(dp2, F32), dp2.stride(0), dp2.shape[1], ptr(dest, I32),
                                    ptr(w, F32), ptr(idx, I32), T, E, k, ptr(dlogits, F32),
                                    stream_handle(stream)), "moe_route_backward")
    return dlogits


# ----------------------------------------------------------------- router

def moe_router_workspace_size(T, H, E):
    return int(lib().moe_router_workspace_size(T, H, E))


def moe_router_forward(x, w_r, k, workspace=None, stream=None, out=None):
    """logits = x @ w_r, top-k routing, aux load-balancing statistics.
    Returns dict with logits [T,E], idx [T,k], w [T,k], aux [1+2E] (loss, f, P)."""
    T, H = x.shape
    E = w_r.shape[1]
    dev = x.device
    if out is None:
        out = {"logits": torch.empty((T, E), dtype=torch.float32, device=dev),
               "idx": torch.empty((T, k), dtype=torch.int32, device=dev),
               "w": torch.empty((T, k), dtype=torch.float32, device=dev),
               "aux": torch.empty(1 + 2 * E, dtype=torch.float32, device=dev)}
    if workspace is None:
        workspace = torch.empty(moe_router_workspace_size(T, H, E), dtype=torch.uint8, device=dev)
    _check(lib().moe_router_forward(ptr(x, BF16), ptr(w_r, BF16), T, H, E, k,
                                    ptr(out["logits"], F32), ptr(out["idx"], I32),
                                    ptr(out["w"], F32), ptr(out["aux"], F32), ptr(workspace, U8),
                                    workspace.numel(), stream_handle(stream)), "moe_router_forward")
    return out


def moe_router_backward(x, w_r, logits, aux, dlogits_route, aux_coeff, dx_in=None, dx_out=None,
                        dlogits=None, dw_r=None, workspace=None, stream=None):
    T, H = x.shape
    E = w_r.shape[1]
    dev = x.device
    dlogits = dlogits if dlogits is not None else torch.empty((T, E), dtype=torch.float32,
                                                              device=dev)
    dx_out = dx_out if dx_out is not None else torch.empty((T, H), dtype=torch.bfloat16,
                                                           device=dev)
    dw_r = dw_r if dw_r is not None else torch.empty((H, E), dtype=torch.bfloat16, device=dev)
    if workspace is None:
        workspace = torch.empty(moe_router_workspace_size(T, H, E), dtype=torch.uint8, device=dev)
    _check(lib().moe_router_backward(ptr(x, BF16), ptr(w_r, BF16), ptr(logits, F32), ptr(aux, F32),
                                     ptr(dlogits_route, F32), float(aux_coeff), T, H, E,
                                     ptr(dlogits, F32), ptr(dx_in, BF16), ptr(dx_out, BF16),
                                     ptr(dw_r, BF16), ptr(workspace, U8), workspace.numel(),
                                     stream_handle(stream)), "moe_router_backward")
    return dlogits, dx_out, dw_r


# ------------------------------------------------------------ expert sort

def moe_rows_padded_max(T, E, k, align):
    return int(lib().moe_rows_padded_max(T, E, k, align))


def moe_permute_plan_workspace_size(T, E, k):
    return int(lib().moe_permute_plan_workspace_size(T, E, k))


def moe_permute_plan(idx, E, align, src_rows=None, workspace=None, stream=None, out=None):
    T, k = idx.shape
    dev = idx.device
    rmax = moe_rows_padded_max(T, E, k, align)
    src_rows = rmax if src_rows is None else src_rows
    if out is None:
        out = {
            "counts": torch.empty(E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "dest": torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
            "src": torch.empty(max(src_rows, 1), dtype=torch.int32, device=dev),
        }
    wsb = moe_permute_plan_workspace_size(T, E, k)
    if workspace is None:
        workspace = torch.empty(wsb, dtype=torch.uint8, device=dev)
    _check(lib().moe_permute_plan(ptr(idx, I32), T, E, k, align, ptr(out["counts"], I32),
                                  ptr(out["offsets"], I32), ptr(out["dest"], I32),
                                  ptr(out["src"], I32), src_rows, ptr(workspace, U8),
                                  workspace.numel(), stream_handle(stream)), "moe_permute_plan")
    return out


PLAN_STATIC_SCRATCH_INTS = 262144


def moe_permute_plan_static(idx, E, align, src_rows=None, stream=None, out=None):
    """moe_permute_plan without a workspace, for callers that cannot allocate
    device memory: the library's fixed 1 MiB scratch array is used instead.
    Raises MoeError when ceil(T*k/1024)*E exceeds that array."""
    T, k = idx.shape
    dev = idx.device
    src_rows = moe_rows_padded_max(T, E, k, align) if src_rows is None else src_rows
    if out is None:
        out = {
            "counts": torch.empty(E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
            "dest": torch.empty(max(T * k, 1), dtype=torch.int32, device=dev),
            "src": torch.empty(max(src_rows, 1), dtype=torch.int32, device=dev),
        }
    st = lib().moe_permute_plan_static(ptr(idx, I32), T, E, k, align, ptr(out["counts"], I32),
                                       ptr(out["offsets"], I32), ptr(out["dest"], I32),
                                       ptr(out["src"], I32), src_rows, stream_handle(stream))
    if st == MOE_ERR_UNSUPPORTED:
        raise MoeError(f"moe_permute_plan_static: ceil(T*k/1024)*E = "
                       f"{-(-T * k // 1024) * E} exceeds the static scratch of "
                       f"{PLAN_STATIC_SCRATCH_INTS} int32")
    _check(st, "moe_permute_plan_static")
    return out


def moe_permute(x, dest, offsets, counts, k, rows, w=None, xp=None, p_rows=None, stream=None):
    T, H = x.shape
    E = counts.numel()
    dev = x.device
    xp = xp if xp is not None else torch.empty((rows, H), dtype=x.dtype, device=dev)
    if w is not None and p_rows is None:
        p_rows = torch.empty(rows, dtype=torch.float32, device=dev)
    _check(lib().moe_permute(ptr(x, BF16), ptr(dest, I32), ptr(offsets, I32), ptr(counts, I32),
                             ptr(w, F32), T, H, E, k, ptr(xp, BF16), ptr(p_rows, F32),
                             stream_handle(stream)), "moe_permute")
    return xp, p_rows


def moe_unpermute(y, dest, T, k, w=None, out=None, stream=None):
    H = y.shape[1]
    out = out if out is not None else torch.empty((T, H), dtype=y.dtype, device=y.device)
    _check(lib().moe_unpermute(ptr(y, BF16), ptr(dest, I32), ptr(w, F32), T, H, k, ptr(out, BF16),
                               stream_handle(stream)), "moe_unpermute")
    return out


# ------------------------------------------------------------------ MXFP8

def mx_scale_bytes(mn, kdim):
    return (mn // 128) * (kdim // 128) * 512


def mxfp8_quantize(x, dirs=QUANT_ROWWISE | QUANT_COLWISE, rows=None, src=None, src_div=1,
                   stream=None, out=None):
    """x: [n, cols] bf16 (row stride x.stride(0)). Returns dict of q_row/s_row/q_col/s_col."""
    cols = x.shape[1]
    rows = x.shape[0] if rows is None else rows
    dev = x.device
    if out is None:
        out = {}
        if dirs & QUANT_ROWWISE:
            out["q_row"] = torch.empty((rows, cols), dtype=torch.uint8, device=dev)
            out["s_row"] = torch.empty(mx_scale_bytes(rows, cols), dtype=torch.uint8, device=dev)
        if dirs & QUANT_COLWISE:
            out["q_col"] = torch.empty((cols, rows), dtype=torch.uint8, device=dev)
            out["s_col"] = torch.empty(mx_scale_bytes(cols, rows), dtype=torch.uint8, device=dev)
    _check(lib().mxfp8_quantize(ptr_rows(x, BF16), rows, cols, x.stride(0), ptr(src, I32), src_div,
                                dirs, ptr(out.get("q_row"), U8), ptr(out.get("s_row"), U8),
                                ptr(out.get("q_col"), U8), ptr(out.get("s_col"), U8),
                                stream_handle(stream)), "mxfp8_quantize")
    return out


def mxfp8_scales_to_canonical(s_tiled, mn, kdim, stream=None, out=None):
    """Tiled scales of an [mn, kdim] MXFP8 operand -> row-major [mn, kdim/32] bytes."""
    out = out if out is not None else torch.empty((mn, kdim // 32), dtype=torch.uint8,
                                                  device=s_tiled.device)
    _check(lib().mxfp8_scales_to_canonical(ptr(s_tiled, U8), mn, kdim, ptr(out, U8),
                                           stream_handle(stream)), "mxfp8_scales_to_canonical")
    return out


# ------------------------------------------------------------------ MXFP4

def _u8(shape, dev):
    return torch.empty(shape, dtype=torch.uint8, device=dev)


def mxfp4_from_mxfp8(q8, s8, stream=None, out=None):
    """Row-wise MXFP8 (q8 [rows, cols] bytes, s8 tiled) -> row-wise MXFP4:
    {"q4": [rows, cols/2] bytes, "s4": tiled scales}."""
    rows, cols = q8.shape
    out = out or {"q4": _u8((rows, cols // 2), q8.device),
                  "s4": _u8(mx_scale_bytes(rows, cols), q8.device)}
    _check(lib().mxfp4_from_mxfp8(ptr(q8, U8), ptr(s8, U8), rows, cols, ptr(out["q4"], U8),
                                  ptr(out["s4"], U8), stream_handle(stream)), "mxfp4_from_mxfp8")
    return out


def mxfp8_from_mxfp4(q4, s4, stream=None, out=None):
    """Row-wise MXFP4 (q4 [rows, cols/2]) -> row-wise MXFP8 {"q8", "s8"}."""
    rows, half = q4.shape
    cols = 2 * half
    out = out or {"q8": _u8((rows, cols), q4.device),
                  "s8": _u8(mx_scale_bytes(rows, cols), q4.device)}
    _check(lib().mxfp8_from_mxfp4(ptr(q4, U8), ptr(s4, U8), rows, cols, ptr(out["q8"], U8),
                                  ptr(out["s8"], U8), stream_handle(stream)), "mxfp8_from_mxfp4")
    return out


def mxfp4_rowwise_to_colwise(q4, s4, stream=None, out=None):
    """Row-wise MXFP4 [rows, cols] -> column-wise MXFP4 stored transposed:
    {"q4c": [cols, rows/2] bytes, "s4c": tiled with MN = cols, K = rows}."""
    rows, half = q4.shape
    cols = 2 * half
    out = out or {"q4c": _u8((cols, rows // 2), q4.device),
                  "s4c": _u8(mx_scale_bytes(cols, rows), q4.device)}
    _check(lib().mxfp4_rowwise_to_colwise(ptr(q4, U8), ptr(s4, U8), rows, cols, ptr(out["q4c"], U8),
                                          ptr(out["s4c"], U8), stream_handle(stream)),
           "mxfp4_rowwise_to_colwise")
    return out


def mxfp8_colwise_from_mxfp4_rowwise(q4, s4, stream=None, out=None):
    """Row-wise MXFP4 [rows, cols] -> column-wise MXFP8 stored transposed:
    {"q8c": [cols, rows] bytes, "s8c": tiled with MN = cols, K = rows}."""
    rows, half = q4.shape
    cols = 2 * half
    out = out or {"q8c": _u8((cols, rows), q4.device),
                  "s8c": _u8(mx_scale_bytes(cols, rows), q4.device)}
    _check(lib().mxfp8_colwise_from_mxfp4_rowwise(ptr(q4, U8), ptr(s4, U8), rows, cols,
                                                  ptr(out["q8c"], U8), ptr(out["s8c"], U8),
                                                  stream_handle(stream)),
           "mxfp8_colwise_from_mxfp4_rowwise")
    return out


# ----------------------------------------------------------- grouped GEMM

def _row_gather(gather, source):
    """(src, src_div) -> (RowGather over `source`'s rows, or None; the number
    of permuted rows, src.numel(), or None)."""
    if gather is None:
        return None, None
    src, src_div = gather
    g = RowGather(ptr(src, I32), int(src_div), int(source.shape[0]))
    return C.byref(g), src.numel()


def moe_grouped_gemm_bf16(mode, A, B, offsets, b_layout=0, M=0, N=0, K=0, C=None, stream=None,
                          gather_a=None, gather_b=None):
    """FPROP: C[rows, N] = A[rows] @ B_e per group (B [E,K,N] or [E,N,K]).
    WGRAD: C[E, M, N] = A_e^T @ B_e over each group's rows (A [rows, M], B [rows, N]).
    gather_a / gather_b = (src, src_div): that operand is its un-permuted source
    and permuted row r is its row src[r] // src_div (rows = src.numel())."""
    E = offsets.numel() - 1
    ga, ra = _row_gather(gather_a, A)
    gb, rb = _row_gather(gather_b, B)
    rows = ra if ra is not None else rb if rb is not None else A.shape[0]
    if mode == GEMM_FPROP:
        K = A.shape[1]
        N = B.shape[2] if b_layout == 0 else B.shape[1]
        C = C if C is not None else torch.empty((rows, N), dtype=torch.bfloat16, device=A.device)
    else:
        M, N = A.shape[1], B.shape[1]
        C = C if C is not None else torch.empty((E, M, N), dtype=torch.bfloat16, device=A.device)
    _check(lib().moe_grouped_gemm_bf16(mode, ptr(A, BF16), ptr(B, BF16), b_layout,
                                       ptr(offsets, I32), E, rows, M, N, K, ptr(C, BF16), ga, gb,
                                       stream_handle(stream)), "moe_grouped_gemm_bf16")
    return C


def moe_fc1_swiglu_bf16(xp, w1, offsets, p_rows, gu=None, h=None, stream=None, gather_x=None):
    """gather_x = (src, src_div): xp is the un-permuted x and permuted row r is
    its row src[r] // src_div (rows = src.numel())."""
    gx, rows = _row_gather(gather_x, xp)
    H = xp.shape[1]
    rows = rows if rows is not None else xp.shape[0]
    E, _, F2 = w1.shape
    F = F2 // 2
    gu = gu if gu is not None else torch.empty((rows, F2), dtype=torch.bfloat16, device=xp.device)
    h = h if h is not None else torch.empty((rows, F), dtype=torch.bfloat16, device=xp.device)
    _check(lib().moe_fc1_swiglu_bf16(ptr(xp, BF16), ptr(w1, BF16), ptr(offsets, I32),
                                     ptr(p_rows, F32), E, rows, H, F, ptr(gu, BF16), ptr(h, BF16),
                                     gx, stream_handle(stream)), "moe_fc1_swiglu_bf16")
    return gu, h


def moe_swiglu_bwd_parts(F):
    return int(lib().moe_swiglu_bwd_parts(F))


def moe_fc2_dgrad_swiglu_bwd_bf16(dy2, w2, offsets, p_rows, gu, dy1=None, dp_part=None,
                                  stream=None, gather_dy=None):
    """gather_dy = (src, src_div): dy2 is the un-permuted dOut and permuted row
    r is its row src[r] // src_div (rows = src.numel())."""
    gdy, rows = _row_gather(gather_dy, dy2)
    H = dy2.shape[1]
    rows = rows if rows is not None else dy2.shape[0]
    E, F, _ = w2.shape
    dev = dy2.device
    dy1 = dy1 if dy1 is not None else torch.empty((rows, 2 * F), dtype=torch.bfloat16, device=dev)
    if dp_part is None:
        dp_part = torch.empty((rows, moe_swiglu_bwd_parts(F)), dtype=torch.float32, device=dev)
    _check(lib().moe_fc2_dgrad_swiglu_bwd_bf16(ptr(dy2, BF16), ptr(w2, BF16), ptr(offsets, I32),
                                               ptr(p_rows, F32), ptr(gu, BF16), E, rows, H, F,
                                               ptr(dy1, BF16), ptr(dp_part, F32), gdy,
                                               stream_handle(stream)),
           "moe_fc2_dgrad_swiglu_bwd_bf16")
    return dy1, dp_part


# ----------------------------------------------------- MXFP8 grouped GEMM

def moe_grouped_gemm_mxfp8(mode, a, sa, b, sb, offsets, b_row_stride=0, b_k_stride=0, M=0, N=0,
                           K=0, C=None, stream=None):
    """a, b: uint8 E4M3 data [rows, cols] (K-major); sa, sb: tiled scales."""
    E = offsets.numel() - 1
    a_rows, a_cols = a.shape
    b_rows, b_cols = b.shape
    if C is None:
        shape = (a_rows, N) if mode == GEMM_FPROP else (E, M, N)
        C = torch.empty(shape, dtype=torch.bfloat16, device=a.device)
    _check(lib().moe_grouped_gemm_mxfp8(mode, ptr(a, U8), ptr(sa, U8), a_rows, a_cols, ptr(b, U8),
                                        ptr(sb, U8), b_rows, b_cols, b_row_stride, b_k_stride,
                                        ptr(offsets, I32), E, M, N, K, ptr(C, BF16),
                                        stream_handle(stream)), "moe_grouped_gemm_mxfp8")
    return C


def moe_fc1_swiglu_mxfp8(xq, sx, w1t, sw1t, offsets, p_rows, F, stream=None, out=None):
    rows, H = xq.shape
    E = offsets.numel() - 1
    dev = xq.device
    if out is None:
        out = {"gu": torch.empty((rows, 2 * F), dtype=torch.bfloat16, device=dev),
               "q_row": torch.empty((rows, F), dtype=torch.uint8, device=dev),
               "s_row": torch.empty(mx_scale_bytes(rows, F), dtype=torch.uint8, device=dev),
               "q_col": torch.empty((F, rows), dtype=torch.uint8, device=dev),
               "s_col": torch.empty(mx_scale_bytes(F, rows), dtype=torch.uint8, device=dev)}
    _check(lib().moe_fc1_swiglu_mxfp8(ptr(xq, U8), ptr(sx, U8), rows, H, ptr(w1t, U8),
                                      ptr(sw1t, U8), ptr(offsets, I32), ptr(p_rows, F32), E, F,
                                      ptr(out["gu"], BF16), ptr(out["q_row"], U8),
                                      ptr(out["s_row"], U8), ptr(out["q_col"], U8),
                                      ptr(out["s_col"], U8), stream_handle(stream)),
           "moe_fc1_swiglu_mxfp8")
    return out


def moe_fc2_dgrad_swiglu_bwd_mxfp8(dy2q, sdy2, w2q, sw2, offsets, p_rows, gu, F, stream=None,
                                   out=None):
    rows, H = dy2q.shape
    E = offsets.numel() - 1
    dev = dy2q.device
    if out is None:
        out = {"q_row": torch.empty((rows, 2 * F), dtype=torch.uint8, device=dev),
               "s_row": torch.empty(mx_scale_bytes(rows, 2 * F), dtype=torch.uint8, device=dev),
               "q_col": torch.empty((2 * F, rows), dtype=torch.uint8, device=dev),
               "s_col": torch.empty(mx_scale_bytes(2 * F, rows), dtype=torch.uint8, device=dev),
               "dp": torch.empty((rows, 2 * -(-F // 256)), dtype=torch.float32, device=dev)}
    _check(lib().moe_fc2_dgrad_swiglu_bwd_mxfp8(ptr(dy2q, U8), ptr(sdy2, U8), rows, H, ptr(w2q, U8),
                                                ptr(sw2, U8), ptr(offsets, I32), ptr(p_rows, F32),
                                                ptr(gu, BF16), E, F, ptr(out["q_row"], U8),
                                                ptr(out["s_row"], U8), ptr(out["q_col"], U8),
                                                ptr(out["s_col"], U8), ptr(out["dp"], F32),
                                                stream_handle(stream)),
           "moe_fc2_dgrad_swiglu_bwd_mxfp8")
    return out


# ------------------------------------------------------------- whole layer

PRECISION = {"bf16": 0, "mxfp8": 1, "mxfp8_act4": 2}
PARTS = {"idx": (0, torch.int32), "w": (1, torch.float32), "counts": (2, torch.int32),
         "offsets": (3, torch.int32), "dest": (4, torch.int32), "src": (5, torch.int32),
         "p_rows": (7, torch.float32), "xp": (8, torch.bfloat16), "gu": (9, torch.bfloat16),
         "h": (10, torch.bfloat16), "y2": (11, torch.bfloat16), "dy2": (12, torch.bfloat16),
         "dy1": (13, torch.bfloat16), "dxp": (14, torch.bfloat16), "dp": (15, torch.float32)}
# MXFP8 parts: four per operand (row-wise data, its scales, column-wise data, its scales)
for _i, _name in enumerate(("x", "w1", "w2", "h", "dy2", "dy1")):
    for _j, _suffix in enumerate(("q_row", "s_row", "q_col", "s_col")):
        PARTS[f"{_name}_{_suffix}"] = (16 + 4 * _i + _j, torch.uint8)
# MXFP8_ACT4 parts: the row-wise MXFP4 copies of x (gathered) and H
PARTS.update({"x4_q_row": (40, torch.uint8), "x4_s_row": (41, torch.uint8),
              "h4_q_row": (42, torch.uint8), "h4_s_row": (43, torch.uint8)})


class LayerConfig(C.Structure):
    _fields_ = [("T", C.c_int), ("H", C.c_int), ("F", C.c_int), ("E", C.c_int), ("k", C.c_int),
                ("align", C.c_int), ("precision", C.c_int)]


def layer_config(T, H, F, E, k, precision="bf16", align=128):
    return LayerConfig(T, H, F, E, k, align, PRECISION[precision])


def moe_layer_workspace_size(cfg):
    return int(lib().moe_layer_workspace_size(C.byref(cfg)))


def moe_layer_workspace_part(cfg, part):
    off, nb = _sz(0), _sz(0)
    _check(lib().moe_layer_workspace_part(C.byref(cfg), part, C.byref(off), C.byref(nb)),
           "moe_layer_workspace_part")
    return off.value, nb.value


def moe_layer_forward(cfg, logits, x, w1, w2, out, workspace, stream=None):
    _check(lib().moe_layer_forward(C.byref(cfg), ptr(logits, F32), ptr(x, BF16), ptr(w1, BF16),
                                   ptr(w2, BF16), ptr(out, BF16), ptr(workspace, U8),
                                   workspace.numel(), stream_handle(stream)), "moe_layer_forward")
    return out


def moe_layer_backward(cfg, dout, w1, w2, dx, dw1, dw2, dlogits, workspace, stream=None):
    _check(lib().moe_layer_backward(C.byref(cfg), ptr(dout, BF16), ptr(w1, BF16), ptr(w2, BF16),
                                    ptr(dx, BF16), ptr(dw1, BF16), ptr(dw2, BF16),
                                    ptr(dlogits, F32), ptr(workspace, U8), workspace.numel(),
                                    stream_handle(stream)), "moe_layer_backward")
    return dx, dw1, dw2, dlogits
