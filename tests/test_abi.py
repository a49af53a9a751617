"""The C-ABI library builds for sm_103a, loads without a GPU and exports every
function declared in include/moe.h (no compute calls are made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]*?\b((?:moe|mxfp8|mxfp4)_\w+)\s*\(", txt)))


@pytest.fixture(scope="module")
def libmoe():
    from mixture_experts_expert_sort_b300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_functions():
    names = _declared()
    assert "moe_route" in names and "mxfp8_quantize" in names and len(names) >= 10


def test_every_declared_symbol_is_exported(libmoe):
    for name in _declared():
        assert hasattr(libmoe, name), name


def test_binding_signatures_cover_header():
    from mixture_experts_expert_sort_b300 import binding
    assert set(binding.SIGNATURES) == set(_declared())


def test_host_only_queries(libmoe):
    from mixture_experts_expert_sort_b300 import binding
    L = binding.lib()
    assert L.moe_rows_padded_max(256, 4, 2, 128) == 256 * 2 + 4 * 127
    assert L.moe_rows_padded_max(-1, 4, 2, 128) == -1
    ws = L.moe_permute_plan_workspace_size(16384, 64, 6)
    assert ws % 256 == 0 and ws >= (16384 * 6 // 1024) * 64 * 4
    assert L.moe_status_string(0) == b"MOE_OK"
    assert b"invalid" in L.moe_status_string(1)


def test_mxfp4_argument_checks(libmoe):
    """The MXFP4 conversions reject bad shapes and null buffers on the host,
    before any CUDA call (MOE_ERR_ARG = 1)."""
    for name in ("mxfp4_from_mxfp8", "mxfp8_from_mxfp4", "mxfp4_rowwise_to_colwise",
                 "mxfp8_colwise_from_mxfp4_rowwise"):
        fn = getattr(libmoe, name)
        fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int,
                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
        assert fn(None, None, 128, 128, None, None, None) == 1, name
        assert fn(16, 16, 100, 128, 16, 16, None) == 1, name   # rows % 128
        assert fn(16, 16, 128, 96, 16, 16, None) == 1, name    # cols % 128
        assert fn(8, 16, 128, 128, 16, 16, None) == 1, name    # misaligned data


def test_layer_workspace_layouts(libmoe):
    """Host-only layout queries: the MXFP4-activation mode adds the row-wise
    MXFP4 copies of x and H (half a byte per element plus scales) to the
    MXFP8 layout and keeps their column-wise FP8 copies in the bytes of the
    row-wise ones, which the backward no longer needs; parts of another
    precision have size 0; unsupported configs report size 0 (H % 256 for
    the MXFP8 modes, align % 128)."""
    from mixture_experts_expert_sort_b300 import binding as B
    T, H, F, E, k = 16384, 4096, 14336, 8, 2
    c8 = B.layer_config(T, H, F, E, k, "mxfp8")
    c4 = B.layer_config(T, H, F, E, k, "mxfp8_act4")
    cb = B.layer_config(T, H, F, E, k, "bf16")
    R = B.moe_rows_padded_max(T, E, k, 128)
    R = -(-R // 128) * 128
    scale = lambda mn, kd: (mn // 128) * (kd // 128) * 512  # noqa: E731
    extra = [R * H // 2, scale(R, H), R * F // 2, scale(R, F)]
    up = lambda b: -(-b // 256) * 256  # noqa: E731
    fp8 = [R * H, scale(H, R), R * F, scale(F, R)]  # the column-wise FP8 copies of x and H
    assert B.moe_layer_workspace_size(c4) == (B.moe_layer_workspace_size(c8) + sum(map(up, extra))
                                              - sum(map(up, fp8)))
    # at this (Mixtral, T = 16384) shape the mode saves about 311 MB of workspace
    saved = B.moe_layer_workspace_size(c8) - B.moe_layer_workspace_size(c4)
    assert 305e6 < saved < 315e6, saved
    for row, col in (("x_q_row", "x_q_col"), ("x_s_row", "x_s_col"), ("h_q_row", "h_q_col"),
                     ("h_s_row", "h_s_col")):
        r_off, r_bytes = B.moe_layer_workspace_part(c4, B.PARTS[row][0])
        c_off, c_bytes = B.moe_layer_workspace_part(c4, B.PARTS[col][0])
        assert (r_off, r_bytes) == (c_off, c_bytes), (row, col)
        assert B.moe_layer_workspace_part(c8, B.PARTS[row][0])[0] != \
            B.moe_layer_workspace_part(c8, B.PARTS[col][0])[0]
    for name, want in zip(("x4_q_row", "x4_s_row", "h4_q_row", "h4_s_row"), extra):
        part = B.PARTS[name][0]
        assert B.moe_layer_workspace_part(c4, part)[1] == want, name
        assert B.moe_layer_workspace_part(c8, part)[1] == 0, name
    assert B.moe_layer_workspace_part(cb, B.PARTS["x_q_row"][0])[1] == 0
    assert B.moe_layer_workspace_part(c8, B.PARTS["xp"][0])[1] == 0
    Rb = B.moe_rows_padded_max(T, E, k, 128)  # BF16 rows are not rounded up to 128
    for name, cols in (("xp", H), ("dy2", H), ("gu", 2 * F)):
        assert B.moe_layer_workspace_part(cb, B.PARTS[name][0])[1] == Rb * cols * 2, name
    assert B.moe_layer_workspace_size(B.layer_config(64, 384, 256, 4, 2, "mxfp8_act4")) == 0
    assert B.moe_layer_workspace_size(B.layer_config(64, 384, 256, 4, 2, "bf16")) > 0
    assert B.moe_layer_workspace_size(B.layer_config(64, 256, 256, 4, 2, "bf16", align=64)) == 0


def test_binding_refuses_host_and_strided_tensors():
    """The library takes plain device pointers: the binding refuses a host
    tensor (it would reach a kernel as an invalid address) and a strided view
    (it would be read as if dense) before any call is made."""
    import torch
    from mixture_experts_expert_sort_b300 import binding as B
    with pytest.raises(B.MoeError, match="cpu tensor"):
        B.ptr(torch.zeros(4, 8))
    with pytest.raises(B.MoeError, match="not contiguous"):
        B.ptr(torch.zeros(8, 4).t())
    with pytest.raises(B.MoeError, match="not contiguous"):
        B.ptr(torch.zeros(4, 8)[:, :4])
    assert B.ptr(None) is None
    # leading-dimension operands: strided rows pass the layout check (and then
    # fail only for being host memory); strided columns do not
    with pytest.raises(B.MoeError, match="cpu tensor"):
        B.ptr_rows(torch.zeros(4, 16)[:, :8])
    with pytest.raises(B.MoeError, match="dense rows"):
        B.ptr_rows(torch.zeros(8, 4).t())
    with pytest.raises(B.MoeError, match="dense rows"):
        B.ptr_rows(torch.zeros(4, 8, 2))


def test_layer_checks_operand_shapes_and_dtypes(libmoe):
    """MoELayer checks every operand against the shapes and dtypes of the
    layer entry points before the library sees a pointer."""
    import torch
    from mixture_experts_expert_sort_b300 import binding as B
    from mixture_experts_expert_sort_b300.layer import MoELayer
    T, H, F, E, k = 64, 128, 256, 4, 2
    L = MoELayer(T, H, F, E, k, device="cpu")
    bf = torch.bfloat16
    lg, x = torch.zeros(T, E), torch.zeros(T, H, dtype=bf)
    w1, w2 = torch.zeros(E, H, 2 * F, dtype=bf), torch.zeros(E, F, H, dtype=bf)
    with pytest.raises(B.MoeError, match="logits: expected"):
        L.forward(lg.to(bf), x, w1, w2)
    with pytest.raises(B.MoeError, match="w1: expected"):
        L.forward(lg, x, w1.transpose(1, 2).contiguous(), w2)
    with pytest.raises(B.MoeError, match="x: expected"):
        L.forward(lg, x[: T - 1], w1, w2)
    with pytest.raises(B.MoeError, match="dw2: expected"):
        L.backward(x, w1, w2, dw2=torch.zeros(E, F, H))
    # right shapes and dtypes, but host memory: refused at the pointer
    with pytest.raises(B.MoeError, match="cpu tensor"):
        L.forward(lg, x, w1, w2)
    # the graph capture checks every buffer the same way before any CUDA call
    dx, dl = torch.zeros(T, H, dtype=bf), torch.zeros(T, E)
    dw1, dw2 = torch.zeros(E, H, 2 * F, dtype=bf), torch.zeros(E, F, H, dtype=bf)
    with pytest.raises(B.MoeError, match="dlogits: expected"):
        L.capture(lg, x, w1, w2, x, x, dx, dw1, dw2, dl.to(bf))
    with pytest.raises(B.MoeError, match="dw1: expected"):
        L.capture(lg, x, w1, w2, x, x, dx, dw2, dw2, dl)


@pytest.fixture
def host_binding(monkeypatch):
    """The binding with a stand-in library that accepts every call, and host
    tensors admitted as device memory: what remains are the binding's own
    checks of element types and layouts."""
    from mixture_experts_expert_sort_b300 import binding as B

    class _AcceptAll:
        def __getattr__(self, name):
            return lambda *args: 0

    monkeypatch.setattr(B, "lib", lambda: _AcceptAll())
    monkeypatch.setattr(B, "_is_device", lambda t: True)
    monkeypatch.setattr(B, "stream_handle", lambda stream=None: None)
    return B


def test_binding_element_types_follow_the_header(host_binding):
    """Every wrapper accepts operands of the element types include/moe.h
    documents for it, and refuses a wrong one."""
    import torch
    B = host_binding
    T, H, F, E, k, rows = 64, 128, 256, 4, 2, 640
    R = T * k

    def bf(*s):
        return torch.zeros(s, dtype=torch.bfloat16)

    def f32(*s):
        return torch.zeros(s, dtype=torch.float32)

    def i32(*s):
        return torch.zeros(s, dtype=torch.int32)

    def u8(*s):
        return torch.zeros(s, dtype=torch.uint8)

    off = i32(E + 1)
    B.moe_route(f32(T, E), k)
    B.moe_route_backward(f32(rows, 3), f32(T, k), i32(T, k), E, dest=i32(R))
    B.moe_router_forward(bf(T, H), bf(H, E), k)
    B.moe_router_backward(bf(T, H), bf(H, E), f32(T, E), f32(1 + 2 * E), f32(T, E), 0.01,
                          dx_in=bf(T, H))
    B.moe_permute_plan(i32(T, k), E, 128)
    B.moe_permute_plan_static(i32(T, k), E, 128)
    B.moe_permute(bf(T, H), i32(R), off, i32(E), k, rows, w=f32(T, k))
    B.moe_unpermute(bf(rows, H), i32(R), T, k, w=f32(T, k))
    B.mxfp8_quantize(bf(T, H), rows=rows, src=i32(rows), src_div=k)
    B.mxfp8_quantize(bf(T, 2 * H)[:, :H])  # strided rows: the leading dimension is passed
    B.mxfp8_scales_to_canonical(u8(rows * H // 32), rows, H)
    B.mxfp4_from_mxfp8(u8(rows, H), u8(rows * H // 32))
    B.mxfp8_from_mxfp4(u8(rows, H // 2), u8(rows * H // 32))
    B.mxfp4_rowwise_to_colwise(u8(rows, H // 2), u8(rows * H // 32))
    B.mxfp8_colwise_from_mxfp4_rowwise(u8(rows, H // 2), u8(rows * H // 32))
    B.moe_grouped_gemm_bf16(B.GEMM_FPROP, bf(rows, H), bf(E, H, F), off)
    B.moe_grouped_gemm_bf16(B.GEMM_WGRAD, bf(rows, H), bf(rows, F), off)
    B.moe_fc1_swiglu_bf16(bf(rows, H), bf(E, H, 2 * F), off, f32(rows))
    B.moe_fc2_dgrad_swiglu_bwd_bf16(bf(rows, H), bf(E, F, H), off, f32(rows), bf(rows, 2 * F))
    # row gathers: the gathered operand is the un-permuted [T, .] source
    B.moe_grouped_gemm_bf16(B.GEMM_FPROP, bf(T, H), bf(E, H, F), off, gather_a=(i32(rows), k))
    B.moe_grouped_gemm_bf16(B.GEMM_WGRAD, bf(T, H), bf(rows, F), off, gather_a=(i32(rows), k))
    B.moe_grouped_gemm_bf16(B.GEMM_WGRAD, bf(rows, F), bf(T, H), off, gather_b=(i32(rows), k))
    B.moe_fc1_swiglu_bf16(bf(T, H), bf(E, H, 2 * F), off, f32(rows), gather_x=(i32(rows), k))
    B.moe_fc2_dgrad_swiglu_bwd_bf16(bf(T, H), bf(E, F, H), off, f32(rows), bf(rows, 2 * F),
                                    gather_dy=(i32(rows), k))
    B.moe_grouped_gemm_mxfp8(B.GEMM_FPROP, u8(rows, H), u8(rows * H // 32), u8(F, E * H),
                             u8(F * E * H // 32), off, N=F)
    B.moe_fc1_swiglu_mxfp8(u8(rows, H), u8(rows * H // 32), u8(2 * F, E * H),
                           u8(2 * F * E * H // 32), off, f32(rows), F)
    B.moe_fc2_dgrad_swiglu_bwd_mxfp8(u8(rows, H), u8(rows * H // 32), u8(E * F, H),
                                     u8(E * F * H // 32), off, f32(rows), bf(rows, 2 * F), F)
    cfg = B.layer_config(T, H, F, E, k)
    B.moe_layer_forward(cfg, f32(T, E), bf(T, H), bf(E, H, 2 * F), bf(E, F, H), bf(T, H), u8(64))
    B.moe_layer_backward(cfg, bf(T, H), bf(E, H, 2 * F), bf(E, F, H), bf(T, H),
                         bf(E, H, 2 * F), bf(E, F, H), f32(T, E), u8(64))

    wrong = [
        lambda: B.moe_route(bf(T, E), k),  # logits are fp32
        lambda: B.moe_route(f32(T, E), k, idx=torch.zeros(T, k, dtype=torch.int64)),
        lambda: B.moe_permute_plan(torch.zeros(T, k, dtype=torch.int64), E, 128),
        lambda: B.moe_permute(f32(T, H), i32(R), off, i32(E), k, rows),  # x is bf16
        lambda: B.mxfp8_quantize(f32(T, H)),
        lambda: B.mxfp8_scales_to_canonical(i32(rows * H // 128), rows, H),
        lambda: B.mxfp4_from_mxfp8(i32(rows, H // 4), u8(rows * H // 32)),
        lambda: B.moe_grouped_gemm_bf16(B.GEMM_FPROP, bf(rows, H), bf(E, H, F), off.long()),
        lambda: B.moe_fc1_swiglu_bf16(bf(rows, H), bf(E, H, 2 * F), off, bf(rows)),
        lambda: B.moe_fc1_swiglu_bf16(bf(T, H), bf(E, H, 2 * F), off, f32(rows),
                                      gather_x=(i32(rows).long(), k)),  # src is int32
        lambda: B.moe_layer_backward(cfg, f32(T, H), bf(E, H, 2 * F), bf(E, F, H), bf(T, H),
                                     bf(E, H, 2 * F), bf(E, F, H), f32(T, E), u8(64)),
        lambda: B.moe_layer_forward(cfg, bf(T, E), bf(T, H), bf(E, H, 2 * F), bf(E, F, H),
                                    bf(T, H), u8(64)),
        lambda: B.moe_layer_forward(cfg, f32(T, E), bf(T, H), bf(E, H, 2 * F), bf(E, F, H),
                                    bf(T, H), f32(16)),  # the workspace is counted in bytes
    ]
    for call in wrong:
        with pytest.raises(B.MoeError, match="element type"):
            call()


@pytest.mark.skipif(__import__("torch").cuda.is_available(),
                    reason="passes made-up device addresses: only on a host with no GPU")
def test_bad_arguments_return_arg_error_before_any_cuda_call(libmoe):
    """Each entry point returns MOE_ERR_ARG (1) for a bad size, count, mode or
    alignment, with non-null buffers, before any CUDA call. On a host without
    a GPU a missed check would show as MOE_ERR_CUDA (3), since every CUDA call
    fails there; nothing can be launched."""
    import ctypes as C
    from mixture_experts_expert_sort_b300 import binding as B
    L = B.lib()
    P = 0x100000  # a made-up, 256-byte aligned address: never dereferenced here
    gather = C.byref(B.RowGather(P, 2, 256))
    div0 = C.byref(B.RowGather(P, 0, 256))
    nosrc = C.byref(B.RowGather(None, 2, 256))
    norows = C.byref(B.RowGather(P, 2, 0))
    cases = {
        "route T < 0": ("moe_route", P, -1, 8, 2, P, P, None),
        "route E = 0": ("moe_route", P, 16, 0, 1, P, P, None),
        "route E > 256": ("moe_route", P, 16, 257, 2, P, P, None),
        "route k > E": ("moe_route", P, 16, 4, 5, P, P, None),
        "route k > 8": ("moe_route", P, 16, 64, 9, P, P, None),
        "route_backward n_part = 0": ("moe_route_backward", P, 1, 0, P, P, P, 16, 8, 2, P, None),
        "route_backward ld < n_part": ("moe_route_backward", P, 1, 2, P, P, P, 16, 8, 2, P, None),
        "plan align = 0": ("moe_permute_plan", P, 16, 8, 2, 0, P, P, P, P, 4096, P, 1 << 20,
                           None),
        "plan workspace too small": ("moe_permute_plan", P, 16, 8, 2, 128, P, P, P, P, 4096, P,
                                     0, None),
        "plan src too short": ("moe_permute_plan", P, 16, 8, 2, 128, P, P, P, P, 1, P, 1 << 20,
                               None),
        "plan_static E = 0": ("moe_permute_plan_static", P, 16, 0, 1, 128, P, P, P, P, 4096,
                              None),
        "permute H % 8": ("moe_permute", P, P, P, P, P, 16, 12, 8, 2, P, P, None),
        "permute x misaligned": ("moe_permute", P + 8, P, P, P, P, 16, 128, 8, 2, P, P, None),
        "unpermute H % 8": ("moe_unpermute", P, P, P, 16, 12, 2, P, None),
        "quantize no direction": ("mxfp8_quantize", P, 128, 128, 128, None, 1, 0, P, P, P, P,
                                  None),
        "quantize ld < cols": ("mxfp8_quantize", P, 128, 256, 128, None, 1, 3, P, P, P, P, None),
        "quantize cols % 128": ("mxfp8_quantize", P, 128, 96, 96, None, 1, 3, P, P, P, P, None),
        "quantize src_div = 0": ("mxfp8_quantize", P, 128, 128, 128, P, 0, 3, P, P, P, P, None),
        "canonical mn % 128": ("mxfp8_scales_to_canonical", P, 100, 128, P + (1 << 20), None),
        "canonical kdim % 128": ("mxfp8_scales_to_canonical", P, 128, 96, P + (1 << 20), None),
        "canonical overlap": ("mxfp8_scales_to_canonical", P, 128, 128, P + 64, None),
        "canonical misaligned": ("mxfp8_scales_to_canonical", P + 2, 128, 128, P + (1 << 20),
                                 None),
        "gemm_bf16 mode": ("moe_grouped_gemm_bf16", 7, P, P, 0, P, 4, 512, 0, 256, 128, P, None,
                           None, None),
        "gemm_bf16 b_layout": ("moe_grouped_gemm_bf16", 0, P, P, 3, P, 4, 512, 0, 256, 128, P,
                               None, None, None),
        "gemm_bf16 E = 0": ("moe_grouped_gemm_bf16", 0, P, P, 0, P, 0, 512, 0, 256, 128, P, None,
                            None, None),
        "gemm_bf16 FPROP gathers B": ("moe_grouped_gemm_bf16", 0, P, P, 0, P, 4, 512, 0, 256, 128,
                                      P, None, gather, None),
        "gemm_bf16 WGRAD gathers both": ("moe_grouped_gemm_bf16", 1, P, P, 0, P, 4, 512, 128, 256,
                                         0, P, gather, gather, None),
        "gemm_bf16 gather src_div = 0": ("moe_grouped_gemm_bf16", 0, P, P, 0, P, 4, 512, 0, 256,
                                         128, P, div0, None, None),
        "gemm_bf16 gather no src": ("moe_grouped_gemm_bf16", 1, P, P, 0, P, 4, 512, 128, 256, 0,
                                    P, nosrc, None, None),
        "fc1_swiglu_bf16 F = 0": ("moe_fc1_swiglu_bf16", P, P, P, P, 4, 512, 128, 0, P, P, None,
                                  None),
        "fc1_swiglu_bf16 gather src_rows = 0": ("moe_fc1_swiglu_bf16", P, P, P, P, 4, 512, 128,
                                                256, P, P, norows, None),
        "fc2_dgrad_bf16 E = 0": ("moe_fc2_dgrad_swiglu_bwd_bf16", P, P, P, P, P, 0, 512, 128,
                                 256, P, P, None, None),
        "fc2_dgrad_bf16 gather src_div = 0": ("moe_fc2_dgrad_swiglu_bwd_bf16", P, P, P, P, P, 4,
                                              512, 128, 256, P, P, div0, None),
        "gemm_mxfp8 mode": ("moe_grouped_gemm_mxfp8", 5, P, P, 512, 128, P, P, 256, 512, 0, 0, P,
                            4, 0, 256, 128, P, None),
        "gemm_mxfp8 FPROP N % 128": ("moe_grouped_gemm_mxfp8", 0, P, P, 512, 128, P, P, 256, 512,
                                     0, 128, P, 4, 0, 100, 128, P, None),
        "gemm_mxfp8 FPROP B too short": ("moe_grouped_gemm_mxfp8", 0, P, P, 512, 128, P, P, 256,
                                         512, 0, 256, P, 4, 0, 256, 128, P, None),
        "gemm_mxfp8 WGRAD K mismatch": ("moe_grouped_gemm_mxfp8", 1, P, P, 256, 512, P, P, 256,
                                        384, 0, 0, P, 4, 128, 128, 0, P, None),
        "fc1_swiglu_mxfp8 rows % 128": ("moe_fc1_swiglu_mxfp8", P, P, 100, 128, P, P, P, P, 4,
                                        256, P, P, P, P, P, None),
        "fc2_dgrad_mxfp8 F % 128": ("moe_fc2_dgrad_swiglu_bwd_mxfp8", P, P, 512, 128, P, P, P, P,
                                    P, 4, 100, P, P, P, P, P, None),
        "router_forward workspace": ("moe_router_forward", P, P, 64, 128, 8, 2, P, P, P, P, P, 0,
                                     None),
        "router_forward k > E": ("moe_router_forward", P, P, 64, 128, 2, 3, P, P, P, P, P,
                                 1 << 24, None),
        "router_backward workspace": ("moe_router_backward", P, P, P, P, P, 0.01, 64, 128, 8, P,
                                      None, P, P, P, 0, None),
    }
    for what, (name, *args) in cases.items():
        assert getattr(L, name)(*args) == 1, what
    good = B.layer_config(256, 128, 256, 4, 2)
    bad = B.layer_config(256, 100, 256, 4, 2)
    assert L.moe_layer_forward(C.byref(bad), P, P, P, P, P, P, 1 << 30, None) == 1
    assert L.moe_layer_forward(C.byref(good), P, P, P, P, P, P, 16, None) == 1
    assert L.moe_layer_backward(C.byref(good), P, P, P, P, P, P, P, P, 16, None) == 1
