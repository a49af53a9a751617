"""The allocation-free expert-sort plan (moe_permute_plan_static).

Callers that cannot allocate device memory use this entry point; it keeps
its scratch in a fixed array inside the library. This test calls it through
the C ABI twice in a row, on different routings, and checks that each result
equals that of moe_permute_plan (which takes a caller workspace) bit for bit.
It lives in a file of its own that is collected last.
"""
import ctypes

import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _idx(T, E, k, seed):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn((T, E), generator=g)
    lg[:, E - 2:] -= 1e4  # two experts with no tokens
    return lg


def _plan_static_via_abi(B, idx, E, align):
    """Direct ctypes call of the C entry point (no Python wrapper logic)."""
    T, k = idx.shape
    rows = B.moe_rows_padded_max(T, E, k, align)
    out = {"counts": torch.full((E,), -7, dtype=torch.int32, device=DEV),
           "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device=DEV),
           "dest": torch.full((T * k,), -7, dtype=torch.int32, device=DEV),
           "src": torch.full((rows,), -7, dtype=torch.int32, device=DEV)}
    st = B.lib().moe_permute_plan_static(
        ctypes.c_void_p(idx.data_ptr()), T, E, k, align, ctypes.c_void_p(out["counts"].data_ptr()),
        ctypes.c_void_p(out["offsets"].data_ptr()), ctypes.c_void_p(out["dest"].data_ptr()),
        ctypes.c_void_p(out["src"].data_ptr()), rows,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, B.lib().moe_status_string(st)
    return out


def test_plan_static_matches_workspace_plan_twice():
    from mixture_experts_expert_sort_b300 import binding as B
    cases = [(16384, 64, 6, 128, 1), (3000, 8, 2, 32, 2)]  # two calls in a row, new shapes
    for T, E, k, align, seed in cases:
        idx, _ = B.moe_route(_idx(T, E, k, seed).to(DEV), k)
        got = _plan_static_via_abi(B, idx, E, align)
        ref = B.moe_permute_plan(idx, E, align)
        torch.cuda.synchronize()
        for name in ("counts", "offsets", "dest", "src"):
            assert torch.equal(got[name], ref[name]), (T, E, k, name)
    assert B.device_error() == 0


def test_plan_static_rejects_oversize():
    from mixture_experts_expert_sort_b300 import binding as B
    T, E, k = 1 << 20, 256, 2  # ceil(T*k/1024) * E = 524288 > 262144
    rows = B.moe_rows_padded_max(T, E, k, 1)
    st = B.lib().moe_permute_plan_static(None, T, E, k, 1, None, None, None, None, rows, None)
    assert st == B.MOE_ERR_ARG  # null pointers are rejected first
    dummy = torch.zeros(1, dtype=torch.int32, device=DEV)
    p = ctypes.c_void_p(dummy.data_ptr())
    st = B.lib().moe_permute_plan_static(p, T, E, k, 1, p, p, p, p, rows, None)
    assert st == B.MOE_ERR_UNSUPPORTED
