"""The allocation-free expert-sort plan (moe_permute_plan_static).

Callers that cannot allocate device memory use this entry point; it keeps
its scratch in a fixed array inside the library. This test calls it through
the C ABI twice in a row, on different routings, and checks that each result
equals that of moe_permute_plan (which takes a caller workspace) bit for bit;
at the largest size the scratch holds it checks the result against the
oracle's plan, and one token more must be rejected. It lives in a file of its
own that is collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O

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


def test_plan_static_at_the_scratch_limit_matches_oracle():
    """ceil(T*k / 1024) * E == 262144 exactly (E = 1024, T*k = 262144): the
    largest case the fixed scratch holds, checked against the oracle's plan;
    one token more is rejected."""
    from mixture_experts_expert_sort_b300 import binding as B
    T, E, k, align = 131072, 1024, 2, 32
    g = torch.Generator().manual_seed(7)
    idx = torch.randint(0, E - 3, (T, k), generator=g, dtype=torch.int32)  # 3 empty experts
    got = _plan_static_via_abi(B, idx.to(DEV), E, align)
    torch.cuda.synchronize()
    counts, offsets, dest, src = O.permute_plan(idx.numpy(), E, align)
    np.testing.assert_array_equal(got["counts"].cpu().numpy(), counts)
    np.testing.assert_array_equal(got["offsets"].cpu().numpy(), offsets)
    np.testing.assert_array_equal(got["dest"].cpu().numpy(), dest)
    gsrc = got["src"].cpu().numpy()
    np.testing.assert_array_equal(gsrc[:len(src)], src)
    assert B.device_error() == 0
    T1 = T + 1  # ceil(262146 / 1024) * 1024 = 263168 > 262144
    idx1 = torch.zeros((T1, k), dtype=torch.int32, device=DEV)
    rows = B.moe_rows_padded_max(T1, E, k, align)
    buf = torch.zeros(max(rows, T1 * k), dtype=torch.int32, device=DEV)
    p = ctypes.c_void_p(buf.data_ptr())
    st = B.lib().moe_permute_plan_static(ctypes.c_void_p(idx1.data_ptr()), T1, E, k, align,
                                         p, p, p, p, rows, None)
    assert st == B.MOE_ERR_UNSUPPORTED
