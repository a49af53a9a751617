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
