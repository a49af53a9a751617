"""Failure detection on the GPU without a fault: the bounded wait that every
pipelined kernel uses runs out on an mbarrier that nothing arrives at; the
kernel records MOE_DEVERR_TIMEOUT and returns, the host reads the bit, and
the context keeps working."""
import time

import numpy as np
import pytest
import torch

from oracle import moe_oracle as O
from tests.helpers import i32

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_bounded_wait_times_out_and_context_survives():
    from mixture_experts_expert_sort_b300 import binding as B
    torch.cuda.synchronize()
    B.device_error()  # read and clear anything left from earlier tests
    t0 = time.perf_counter()
    B.selftest_wait_timeout()
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    flags = B.device_error()
    assert flags & B.MOE_DEVERR_TIMEOUT, flags
    assert 1.5 < elapsed < 30.0, elapsed  # the 2 s limit, then a return
    assert B.device_error() == 0  # reading cleared it
    # the context is still usable: a routing call afterwards is exact
    lg = torch.randn((64, 8), generator=torch.Generator().manual_seed(5))
    idx, w = B.moe_route(lg.to(DEV), 2)
    torch.cuda.synchronize()
    ridx, _ = O.route(lg.double().numpy(), 2)
    np.testing.assert_array_equal(i32(idx), ridx)
    assert B.device_error() == 0
