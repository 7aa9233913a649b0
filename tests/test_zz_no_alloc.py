"""The allocation-free dispatch planner (mm_plan_dispatch_static).

It exists for callers that cannot allocate device memory where they need a
dispatch plan -- code running under another framework's memory pool or an
allocator-free runtime, or a serving loop that must not call cudaMalloc in its
steady state.  Its scratch is an array compiled into the library, shared by
every call, so this test makes two calls in a row with different inputs (the
second call must not see the first call's leftovers) and checks each against
the plan that mm_forward itself built for the same routing.  The plan is
integer work, so the comparison is exact.  This file is collected last.
"""
import ctypes as C
import dataclasses

import numpy as np
import pytest

import synthetic
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch


def _forward_plan(cfg, T):
    """phys, pos, offsets of one mm_forward (the existing entry point)."""
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    run = gpu_util.Run(cfg, cap=T)
    res = run.forward(hidden, logits, bias)
    run.close()
    assert res["status"] == 0
    return res["phys"].ravel().copy(), res["pos"].ravel().copy(), res["offsets"].copy()


def _static_plan(torch, phys, P):
    import moe_layer_serving_gb300 as mm
    n = phys.size
    d_phys = torch.from_numpy(phys.astype(np.int32)).cuda()
    d_pos = torch.full((max(n, 1),), -7, dtype=torch.int32, device="cuda")
    d_off = torch.full((P + 1,), -7, dtype=torch.int32, device="cuda")
    st = mm.lib().mm_plan_dispatch_static(d_phys.data_ptr(), n, P, d_pos.data_ptr(), d_off.data_ptr(), None)
    assert st == mm.MM_OK, mm.lib().mm_status_string(st)
    torch.cuda.synchronize()
    return d_pos[:n].cpu().numpy(), d_off.cpu().numpy()


def test_static_plan_matches_forward_twice_in_a_row(torch):
    cfg = dataclasses.replace(synthetic.CONFIGS[0], P=12)
    # two different routings: the second, smaller one runs after the first
    # left its counts in the shared scratch array
    for T in (1500, 300):
        phys, pos, off = _forward_plan(cfg, T)
        got_pos, got_off = _static_plan(torch, phys, cfg.P)
        assert np.array_equal(got_off, off)
        assert np.array_equal(got_pos, pos)


def test_static_plan_rejects_oversized_input(torch):
    import moe_layer_serving_gb300 as mm
    L = mm.lib()
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    assert L.mm_plan_dispatch_static(dummy.data_ptr(), 131073, 8, dummy.data_ptr(), dummy.data_ptr(), None) == \
        mm.MM_ERR_CAPACITY
    assert L.mm_plan_dispatch_static(dummy.data_ptr(), 16, 513, dummy.data_ptr(), dummy.data_ptr(), None) == \
        mm.MM_ERR_INVALID_ARG
