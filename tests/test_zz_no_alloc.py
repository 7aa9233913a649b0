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


def _expected_plan(phys, P):
    """The plan from the oracle's permute over the ids inside [0, P): segments
    padded to 16 rows, pairs in pair order inside a segment, -1 elsewhere."""
    import oracle
    valid = (phys >= 0) & (phys < P)
    off_o, _, pos_o = oracle.permute(phys[valid].astype(np.int32), P)
    padded = (np.diff(off_o) + 15) // 16 * 16
    off = np.concatenate([[0], np.cumsum(padded)]).astype(np.int64)
    pos = np.full(phys.size, -1, np.int64)
    pv = phys[valid]
    pos[valid] = off[pv] + (pos_o - off_o[pv])
    return pos, off


def test_static_plan_leaves_out_ids_outside_the_expert_range(torch):
    rng = np.random.default_rng(3)
    P = 40
    phys = rng.integers(0, P, size=5000).astype(np.int32)
    phys[::97] = P                  # one past the last expert
    phys[5::131] = -3               # negative
    phys[7::1009] = 1 << 20         # far outside
    got_pos, got_off = _static_plan(torch, phys, P)
    pos, off = _expected_plan(phys, P)
    assert np.array_equal(got_off, off)
    assert np.array_equal(got_pos, pos)
    assert np.all(got_pos[(phys < 0) | (phys >= P)] == -1)


def test_static_plan_at_its_limits_then_a_small_call(torch):
    # 512 experts (the limit) and 131,072 pairs (the cap): 128 chunks x 512
    # experts of counts fill the whole 256 KB scratch array.  A small call on
    # the same stream right after must not see those leftovers.
    rng = np.random.default_rng(4)
    P = 512
    # skewed ids so that some chunks hit every expert and some experts get many rows
    big = np.minimum(rng.zipf(1.3, size=131072) - 1, P - 1).astype(np.int32)
    big[:P] = np.arange(P, dtype=np.int32)
    got_pos, got_off = _static_plan(torch, big, P)
    pos, off = _expected_plan(big, P)
    assert np.array_equal(got_off, off)
    assert np.array_equal(got_pos, pos)
    small = rng.integers(0, 7, size=333).astype(np.int32)
    got_pos, got_off = _static_plan(torch, small, P)
    pos, off = _expected_plan(small, P)
    assert np.array_equal(got_off, off)
    assert np.array_equal(got_pos, pos)
    assert got_off[-1] == off[7] and np.all(got_off[7:] == got_off[7])
