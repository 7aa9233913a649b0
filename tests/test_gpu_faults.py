"""Failure detection without a GPU fault.

MM_FAULT (read when a handle is created) makes one device-side wait
unsatisfiable: one CTA withholds its arrival at a grid barrier of the fused
kernel, or GEMM2 waits for a GEMM1 unit that never exists.  Every wait in the
kernels is bounded, so the forward must come back with MM_ERR_TIMEOUT latched
and the site that raised it, and the CUDA context must stay usable: a handle
without the fault then runs the same layer and matches the oracle.
"""
import os

import numpy as np
import pytest

import oracle
import synthetic
from tests import gpu_util

pytestmark = pytest.mark.gpu

SITE_PRODUCER_DONE1, SITE_GRID_BARRIER = 5, 6


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch


def _faulty_run(cfg, T, fault, act=0, gemm=None):
    os.environ["MM_FAULT"] = fault
    if gemm is not None:
        os.environ["MM_GEMM_2SM"] = gemm
    try:
        run = gpu_util.Run(cfg, cap=T, act=act)
    finally:
        del os.environ["MM_FAULT"]
        os.environ.pop("MM_GEMM_2SM", None)
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    res = run.forward(hidden, logits, bias, dumps=False)
    route, _, site = run.op.last_info()
    kind = run.op.last_gemm()
    run.close()
    if gemm is not None and route == 2:
        assert kind == int(gemm) + 1          # the GEMM kernel the test means to time out
    return res["status"], route, site, (hidden, logits, bias)


@pytest.mark.parametrize("fault,T,site,route,gemm", [("grid_barrier", 64, SITE_GRID_BARRIER, 1, None),
                                                     ("gemm_dependency", 64, SITE_PRODUCER_DONE1, 1, None),
                                                     ("gemm_dependency", 1200, SITE_PRODUCER_DONE1, 2, "0"),
                                                     ("gemm_dependency", 1200, SITE_PRODUCER_DONE1, 2, "1")])
def test_injected_wait_times_out_and_context_survives(torch, fault, T, site, route, gemm):
    # gemm: MM_GEMM_2SM for the large path ("0" the one-CTA kernel, "1" CTA pairs)
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    status, took, got_site, inputs = _faulty_run(cfg, T, fault, gemm=gemm)
    assert took == route
    assert status == mm.MM_ERR_TIMEOUT
    assert got_site == site
    # the context is still usable: a clean handle runs the layer correctly
    run = gpu_util.Run(cfg, cap=T)
    res = run.forward(*inputs, dumps=False)
    run.close()
    assert res["status"] == 0
    ref = oracle.forward(*inputs, cfg.k, gpu_util.weights(cfg))
    gpu_util.assert_out_close(res["out"], ref["out"])


@pytest.mark.parametrize("T", [64, 1200])
def test_injected_wait_times_out_in_the_a16w4_gemm(torch, T):
    # the bf16 x MXFP4 GEMM's token producer waits for GEMM1 units that never come
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    status, took, got_site, inputs = _faulty_run(cfg, T, "gemm_dependency", act=mm.ACT_BF16)
    assert took == 2
    assert status == mm.MM_ERR_TIMEOUT
    assert got_site == SITE_PRODUCER_DONE1
    run = gpu_util.Run(cfg, cap=T, act=mm.ACT_BF16)
    res = run.forward(*inputs, dumps=False)
    run.close()
    assert res["status"] == 0
    ref = oracle.forward(*inputs, cfg.k, gpu_util.weights(cfg), act="bf16")
    gpu_util.assert_out_close_a16(res["out"], ref["out"], mag=gpu_util.pair_magnitude(ref, cfg.k))


def test_forward_after_unread_failure_does_no_work(torch):
    # A timed-out fused launch leaves the grid-barrier count short of a multiple
    # of the grid.  A second forward made before mm_get_status must not run on
    # that count (its barriers would release early and its output be wrong):
    # it does no work, leaves its output untouched, and the error stays latched.
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    T = 64
    os.environ["MM_FAULT"] = "grid_barrier"
    try:
        run = gpu_util.Run(cfg, cap=T)
    finally:
        del os.environ["MM_FAULT"]
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    x, lg, b = run.to_dev(hidden, logits, bias)
    out = torch.empty_like(x)
    run.op.forward(x, lg, b, out)                    # times out on the device
    torch.cuda.synchronize()
    out.view(torch.int16).fill_(0x7F7F)
    run.op.forward(x, lg, b, out)                    # no mm_get_status in between
    torch.cuda.synchronize()
    assert run.op.last_info()[0] == 1
    assert bool((out.view(torch.int16) == 0x7F7F).all()), "a forward after an unread failure wrote output"
    assert run.op.get_status() == mm.MM_ERR_TIMEOUT
    assert run.op.last_info()[2] == SITE_GRID_BARRIER
    assert run.op.get_status() == 0                  # read and cleared
    run.close()


SITE_ROUTE_MAP = 8


@pytest.mark.parametrize("route", [1, 2])
def test_corrupt_map_entry_is_caught_at_the_route_in_the_debug_build(torch, route):
    # The build with device-side bounds checks (libmegamoe_debug.so): after
    # mm_set_eplb_map validated the map, MM_FAULT=map_entry overwrites the
    # device entry of logical expert 0 with a physical id past the last expert.
    # The route's check must catch it before any later stage indexes with it:
    # MM_ERR_DEVICE with the route's site, the pairs of expert 0 left out
    # (physical id -1), every other pair placed as the oracle places it.
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    T = 64
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    idx, _ = oracle.route(logits, bias, cfg.k)
    assert (idx == 0).any()
    os.environ["MM_FAULT"] = "map_entry"
    try:
        op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I, debug=True)
    finally:
        del os.environ["MM_FAULT"]
    dev = torch.device("cuda:0")
    op.set_weights(*[torch.from_numpy(a).to(dev) for a in gpu_util.weights(cfg)])
    op.reserve(T)
    op.set_route(mm.ROUTE_SMALL if route == 1 else mm.ROUTE_LARGE)
    x = torch.from_numpy(hidden.view(np.int16)).to(dev).view(torch.bfloat16)
    lg, b = torch.from_numpy(logits).to(dev), torch.from_numpy(bias).to(dev)
    out = torch.empty_like(x)
    op.forward(x, lg, b, out)
    torch.cuda.synchronize()
    assert op.last_info()[0] == route
    phys = op.debug_dump(2).reshape(T, cfg.k)
    assert op.get_status() == mm.MM_ERR_DEVICE
    assert op.last_info()[2] == SITE_ROUTE_MAP
    assert np.array_equal(phys == -1, idx == 0)
    assert np.array_equal(phys[idx != 0], idx[idx != 0])        # identity map elsewhere
    op.close()


@pytest.mark.parametrize("route", [1, 2])
def test_debug_build_runs_the_layer_and_release_ignores_the_debug_fault(torch, route):
    # without a fault the bounds-checked build computes the same layer; the
    # release build ignores MM_FAULT=map_entry (it has no checks to catch it)
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    T = 64
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    ref = oracle.forward(hidden, logits, bias, cfg.k, gpu_util.weights(cfg))
    dev = torch.device("cuda:0")
    outs = []
    for debug, fault in ((True, None), (False, "map_entry")):
        if fault:
            os.environ["MM_FAULT"] = fault
        try:
            op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I, debug=debug)
        finally:
            os.environ.pop("MM_FAULT", None)
        op.set_weights(*[torch.from_numpy(a).to(dev) for a in gpu_util.weights(cfg)])
        op.reserve(T)
        op.set_route(mm.ROUTE_SMALL if route == 1 else mm.ROUTE_LARGE)
        x = torch.from_numpy(hidden.view(np.int16)).to(dev).view(torch.bfloat16)
        lg, b = torch.from_numpy(logits).to(dev), torch.from_numpy(bias).to(dev)
        out = torch.empty_like(x)
        op.forward(x, lg, b, out)
        torch.cuda.synchronize()
        assert op.get_status() == 0
        outs.append(out.view(torch.int16).cpu().numpy().view(np.uint16))
        op.close()
    gpu_util.assert_out_close(outs[0], ref["out"])
    assert np.array_equal(outs[0], outs[1])            # the checks change no result
