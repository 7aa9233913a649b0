"""Behaviour of the C ABI on the GPU: idle batches, capacity and route
checks, per-layer recording slots, EPLB map validation, replica invariance,
determinism and CUDA-graph capture."""
import ctypes as C
import dataclasses

import numpy as np
import pytest

import oracle
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


@pytest.fixture
def small(torch):
    cfg = dataclasses.replace(synthetic.CONFIGS[0], P=12, recording=True)
    run = gpu_util.Run(cfg, cap=64)
    yield cfg, run
    run.close()


def test_idle_batch_is_a_noop(torch, small):
    cfg, run = small
    import moe_layer_serving_gb300 as mm
    out = torch.full((4, cfg.H), 3.0, dtype=torch.bfloat16, device="cuda")
    st = mm.lib().mm_forward(run.op.handle, None, None, None, None, 0, None)
    assert st == mm.MM_OK
    run.op.forward(out, torch.zeros(4, cfg.E, device="cuda"), None, out, num_tokens=0)
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)
    assert run.op.read_counts(0).sum() == 0


def test_capacity_and_route_limits(torch, small):
    cfg, run = small
    import moe_layer_serving_gb300 as mm
    x = torch.zeros(65, cfg.H, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(65, cfg.E, device="cuda")
    L = mm.lib()
    assert L.mm_forward(run.op.handle, x.data_ptr(), lg.data_ptr(), None, x.data_ptr(), 65, None) == \
        mm.MM_ERR_CAPACITY
    run.op.reserve(1024)
    run.op.set_route(mm.ROUTE_SMALL)
    x2 = torch.zeros(600, cfg.H, dtype=torch.bfloat16, device="cuda")
    lg2 = torch.zeros(600, cfg.E, device="cuda")
    out = torch.empty_like(x2)
    assert L.mm_forward(run.op.handle, x2.data_ptr(), lg2.data_ptr(), None, out.data_ptr(), 600, None) == \
        mm.MM_ERR_CAPACITY
    run.op.set_route(mm.ROUTE_LARGE)
    assert L.mm_forward(run.op.handle, x2.data_ptr(), lg2.data_ptr(), None, out.data_ptr(), 600, None) == mm.MM_OK
    torch.cuda.synchronize()
    assert L.mm_forward(run.op.handle, x2.data_ptr() + 2, lg2.data_ptr(), None, out.data_ptr(), 8, None) == \
        mm.MM_ERR_INVALID_ARG
    assert L.mm_set_route(run.op.handle, 7) == mm.MM_ERR_INVALID_ARG


def test_forced_routes_agree(torch):
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    hidden, logits, bias = synthetic.make_activations(cfg, 200)
    run = gpu_util.Run(cfg, cap=200)
    outs = []
    # the large route: route, hist, scan, scatter, quantise/dispatch, the two
    # grouped GEMM kernels (H = 256 allows CTA pairs: both are launched, the
    # tile scan picks one), combine
    for r, expect in ((mm.ROUTE_SMALL, (1, 1)), (mm.ROUTE_LARGE, (2, 8)), (mm.ROUTE_AUTO, (1, 1))):
        run.op.set_route(r)
        outs.append(run.forward(hidden, logits, bias, dumps=False)["out"])
        route, launches, site = run.op.last_info()
        assert (route, launches) == expect and site == 0
    run.close()
    # the fused small-input kernel and the multi-kernel large-input path agree bit for bit
    assert np.array_equal(outs[0], outs[1])
    ref = oracle.forward(hidden, logits, bias, cfg.k, gpu_util.weights(cfg))["out"]
    for o in outs:
        gpu_util.assert_out_close(o, ref)


def test_recording_slots_and_reset(torch, small):
    cfg, run = small
    hidden, logits, bias = synthetic.make_activations(cfg, 40)
    idx, _ = oracle.route(logits, bias, cfg.k)
    hist = np.bincount(idx.ravel(), minlength=cfg.E)
    run.op.set_recording(False)
    run.forward(hidden, logits, bias, dumps=False)
    assert run.op.read_counts(0).sum() == 0
    run.op.set_recording(True)
    run.op.bind_layer(3)
    run.forward(hidden, logits, bias, dumps=False)
    run.forward(hidden, logits, bias, dumps=False)
    run.op.bind_layer(7)
    run.forward(hidden, logits, bias, dumps=False)
    assert np.array_equal(run.op.read_counts(3), 2 * hist)
    assert np.array_equal(run.op.read_counts(7), hist)
    assert run.op.read_counts(0).sum() == 0
    run.op.reset_counts(3)
    assert run.op.read_counts(3).sum() == 0 and np.array_equal(run.op.read_counts(7), hist)
    run.op.reset_counts(-1)
    assert run.op.read_counts(7).sum() == 0


def test_eplb_map_validation(torch):
    import moe_layer_serving_gb300 as mm
    cfg = dataclasses.replace(synthetic.CONFIGS[0], P=12)
    op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I)
    W = [torch.from_numpy(a).cuda() for a in gpu_util.weights(cfg)]
    op.set_weights(*W)
    op.reserve(16)
    hidden, logits, bias = synthetic.make_activations(cfg)
    x = torch.from_numpy(hidden.view(np.int16)).cuda().view(torch.bfloat16)
    lg = torch.from_numpy(logits).cuda()
    out = torch.empty_like(x)
    L = mm.lib()
    # no map yet with P > E
    assert L.mm_forward(op.handle, x.data_ptr(), lg.data_ptr(), None, out.data_ptr(), 16, None) == mm.MM_ERR_NOT_READY
    m, rc, R = synthetic.make_eplb_map(cfg)
    bad = m.copy()
    bad[1, 0] = 0                              # physical 0 twice, physical 1 never
    for mm_, rc_ in ((bad, rc), (m, np.where(rc == 2, 3, rc).astype(np.int32)), (m, np.zeros_like(rc))):
        with pytest.raises(mm.MegaMoEError):
            op.set_eplb_map(mm_, rc_)
    op.set_eplb_map(m, rc)
    assert L.mm_forward(op.handle, x.data_ptr(), lg.data_ptr(), None, out.data_ptr(), 16, None) == mm.MM_OK
    torch.cuda.synchronize()
    op.close()


def test_replicas_give_identical_output(torch):
    base = synthetic.CONFIGS[0]
    hidden, logits, bias = synthetic.make_activations(base, 300)
    a = gpu_util.Run(base, cap=300)
    ra = a.forward(hidden, logits, bias)
    a.close()
    rep = dataclasses.replace(base, P=12)
    b = gpu_util.Run(rep, cap=300)
    rb = b.forward(hidden, logits, bias)
    b.close()
    assert np.any(rb["phys"] >= base.E)
    assert np.array_equal(ra["out"], rb["out"])


def test_deterministic_across_runs(torch):
    cfg = synthetic.CONFIGS[0]
    hidden, logits, bias = synthetic.make_activations(cfg, 257)
    run = gpu_util.Run(cfg, cap=257)
    o1 = run.forward(hidden, logits, bias, dumps=False)["out"]
    o2 = run.forward(hidden, logits, bias, dumps=False)["out"]
    run.close()
    assert np.array_equal(o1, o2)


@pytest.mark.parametrize("T", [96, 1100])          # fused small path, and the 7-launch large path
def test_graph_capture_replay_matches_eager(torch, T):
    cfg = synthetic.CONFIGS[0]
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    run = gpu_util.Run(cfg, cap=T)
    x, lg, b = run.to_dev(hidden, logits, bias)
    eager = torch.empty_like(x)
    run.op.forward(x, lg, b, eager)
    torch.cuda.synchronize()
    out = torch.zeros_like(x)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            run.op.forward(x, lg, b, out, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    lg.copy_(torch.flip(lg, dims=[0]))
    g.replay()
    run.op.forward(x, lg, b, eager)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    assert run.op.get_status() == 0
    run.close()


def test_routing_bit_exact_wide_experts(torch):
    # E = 512, k = 8, logits over a wide range with ties: the score sequence
    # must select exactly the oracle's experts and reproduce its weights.
    cfg = dataclasses.replace(synthetic.CONFIGS[0], E=512, P=512, k=8, H=128, I=128)
    T = 2048
    rng = np.random.default_rng(11)
    logits = (rng.standard_normal((T, cfg.E)) * rng.choice([0.01, 1, 10, 60], (T, 1))).astype(np.float32)
    logits[::5, 1::2] = logits[::5, 0::2]
    bias = (0.05 * rng.standard_normal(cfg.E)).astype(np.float32)
    hidden = synthetic.bf16_bits_from_f32(rng.standard_normal((T, cfg.H)).astype(np.float32))
    W = synthetic.make_all_weights(dataclasses.replace(cfg, E=cfg.E))
    run = gpu_util.Run(cfg, W, cap=T)
    res = run.forward(hidden, logits, bias)
    run.close()
    idx, w = oracle.route(logits, bias, cfg.k)
    assert np.array_equal(res["idx"], idx)
    assert np.array_equal(res["weights"].view(np.uint32), w.view(np.uint32))


@pytest.mark.parametrize("T", [400, 1500])
def test_rebalance_keeps_outputs_and_spreads_load(torch, T):
    # skewed routing, replicas first placed on experts 0..3; recorded counts
    # drive a new plan with up to 4 replicas per expert
    cfg = dataclasses.replace(synthetic.CONFIGS[0], P=12, zipf_s=1.4, recording=True)
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    run = gpu_util.Run(cfg, cap=T)
    run.op.set_recording(True)
    r1 = run.forward(hidden, logits, bias)
    counts = run.op.read_counts(0)
    run.op.rebalance(0, 4)
    run.op.set_recording(False)
    r2 = run.forward(hidden, logits, bias)
    run.close()
    assert r1["status"] == 0 and r2["status"] == 0
    assert np.array_equal(r1["idx"], r2["idx"])
    assert not np.array_equal(r1["phys"], r2["phys"])          # the map really changed
    assert np.array_equal(r1["out"], r2["out"])                # replicas are byte copies
    load1 = np.bincount(r1["phys"].ravel(), minlength=cfg.P)
    load2 = np.bincount(r2["phys"].ravel(), minlength=cfg.P)
    assert load2.max() < load1.max()
    pol, rc = oracle.plan_replicas(counts, cfg.P, 4)
    assert np.array_equal(r2["phys"], oracle.eplb(r2["idx"], pol, rc))


def _check_tiles(res, P, tile):
    """Token tiles cut each expert's segment into consecutive `tile`-row pieces."""
    tiles = res["tiles"].reshape(-1, 3)
    off = res["offsets"]
    count = np.bincount(res["phys"].ravel(), minlength=P)
    want = []
    for p in range(P):
        for j in range((count[p] + tile - 1) // tile):
            want.append((p, off[p] + j * tile, min(tile, count[p] - j * tile)))
    assert tiles.tolist() == [list(w) for w in want]


@pytest.mark.parametrize("case", ["short", "full_small", "large"])
def test_tile_table_and_tile_size_choice(torch, case):
    # short: one hot expert of 100 rows among many small ones; 64-row tiles add
    # one tile in 33, so the fused kernel takes them.  full_small: eight
    # experts of 512 rows; 64-row tiles would double the tiles, so it takes
    # 128.  large: the large-input path always cuts 128-row tiles.
    T = {"short": 200, "full_small": 512, "large": 1100}[case]
    k = 2 if case == "short" else 8
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, H=256, I=128, E=32, P=32, k=k)
    hidden, logits, bias = synthetic.make_activations(cfg)
    if case == "short":
        logits[:100, 0] += 20.0
    elif case == "full_small":
        logits[:, :8] += 20.0
    W = synthetic.make_all_weights(cfg)
    run = gpu_util.Run(cfg, W, cap=T)
    res = run.forward(hidden, logits, bias)
    route = run.op.last_info()[0]
    run.close()
    assert res["status"] == 0
    assert route == (2 if case == "large" else 1)
    if case == "short":
        assert np.bincount(res["phys"].ravel(), minlength=cfg.P)[0] > 64
    _check_tiles(res, cfg.P, 64 if case == "short" else 128)
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None, gpu_util.sample_tokens(T, 32))


def test_shared_expert_limits_and_weight_reset(torch):
    # k + S <= MM_MAX_TOPK and P + S <= MM_MAX_EXPERTS; changing S drops the
    # weights (forward is not ready until they are set again)
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I)
    L = mm.lib()
    assert L.mm_set_shared_experts(op.handle, -1) == mm.MM_ERR_INVALID_ARG
    assert L.mm_set_shared_experts(op.handle, 8 - cfg.k + 1) == mm.MM_ERR_INVALID_ARG
    assert L.mm_set_shared_experts(op.handle, 8 - cfg.k) == mm.MM_OK
    op.set_shared_experts(1)
    op.reserve(cfg.T)
    x = torch.zeros(cfg.T, cfg.H, dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros(cfg.T, cfg.E, device="cuda")
    assert L.mm_forward(op.handle, x.data_ptr(), lg.data_ptr(), None, x.data_ptr(), cfg.T, None) == \
        mm.MM_ERR_NOT_READY
    op.close()
