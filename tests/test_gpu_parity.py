"""Parity of the CUDA path with the CPU oracle on every workload.

Bit-exact: routing indices and weights, physical experts, recorded counts,
segment offsets and dispatch order, MXFP8 activation codes and scales.
GEMM1 requantised codes: >= 99.9% identical, the rest one e4m3 step apart.
GEMM2 + combine fed with the GPU's hq: within bf16 rounding.
Layer output: relative L2 <= 1e-2 and every |err| <= 0.05 rms(out).
The decode batch is compared end to end on every token; the 512-token
workload on sampled tokens; the 8192- and 16384-token workloads on the tokens
of the first and the last row of every token tile (every tile of every
expert); all workloads on all tokens for routing, remap, counts and dispatch.
"""
import numpy as np
import pytest

import oracle
import synthetic
from tests import gpu_util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


def _cfg_run(cid, T=None, sample=None, tiles=False):
    cfg = synthetic.CONFIGS[cid]
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    W = gpu_util.weights(cfg)
    run = gpu_util.Run(cfg, W, cap=hidden.shape[0])
    run.op.set_recording(cfg.recording)
    res = run.forward(hidden, logits, bias)
    assert res["status"] == 0
    if cfg.recording:
        idx, _ = oracle.route(logits, bias, cfg.k)
        assert np.array_equal(run.op.read_counts(0), np.bincount(idx.ravel(), minlength=cfg.E)), "counts differ"
    sel = None if sample is None else gpu_util.sample_tokens(hidden.shape[0], sample)
    if tiles:
        # the first and the last row of every token tile, end to end
        sel = gpu_util.tile_edge_tokens(res, hidden.shape[0])
        assert sel.size >= res["tiles"].size // 3
    rel, _ = gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, run.map, sel)
    run.close()
    return rel


def test_config0_tiny_all_tokens():
    _cfg_run(0)


@pytest.mark.parametrize("T", [1, 5, 37, 130, 300])
def test_config0_shapes_ragged_token_counts(T):
    _cfg_run(0, T=T)


def test_config1_decode_t64():
    _cfg_run(1)             # every token of the decode batch


def test_config2_eplb_t512():
    _cfg_run(2, sample=128)


def test_config3_prefill_t8192():
    _cfg_run(3, tiles=True)         # every token tile of the layer


def test_config4_skewed_eplb_t16384():
    _cfg_run(4, tiles=True)


def test_ragged_hidden_and_odd_shapes():
    # H = 384: the last GEMM2 block has 128 output features (one weight block);
    # I = 256: two GEMM1 n-blocks; 37 tokens spread over 6 experts, top-3
    import dataclasses
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=37, H=384, I=256, E=6, P=6, k=3)
    hidden, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    run = gpu_util.Run(cfg, W, cap=cfg.T)
    res = run.forward(hidden, logits, bias)
    run.close()
    assert res["status"] == 0
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None)


def test_maximum_experts_and_topk_small_path():
    # E = P = 512 (the limit), top-8, T = 512 (the fused kernel's limit)
    import dataclasses
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=512, H=256, I=128, E=512, P=512, k=8, bias_std=0.1)
    hidden, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    run = gpu_util.Run(cfg, W, cap=cfg.T)
    res = run.forward(hidden, logits, bias)
    assert run.op.last_info()[:2] == (1, 1)
    run.close()
    assert res["status"] == 0
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None, gpu_util.sample_tokens(cfg.T, 48))


@pytest.mark.parametrize("T", [512, 513])
def test_concentrated_routing_many_tiles_per_expert(T):
    # every token prefers the same 8 experts: 8 segments of T rows each, several
    # 128-row tiles per expert, the rest of the experts idle
    import dataclasses
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, H=256, I=256, E=64, P=64, k=8)
    hidden, logits, bias = synthetic.make_activations(cfg)
    logits[:, :8] += 20.0
    W = synthetic.make_all_weights(cfg)
    run = gpu_util.Run(cfg, W, cap=T)
    res = run.forward(hidden, logits, bias)
    route = run.op.last_info()[0]
    run.close()
    assert route == (1 if T <= 512 else 2)
    assert res["status"] == 0
    assert np.all(np.sort(res["idx"], axis=1) == np.arange(8))
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None, gpu_util.sample_tokens(T, 40))


@pytest.mark.parametrize("T,E,route", [(37, 1, 1), (1100, 1, 2), (300, 8, 1)])
def test_top1_degenerate_routing(T, E, route):
    # top-1: every weight is 1.0; with one expert the layer is a dense SwiGLU
    # MLP over all tokens (one segment of T rows: one tile in the fused
    # kernel at T = 37, nine 128-row tiles on the large path at T = 1100)
    import dataclasses
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, E=E, P=E, k=1)
    hidden, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    run = gpu_util.Run(cfg, W, cap=T)
    res = run.forward(hidden, logits, bias)
    info = run.op.last_info()
    run.close()
    assert res["status"] == 0
    assert info[0] == route
    assert np.all(res["weights"] == 1.0)
    if E == 1:
        assert np.all(res["idx"] == 0)
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None)


@pytest.mark.parametrize("route", [1, 2])
def test_special_values_and_routing_ties(route):
    # token rows that are all zero, hold a zero 32-block, or sit far from unit
    # scale; logits that tie across all experts (top-k = the lowest indices) or
    # between the two best; both paths (fused kernel, large path)
    import dataclasses
    import moe_layer_serving_gb300 as mm
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=40)
    hidden, logits, bias = synthetic.make_activations(cfg)
    x = synthetic.f32_from_bf16_bits(hidden)
    x[0] = 0.0
    x[1, :32] = 0.0
    x[2] *= 1.0e4
    x[3] *= 1.0e-6
    hidden = synthetic.bf16_bits_from_f32(x)
    logits[5] = 0.25
    logits[6, 3] = logits[6, 6] = logits[6].max() + 1.0
    W = synthetic.make_all_weights(cfg)
    run = gpu_util.Run(cfg, W, cap=cfg.T)
    run.op.set_route(mm.ROUTE_SMALL if route == 1 else mm.ROUTE_LARGE)
    res = run.forward(hidden, logits, bias)
    assert run.op.last_info()[0] == route
    run.close()
    assert res["status"] == 0
    assert list(res["idx"][5]) == list(range(cfg.k))
    assert list(res["idx"][6][:2]) == [3, 6]
    assert not np.any(synthetic.f32_from_bf16_bits(res["out"][0]))      # a zero token gives a zero output
    # the row scaled by 1e4 has outputs ~1e6 and would set the rms of the whole
    # batch: each magnitude regime is held to the tolerance against its own rms
    rest = np.array([t for t in range(cfg.T) if t != 2])
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None, rest)
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None, np.array([2]))


def _shared_weights(cfg, shared, physical_map=False):
    # routed physical experts' weights, then `shared` further experts' weights
    import dataclasses
    wide = dataclasses.replace(cfg, E=cfg.E + shared, P=cfg.E + shared)
    Wl = synthetic.make_all_weights(wide, physical=False)
    if physical_map:
        p2l = synthetic.physical_to_logical(cfg)
        routed = [a[p2l] for a in Wl]
    else:
        routed = [a[:cfg.E] for a in Wl]
    return tuple(np.concatenate([r, a[cfg.E:]]) for r, a in zip(routed, Wl))


@pytest.mark.parametrize("T,route,shared", [(40, 1, 1), (40, 2, 1), (300, 1, 2), (1100, 2, 1)])
def test_fused_shared_experts(T, route, shared):
    # every token also goes to the shared experts (weight 1) on both paths
    import dataclasses
    import moe_layer_serving_gb300 as mm
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T)
    W = _shared_weights(cfg, shared)
    hidden, logits, bias = synthetic.make_activations(cfg)
    run = gpu_util.Run(cfg, W, cap=T, shared=shared)
    run.op.set_route(mm.ROUTE_SMALL if route == 1 else mm.ROUTE_LARGE)
    res = run.forward(hidden, logits, bias)
    info = run.op.last_info()
    run.close()
    assert res["status"] == 0 and info[0] == route
    assert np.all(res["idx"][:, cfg.k:] == cfg.E + np.arange(shared))
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None, shared=shared)


def test_fused_shared_expert_with_replicas_and_recording():
    # P > E (two redundant replicas) with the recorder on: the counts hold the
    # routed selections only
    import dataclasses
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=200, P=10, recording=True)
    W = _shared_weights(cfg, 1, physical_map=True)
    hidden, logits, bias = synthetic.make_activations(cfg)
    run = gpu_util.Run(cfg, W, cap=cfg.T, shared=1)
    run.op.set_recording(True)
    res = run.forward(hidden, logits, bias)
    counts = run.op.read_counts(0)
    run_map = run.map
    run.close()
    assert res["status"] == 0
    idx, _ = oracle.route(logits, bias, cfg.k)
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=cfg.E))
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, run_map, shared=1)


def test_fused_shared_expert_decode_shapes():
    # the decode layer (H = 7168, I = 2048, 256 experts, top-6) plus one shared expert
    cfg = synthetic.CONFIGS[1]
    W = _shared_weights(cfg, 1)
    hidden, logits, bias = synthetic.make_activations(cfg)
    run = gpu_util.Run(cfg, W, cap=cfg.T, shared=1)
    res = run.forward(hidden, logits, bias)
    run.close()
    assert res["status"] == 0
    gpu_util.check_against_oracle(cfg, res, hidden, logits, bias, W, None, gpu_util.sample_tokens(cfg.T, 16), shared=1)


@pytest.mark.parametrize("H,I,T,E,k", [(512, 256, 1500, 12, 4), (512, 512, 1100, 8, 2), (768, 256, 600, 16, 3),
                                       (384, 256, 1100, 8, 2)])
def test_two_sm_gemm_matches_one_cta_gemm(H, I, T, E, k):
    # The large-input GEMM runs on CTA pairs (one 2-SM MMA over two token
    # tiles of an expert) when H is a multiple of 256; MM_GEMM_2SM=0 runs the
    # one-CTA kernel.  Experts with an odd number of tiles leave the second
    # CTA of their last pair without a tile.  Both kernels must give identical
    # intermediates and outputs (each row's MMAs and epilogue are the same),
    # and match the oracle.  H = 384 takes the one-CTA kernel either way.
    import dataclasses
    import os
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, H=H, I=I, E=E, P=E, k=k)
    hidden, logits, bias = synthetic.make_activations(cfg)
    logits[:, 0] += 3.0                 # one hot expert: many tiles
    W = synthetic.make_all_weights(cfg)
    res = {}
    for two_sm in ("1", "0"):
        os.environ["MM_GEMM_2SM"] = two_sm
        try:
            run = gpu_util.Run(cfg, W, cap=cfg.T)
        finally:
            del os.environ["MM_GEMM_2SM"]
        run.op.set_route(2)
        res[two_sm] = run.forward(hidden, logits, bias)
        run.close()
        assert res[two_sm]["status"] == 0
    tiles = res["1"]["tiles"].reshape(-1, 3)
    per_expert = np.bincount(tiles[:, 0], minlength=cfg.P)
    assert (per_expert >= 2).any()
    if T != 1500:
        assert (per_expert % 2 == 1).any()          # an expert with an odd number of tiles
    for name in ("hq", "hs", "y", "out"):
        assert np.array_equal(res["1"][name], res["0"][name]), name
    gpu_util.check_against_oracle(cfg, res["1"], hidden, logits, bias, W, None, gpu_util.tile_edge_tokens(res["1"], T))


@pytest.mark.parametrize("T,kind", [(1024, 2), (400, 1)])
def test_gemm_kernel_chosen_per_batch(T, kind):
    # By default both large-input GEMM kernels are launched and the tile scan
    # picks one per batch on the device: the pair kernel when the experts' odd
    # tile counts add at most 1/64 to its MMA work.  Token t goes to experts
    # t % 8 and (t + 1) % 8: at T = 1024 every expert has two full tiles (the
    # pairs are chosen), at T = 400 every expert has one tile of 100 rows (the
    # one-CTA kernel is).  The default run equals the fixed choice bit for bit.
    import dataclasses
    import os
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, H=512, I=256, E=8, P=8, k=2)
    hidden, _, _ = synthetic.make_activations(cfg)
    logits = np.full((T, cfg.E), -8.0, np.float32)
    t = np.arange(T)
    logits[t, t % 8] = 6.0
    logits[t, (t + 1) % 8] = 5.0
    bias = np.zeros(cfg.E, np.float32)
    W = synthetic.make_all_weights(cfg)
    res = {}
    for mode in (None, str(kind - 1)):
        if mode is not None:
            os.environ["MM_GEMM_2SM"] = mode
        try:
            run = gpu_util.Run(cfg, W, cap=T)
        finally:
            os.environ.pop("MM_GEMM_2SM", None)
        run.op.set_route(2)
        res[mode] = run.forward(hidden, logits, bias)
        info = run.op.debug_dump(10)
        run.close()
        assert res[mode]["status"] == 0
        assert int(info[3]) == kind
        assert int(info[1]) == (8 if mode is None else 7)      # the default launches both kernels
    per_expert = np.bincount(res[None]["tiles"].reshape(-1, 3)[:, 0], minlength=cfg.P)
    assert np.all(per_expert == (2 if kind == 2 else 1))
    for name in ("hq", "hs", "y", "out"):
        assert np.array_equal(res[None][name], res[str(kind - 1)][name]), name
    gpu_util.check_against_oracle(cfg, res[None], hidden, logits, bias, W, None, gpu_util.tile_edge_tokens(res[None], T))
