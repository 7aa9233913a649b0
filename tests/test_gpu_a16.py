"""Parity of the a16w4 variant (bf16 activations x MXFP4 experts) with the
oracle's bf16 variant, and its behaviour at the C ABI.

Bit-exact: routing, physical experts, recorded counts, segment offsets,
dispatch order and the dispatched bf16 rows.  h in bf16: every element within
one bf16 step of the oracle's, >= 99.5% identical.  GEMM2 + combine fed with
the GPU's h: within bf16 rounding.  Layer output: relative L2 <= 4e-3 and
every |err| within 2^-7 (|out| + sum_j |w_j y_j|) + 0.01 rms(out).
"""
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


def _run(cfg, hidden, logits, bias, W, sample=None, recording=False, tiles=False):
    import moe_layer_serving_gb300 as mm
    run = gpu_util.Run(cfg, W, cap=hidden.shape[0], act=mm.ACT_BF16)
    run.op.set_recording(recording)
    res = run.forward(hidden, logits, bias)
    info = run.op.last_info()
    if recording:
        idx, _ = oracle.route(logits, bias, cfg.k)
        assert np.array_equal(run.op.read_counts(0), np.bincount(idx.ravel(), minlength=cfg.E)), "counts differ"
    run_map = run.map
    run.close()
    assert res["status"] == 0
    assert info[:2] == (2, 7)
    sel = None if sample is None else gpu_util.sample_tokens(hidden.shape[0], sample)
    if tiles:
        # the first and the last row of every token tile, end to end
        sel = gpu_util.tile_edge_tokens(res, hidden.shape[0])
    rel, _ = gpu_util.check_against_oracle_a16(cfg, res, hidden, logits, bias, W, run_map, sel)
    return res, rel


def _cfg(cid, T=None, sample=None, tiles=False):
    cfg = synthetic.CONFIGS[cid]
    hidden, logits, bias = synthetic.make_activations(cfg, T)
    W = gpu_util.weights(cfg)
    return _run(cfg, hidden, logits, bias, W, sample, cfg.recording, tiles)


def test_tiny_all_tokens(torch):
    _cfg(0)


@pytest.mark.parametrize("T", [1, 5, 37, 300])
def test_ragged_token_counts(torch, T):
    _cfg(0, T=T)


def test_ragged_hidden_and_odd_shapes(torch):
    # H = 384: the last GEMM2 unit is the first member of a W2 pair whose
    # second member is absent; I = 256: four GEMM1 units per tile
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=37, H=384, I=256, E=6, P=6, k=3)
    hidden, logits, bias = synthetic.make_activations(cfg)
    _run(cfg, hidden, logits, bias, synthetic.make_all_weights(cfg))


def test_many_tiles_per_expert(torch):
    # every token prefers the same 8 experts: 4 full 128-row tiles each
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=512, H=256, I=256, E=64, P=64, k=8)
    hidden, logits, bias = synthetic.make_activations(cfg)
    logits[:, :8] += 20.0
    res, _ = _run(cfg, hidden, logits, bias, synthetic.make_all_weights(cfg), sample=40)
    assert np.all(np.sort(res["idx"], axis=1) == np.arange(8))


def test_decode_t64(torch):
    _cfg(1)                 # every token of the decode batch


def test_eplb_t512(torch):
    _cfg(2, sample=24)


def test_prefill_t8192(torch):
    _cfg(3, tiles=True)             # every token tile of the layer


def test_skewed_eplb_t16384(torch):
    # skewed routing with 64 redundant replicas and the recorder on
    _cfg(4, tiles=True)


def test_format_switch_and_route_rules(torch):
    import moe_layer_serving_gb300 as mm
    cfg = synthetic.CONFIGS[0]
    hidden, logits, bias = synthetic.make_activations(cfg)
    W = gpu_util.weights(cfg)
    run = gpu_util.Run(cfg, W, cap=cfg.T)
    a8 = run.forward(hidden, logits, bias)["out"]
    x, lg, b = run.to_dev(hidden, logits, bias)
    out = torch.empty_like(x)
    lib, h = mm.lib(), run.op.handle
    assert lib.mm_set_activation_format(h, 7) == mm.MM_ERR_INVALID_ARG
    run.op.set_activation_format(mm.ACT_BF16)
    # the format change dropped the workspace
    assert lib.mm_forward(h, x.data_ptr(), lg.data_ptr(), b.data_ptr(), out.data_ptr(), cfg.T, None) == \
        mm.MM_ERR_CAPACITY
    run.op.reserve(cfg.T)
    run.act = mm.ACT_BF16
    a16 = run.forward(hidden, logits, bias)
    assert a16["status"] == 0
    ref = oracle.forward(hidden, logits, bias, cfg.k, W, act="bf16")
    gpu_util.assert_out_close_a16(a16["out"], ref["out"], mag=gpu_util.pair_magnitude(ref, cfg.k))
    # stages 6 and 8 (activation scales) are empty in the bf16 format; 5 and 7 hold bf16 rows
    rows = int(a16["offsets"][-1])
    assert C_size(lib, h, 6) == 0 and C_size(lib, h, 8) == 0
    assert C_size(lib, h, 5) == rows * cfg.H * 2 and C_size(lib, h, 7) == rows * cfg.I * 2
    run.op.set_route(mm.ROUTE_SMALL)
    assert lib.mm_forward(h, x.data_ptr(), lg.data_ptr(), b.data_ptr(), out.data_ptr(), cfg.T, None) == \
        mm.MM_ERR_UNSUPPORTED
    run.op.set_route(mm.ROUTE_AUTO)
    run.op.set_activation_format(mm.ACT_MXFP8)
    run.op.reserve(cfg.T)
    run.act = mm.ACT_MXFP8
    again = run.forward(hidden, logits, bias)
    run.close()
    assert np.array_equal(again["out"], a8)           # back to a8w4: the same bits as before


def C_size(lib, h, stage):
    import ctypes as C
    n = C.c_size_t(0)
    assert lib.mm_debug_size(h, stage, C.byref(n)) == 0
    return n.value


def test_graph_capture_replay_matches_eager(torch):
    import moe_layer_serving_gb300 as mm
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=96)
    hidden, logits, bias = synthetic.make_activations(cfg)
    W = gpu_util.weights(cfg)
    run = gpu_util.Run(cfg, W, cap=cfg.T, act=mm.ACT_BF16)
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
    assert run.op.get_status() == 0
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
    run.close()


@pytest.mark.parametrize("T", [40, 1100])
def test_fused_shared_expert(torch, T):
    import moe_layer_serving_gb300 as mm
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T)
    wide = dataclasses.replace(cfg, E=cfg.E + 1, P=cfg.P + 1)
    W = synthetic.make_all_weights(wide)
    hidden, logits, bias = synthetic.make_activations(cfg)
    run = gpu_util.Run(cfg, W, cap=T, act=mm.ACT_BF16, shared=1)
    res = run.forward(hidden, logits, bias)
    run.close()
    assert res["status"] == 0
    assert np.all(res["idx"][:, cfg.k] == cfg.E) and np.all(res["weights"][:, cfg.k] == 1.0)
    gpu_util.check_against_oracle_a16(cfg, res, hidden, logits, bias, W, None, shared=1)
