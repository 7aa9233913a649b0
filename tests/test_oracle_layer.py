"""Pins of the oracle's layer stages: EPLB remap and recording, permute,
GEMM1/SwiGLU/requant, GEMM2 and combine.

Anchors: hand-derived worked examples, the E=1/k=1 reduction to a dense
SwiGLU MLP computed with torch fp64 matmuls, a second (dense numpy einsum)
formulation on tiny shapes, replica invariance, invariants of the permute
and of the counts, and the skew the workload recipe asks for.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests import helpers


# ---- EPLB remap and recording ---------------------------------------------
def test_eplb_identity_map_is_identity():
    rng = np.random.default_rng(0)
    idx = rng.integers(0, 16, (40, 3)).astype(np.int32)
    phys = oracle.eplb(idx, np.arange(16, dtype=np.int32)[:, None], np.ones(16, np.int32))
    assert np.array_equal(phys, idx)


def test_eplb_replica_rule_worked_example():
    # logical 0 -> {0, 3}, logical 1 -> {1}, logical 2 -> {2, 4}
    m = np.array([[0, 3], [1, -1], [2, 4]], np.int32)
    rc = np.array([2, 1, 2], np.int32)
    idx = np.array([[0, 2], [0, 1], [2, 0]], np.int32)
    # slot = (t + j) mod rc: t0: e0 s0 -> 0, e2 s1 -> 4; t1: e0 s1 -> 3, e1 -> 1;
    # t2: e2 s0 -> 2, e0 s1 -> 3
    assert oracle.eplb(idx, m, rc).tolist() == [[0, 4], [3, 1], [2, 3]]
    # the same tokens at positions 5, 6, 7 of their forward call
    assert oracle.eplb(idx, m, rc, token_ids=[5, 6, 7]).tolist() == [[3, 2], [0, 1], [4, 0]]


def test_eplb_replicas_share_load_evenly():
    m = np.array([[0, 1]], np.int32)
    idx = np.zeros((1000, 1), np.int32)
    phys = oracle.eplb(idx, m, np.array([2], np.int32))
    assert np.bincount(phys.ravel()).tolist() == [500, 500]


def test_counts_are_histogram_and_accumulate():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((100, 32)).astype(np.float32)
    idx, _ = oracle.route(logits, None, 4)
    c = oracle.record(idx, 32)
    assert c.sum() == 100 * 4
    assert np.array_equal(c, np.bincount(idx.ravel(), minlength=32))
    oracle.record(idx, 32, c)
    assert np.array_equal(c, 2 * np.bincount(idx.ravel(), minlength=32))


# ---- permute ---------------------------------------------------------------
@pytest.mark.parametrize("n,P", [(1, 4), (384, 256), (3072, 320), (5000, 7)])
def test_permute_is_stable_bijection(n, P):
    rng = np.random.default_rng(n)
    phys = rng.integers(0, P, n).astype(np.int32)
    off, order, pos = oracle.permute(phys, P)
    assert np.array_equal(np.sort(order), np.arange(n))
    assert np.array_equal(order[pos], np.arange(n))
    assert np.array_equal(np.diff(off), np.bincount(phys, minlength=P))
    assert off[0] == 0 and off[-1] == n
    for p in range(P):
        seg = order[off[p]:off[p + 1]]
        assert np.all(phys[seg] == p) and np.all(np.diff(seg) > 0)


# ---- worked examples (hand-derived) ---------------------------------------
def _const_weights(E, H, I, nib):
    """every element = the e2m1 value of nib, scale byte 127 (x 1)"""
    b = np.uint8(nib | (nib << 4))
    return (np.full((E, 2 * I, H // 2), b, np.uint8), np.full((E, 2 * I, H // 32), 127, np.uint8),
            np.full((E, H, I // 2), b, np.uint8), np.full((E, H, I // 32), 127, np.uint8))


def test_worked_example_all_ones():
    # x = 1 everywhere, W1 = W2 = 1 (e2m1 code 2), one expert, top-1.
    # quant(x): amax 1 -> X = -8 -> scale byte 119, codes e4m3(256) = 0x78.
    # G = sum_h 1*1 = H = 32 for gate and up; h = 32/(1+e^-32) * 32 -> 1024.0 in fp32.
    # quant(h): amax 1024 -> X = 2 -> byte 129, codes e4m3(256) = 0x78.
    # y = sum_i 1024 * 1 = 32768; w = 1; out = bf16(32768) = 0x4700.
    H, I = 32, 32
    x = np.full((2, H), 0x3F80, np.uint16)
    r = oracle.forward(x, np.zeros((2, 1), np.float32), None, 1, _const_weights(1, H, I, 2))
    assert np.all(r["xs"] == 119) and np.all(r["xq"] == 0x78)
    assert np.all(r["h"] == 1024.0)
    assert np.all(r["hs"] == 129) and np.all(r["hq"] == 0x78)
    assert np.all(r["y"] == 32768.0)
    assert np.all(r["out"] == 0x4700)


def test_worked_example_two_experts_tie_and_combine():
    # E=2, top-2, equal logits: tie -> idx (0, 1), s = 0.5 each -> w = (0.5, 0.5).
    # Expert 0 as above gives y = 32768; expert 1 has W1 = W2 = -1 (code 0xA):
    # gate = up = -32, h = silu(-32) * -32 ~ 1.3e-11, y1 = -32 * h ~ -4e-10.
    # out = bf16(0.5 * 32768 + 0.5 * y1) = bf16(16384 - 2e-10) = 16384 = 0x4680.
    H, I = 32, 32
    w_pos = _const_weights(1, H, I, 2)
    w_neg = _const_weights(1, H, I, 0xA)
    W = tuple(np.concatenate([a, b]) for a, b in zip(w_pos, w_neg))
    x = np.full((1, H), 0x3F80, np.uint16)
    r = oracle.forward(x, np.zeros((1, 2), np.float32), None, 2, W)
    assert r["idx"].tolist() == [[0, 1]]
    assert r["w"].tolist() == [[0.5, 0.5]]
    assert np.all(r["y"][0] == 32768.0) and np.all((r["y"][1] < 0) & (r["y"][1] > -1e-9))
    assert np.all(r["out"] == 0x4680)


def test_nibble_order_low_is_even_element():
    # a single nonzero weight at odd position h = 1 must pick x[1]
    H, I = 32, 32
    W = list(_const_weights(1, H, I, 0))
    W[0][0, 0, 0] = 0x20                      # high nibble = element 1 = 1.0 (gate row 0)
    W[0][0, I, 0] = 0x20                      # up row 0 too
    x = np.zeros((1, H), np.float32)
    x[0, 1] = 2.0
    x[0, 0] = 1.0
    r = oracle.forward(helpers.bf16_bits(x), np.zeros((1, 1), np.float32), None, 1, tuple(W), want_g=True)
    assert r["g"][0, 0] == 2.0 and r["g"][0, I] == 2.0
    assert np.all(r["g"][0, 1:I] == 0)


def test_zero_input_gives_exact_zero():
    cfg = synthetic.CONFIGS[0]
    _, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    x = np.zeros((cfg.T, cfg.H), np.uint16)
    r = oracle.forward(x, logits, bias, cfg.k, W)
    assert np.all(r["out"] == 0)


# ---- E=1, k=1 reduces to a dense SwiGLU MLP ---------------------------------
def test_single_expert_is_dense_swiglu_mlp(e2m1_table):
    cfg = dataclasses.replace(synthetic.CONFIGS[0], E=1, P=1, k=1)
    T, H, I = 12, cfg.H, cfg.I
    rng = np.random.default_rng(7)
    x = helpers.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    W = synthetic.make_all_weights(cfg)
    r = oracle.forward(x, np.zeros((T, 1), np.float32), None, 1, W, want_g=True)
    w1 = torch.from_numpy(helpers.deq_mxfp4(W[0][0], W[1][0], e2m1_table))
    w2 = torch.from_numpy(helpers.deq_mxfp4(W[2][0], W[3][0], e2m1_table))
    xq, xs = helpers.quant_mxfp8(helpers.bf16_to_f64(x))
    assert np.array_equal(xq, r["xq"]) and np.array_equal(xs, r["xs"])
    a = torch.from_numpy(helpers.deq_mxfp8(xq, xs))
    G = (a @ w1.T).to(torch.float32)
    assert torch.allclose(torch.from_numpy(r["g"]), G, rtol=2 ** -22, atol=0)
    G = torch.from_numpy(r["g"]).double()
    h = (torch.nn.functional.silu(G[:, :I]) * G[:, I:]).to(torch.float32)
    assert torch.allclose(torch.from_numpy(r["h"]), h, rtol=2 ** -22, atol=1e-30)
    hq, hs = helpers.quant_mxfp8(r["h"].astype(np.float64))
    assert np.array_equal(hq, r["hq"]) and np.array_equal(hs, r["hs"])
    y = (torch.from_numpy(helpers.deq_mxfp8(hq, hs)) @ w2.T).to(torch.float32)
    assert torch.allclose(torch.from_numpy(r["y"]), y, rtol=2 ** -22, atol=0)
    out = helpers.bf16_bits(r["y"])          # w = 1: out = bf16(y)
    assert np.array_equal(out, r["out"])


# ---- second formulation: dense numpy einsum over all experts ----------------
def test_bruteforce_dense_formulation_tiny(e2m1_table):
    E, P, k, T, H, I = 4, 4, 2, 6, 64, 64
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, H=H, I=I, E=E, P=P, k=k)
    x, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    r = oracle.forward(x, logits, bias, k, W, want_g=True)
    w1 = np.stack([helpers.deq_mxfp4(W[0][p], W[1][p], e2m1_table) for p in range(P)])
    w2 = np.stack([helpers.deq_mxfp4(W[2][p], W[3][p], e2m1_table) for p in range(P)])
    a = helpers.deq_mxfp8(*helpers.quant_mxfp8(helpers.bf16_to_f64(x)))
    G_all = np.einsum("th,pnh->tpn", a, w1).astype(np.float32)        # every token x expert
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            p = r["phys"][t, j]
            g = G_all[t, p].astype(np.float64)
            assert np.allclose(g, r["g"][t * k + j], rtol=2 ** -22, atol=0)
            h = (g[:I] / (1 + np.exp(-g[:I])) * g[I:]).astype(np.float32)
            hq, hs = helpers.quant_mxfp8(h[None].astype(np.float64))
            y = (helpers.deq_mxfp8(hq, hs)[0] @ w2[p].T).astype(np.float32)
            out[t] += np.float64(r["w"][t, j]) * y
    ref = helpers.bf16_to_f64(helpers.bf16_bits(out.astype(np.float32)))
    got = helpers.bf16_to_f64(r["out"])
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


# ---- replicas are byte copies: EPLB does not change the result ------------
def test_replica_invariance():
    cfg = dataclasses.replace(synthetic.CONFIGS[0], P=12)
    x, logits, bias = synthetic.make_activations(cfg)
    Wl = synthetic.make_all_weights(cfg, physical=False)
    Wp = synthetic.make_all_weights(cfg, physical=True)
    m, rc, R = synthetic.make_eplb_map(cfg)
    a = oracle.forward(x, logits, bias, cfg.k, Wl)
    b = oracle.forward(x, logits, bias, cfg.k, Wp, m, rc)
    assert np.any(b["phys"] >= cfg.E)            # some pairs really went to replicas
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(a["idx"], b["idx"]) and np.array_equal(a["counts"], b["counts"])


def test_token_subset_matches_full_forward():
    cfg = dataclasses.replace(synthetic.CONFIGS[0], P=12)
    x, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    m, rc, R = synthetic.make_eplb_map(cfg)
    full = oracle.forward(x, logits, bias, cfg.k, W, m, rc)
    sel = np.array([3, 7, 8, 15])
    sub = oracle.forward(x[sel], logits[sel], bias, cfg.k, W, m, rc, token_ids=sel)
    assert np.array_equal(sub["out"], full["out"][sel])
    assert np.array_equal(sub["phys"], full["phys"][sel])


# ---- workload recipe -------------------------------------------------------
def test_skewed_workload_hot_expert_load():
    cfg = synthetic.CONFIGS[4]
    _, logits, bias = synthetic.make_activations(cfg)
    idx, _ = oracle.route(logits, bias, cfg.k)
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    assert counts.max() >= 8 * cfg.T * cfg.k / cfg.E


def test_zipf_workload_replicates_the_hottest_experts():
    cfg = synthetic.CONFIGS[2]
    _, logits, bias = synthetic.make_activations(cfg)
    idx, _ = oracle.route(logits, bias, cfg.k)
    counts = np.bincount(idx.ravel(), minlength=cfg.E)
    hot = set(np.argsort(-counts, kind="stable")[:64].tolist())
    assert len(hot & set(range(64))) >= 56        # replicas sit on the popular experts


# ---- fused shared experts ----------------------------------------------------
def _shared_case(ns=1, T=24):
    # E routed experts plus ns shared ones: the shared experts' weights are the
    # last ns of E + ns independently drawn experts
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, E=8, P=8, k=2)
    wide = dataclasses.replace(cfg, E=cfg.E + ns, P=cfg.P + ns)
    W = synthetic.make_all_weights(wide)
    hidden, logits, bias = synthetic.make_activations(cfg)
    return cfg, W, hidden, logits, bias


@pytest.mark.parametrize("act", ["mxfp8", "bf16"])
def test_shared_slots_leave_the_routed_part_alone(act):
    cfg, W, hidden, logits, bias = _shared_case(ns=2)
    base = oracle.forward(hidden, logits, bias, cfg.k, tuple(a[:cfg.P] for a in W), act=act)
    res = oracle.forward(hidden, logits, bias, cfg.k, W, act=act, shared=2)
    k = cfg.k
    assert np.array_equal(res["idx"][:, :k], base["idx"]) and np.array_equal(res["w"][:, :k], base["w"])
    assert np.array_equal(res["phys"][:, :k], base["phys"]) and np.array_equal(res["counts"], base["counts"])
    assert np.all(res["idx"][:, k:] == cfg.E + np.arange(2)) and np.all(res["w"][:, k:] == 1.0)
    assert np.all(res["phys"][:, k:] == cfg.P + np.arange(2))


def test_shared_expert_alone_is_its_dense_ffn():
    # routed down projections all zero: every routed y is exactly 0, so the
    # layer output is the shared expert's own output for each token, computed
    # here per token straight from the expert FFN (no permute, no combine)
    cfg, W, hidden, logits, bias = _shared_case(ns=1)
    w1, w1s, w2, w2s = (a.copy() for a in W)
    w2[:cfg.P] = 0
    res = oracle.forward(hidden, logits, bias, cfg.k, (w1, w1s, w2, w2s), shared=1)
    xq, xs = oracle.mxfp8_quant_bf16(hidden)
    y = oracle.expert_ffn(xq, xs, w1[cfg.P], w1s[cfg.P], w2[cfg.P], w2s[cfg.P])["y"]
    assert np.any(y != 0)
    assert np.array_equal(res["out"], synthetic.bf16_bits_from_f32(y))


def test_shared_expert_alone_is_its_dense_ffn_a16():
    cfg, W, hidden, logits, bias = _shared_case(ns=1)
    w1, w1s, w2, w2s = (a.copy() for a in W)
    w2[:cfg.P] = 0
    res = oracle.forward(hidden, logits, bias, cfg.k, (w1, w1s, w2, w2s), act="bf16", shared=1)
    y = oracle.expert_ffn_a16(hidden, w1[cfg.P], w1s[cfg.P], w2[cfg.P], w2s[cfg.P])["y"]
    assert np.any(y != 0)
    assert np.array_equal(res["out"], synthetic.bf16_bits_from_f32(y))
