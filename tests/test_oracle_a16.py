"""Pins of the oracle's a16w4 variant (bf16 activations x MXFP4 experts).

Anchors: hand-derived worked examples, the E=1/k=1 reduction to a dense
SwiGLU MLP on bf16 inputs computed with torch fp64 matmuls, a dense numpy
einsum formulation over all experts on tiny shapes, exact agreement with the
(separately pinned) a8w4 GEMM1 when the activations are exactly MXFP8
values, the nibble order of the packed weights, and replica invariance.
"""
import dataclasses

import numpy as np
import torch

import oracle
import synthetic
from tests import helpers


def _const_weights(E, H, I, nib):
    """every element = the e2m1 value of nib, scale byte 127 (x 1)"""
    b = np.uint8(nib | (nib << 4))
    return (np.full((E, 2 * I, H // 2), b, np.uint8), np.full((E, 2 * I, H // 32), 127, np.uint8),
            np.full((E, H, I // 2), b, np.uint8), np.full((E, H, I // 32), 127, np.uint8))


def test_worked_example_all_ones():
    # x = 1, W1 = W2 = 1 (e2m1 code 2), one expert, top-1, H = I = 32:
    # G = 32 for gate and up; h = 32 / (1 + e^-32) * 32 = 1024.0 in fp32, bf16 0x4480;
    # y = sum_i 1024 * 1 = 32768; w = 1; out = bf16(32768) = 0x4700.
    H, I = 32, 32
    x = np.full((2, H), 0x3F80, np.uint16)
    r = oracle.forward(x, np.zeros((2, 1), np.float32), None, 1, _const_weights(1, H, I, 2), act="bf16")
    assert np.all(r["h"] == 1024.0) and np.all(r["hb"] == 0x4480)
    assert np.all(r["y"] == 32768.0)
    assert np.all(r["out"] == 0x4700)


def test_worked_example_h_is_rounded_to_bf16():
    # x = 1 in the first 3 positions only, W1 = W2 = 1: gate = up = 3, so
    # h = 3 * 3 / (1 + e^-3) = 8.573167...; in bf16 (8 significant bits) that is
    # 8.5625 (0x4109: 8.5625 = 1.0001001b * 2^3, the next value up is 8.625).
    # y = I * 8.5625 = 274.0 exactly; out = bf16(274) = 0x4389.
    H, I = 32, 32
    x = np.zeros((1, H), np.uint16)
    x[0, :3] = 0x3F80
    r = oracle.forward(x, np.zeros((1, 1), np.float32), None, 1, _const_weights(1, H, I, 2), act="bf16")
    assert abs(float(r["h"][0, 0]) - 8.573167) < 1e-5
    assert np.all(r["hb"] == 0x4109)
    assert np.all(r["y"] == 274.0)
    assert np.all(r["out"] == 0x4389)


def test_nibble_order_low_is_even_element():
    H, I = 32, 32
    W = list(_const_weights(1, H, I, 0))
    W[0][0, 0, 0] = 0x20                      # high nibble = element 1 = 1.0 (gate row 0)
    W[0][0, I, 0] = 0x20                      # up row 0 too
    x = np.zeros((1, H), np.float32)
    x[0, 1] = 2.0
    x[0, 0] = 1.0
    r = oracle.forward(helpers.bf16_bits(x), np.zeros((1, 1), np.float32), None, 1, tuple(W), want_g=True,
                       act="bf16")
    assert r["g"][0, 0] == 2.0 and r["g"][0, I] == 2.0
    assert np.all(r["g"][0, 1:I] == 0)


def test_zero_input_gives_exact_zero():
    cfg = synthetic.CONFIGS[0]
    _, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    x = np.zeros((cfg.T, cfg.H), np.uint16)
    r = oracle.forward(x, logits, bias, cfg.k, W, act="bf16")
    assert np.all(r["out"] == 0)


def test_single_expert_is_dense_swiglu_mlp_on_bf16(e2m1_table):
    cfg = dataclasses.replace(synthetic.CONFIGS[0], E=1, P=1, k=1)
    T, H, I = 12, cfg.H, cfg.I
    rng = np.random.default_rng(7)
    x = helpers.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    W = synthetic.make_all_weights(cfg)
    r = oracle.forward(x, np.zeros((T, 1), np.float32), None, 1, W, want_g=True, act="bf16")
    w1 = torch.from_numpy(helpers.deq_mxfp4(W[0][0], W[1][0], e2m1_table))
    w2 = torch.from_numpy(helpers.deq_mxfp4(W[2][0], W[3][0], e2m1_table))
    a = torch.from_numpy(helpers.bf16_to_f64(x))
    G = (a @ w1.T).to(torch.float32)
    assert torch.allclose(torch.from_numpy(r["g"]), G, rtol=2 ** -22, atol=0)
    G = torch.from_numpy(r["g"]).double()
    h = (torch.nn.functional.silu(G[:, :I]) * G[:, I:]).to(torch.float32)
    assert torch.allclose(torch.from_numpy(r["h"]), h, rtol=2 ** -22, atol=1e-30)
    hb = helpers.bf16_bits(r["h"])
    assert np.array_equal(hb, r["hb"])
    y = (torch.from_numpy(helpers.bf16_to_f64(hb)) @ w2.T).to(torch.float32)
    assert torch.allclose(torch.from_numpy(r["y"]), y, rtol=2 ** -22, atol=0)
    assert np.array_equal(helpers.bf16_bits(r["y"]), r["out"])      # w = 1: out = bf16(y)


def test_bruteforce_dense_formulation_tiny(e2m1_table):
    E, P, k, T, H, I = 4, 4, 2, 6, 64, 64
    cfg = dataclasses.replace(synthetic.CONFIGS[0], T=T, H=H, I=I, E=E, P=P, k=k)
    x, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    r = oracle.forward(x, logits, bias, k, W, want_g=True, act="bf16")
    w1 = np.stack([helpers.deq_mxfp4(W[0][p], W[1][p], e2m1_table) for p in range(P)])
    w2 = np.stack([helpers.deq_mxfp4(W[2][p], W[3][p], e2m1_table) for p in range(P)])
    a = helpers.bf16_to_f64(x)
    G_all = np.einsum("th,pnh->tpn", a, w1).astype(np.float32)        # every token x expert
    out = np.zeros((T, H))
    for t in range(T):
        for j in range(k):
            p = r["phys"][t, j]
            g = G_all[t, p].astype(np.float64)
            assert np.allclose(g, r["g"][t * k + j], rtol=2 ** -22, atol=0)
            h = (g[:I] / (1 + np.exp(-g[:I])) * g[I:]).astype(np.float32)
            hb = helpers.bf16_to_f64(helpers.bf16_bits(h))
            y = (hb @ w2[p].T).astype(np.float32)
            out[t] += np.float64(r["w"][t, j]) * y
    ref = helpers.bf16_to_f64(helpers.bf16_bits(out.astype(np.float32)))
    got = helpers.bf16_to_f64(r["out"])
    assert np.all(np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-30)


def test_gemm1_equals_a8w4_when_activations_are_mxfp8_values():
    # x built from e4m3 codes and one power-of-two scale per 32 values: MXFP8
    # quantisation reproduces it exactly, so both variants sum the same products
    # in the same order and GEMM1 agrees bit for bit.
    cfg = dataclasses.replace(synthetic.CONFIGS[0], E=1, P=1, k=1)
    T, H = 5, cfg.H
    rng = np.random.default_rng(11)
    codes = rng.integers(0, 0x7F, (T, H)).astype(np.uint8) | (rng.integers(0, 2, (T, H)).astype(np.uint8) << 7)
    codes[(codes & 0x7F) == 0x7F] = 0x30                  # no NaN codes
    codes[:, ::32] = 0x7E                                 # every block reaches 448: its scale is 2^X exactly
    X = rng.integers(-12, -4, (T, H // 32))
    v = helpers.e4m3_to_f64(codes) * np.repeat(2.0 ** X, 32, axis=1)
    x = helpers.bf16_bits(v.astype(np.float32))
    assert np.array_equal(helpers.bf16_to_f64(x), v)       # e4m3 x 2^X is exact in bf16
    W = synthetic.make_all_weights(cfg)
    a16 = oracle.forward(x, np.zeros((T, 1), np.float32), None, 1, W, want_g=True, act="bf16")
    a8 = oracle.forward(x, np.zeros((T, 1), np.float32), None, 1, W, want_g=True)
    assert np.array_equal(helpers.deq_mxfp8(a8["xq"], a8["xs"]), v)
    assert np.array_equal(a16["g"], a8["g"])
    assert np.array_equal(a16["h"], a8["h"])


def test_replica_invariance():
    cfg = dataclasses.replace(synthetic.CONFIGS[0], P=12)
    x, logits, bias = synthetic.make_activations(cfg)
    Wl = synthetic.make_all_weights(cfg, physical=False)
    Wp = synthetic.make_all_weights(cfg, physical=True)
    m, rc, R = synthetic.make_eplb_map(cfg)
    a = oracle.forward(x, logits, bias, cfg.k, Wl, act="bf16")
    b = oracle.forward(x, logits, bias, cfg.k, Wp, m, rc, act="bf16")
    assert np.any(b["phys"] >= cfg.E)
    assert np.array_equal(a["out"], b["out"])


def test_token_subset_matches_full_forward():
    cfg = synthetic.CONFIGS[0]
    x, logits, bias = synthetic.make_activations(cfg)
    W = synthetic.make_all_weights(cfg)
    full = oracle.forward(x, logits, bias, cfg.k, W, act="bf16")
    sel = np.array([3, 7, 11])
    sub = oracle.forward(x[sel], logits[sel], bias, cfg.k, W, token_ids=sel, act="bf16")
    assert np.array_equal(sub["out"], full["out"][sel])
