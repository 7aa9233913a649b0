"""Pins of the oracle's element formats, quantiser and routing score.

Each check compares the oracle with something other than itself: torch's
float8_e4m3fn codec, the OCP e2m1 table, libm's exp in double, closed-form
scale rules, or a full sort.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import helpers

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def test_e2m1_values_match_ocp_table(e2m1_table):
    got = oracle.e2m1_value(np.arange(16))
    assert np.array_equal(got, np.array(e2m1_table))
    assert np.array_equal(np.signbit(got), np.signbit(np.array(e2m1_table)))


def test_e8m0_values_closed_form():
    got = oracle.e8m0_value(np.arange(256))
    assert np.isnan(got[255])
    assert np.array_equal(got[:255], [math.ldexp(1.0, c - 127) for c in range(255)])


def test_e4m3_decode_all_codes_vs_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = helpers.e4m3_to_f64(codes)
    got = oracle.e4m3_value(codes)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], got[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(got[ok]))


def _e4m3_finite_values():
    v = helpers.e4m3_to_f64(np.arange(128, dtype=np.uint8))
    return np.unique(v[~np.isnan(v)])       # 0 .. 448, ascending


def test_e4m3_encode_vs_torch_cast():
    pos = _e4m3_finite_values()
    mids = (pos[:-1] + pos[1:]) / 2           # every tie, exact in binary32
    rng = np.random.default_rng(1)
    rand = np.ldexp(rng.uniform(1, 2, 4000), rng.integers(-14, 9, 4000))
    rand = rand.astype(np.float32).astype(np.float64)
    rand = rand[rand <= 448]
    vals = np.concatenate([pos, mids, rand, -pos[1:], -mids, -rand])
    ref = helpers.f64_to_e4m3_sat(vals)
    got = oracle.e4m3_encode(vals)
    assert np.array_equal(ref, got)


def test_e4m3_encode_saturates_and_keeps_zero_sign():
    assert list(oracle.e4m3_encode([448.0, 449.0, 464.0, 479.9, 480.0, 1e6])) == [0x7E] * 6
    assert list(oracle.e4m3_encode([-449.0, -1e30])) == [0xFE] * 2
    assert list(oracle.e4m3_encode([0.0, -0.0])) == [0x00, 0x80]
    # below half of the smallest subnormal (2^-9) rounds to zero, the half itself to even (zero)
    assert list(oracle.e4m3_encode([2.0 ** -11, 2.0 ** -10, -2.0 ** -10, 2.0 ** -10 * 1.0001])) == [0, 0, 0x80, 1]


def test_e4m3_decode_encode_roundtrip():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(oracle.e4m3_encode(oracle.e4m3_value(codes)), codes)


def _all_finite_bf16():
    bits = np.arange(65536, dtype=np.uint32)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF].astype(np.uint16)
    return bits


def test_mxfp8_quant_exhaustive_bf16_single_value_blocks():
    bits = _all_finite_bf16()
    vals = helpers.bf16_to_f64(bits)
    n = vals.size
    blocks = np.zeros((n, 32))
    blocks[np.arange(n), np.arange(n) % 32] = vals
    q, s = oracle.mxfp8_quant(blocks.reshape(-1, 32).astype(np.float32))
    rq, rs = helpers.quant_mxfp8(blocks)
    assert np.array_equal(s[:, 0], rs[:, 0])
    assert np.array_equal(q, rq)
    # the largest element always lands in [256, 448] after scaling (unless clamped)
    nz = vals != 0
    top = q[np.arange(n), np.arange(n) % 32][nz]
    scaled = np.abs(helpers.e4m3_to_f64(top))
    X = s[nz, 0].astype(int) - 127
    unclamped = X > -127
    assert np.all((scaled[unclamped] >= 256) & (scaled[unclamped] <= 448))


def test_mxfp8_quant_exhaustive_bf16_mixed_blocks():
    bits = _all_finite_bf16()
    rng = np.random.default_rng(2)
    bits = rng.permutation(bits)
    bits = bits[: bits.size // 32 * 32].reshape(-1, 32)
    vals = helpers.bf16_to_f64(bits)
    q, s = oracle.mxfp8_quant_bf16(bits)
    rq, rs = helpers.quant_mxfp8(vals)
    assert np.array_equal(s[:, 0], rs[:, 0])
    assert np.array_equal(q, rq)


def test_mxfp8_quant_error_bound_and_pow2_invariance():
    rng = np.random.default_rng(3)
    v = rng.standard_normal((256, 64)).astype(np.float32)
    q, s = oracle.mxfp8_quant(v)
    deq = helpers.deq_mxfp8(q, s)
    X = np.repeat(s.astype(int) - 127, 32, axis=1)
    sat = np.abs(v.astype(np.float64)) * np.ldexp(1.0, -X) > 448
    ev = np.frexp(np.abs(v.astype(np.float64)))[1] - 1
    bound = np.maximum(np.ldexp(1.0, ev - 4), np.ldexp(1.0, X - 10))
    err = np.abs(deq - v)
    assert np.all(err[~sat] <= bound[~sat])
    assert np.all(err[sat] <= np.abs(v[sat]) - 448 * np.ldexp(1.0, X[sat]) + 1e-30)
    for m in (-20, -3, 5, 30):
        q2, s2 = oracle.mxfp8_quant((v * np.float32(2.0 ** m)).astype(np.float32))
        assert np.array_equal(q2, q)
        assert np.array_equal(s2.astype(int), s.astype(int) + m)


def test_mxfp8_zero_block():
    q, s = oracle.mxfp8_quant(np.zeros((2, 64), np.float32))
    assert not q.any() and not s.any()
    v = np.zeros((1, 32), np.float32)
    v[0, 3] = -0.0
    q, s = oracle.mxfp8_quant(v)
    assert not q.any() and s[0, 0] == 0


# ---- routing score ---------------------------------------------------------
def _ulp_err(got, ref):
    """|got - ref| in units of the binary32 ulp of ref's binade."""
    e = np.frexp(np.abs(ref))[1] - 1
    ulp = np.ldexp(1.0, np.maximum(e - 23, -149))
    return np.abs(got.astype(np.float64) - ref) / ulp


def _sweep(lo, hi, stride):
    a = np.float32(lo).view(np.uint32)
    b = np.float32(hi).view(np.uint32)
    lo_b, hi_b = min(a, b), max(a, b)
    return np.arange(lo_b, hi_b, stride, dtype=np.uint32).view(np.float32)


@pytest.mark.parametrize("lo,hi", [(-87.0, -1e-30), (1e-30, 88.0)])
def test_exp_spec_within_2ulp_of_libm(lo, hi):
    y = _sweep(lo, hi, 211)
    got = oracle.exp_spec(y)
    ref = np.exp(y.astype(np.float64))
    assert _ulp_err(got, ref).max() <= 2.0


@pytest.mark.parametrize("lo,hi", [(-80.0, -1e-30), (1e-30, 80.0)])
def test_sigmoid_spec_within_3ulp_and_monotone(lo, hi):
    x = _sweep(lo, hi, 211)
    x = np.sort(x)
    got = oracle.sigmoid_spec(x)
    ref = 1.0 / (1.0 + np.exp(-x.astype(np.float64)))
    assert _ulp_err(got, ref).max() <= 3.0
    assert np.all(np.diff(got) >= 0)


def test_sigmoid_spec_special_values():
    got = oracle.sigmoid_spec(np.array([0.0, -0.0, 100.0, 1e30, -1e30], np.float32))
    assert got[0] == 0.5 and got[1] == 0.5
    assert got[2] == 1.0 and got[3] == 1.0
    assert 0.0 < got[4] < 1e-37


@pytest.mark.slow
def test_exp_spec_exhaustive_c_sweep():
    L = oracle.lib()
    assert L.orc_exp_spec_max_ulp(-87.0, -1e-38, 1, 0) <= 2.0
    assert L.orc_exp_spec_max_ulp(1e-38, 88.0, 1, 0) <= 2.0


# ---- top-k -----------------------------------------------------------------
@pytest.mark.parametrize("T,E,k,with_bias", [(64, 8, 2, False), (200, 256, 6, True),
                                             (50, 512, 8, True), (30, 16, 1, True),
                                             (20, 8, 8, False)])
def test_topk_matches_full_sort(T, E, k, with_bias):
    rng = np.random.default_rng(T * 1000 + E)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[::3, 1::2] = logits[::3, 0:E - 1:2]          # equal scores -> ties
    bias = (0.1 * rng.standard_normal(E)).astype(np.float32) if with_bias else None
    idx, w = oracle.route(logits, bias, k)
    s = oracle.sigmoid_spec(logits)
    key = s + (bias if bias is not None else np.float32(0))
    assert key.dtype == np.float32
    e = np.broadcast_to(np.arange(E), (T, E))
    ref = np.array([np.lexsort((e[t], -key[t])) for t in range(T)])[:, :k]
    assert np.array_equal(idx, ref)


def test_topk_tie_prefers_lower_expert():
    logits = np.zeros((1, 6), np.float32)
    logits[0, [1, 4]] = 2.0
    idx, _ = oracle.route(logits, None, 3)
    assert idx.tolist() == [[1, 4, 0]]


def test_route_weights_normalised():
    rng = np.random.default_rng(5)
    for k in (1, 2, 6, 8):
        logits = rng.standard_normal((300, 64)).astype(np.float32)
        idx, w = oracle.route(logits, None, k)
        if k == 1:
            assert np.all(w == 1.0)
        assert np.all(np.abs(w.astype(np.float64).sum(1) - 1.0) <= k * 2.0 ** -23)
        assert np.all(np.diff(w, axis=1) <= 0)         # no bias: score order = key order


def test_route_weights_use_unbiased_scores():
    # Reading: the selection uses s + bias, the weights normalise s alone.  A
    # large bias flips the selection order but must not leak into the weights.
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((100, 32)).astype(np.float32)
    bias = np.where(np.arange(32) % 2 == 0, 0.5, -0.5).astype(np.float32)
    idx, w = oracle.route(logits, bias, 4)
    s = np.take_along_axis(oracle.sigmoid_spec(logits), idx, axis=1).astype(np.float64)
    assert np.allclose(w, s / s.sum(1, keepdims=True), rtol=4 * 2.0 ** -24, atol=0)
    assert np.all(idx % 2 == 0)                # the bias decided the selection
