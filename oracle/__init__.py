"""CPU oracle for the fused MoE layer forward (a8w4, and the a16w4 variant) --
TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (``moe_layer_serving_gb300``)
never imports it and shares no code with it; the two meet only in the seeded
input generator (``synthetic``).

The arithmetic lives in ``oracle.c`` (plain C, fp64 accumulation, one
function per stage).  This module marshals numpy arrays into it and composes
the stages in the order the pages give for the fused operator: route, fused
EPLB remap + record, quant, dispatch (permute), GEMM1 (+SwiGLU, requant),
GEMM2, combine ("sglang PR #47065", Title/switches; "sglang PR #35619",
Summary).  Parity of every function here is pinned by ``tests/test_oracle_*``
against closed forms, library routines, invariants and brute force.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = C.CDLL(path)
        f32, f64, i32, i64, u8 = C.c_float, C.c_double, C.c_int, C.c_int64, C.c_uint8
        p = C.c_void_p
        sig = {
            "orc_exp_spec": (f32, [f32]),
            "orc_sigmoid_spec": (f32, [f32]),
            "orc_sigmoid_spec_vec": (None, [i64, p, p]),
            "orc_exp_spec_vec": (None, [i64, p, p]),
            "orc_exp_spec_max_ulp": (f64, [f32, f32, i32, i32]),
            "orc_route": (None, [i64, i32, i32, p, p, p, p]),
            "orc_eplb": (None, [i64, i32, p, p, p, p, i32, p]),
            "orc_record": (None, [i64, p, p]),
            "orc_e4m3_value": (f64, [u8]),
            "orc_e2m1_value": (f64, [u8]),
            "orc_e8m0_value": (f64, [u8]),
            "orc_e4m3_encode": (u8, [f64]),
            "orc_mxfp8_quant": (None, [i64, i32, p, p, p]),
            "orc_mxfp8_quant_bf16": (None, [i64, i32, p, p, p]),
            "orc_permute": (None, [i64, i32, p, p, p, p]),
            "orc_expert_down": (None, [i64, i32, i32, p, p, p, p, p]),
            "orc_expert_ffn": (None, [i64, i32, i32, p, p, p, p, p, p, p, p, p, p, p]),
            "orc_combine": (None, [i64, i32, i32, p, p, p]),
            "orc_expert_down_a16": (None, [i64, i32, i32, p, p, p, p]),
            "orc_expert_ffn_a16": (None, [i64, i32, i32, p, p, p, p, p, p, p, p, p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---- scalar helpers -------------------------------------------------------
def exp_spec(y) -> np.ndarray:
    y = _c(y, np.float32)
    out = np.empty_like(y)
    lib().orc_exp_spec_vec(y.size, _ptr(y), _ptr(out))
    return out


def sigmoid_spec(x) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty_like(x)
    lib().orc_sigmoid_spec_vec(x.size, _ptr(x), _ptr(out))
    return out


def e4m3_value(codes) -> np.ndarray:
    return np.array([lib().orc_e4m3_value(int(c)) for c in np.ravel(codes)]).reshape(np.shape(codes))


def e2m1_value(nibs) -> np.ndarray:
    return np.array([lib().orc_e2m1_value(int(c)) for c in np.ravel(nibs)]).reshape(np.shape(nibs))


def e8m0_value(s) -> np.ndarray:
    return np.array([lib().orc_e8m0_value(int(c)) for c in np.ravel(s)]).reshape(np.shape(s))


def e4m3_encode(values) -> np.ndarray:
    return np.array([lib().orc_e4m3_encode(float(v)) for v in np.ravel(values)],
                    np.uint8).reshape(np.shape(values))


# ---- stages ----------------------------------------------------------------
def route(logits, bias, k):
    """-> idx int32 [T,k], w float32 [T,k]"""
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float32)
    b = None if bias is None else _c(bias, np.float32)
    lib().orc_route(T, E, k, _ptr(logits), _ptr(b), _ptr(idx), _ptr(w))
    return idx, w


def eplb(idx, phys_of_logical, replica_counts, token_ids=None):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    m = _c(phys_of_logical, np.int32)
    rc = _c(replica_counts, np.int32)
    tid = None if token_ids is None else _c(token_ids, np.int64)
    phys = np.empty_like(idx)
    lib().orc_eplb(T, k, _ptr(tid), _ptr(idx), _ptr(m), _ptr(rc), m.shape[1], _ptr(phys))
    return phys


def record(idx, E, counts=None):
    idx = _c(idx, np.int32)
    counts = np.zeros(E, np.int64) if counts is None else counts
    assert counts.dtype == np.int64 and counts.flags.c_contiguous
    lib().orc_record(idx.size, _ptr(idx), _ptr(counts))
    return counts


def mxfp8_quant(values):
    """exact float32 values [R,K] -> (codes u8 [R,K], scales u8 [R,K/32])"""
    v = _c(values, np.float32)
    R, K = v.shape
    q = np.empty((R, K), np.uint8)
    s = np.empty((R, K // 32), np.uint8)
    lib().orc_mxfp8_quant(R, K, _ptr(v), _ptr(q), _ptr(s))
    return q, s


def mxfp8_quant_bf16(bits):
    x = _c(bits, np.uint16)
    R, K = x.shape
    q = np.empty((R, K), np.uint8)
    s = np.empty((R, K // 32), np.uint8)
    lib().orc_mxfp8_quant_bf16(R, K, _ptr(x), _ptr(q), _ptr(s))
    return q, s


def permute(phys, P):
    """-> offsets int64 [P+1] (unpadded), order int64 [N], pos int64 [N]"""
    ph = _c(phys, np.int32).ravel()
    n = ph.size
    off = np.empty(P + 1, np.int64)
    order = np.empty(n, np.int64)
    pos = np.empty(n, np.int64)
    lib().orc_permute(n, P, _ptr(ph), _ptr(off), _ptr(order), _ptr(pos))
    return off, order, pos


def expert_down(hq, hs, w2, w2s):
    hq, hs = _c(hq, np.uint8), _c(hs, np.uint8)
    w2, w2s = _c(w2, np.uint8), _c(w2s, np.uint8)
    rows, I = hq.shape
    H = w2.shape[0]
    y = np.empty((rows, H), np.float32)
    lib().orc_expert_down(rows, H, I, _ptr(hq), _ptr(hs), _ptr(w2), _ptr(w2s), _ptr(y))
    return y


def expert_ffn(xq, xs, w1, w1s, w2, w2s, want_g=False):
    """One expert on its rows -> dict(hq, hs, h, y[, g])."""
    xq, xs = _c(xq, np.uint8), _c(xs, np.uint8)
    w1, w1s, w2, w2s = (_c(a, np.uint8) for a in (w1, w1s, w2, w2s))
    rows, H = xq.shape
    I = w2.shape[1] * 2
    hq = np.empty((rows, I), np.uint8)
    hs = np.empty((rows, I // 32), np.uint8)
    h = np.empty((rows, I), np.float32)
    g = np.empty((rows, 2 * I), np.float32) if want_g else None
    y = np.empty((rows, H), np.float32)
    lib().orc_expert_ffn(rows, H, I, _ptr(xq), _ptr(xs), _ptr(w1), _ptr(w1s), _ptr(w2),
                         _ptr(w2s), _ptr(hq), _ptr(hs), _ptr(g), _ptr(h), _ptr(y))
    out = dict(hq=hq, hs=hs, h=h, y=y)
    if want_g:
        out["g"] = g
    return out


def expert_down_a16(hb, w2, w2s):
    """bf16 bits hb [rows,I] -> y float32 [rows,H] (fp64 sums rounded to fp32)"""
    hb = _c(hb, np.uint16)
    w2, w2s = _c(w2, np.uint8), _c(w2s, np.uint8)
    rows, I = hb.shape
    H = w2.shape[0]
    y = np.empty((rows, H), np.float32)
    lib().orc_expert_down_a16(rows, H, I, _ptr(hb), _ptr(w2), _ptr(w2s), _ptr(y))
    return y


def expert_ffn_a16(x, w1, w1s, w2, w2s, want_g=False):
    """One expert on bf16 rows x [rows,H] (bits) -> dict(hb, h, y[, g])."""
    x = _c(x, np.uint16)
    w1, w1s, w2, w2s = (_c(a, np.uint8) for a in (w1, w1s, w2, w2s))
    rows, H = x.shape
    I = w2.shape[1] * 2
    hb = np.empty((rows, I), np.uint16)
    h = np.empty((rows, I), np.float32)
    g = np.empty((rows, 2 * I), np.float32) if want_g else None
    y = np.empty((rows, H), np.float32)
    lib().orc_expert_ffn_a16(rows, H, I, _ptr(x), _ptr(w1), _ptr(w1s), _ptr(w2), _ptr(w2s),
                             _ptr(hb), _ptr(g), _ptr(h), _ptr(y))
    out = dict(hb=hb, h=h, y=y)
    if want_g:
        out["g"] = g
    return out


def append_shared(idx, w, phys, E, P, shared):
    """Fused shared experts ("sglang PR #35619", settings that silently break it:
    fusion sizes the operator with top-k plus the shared experts): every token
    gets `shared` more slots after its k routed ones; slot k + s holds shared
    expert s, logical id E + s (outside the routed experts, so the recorder
    never counts it), weight 1 (its output is added as is) and physical id
    P + s (after the P routed physical experts).  Reading: the pages give the
    slot count only; weight 1 is the plain sum of a shared expert's output."""
    T = idx.shape[0]
    s = np.arange(shared, dtype=np.int32)
    idx = np.concatenate([idx, np.broadcast_to(E + s, (T, shared))], axis=1).astype(np.int32)
    w = np.concatenate([w, np.ones((T, shared), np.float32)], axis=1)
    phys = np.concatenate([phys, np.broadcast_to(P + s, (T, shared))], axis=1).astype(np.int32)
    return np.ascontiguousarray(idx), np.ascontiguousarray(w), np.ascontiguousarray(phys)


def combine(w, ypair):
    """w [T,k] f32, ypair [T*k, H] f32 in pair order -> bf16 bits [T,H]"""
    w = _c(w, np.float32)
    T, k = w.shape
    yp = _c(ypair, np.float32)
    H = yp.shape[1]
    out = np.empty((T, H), np.uint16)
    lib().orc_combine(T, k, H, _ptr(w), _ptr(yp), _ptr(out))
    return out


def forward(hidden, logits, bias, k, weights, phys_of_logical=None, replica_counts=None,
            token_ids=None, want_g=False, act="mxfp8", shared=0):
    """The whole layer for the given tokens.

    hidden bf16 bits [n,H], logits [n,E] for tokens ``token_ids`` (their index
    in the forward call; default 0..n-1).  weights = (w1, w1s, w2, w2s) indexed
    by physical expert.  ``act``: "mxfp8" (a8w4: activations quantised to
    MXFP8 before each GEMM) or "bf16" (a16w4: bf16 activations, h rounded to
    bf16).  ``shared``: fused shared experts, the last ``shared`` physical
    experts of ``weights`` (see append_shared).  Returns a dict of every
    intermediate (pair order is (token, slot)) plus ``out`` (bf16 bits [n,H])
    and ``counts`` (int64 [E]).
    """
    if act == "bf16":
        return _forward_a16(hidden, logits, bias, k, weights, phys_of_logical, replica_counts,
                            token_ids, want_g, shared)
    assert act == "mxfp8", act
    w1, w1s, w2, w2s = weights
    n, H = hidden.shape
    E = logits.shape[1]
    P = w1.shape[0]
    if phys_of_logical is None:
        phys_of_logical = np.arange(E, dtype=np.int32)[:, None]
        replica_counts = np.ones(E, np.int32)
    idx, w = route(logits, bias, k)
    phys = eplb(idx, phys_of_logical, replica_counts, token_ids)
    counts = record(idx, E)
    if shared:
        idx, w, phys = append_shared(idx, w, phys, E, P - shared, shared)
    k += shared                       # slots per token from here on
    xq, xs = mxfp8_quant_bf16(hidden)
    off, order, pos = permute(phys, P)
    I = w2.shape[2] * 2
    npairs = n * k
    hq = np.zeros((npairs, I), np.uint8)
    hs = np.zeros((npairs, I // 32), np.uint8)
    h = np.zeros((npairs, I), np.float32)
    g = np.zeros((npairs, 2 * I), np.float32) if want_g else None
    ypair = np.zeros((npairs, H), np.float32)
    for p in range(P):
        pairs = order[off[p]:off[p + 1]]
        if pairs.size == 0:
            continue
        toks = pairs // k
        r = expert_ffn(xq[toks], xs[toks], w1[p], w1s[p], w2[p], w2s[p], want_g=want_g)
        hq[pairs], hs[pairs], h[pairs], ypair[pairs] = r["hq"], r["hs"], r["h"], r["y"]
        if want_g:
            g[pairs] = r["g"]
    out = combine(w, ypair)
    res = dict(idx=idx, w=w, phys=phys, counts=counts, xq=xq, xs=xs, offsets=off,
               order=order, pos=pos, hq=hq, hs=hs, h=h, y=ypair, out=out)
    if want_g:
        res["g"] = g
    return res


def _forward_a16(hidden, logits, bias, k, weights, phys_of_logical, replica_counts, token_ids,
                 want_g, shared=0):
    w1, w1s, w2, w2s = weights
    n, H = hidden.shape
    E = logits.shape[1]
    P = w1.shape[0]
    if phys_of_logical is None:
        phys_of_logical = np.arange(E, dtype=np.int32)[:, None]
        replica_counts = np.ones(E, np.int32)
    idx, w = route(logits, bias, k)
    phys = eplb(idx, phys_of_logical, replica_counts, token_ids)
    counts = record(idx, E)
    if shared:
        idx, w, phys = append_shared(idx, w, phys, E, P - shared, shared)
    k += shared
    off, order, pos = permute(phys, P)
    I = w2.shape[2] * 2
    npairs = n * k
    hb = np.zeros((npairs, I), np.uint16)
    h = np.zeros((npairs, I), np.float32)
    g = np.zeros((npairs, 2 * I), np.float32) if want_g else None
    ypair = np.zeros((npairs, H), np.float32)
    for p in range(P):
        pairs = order[off[p]:off[p + 1]]
        if pairs.size == 0:
            continue
        r = expert_ffn_a16(hidden[pairs // k], w1[p], w1s[p], w2[p], w2s[p], want_g=want_g)
        hb[pairs], h[pairs], ypair[pairs] = r["hb"], r["h"], r["y"]
        if want_g:
            g[pairs] = r["g"]
    out = combine(w, ypair)
    res = dict(idx=idx, w=w, phys=phys, counts=counts, offsets=off, order=order, pos=pos,
               hb=hb, h=h, y=ypair, out=out)
    if want_g:
        res["g"] = g
    return res


def threads() -> int:
    """OpenMP threads the oracle will use (OMP_NUM_THREADS or all cores)."""
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else (os.cpu_count() or 1)


def plan_replicas(load, num_physical, max_replicas):
    """EPLB replica plan.

    Every logical expert e keeps physical slot e; the redundant slots E..P-1 are
    handed out one at a time, each to the expert whose recorded load per replica
    is highest (exact rational comparison; the lower index on ties), among the
    experts that are below max_replicas.  The pages rebalance periodically from
    the recorder's per-expert statistics ("sglang PR #35619", EPLB arm
    settings) but do not spell out the placement rule; this greedy rule is the
    reading taken here.  Returns (phys_of_logical [E, R] with -1 for unused
    entries, replica_counts [E]).
    """
    from fractions import Fraction
    load = [int(v) for v in np.asarray(load).ravel()]
    E = len(load)
    pol = np.full((E, max_replicas), -1, np.int32)
    rc = np.ones(E, np.int32)
    pol[:, 0] = np.arange(E)
    for slot in range(E, num_physical):
        cands = [e for e in range(E) if rc[e] < max_replicas]
        best = max(cands, key=lambda e: (Fraction(load[e], int(rc[e])), -e))
        pol[best, rc[best]] = slot
        rc[best] += 1
    return pol, rc
