"""Shared plumbing of the GPU tests: run the library on seeded inputs and
compare each stage with the CPU oracle (tests only)."""
import numpy as np

import oracle
import synthetic
from tests import helpers

_WEIGHT_CACHE = {}


def weights(cfg, physical=True):
    key = (cfg.seed, cfg.E, cfg.H, cfg.I)
    if key not in _WEIGHT_CACHE:
        _WEIGHT_CACHE[key] = synthetic.make_all_weights(cfg, physical=False)
    w = _WEIGHT_CACHE[key]
    if physical and cfg.P != cfg.E:
        p2l = synthetic.physical_to_logical(cfg)
        return tuple(a[p2l] for a in w)
    return w


class Run:
    """One handle with weights uploaded; forward() runs and collects dumps."""

    def __init__(self, cfg, W=None, eplb=True, cap=None, act=0, shared=0):
        import torch
        import moe_layer_serving_gb300 as mm
        self.torch, self.mm, self.cfg = torch, mm, cfg
        self.dev = torch.device("cuda:0")
        self.op = mm.MegaMoE(cfg.E, cfg.P, cfg.k, cfg.H, cfg.I)
        self.act, self.shared = act, shared
        if act:
            self.op.set_activation_format(act)
        if shared:
            self.op.set_shared_experts(shared)
        W = weights(cfg) if W is None else W
        wt = [torch.from_numpy(np.ascontiguousarray(a)).to(self.dev) for a in W]
        self.op.set_weights(*wt)
        del wt
        self.map = None
        if cfg.P != cfg.E and eplb:
            m, rc, _ = synthetic.make_eplb_map(cfg)
            self.op.set_eplb_map(m, rc)
            self.map = (m, rc)
        self.op.reserve(cap or cfg.T)

    def to_dev(self, hidden, logits, bias):
        t = self.torch
        x = t.from_numpy(np.ascontiguousarray(hidden).view(np.int16)).to(self.dev).view(t.bfloat16)
        lg = t.from_numpy(np.ascontiguousarray(logits)).to(self.dev)
        b = None if bias is None else t.from_numpy(np.ascontiguousarray(bias)).to(self.dev)
        return x, lg, b

    def forward(self, hidden, logits, bias, dumps=True):
        t = self.torch
        x, lg, b = self.to_dev(hidden, logits, bias)
        out = t.empty_like(x)
        self.op.forward(x, lg, b, out)
        t.cuda.synchronize()
        status = self.op.get_status()
        res = {"out": out.view(t.int16).cpu().numpy().view(np.uint16), "status": status}
        if dumps:
            T, k = hidden.shape[0], self.cfg.k + self.shared
            for stage, (name, _) in self.mm.DUMP_STAGES.items():
                a = self.op.debug_dump(stage)
                if stage <= 3:
                    a = a.reshape(T, k)
                res[name] = a
            rows = int(res["offsets"][-1])
            H, I = self.cfg.H, self.cfg.I
            if self.act:
                res["xd"] = res.pop("xq").view(np.uint16).reshape(rows, H)
                res["hb"] = res.pop("hq").view(np.uint16).reshape(rows, I)
                res["y"] = res["y"].reshape(rows, H)
                del res["xs"], res["hs"]
                return res
            res["xq"] = res["xq"].reshape(rows, H)
            res["xs"] = res["xs"].reshape(rows, H // 32)
            res["hq"] = res["hq"].reshape(rows, I)
            res["hs"] = res["hs"].reshape(rows, I // 32)
            res["y"] = res["y"].reshape(rows, H)
        return res

    def close(self):
        self.op.close()


def sample_tokens(T, n=24, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, T // 2, T - 1]
    rest = rng.choice(T, size=min(T, n), replace=False)
    return np.unique(np.clip(np.concatenate([fixed, rest]), 0, T - 1))


def tile_edge_tokens(res, T):
    """Tokens whose (token, slot) pairs sit in the first or the last row of
    every token tile of one GPU forward (the tile table of debug stage 12):
    checking them end to end covers every tile of every expert, however late
    its units ran, with about two tokens per tile."""
    pos = res["pos"]
    k = pos.shape[1]
    token_of_row = {int(r): t for t, r in zip(np.repeat(np.arange(T), k), pos.ravel())}
    tiles = res["tiles"].reshape(-1, 3)
    assert tiles.shape[0] > 0
    sel = set()
    for _, row0, rows in tiles:
        assert rows >= 1
        sel.add(token_of_row[int(row0)])
        sel.add(token_of_row[int(row0 + rows - 1)])
    return np.array(sorted(sel), dtype=np.int64)


def bf16_f64(bits):
    return synthetic.f32_from_bf16_bits(bits).astype(np.float64)


def assert_out_close(got_bits, ref_bits, what=""):
    """The layer tolerance: relative L2 <= 1e-2 and every |err| <= 0.05 rms(ref)."""
    got, ref = bf16_f64(got_bits), bf16_f64(ref_bits)
    err = got - ref
    rms = np.sqrt(np.mean(ref ** 2))
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= 1e-2, f"{what} relative L2 {rel:.3e}"
    assert np.abs(err).max() <= 0.05 * rms, f"{what} max |err| {np.abs(err).max():.3e} > 0.05 rms {rms:.3e}"
    return rel


def assert_mxfp8_close(q_gpu, s_gpu, q_ref, s_ref, min_equal=0.999):
    """Requantised codes: nearly all identical, the rest one e4m3 step apart."""
    a = helpers.deq_mxfp8(q_gpu, s_gpu)
    b = helpers.deq_mxfp8(q_ref, s_ref)
    X = np.repeat(np.maximum(s_gpu.astype(int), s_ref.astype(int)) - 127, 32, axis=-1)
    step = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -3 + np.ldexp(1.0, X - 9)
    assert np.all(np.abs(a - b) <= step * (1 + 1e-12)), "codes more than one e4m3 step apart"
    same = np.mean((q_gpu == q_ref) & (np.repeat(s_gpu, 32, axis=-1) == np.repeat(s_ref, 32, axis=-1)))
    assert same >= min_equal, f"only {same:.5f} of codes identical"
    return same


def _check_routing(cfg, res, logits, bias, map_rc, shared=0):
    """Routing, physical ids, segment offsets and dispatch order (all tokens, exact)."""
    k, P = cfg.k, cfg.P
    m, rc = map_rc if map_rc is not None else (None, None)
    idx, w = oracle.route(logits, bias, k)
    if m is None:
        m_, rc_ = np.arange(cfg.E, dtype=np.int32)[:, None], np.ones(cfg.E, np.int32)
    else:
        m_, rc_ = m, rc
    phys = oracle.eplb(idx, m_, rc_)
    if shared:
        idx, w, phys = oracle.append_shared(idx, w, phys, cfg.E, P, shared)
    assert np.array_equal(res["idx"], idx), "routing indices differ"
    assert np.array_equal(res["weights"].view(np.uint32), w.view(np.uint32)), "routing weights differ"
    assert np.array_equal(res["phys"], phys), "physical experts differ"
    off_o, order, pos_o = oracle.permute(phys, P + shared)
    cnt = np.diff(off_o)
    padded = (cnt + 15) // 16 * 16
    off_g = np.concatenate([[0], np.cumsum(padded)])
    assert np.array_equal(res["offsets"], off_g), "segment offsets differ"
    p_flat = phys.ravel()
    assert np.array_equal(res["pos"].ravel() - off_g[p_flat], pos_o - off_o[p_flat]), "dispatch order differs"
    return idx, w, phys


def pair_magnitude(ref, k):
    """sum_j |w[t,j] * y[t,j]| per output element, from an oracle result."""
    w = np.abs(ref["w"].astype(np.float64))
    y = np.abs(ref["y"].astype(np.float64)).reshape(w.shape[0], k, -1)
    return (w[:, :, None] * y).sum(1)


def assert_out_close_a16(got_bits, ref_bits, what="", mag=None):
    """a16w4 layer tolerance: relative L2 <= 4e-3, and every |err| within one
    bf16 step of the element and of the summed terms, 2^-7 (|ref| + sum_j
    |w_j y_j|), plus 0.01 rms(ref).  The GPU path rounds y to bf16 before the
    combine (the oracle keeps fp32), which moves a sum by up to 2^-9 of its
    terms' magnitude -- large next to a sum whose terms cancel -- and the
    output may land on the neighbouring bf16 value; the rms term covers the
    rare h that rounds to the other bf16 neighbour."""
    got, ref = bf16_f64(got_bits), bf16_f64(ref_bits)
    err = got - ref
    rms = np.sqrt(np.mean(ref ** 2))
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= 4e-3, f"{what} relative L2 {rel:.3e}"
    bound = 2.0 ** -7 * (np.abs(ref) + (0.0 if mag is None else mag)) + 0.01 * rms
    worst = np.argmax(np.abs(err) - bound)
    assert np.all(np.abs(err) <= bound), \
        f"{what} |err| {np.abs(err).flat[worst]:.3e} at |ref| {np.abs(ref).flat[worst]:.3e}, rms {rms:.3e}"
    return rel


def check_against_oracle_a16(cfg, res, hidden, logits, bias, W, map_rc, token_sel=None, shared=0):
    """Every stage of one a16w4 GPU forward against the oracle's bf16 variant.

    Routing and dispatch exact for all tokens; for token_sel: the dispatched
    bf16 rows exact, h in bf16 within one bf16 step (nearly all identical),
    GEMM2 + combine teacher-forced on the GPU's h within bf16 rounding, and
    the output end to end.
    """
    T, k = hidden.shape[0], cfg.k + shared
    m, rc = map_rc if map_rc is not None else (None, None)
    idx, w, phys = _check_routing(cfg, res, logits, bias, map_rc, shared)
    sel = np.arange(T) if token_sel is None else np.asarray(token_sel)
    for j in range(k):
        assert np.array_equal(res["xd"][res["pos"][sel, j]], hidden[sel]), "dispatched rows differ"
    ref = oracle.forward(hidden[sel], logits[sel], bias, cfg.k, W, m, rc, token_ids=sel, act="bf16", shared=shared)
    rows = res["pos"][sel].ravel()                        # pair order (t, j)
    a, b = bf16_f64(res["hb"][rows]), bf16_f64(ref["hb"])
    # one bf16 step of the element, plus an absolute 2^-14 rms(h) for elements
    # near zero: gate and up are K-term fp32 sums on the GPU (fp64 in the
    # oracle), whose absolute error (~1e-5 rms at K = 7168) exceeds a bf16
    # step of an h that cancellation left far below its row's scale
    rms = np.sqrt(np.mean(b ** 2)) + 1e-30
    step = np.maximum(np.abs(a), np.abs(b)) * 2.0 ** -7 + 2.0 ** -14 * rms
    over = np.abs(a - b) > step
    assert not over.any(), (f"h: {over.sum()} of {over.size} elements beyond one bf16 step + 2^-14 rms; "
                            f"max |err| / rms {np.abs(a - b).max() / rms:.3e}")
    same = np.mean(res["hb"][rows] == ref["hb"])
    assert same >= 0.995, f"only {same:.5f} of h identical"
    ypair = np.empty((rows.size, cfg.H), np.float32)
    psel = phys[sel].ravel()
    for p in np.unique(psel):
        at = np.nonzero(psel == p)[0]
        ypair[at] = oracle.expert_down_a16(res["hb"][rows[at]], W[2][p], W[3][p])
    tf = oracle.combine(w[sel], ypair)
    got, exp = bf16_f64(res["out"][sel]), bf16_f64(tf)
    mag = np.abs(w[sel].astype(np.float64)[:, :, None] * ypair.reshape(len(sel), k, cfg.H)).sum(1)
    bound = 2.0 ** -7 * mag + 2.0 ** -8 * np.abs(exp) + 1e-30
    assert np.all(np.abs(got - exp) <= bound), "GEMM2/combine off beyond bf16 rounding"
    rel = assert_out_close_a16(res["out"][sel], ref["out"], "end to end", pair_magnitude(ref, k))
    return rel, ref


def check_against_oracle(cfg, res, hidden, logits, bias, W, map_rc, token_sel=None, check_hq=True, shared=0):
    """Every stage of one GPU forward against the oracle.

    Routing, physical ids and the dispatch order are checked for all tokens;
    the expert FFN and the output for token_sel (all tokens when None).
    ``shared``: fused shared experts (the last ``shared`` experts of W).
    """
    T, k, P = hidden.shape[0], cfg.k, cfg.P
    m, rc = map_rc if map_rc is not None else (None, None)
    idx, w = oracle.route(logits, bias, k)
    if m is None:
        m_, rc_ = np.arange(cfg.E, dtype=np.int32)[:, None], np.ones(cfg.E, np.int32)
    else:
        m_, rc_ = m, rc
    phys = oracle.eplb(idx, m_, rc_)
    if shared:
        idx, w, phys = oracle.append_shared(idx, w, phys, cfg.E, P, shared)
    k, P = k + shared, P + shared                           # slots per token, physical experts
    assert np.array_equal(res["idx"], idx), "routing indices differ"
    assert np.array_equal(res["weights"].view(np.uint32), w.view(np.uint32)), "routing weights differ"
    assert np.array_equal(res["phys"], phys), "physical experts differ"
    off_o, order, pos_o = oracle.permute(phys, P)
    cnt = np.diff(off_o)
    padded = (cnt + 15) // 16 * 16
    off_g = np.concatenate([[0], np.cumsum(padded)])
    assert np.array_equal(res["offsets"], off_g), "segment offsets differ"
    p_flat = phys.ravel()
    rank_o = pos_o - off_o[p_flat]
    rank_g = res["pos"].ravel() - off_g[p_flat]
    assert np.array_equal(rank_g, rank_o), "dispatch order differs"

    sel = np.arange(T) if token_sel is None else np.asarray(token_sel)
    xq, xs = oracle.mxfp8_quant_bf16(hidden[sel])
    for j in range(k):
        rows = res["pos"][sel, j]
        assert np.array_equal(res["xq"][rows], xq), "activation codes differ"
        assert np.array_equal(res["xs"][rows], xs), "activation scales differ"

    ref = oracle.forward(hidden[sel], logits[sel], bias, cfg.k, W, m, rc, token_ids=sel, shared=shared)
    assert np.array_equal(ref["idx"], idx[sel])
    rows = res["pos"][sel].ravel()                        # pair order (t, j)
    if check_hq:
        assert_mxfp8_close(res["hq"][rows], res["hs"][rows], ref["hq"], ref["hs"],
                           min_equal=0.999 if rows.size * cfg.I >= 100000 else 0.995)
    # teacher-forced GEMM2 + combine: the oracle consumes the GPU's hq/hs
    ypair = np.empty((rows.size, cfg.H), np.float32)
    psel = phys[sel].ravel()
    for p in np.unique(psel):
        at = np.nonzero(psel == p)[0]
        ypair[at] = oracle.expert_down(res["hq"][rows[at]], res["hs"][rows[at]], W[2][p], W[3][p])
    tf = oracle.combine(w[sel], ypair)
    got, exp = bf16_f64(res["out"][sel]), bf16_f64(tf)
    mag = np.abs(w[sel].astype(np.float64)[:, :, None] * ypair.reshape(len(sel), k, cfg.H)).sum(1)
    bound = 2.0 ** -7 * mag + 2.0 ** -8 * np.abs(exp) + 1e-30
    assert np.all(np.abs(got - exp) <= bound), "GEMM2/combine off beyond bf16 rounding"
    rel = assert_out_close(res["out"][sel], ref["out"], "end to end")
    return rel, ref
