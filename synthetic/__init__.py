"""Seeded synthetic inputs for the a8w4 fused MoE layer forward.

This module is shared by the CPU oracle (``oracle/``) and by the CUDA path's
tests and benchmark.  It holds only input preparation: random draws, the
bf16 rounding of those draws, the MXFP4 encoding that turns bf16 weights into
the checkpoint format the layer consumes, and the EPLB replica map.  None of
the layer's own arithmetic (routing, remap, activation quantisation, GEMMs,
combine) lives here.

Workloads (the pages serve DeepSeek-V4-Pro's routed experts as a8w4 with
MXFP4 weights; "sglang PR #47065", Title/switches and "InferenceX PR #3430",
draft-precision notes):

  id  T      H     I     E->P      k  routing
  0   16     256   128   8->8      2  logits N(0,1), bias 0
  1   64     7168  2048  256->256  6  logits N(0,1), bias N(0,0.1)
  2   512    7168  2048  256->320  6  logits N(0,1) - 1.1 ln(e+1), bias 0, EPLB
  3   8192   7168  2048  256->256  6  logits N(0,1), bias 0
  4   16384  7168  2048  256->320  6  logits N(0,1) - 1.4 ln(e+1), bias 0, EPLB

Every draw comes from numpy's Philox-4x32 counter-based generator keyed by
(seed, tensor id, index), so any expert's weights can be regenerated alone.
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np

__all__ = [
    "Config", "CONFIGS", "make_activations", "make_expert_weights",
    "make_all_weights", "make_eplb_map", "physical_to_logical",
    "bf16_bits_from_f32", "f32_from_bf16_bits", "mxfp4_encode_rows",
]

# tensor ids for the generator key
_TID_HIDDEN, _TID_LOGITS, _TID_BIAS, _TID_W1, _TID_W2 = 1, 2, 3, 4, 5


@dataclasses.dataclass(frozen=True)
class Config:
    cid: int
    T: int
    H: int
    I: int
    E: int
    P: int
    k: int
    zipf_s: float        # logit offset -zipf_s * ln(e+1); 0 = uniform-ish
    bias_std: float      # routing bias ~ N(0, bias_std); 0 = zeros
    recording: bool      # per-logical-expert count recording on
    seed: int = 0

    @property
    def redundant(self) -> int:
        return self.P - self.E


CONFIGS = {
    0: Config(0, 16, 256, 128, 8, 8, 2, 0.0, 0.0, False),
    1: Config(1, 64, 7168, 2048, 256, 256, 6, 0.0, 0.1, False),
    2: Config(2, 512, 7168, 2048, 256, 320, 6, 1.1, 0.0, True),
    3: Config(3, 8192, 7168, 2048, 256, 256, 6, 0.0, 0.0, False),
    4: Config(4, 16384, 7168, 2048, 256, 320, 6, 1.4, 0.0, True),
}


def _gen(seed: int, tid: int, index: int = 0) -> np.random.Generator:
    key = (int(seed) << 64) | (int(tid) << 32) | int(index)
    return np.random.Generator(np.random.Philox(key=key))


def bf16_bits_from_f32(a: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (round to nearest, ties to even); uint16 bits."""
    b = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    return ((b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def f32_from_bf16_bits(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def make_activations(cfg: Config, T: int | None = None):
    """hidden bf16 bits [T,H], router logits f32 [T,E], bias f32 [E]."""
    T = cfg.T if T is None else T
    hidden = _gen(cfg.seed, _TID_HIDDEN).standard_normal((T, cfg.H), dtype=np.float32)
    hidden = bf16_bits_from_f32(hidden)
    logits = _gen(cfg.seed, _TID_LOGITS).standard_normal((T, cfg.E), dtype=np.float32)
    if cfg.zipf_s:
        off = (cfg.zipf_s * np.log(np.arange(1, cfg.E + 1, dtype=np.float64))).astype(np.float32)
        logits = (logits - off[None, :]).astype(np.float32)
    if cfg.bias_std:
        bias = (cfg.bias_std * _gen(cfg.seed, _TID_BIAS).standard_normal(cfg.E)).astype(np.float32)
    else:
        bias = np.zeros(cfg.E, np.float32)
    return hidden, logits, bias


# --- MXFP4 weight encoding (input preparation: the checkpoint format) -------
# OCP Microscaling v1.0: one e8m0 scale per 32 elements, X = floor(log2 amax)
# - emax(e2m1) with emax = 2, elements rounded to nearest-even on the e2m1 grid
# {0, .5, 1, 1.5, 2, 3, 4, 6} and saturated at 6.  Packing: element 2i in the
# low nibble of byte i, sign in bit 3 of the nibble.
#
# After scaling, |v| / 2^X lies in [0, 8) and every rounding midpoint of the
# grid is a multiple of 1/4, so the code is a function of (floor(4a), whether
# 4a is an integer): a 64-entry table indexed by 2*floor(4a) + (4a not integer).
_E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def _e2m1_rne_code(a: float) -> int:
    """Nearest grid code for a >= 0, ties to the even code, saturating at 6."""
    best = min(range(8), key=lambda c: (abs(_E2M1_GRID[c] - a), c % 2))
    return best


_E2M1_TABLE = np.array(
    [_e2m1_rne_code(i / 4 if inexact == 0 else (i + 0.5) / 4)
     for i in range(32) for inexact in (0, 1)], np.uint8)


def mxfp4_encode_rows(v: np.ndarray):
    """v: float32 [R, K] (exact bf16 values), K % 32 == 0 -> (packed u8 [R,K/2], scale u8 [R,K/32])."""
    R, K = v.shape
    blk = np.ascontiguousarray(v, dtype=np.float32).reshape(R, K // 32, 32)
    amax = np.abs(blk).max(axis=2)
    _, ex = np.frexp(amax)                    # amax = m * 2**ex, m in [0.5, 1)
    X = np.where(amax > 0, ex - 1 - 2, -127).clip(-127, 127)
    a4 = np.abs(blk)
    a4 *= (np.ldexp(np.float32(1.0), -X).astype(np.float32) * np.float32(4.0))[:, :, None]
    fl = np.minimum(a4.astype(np.int32), 31)
    j = 2 * fl + (a4 > fl)
    code = _E2M1_TABLE[j]
    code |= (blk.view(np.uint32) >> 28).astype(np.uint8) & np.uint8(8)
    code = code.reshape(R, K)
    packed = code[:, 0::2] | (code[:, 1::2] << np.uint8(4))
    return packed, (X + 127).astype(np.uint8)


_CHUNK_ROWS = 64     # rows per draw/encode step; keeps temporaries small


def _normal_bf16_mxfp4(gen: np.random.Generator, R: int, K: int, std: float):
    """R x K draws of bf16(N(0, std^2)), MXFP4-encoded row chunk by row chunk."""
    packed = np.empty((R, K // 2), np.uint8)
    scale = np.empty((R, K // 32), np.uint8)
    for r0 in range(0, R, _CHUNK_ROWS):
        r1 = min(R, r0 + _CHUNK_ROWS)
        a = gen.standard_normal((r1 - r0, K), dtype=np.float32)
        a *= np.float32(std)
        packed[r0:r1], scale[r0:r1] = mxfp4_encode_rows(f32_from_bf16_bits(bf16_bits_from_f32(a)))
    return packed, scale


def make_expert_weights(cfg: Config, e: int):
    """Logical expert e: (w1 [2I,H/2], w1s [2I,H/32], w2 [H,I/2], w2s [H,I/32]) uint8.

    W1 rows 0..I-1 are the gate projection and rows I..2I-1 the up projection.
    """
    w1p, w1s = _normal_bf16_mxfp4(_gen(cfg.seed, _TID_W1, e), 2 * cfg.I, cfg.H, 0.02)
    w2p, w2s = _normal_bf16_mxfp4(_gen(cfg.seed, _TID_W2, e), cfg.H, cfg.I, 0.02)
    return w1p, w1s, w2p, w2s


def physical_to_logical(cfg: Config) -> np.ndarray:
    """Physical expert p holds logical expert p (p < E) or replica of p - E."""
    return np.concatenate([np.arange(cfg.E), np.arange(cfg.P - cfg.E)]).astype(np.int32)


def make_eplb_map(cfg: Config):
    """(phys_of_logical int32 [E,R], replica_counts int32 [E], R).

    The P - E redundant slots replicate the most popular logical experts, which
    under the Zipf logit offset are the lowest-indexed ones: physical E+i is the
    second replica of logical i.
    """
    R = 2 if cfg.P > cfg.E else 1
    m = np.full((cfg.E, R), -1, np.int32)
    m[:, 0] = np.arange(cfg.E)
    rc = np.ones(cfg.E, np.int32)
    for i in range(cfg.P - cfg.E):
        m[i, 1] = cfg.E + i
        rc[i] = 2
    return m, rc, R


def make_all_weights(cfg: Config, threads: int | None = None, physical: bool = True,
                     cache_dir: str | None = None):
    """All weights, stacked [P,...] (physical=True, replicas are byte copies) or [E,...].

    cache_dir (default: $MM_SYNTH_CACHE, unset = no cache) keeps the logical
    experts' arrays as .npy files keyed by (seed, E, H, I) so that several
    processes on one machine draw them once.
    """
    E, H, I = cfg.E, cfg.H, cfg.I
    cache_dir = cache_dir if cache_dir is not None else os.environ.get("MM_SYNTH_CACHE")
    names = ("w1", "w1s", "w2", "w2s")
    paths = None
    if cache_dir:
        tag = f"s{cfg.seed}_E{E}_H{H}_I{I}"
        paths = [os.path.join(cache_dir, f"{tag}_{n}.npy") for n in names]
    if paths and all(os.path.exists(p) for p in paths):
        w1, w1s, w2, w2s = (np.load(p) for p in paths)
    else:
        w1 = np.empty((E, 2 * I, H // 2), np.uint8)
        w1s = np.empty((E, 2 * I, H // 32), np.uint8)
        w2 = np.empty((E, H, I // 2), np.uint8)
        w2s = np.empty((E, H, I // 32), np.uint8)

        def one(e):
            w1[e], w1s[e], w2[e], w2s[e] = make_expert_weights(cfg, e)

        threads = threads or min(32, os.cpu_count() or 1)
        if E > 1 and threads > 1:
            with _cf.ThreadPoolExecutor(threads) as ex:
                list(ex.map(one, range(E)))
        else:
            for e in range(E):
                one(e)
        if paths:
            os.makedirs(cache_dir, exist_ok=True)
            for p, a in zip(paths, (w1, w1s, w2, w2s)):
                tmp = p + f".{os.getpid()}.tmp"
                with open(tmp, "wb") as f:
                    np.save(f, a)
                os.replace(tmp, p)
    if physical and cfg.P != cfg.E:
        p2l = physical_to_logical(cfg)
        return w1[p2l], w1s[p2l], w2[p2l], w2s[p2l]
    return w1, w1s, w2, w2s
