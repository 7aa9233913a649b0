"""Independent decoders/encoders used to pin the oracle (tests only).

Nothing here is shared with the oracle or with the CUDA library: e4m3 goes
through torch's float8_e4m3fn codec (a library routine), e2m1 through the
OCP table in tests/golden/e2m1_values.txt, and the MX scale rule through
Python's math.frexp.
"""
import math

import numpy as np
import torch


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def f64_to_e4m3_sat(v: np.ndarray) -> np.ndarray:
    """torch cast (nearest-even) after clamping to the finite range."""
    t = torch.from_numpy(np.clip(np.asarray(v, np.float64), -448.0, 448.0))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e8m0_to_f64(s: np.ndarray) -> np.ndarray:
    s = np.asarray(s)
    return np.array([math.ldexp(1.0, int(c) - 127) for c in s.ravel()]).reshape(s.shape)


def deq_mxfp8(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    v = e4m3_to_f64(q)
    return v * np.repeat(e8m0_to_f64(s), 32, axis=-1)


def deq_mxfp4(packed: np.ndarray, scale: np.ndarray, table) -> np.ndarray:
    lo = packed & 0xF
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    vals = np.asarray(table, np.float64)[codes]
    return vals * np.repeat(e8m0_to_f64(scale), 32, axis=-1)


def quant_mxfp8(v: np.ndarray):
    """MX scale rule via frexp, element codes via torch's e4m3 cast."""
    v = np.asarray(v, np.float64)
    R, K = v.shape
    blk = v.reshape(R, K // 32, 32)
    amax = np.abs(blk).max(axis=2)
    X = np.clip(np.frexp(amax)[1] - 1 - 8, -127, 127)
    X = np.where(amax == 0.0, -127, X)
    q = f64_to_e4m3_sat(blk * np.ldexp(1.0, -X)[:, :, None])
    q = np.where((amax == 0.0)[:, :, None], np.uint8(0), q).reshape(R, K)
    return q.astype(np.uint8), (X + 127).astype(np.uint8)


def bf16_bits(v: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()
