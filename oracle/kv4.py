"""Oracle of a 4-bit KV page format (test infrastructure: only the tests use
it; it shares no code with the library, which does not implement the format
yet).

What the pages fix ("Dendrite", section on FlashInfer and TurboQuant
integration): 4-bit KV compression that cuts KV memory 3.88x and is computed
on directly instead of being dequantised on every call.  They leave the
quantiser open.  Reading adopted: symmetric 4-bit integer codes with one
power-of-two scale per (token, kv head) row of d values, the scale stored as
an 8-bit exponent (as in the OCP microscaling formats).  That is
4 + 8 / d bits per value, i.e. 16 / 4.125 = 3.88x at TinyLlama's d = 64 --
the pages' figure -- and 3.94x at d = 128.

  e(row)  = the smallest integer with max|x| <= 7 * 2^e  (-127 for a zero row)
  code(x) = round-half-even(x / 2^e), in [-7, 7]
  x'      = code * 2^e
"""
from __future__ import annotations

import math

import numpy as np

E_MIN, E_MAX = -127, 127


def row_exponent(row: np.ndarray) -> int:
    m = float(np.max(np.abs(row))) if row.size else 0.0
    if m == 0.0:
        return E_MIN
    e = math.ceil(math.log2(m / 7.0))
    # guard the log against rounding at exact powers of two
    while m > 7.0 * 2.0 ** e:
        e += 1
    while e > E_MIN and m <= 7.0 * 2.0 ** (e - 1):
        e -= 1
    return max(E_MIN, min(E_MAX, e))


def quantize(x: np.ndarray):
    """x [..., d] (float) -> (codes int8 [..., d] in [-7, 7], exponents int16 [...])."""
    x = np.asarray(x, np.float64)
    rows = x.reshape(-1, x.shape[-1])
    exps = np.array([row_exponent(r) for r in rows], np.int16)
    codes = np.rint(rows / np.ldexp(1.0, exps.astype(np.int64))[:, None])   # rint: half to even
    codes = np.clip(codes, -7, 7).astype(np.int8)
    return codes.reshape(x.shape), exps.reshape(x.shape[:-1])


def dequantize(codes: np.ndarray, exps: np.ndarray) -> np.ndarray:
    return codes.astype(np.float64) * np.ldexp(1.0, exps.astype(np.int64))[..., None]


def bits_per_value(d: int) -> float:
    return 4.0 + 8.0 / d


def compression_vs_bf16(d: int) -> float:
    return 16.0 / bits_per_value(d)
