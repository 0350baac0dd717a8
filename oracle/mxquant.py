"""OCP MX quantisation of activations to MXFP4, in fp64 (the A-quantised
prefill mode).  TEST INFRASTRUCTURE ONLY (see the package docstring).

Every page runs its experts W4A16: the activations stay bf16.  The tensor
cores' block-scaled FP4 product (FP4 x FP4 with one E8M0 scale per 32
elements along K) needs the activations in MXFP4 as well, which is not on the
pages; the reading taken for that mode follows the OCP Microscaling Formats
(MX) Specification v1.0 conversion:

* blocks of 32 consecutive elements along K (the reduction dimension);
* shared scale X = 2^(floor(log2 amax) - 2), amax = the block's largest
  magnitude, stored as the E8M0 byte floor(log2 amax) - 2 + 127 clamped to
  [0, 254]; an all-zero block takes X = 2^-127 (byte 0);
* each element becomes the E2M1 value nearest to v / X, ties to the code whose
  mantissa bit is 0 (round half to even), magnitudes above 6 saturated to 6;
  a magnitude that rounds to 0 is stored as +0 (code 0).

Element 2j of a block row goes in the low nibble of byte j, as in the
weights' codes.  In the prefill mode both x (along H, per token) and h (along
I, per routed pair) are quantised; the oracle applies it to its own fp64 h.
"""
from __future__ import annotations

import math

import numpy as np

from .formats import E2M1_TABLE

# E2M1 magnitudes by code 0..7
_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_code(r: float) -> int:
    """E2M1 code (0..15) of the value nearest to r, ties to the even code, |r| > 6 saturated."""
    m = abs(r)
    c = 7
    for i in range(7):
        lo, hi = _GRID[i], _GRID[i + 1]
        if m <= hi:
            mid = 0.5 * (lo + hi)
            if m < mid:
                c = i
            elif m > mid:
                c = i + 1
            else:
                c = i if i % 2 == 0 else i + 1
            break
    if c == 0:
        return 0
    return c | 8 if r < 0 else c


def block_scale_byte(amax: float) -> int:
    """E8M0 byte of the shared scale of a block whose largest magnitude is amax."""
    if amax == 0.0:
        return 0
    _, ex = math.frexp(amax)          # amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1
    return min(254, max(0, ex - 1 - 2 + 127))


def mx_quantize(v: np.ndarray):
    """v [rows, K] (K a multiple of 32) -> (codes uint8 [rows, K/2], scales uint8 [rows, K/32])."""
    v = np.asarray(v, dtype=np.float64)
    rows, K = v.shape
    if K % 32:
        raise ValueError("K must be a multiple of 32")
    codes = np.zeros((rows, K // 2), dtype=np.uint8)
    scales = np.zeros((rows, K // 32), dtype=np.uint8)
    for r in range(rows):
        for b in range(K // 32):
            blk = v[r, 32 * b:32 * b + 32]
            e = block_scale_byte(float(np.max(np.abs(blk))))
            scales[r, b] = e
            X = math.ldexp(1.0, e - 127)
            for i in range(32):
                c = e2m1_code(float(blk[i]) / X)
                j = 32 * b + i
                if j % 2 == 0:
                    codes[r, j // 2] |= c
                else:
                    codes[r, j // 2] |= c << 4
    return codes, scales


def mx_dequantize(codes: np.ndarray, scales: np.ndarray, K: int) -> np.ndarray:
    """Inverse view of mx_quantize: the exact fp64 values the codes stand for."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows = codes.shape[0]
    lo = (codes & 0xF).astype(np.int64)
    hi = (codes >> 4).astype(np.int64)
    el = np.empty((rows, K), dtype=np.int64)
    el[:, 0::2] = lo
    el[:, 1::2] = hi
    X = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return E2M1_TABLE[el] * np.repeat(X, 32, axis=1)


def mx_round(v: np.ndarray) -> np.ndarray:
    """v replaced by its MXFP4 quantisation (rows of K, blocks of 32 along K)."""
    v = np.asarray(v, dtype=np.float64)
    c, s = mx_quantize(v)
    return mx_dequantize(c, s, v.shape[1])
