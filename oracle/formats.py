"""Decoders for the weight formats, by table, in fp64.

* E2M1 (4-bit float, OCP Microscaling Formats (MX) Specification v1.0, the
  element type of MXFP4): sign bit, 2 exponent bits with bias 1, 1 mantissa
  bit; exponent field 0 is subnormal (0 or 0.5).  Magnitudes 0, 0.5, 1, 1.5,
  2, 3, 4, 6.
* E8M0 (the MX shared scale): value 2^(e - 127); 255 is NaN.
* E4M3 (OCP 8-bit float, "FN" variant): sign, 4 exponent bits with bias 7,
  3 mantissa bits; exponent field 0 is subnormal; S.1111.111 is NaN (no
  infinities); largest finite 448.
* The 2-bit copy's codes ("An elephant through a straw": 2-bit codes with one
  fp8 scale per group of 32 weights): the pages do not print the level
  values; the reading taken is a symmetric mid-rise quantiser, code q maps to
  (q - 1.5) times the group scale.

The routed MXFP4 experts are the checkpoint's format ("Running
DeepSeek-V4-Flash across four free GPUs", section "The model": FP4 experts
packed into I8 tensors with F8_E8M0 scale tensors alongside), with one scale
per 32 weights along K, and element 2j in the low nibble of byte j.
"""
from __future__ import annotations

import math

import numpy as np

# E2M1 magnitudes by the 3 low bits (exponent, mantissa): the subnormal
# pair 0, 0.5 then 2^(e-1) * (1 + m/2) for e = 1..3.
_E2M1_MAG = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)


def e2m1_value(code: int) -> float:
    mag = _E2M1_MAG[code & 7]
    return -mag if code & 8 else mag          # code 8 is -0.0


def e8m0_value(e: int) -> float:
    if e == 255:
        return math.nan
    return math.ldexp(1.0, e - 127)


def e4m3_value(b: int) -> float:
    s, ex, m = (b >> 7) & 1, (b >> 3) & 0xF, b & 7
    if ex == 0xF and m == 7:
        return math.nan
    if ex == 0:
        mag = math.ldexp(m / 8.0, -6)
    else:
        mag = math.ldexp(1.0 + m / 8.0, ex - 7)
    return -mag if s else mag


def int2_value(q: int) -> float:
    return (q & 3) - 1.5


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E8M0_TABLE = np.array([e8m0_value(e) for e in range(256)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)
INT2_TABLE = np.array([int2_value(q) for q in range(4)], dtype=np.float64)


# ----------------------------------------------------------------------------
# expert byte layout (canonical order: gate w1 [I,H], up w3 [I,H], down w2 [H,I])
# ----------------------------------------------------------------------------

MATRICES = ("w1", "w3", "w2")


def matrix_shape(name: str, H: int, I: int):
    return (I, H) if name in ("w1", "w3") else (H, I)


def fp4_layout(H: int, I: int):
    """{matrix: (codes_offset, scales_offset, N, K)} and total bytes of one MXFP4 expert."""
    if H % 32 or I % 32:
        raise ValueError("H and I must be multiples of 32 (one E8M0 scale per 32 weights)")
    off, lay = 0, {}
    for m in MATRICES:
        N, K = matrix_shape(m, H, I)
        c = off
        off += N * K // 2
        s = off
        off += N * K // 32
        lay[m] = (c, s, N, K)
    return lay, off


def int2_layout(H: int, I: int):
    if H % 32 or I % 32:
        raise ValueError("H and I must be multiples of 32")
    off, lay = 0, {}
    for m in MATRICES:
        N, K = matrix_shape(m, H, I)
        c = off
        off += N * K // 4
        s = off
        off += N * K // 32
        lay[m] = (c, s, N, K)
    return lay, off


def fp8_layout(H: int, I: int):
    off, lay = 0, {}
    for m in MATRICES:
        N, K = matrix_shape(m, H, I)
        c = off
        off += N * K
        s = off
        off += N * 4
        lay[m] = (c, s, N, K)
    return lay, off


def fp4_expert_nbytes(H: int, I: int) -> int:
    return fp4_layout(H, I)[1]


def int2_expert_nbytes(H: int, I: int) -> int:
    return int2_layout(H, I)[1]


def fp8_expert_nbytes(H: int, I: int) -> int:
    return fp8_layout(H, I)[1]


# ----------------------------------------------------------------------------
# matrix decoders
# ----------------------------------------------------------------------------

def decode_mxfp4(codes: np.ndarray, scales: np.ndarray, N: int, K: int) -> np.ndarray:
    """W[n, k] = E2M1(code of element k of row n) * E8M0(scale[n, k // 32])."""
    codes = np.asarray(codes, dtype=np.uint8).reshape(N, K // 2)
    scales = np.asarray(scales, dtype=np.uint8).reshape(N, K // 32)
    el = np.empty((N, K), dtype=np.float64)
    el[:, 0::2] = E2M1_TABLE[codes & 0xF]
    el[:, 1::2] = E2M1_TABLE[codes >> 4]
    return el * np.repeat(E8M0_TABLE[scales], 32, axis=1)


def decode_int2(codes: np.ndarray, scales: np.ndarray, N: int, K: int) -> np.ndarray:
    """W[n, k] = level(2-bit code of element k) * E4M3(scale[n, k // 32]); element 4j+q at bits 2q."""
    codes = np.asarray(codes, dtype=np.uint8).reshape(N, K // 4)
    scales = np.asarray(scales, dtype=np.uint8).reshape(N, K // 32)
    el = np.empty((N, K), dtype=np.float64)
    for q in range(4):
        el[:, q::4] = INT2_TABLE[(codes >> (2 * q)) & 3]
    return el * np.repeat(E4M3_TABLE[scales], 32, axis=1)


def decode_fp8_rows(codes: np.ndarray, rowscale_bytes: np.ndarray, N: int, K: int) -> np.ndarray:
    """W[n, k] = E4M3(code[n, k]) * rowscale[n] (rowscale stored as little-endian fp32)."""
    codes = np.asarray(codes, dtype=np.uint8).reshape(N, K)
    rs = np.frombuffer(np.ascontiguousarray(rowscale_bytes, dtype=np.uint8).tobytes(),
                       dtype="<f4").astype(np.float64)
    return E4M3_TABLE[codes] * rs[:, None]


def _decode_expert(blob: np.ndarray, H: int, I: int, layout_fn, dec):
    lay, total = layout_fn(H, I)
    blob = np.asarray(blob, dtype=np.uint8)
    if blob.size != total:
        raise ValueError(f"expert blob has {blob.size} bytes, expected {total}")
    res = {}
    names = list(lay.keys())
    for i, m in enumerate(names):
        c, s, N, K = lay[m]
        nxt = lay[names[i + 1]][0] if i + 1 < len(names) else total
        res[m] = dec(blob[c:s], blob[s:nxt], N, K)
    return res


def decode_fp4_expert(blob, H, I):
    """{'w1','w3','w2'} -> fp64 matrices of one canonical MXFP4 expert."""
    return _decode_expert(blob, H, I, fp4_layout, decode_mxfp4)


def decode_int2_expert(blob, H, I):
    return _decode_expert(blob, H, I, int2_layout, decode_int2)


def decode_fp8_expert(blob, H, I):
    return _decode_expert(blob, H, I, fp8_layout, decode_fp8_rows)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) widened exactly to fp64."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)
