"""Seeded synthetic inputs for the routed MoE layer.

This module draws bytes and numbers; it computes no part of the MoE layer
(no decoding, routing, caching or matrix work).  Both the CUDA path and the
CPU oracle consume exactly the bytes it returns.

Routed-expert weight bytes come from a counter-based generator (SplitMix64,
G. Steele, D. Lea, C. Flood, "Fast splittable pseudorandom number
generators", OOPSLA 2014) so that any byte range of any expert can be
produced independently, on the host with NumPy or on a device with torch
integer ops, with identical results.  Everything small (activations, router
logits, the 2-bit copy's fp8 scales, the shared expert) comes from NumPy's
PCG64 keyed by a SeedSequence per (seed, stream, layer, step).

Byte formats (the canonical layout that both sides read):

* MXFP4 expert: for each matrix in the order gate ``w1`` [I,H], up ``w3``
  [I,H], down ``w2`` [H,I]: codes ``[N][K/2]`` (two E2M1 codes per byte,
  element 2j in the low nibble), then E8M0 scales ``[N][K/32]``.
* 2-bit copy: same matrix order, codes ``[N][K/4]`` (element 4j+q at bits
  2q..2q+1), then E4M3 scales ``[N][K/32]``.
* Shared expert: same matrix order, E4M3 codes ``[N][K]``, then fp32 row
  scales ``[N]``.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np

from .configs import Workload

_M64 = (1 << 64) - 1
_GOLDEN = 0x9E3779B97F4A7C15
_MIX1 = 0xBF58476D1CE4E5B9
_MIX2 = 0x94D049BB133111EB


# ----------------------------------------------------------------------------
# SplitMix64, three implementations of one published definition
# ----------------------------------------------------------------------------

def splitmix64_int(x: int) -> int:
    """SplitMix64 finaliser of (x + golden gamma), on Python ints."""
    z = (x + _GOLDEN) & _M64
    z = ((z ^ (z >> 30)) * _MIX1) & _M64
    z = ((z ^ (z >> 27)) * _MIX2) & _M64
    return z ^ (z >> 31)


def splitmix64_np(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.uint64, copy=False)
    with np.errstate(over="ignore"):
        z = x + np.uint64(_GOLDEN)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(_MIX1)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(_MIX2)
        return z ^ (z >> np.uint64(31))


def _signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def splitmix64_torch(x):
    """Same function on int64 torch tensors (two's-complement wrap; logical shifts by mask)."""
    def srl(z, s):
        return (z >> s) & ((1 << (64 - s)) - 1)
    z = x + _signed(_GOLDEN)
    z = (z ^ srl(z, 30)) * _signed(_MIX1)
    z = (z ^ srl(z, 27)) * _signed(_MIX2)
    return z ^ srl(z, 31)


def stream_base(*key: int) -> int:
    h = 0
    for v in key:
        h = splitmix64_int(h ^ (int(v) & _M64))
    return h


def _words_np(base: int, start: int, n: int) -> np.ndarray:
    idx = np.arange(start, start + n, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return splitmix64_np(idx + np.uint64(base))


def _words_torch(base: int, start: int, n: int, device):
    import torch
    idx = torch.arange(start, start + n, dtype=torch.int64, device=device)
    return splitmix64_torch(idx + _signed(base))


def counter_bytes(base: int, nbytes: int, device=None):
    """``nbytes`` uniform bytes of stream ``base``: byte i is byte (i mod 8) of word i//8."""
    nw = (nbytes + 7) // 8
    if device is None:
        return _words_np(base, 0, nw).view(np.uint8)[:nbytes]
    return _words_torch(base, 0, nw, device).view(__import__("torch").uint8)[:nbytes]


def counter_range_bytes(base: int, n: int, lo: int, hi: int, device=None):
    """``n`` bytes uniform in [lo, hi]: lo + (high 32 bits of word i) mod (hi - lo + 1)."""
    span = hi - lo + 1
    if device is None:
        w = _words_np(base, 0, n)
        return (lo + ((w >> np.uint64(32)) % np.uint64(span))).astype(np.uint8)
    import torch
    w = _words_torch(base, 0, n, device)
    hi32 = (w >> 32) & 0xFFFFFFFF
    return (lo + hi32 % span).to(torch.uint8)


# ----------------------------------------------------------------------------
# byte-layout sizes (format definitions, not arithmetic of the method)
# ----------------------------------------------------------------------------

def fp4_regions(H: int, I: int):
    """(name, nbytes, kind) for the canonical MXFP4 expert, in storage order."""
    out = []
    for name, N, K in (("w1", I, H), ("w3", I, H), ("w2", H, I)):
        out.append((name + ".codes", N * K // 2, "codes"))
        out.append((name + ".scales", N * K // 32, "scales"))
    return out


def int2_regions(H: int, I: int):
    out = []
    for name, N, K in (("w1", I, H), ("w3", I, H), ("w2", H, I)):
        out.append((name + ".codes", N * K // 4, "codes"))
        out.append((name + ".scales", N * K // 32, "scales"))
    return out


def fp4_expert_nbytes(H: int, I: int) -> int:
    return sum(n for _, n, _ in fp4_regions(H, I))


def int2_expert_nbytes(H: int, I: int) -> int:
    return sum(n for _, n, _ in int2_regions(H, I))


def shared_nbytes(H: int, I: int) -> int:
    return 3 * H * I + (2 * I + H) * 4


_TAG_FP4 = 0x46503400
_TAG_INT2 = 0x494E5432


def fp4_expert(wl: Workload, layer: int, expert: int, device=None):
    """Canonical MXFP4 bytes of routed expert ``expert`` of ``layer``."""
    parts = []
    for ri, (_, n, kind) in enumerate(fp4_regions(wl.H, wl.I)):
        base = stream_base(wl.seed, _TAG_FP4, layer, expert, ri)
        if kind == "codes":
            parts.append(counter_bytes(base, n, device))
        else:
            parts.append(counter_range_bytes(base, n, wl.scale_lo, wl.scale_hi, device))
    if device is None:
        return np.concatenate(parts)
    import torch
    return torch.cat(parts)


def fp4_bank_into(wl: Workload, layer: int, out, experts: Optional[Iterable[int]] = None,
                  device=None, first_expert_offset: int = 0):
    """Write experts of ``layer`` into ``out`` (uint8, indexed ``[(e - first) * B ...]``)."""
    B = fp4_expert_nbytes(wl.H, wl.I)
    experts = range(wl.E) if experts is None else experts
    for e in experts:
        o = (e - first_expert_offset) * B
        out[o:o + B] = fp4_expert(wl, layer, e, device)
    return out


def _rng(seed: int, *stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


_S_X, _S_LOGIT, _S_ZIPF, _S_INT2S, _S_SHARED, _S_REUSE = 11, 12, 13, 14, 15, 16


def _f32_to_e4m3_bytes(v: np.ndarray) -> np.ndarray:
    """OCP E4M3 bytes of float32 values by the library cast (round to nearest even)."""
    import torch
    v = np.clip(v, -448.0, 448.0).astype(np.float32)
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def int2_expert(wl: Workload, layer: int, expert: int) -> np.ndarray:
    """Canonical 2-bit-copy bytes: uniform codes, E4M3 scales of |N(0,1)|."""
    parts = []
    rng = _rng(wl.seed, _S_INT2S, layer, expert)
    for ri, (_, n, kind) in enumerate(int2_regions(wl.H, wl.I)):
        if kind == "codes":
            parts.append(counter_bytes(stream_base(wl.seed, _TAG_INT2, layer, expert, ri), n))
        else:
            parts.append(_f32_to_e4m3_bytes(np.abs(rng.standard_normal(n, dtype=np.float32))))
    return np.concatenate(parts)


def shared_expert(wl: Workload, layer: int) -> np.ndarray:
    """Shared expert bytes: E4M3 codes of N(0,1) and fp32 row scales uniform in [1, 4)."""
    rng = _rng(wl.seed, _S_SHARED, layer)
    H, I = wl.H, wl.I
    parts = []
    for N, K in ((I, H), (I, H), (H, I)):
        parts.append(_f32_to_e4m3_bytes(rng.standard_normal(N * K, dtype=np.float32)))
        parts.append(rng.uniform(1.0, 4.0, N).astype(np.float32).view(np.uint8))
    return np.concatenate(parts)


def activations(wl: Workload, layer: int, step: int, T: Optional[int] = None) -> np.ndarray:
    """bf16 N(0,1) activations [T, H] as uint16 bit patterns (library cast, RNE)."""
    import torch
    T = wl.T if T is None else T
    v = _rng(wl.seed, _S_X, layer, step, T).standard_normal((T, wl.H), dtype=np.float32)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def zipf_bias(wl: Workload, layer: int) -> np.ndarray:
    """Per-expert popularity bias -s*ln(rank), ranks from a seeded permutation."""
    E = wl.E
    if wl.zipf_s is None:
        return np.zeros(E, dtype=np.float32)
    rank = np.empty(E, dtype=np.int64)
    rank[_rng(wl.seed, _S_ZIPF, layer).permutation(E)] = np.arange(1, E + 1)
    return (-wl.zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)


def router_logits(wl: Workload, layer: int, step: int, T: Optional[int] = None) -> np.ndarray:
    """fp32 logits [T, E] = N(0,1) + popularity bias (+ reuse boost for the stack)."""
    T = wl.T if T is None else T
    base = _rng(wl.seed, _S_LOGIT, layer, step, T).standard_normal((T, wl.E), dtype=np.float32)
    out = base + zipf_bias(wl, layer)[None, :]
    if wl.reuse is not None:
        out = out + (wl.reuse_boost * preferred_sets(wl, layer, step, T)).astype(np.float32)
    return out.astype(np.float32)


def preferred_sets(wl: Workload, layer: int, step: int, T: Optional[int] = None) -> np.ndarray:
    """Multi-hot [T, E] of each token's preferred experts at ``step``.

    Step 0 draws k experts per token by popularity without replacement; at each
    later step every member is kept with probability ``reuse`` and otherwise
    replaced by a fresh popularity draw outside the set.  This evolves without
    ever running the router.
    """
    T = wl.T if T is None else T
    E, k = wl.E, wl.k
    p = np.exp(zipf_bias(wl, layer).astype(np.float64))
    p /= p.sum()
    rng = _rng(wl.seed, _S_REUSE, layer, T)
    sets = [list(rng.choice(E, size=k, replace=False, p=p)) for _ in range(T)]
    for _ in range(step):
        for t in range(T):
            cur = sets[t]
            for j in range(k):
                if rng.random() >= wl.reuse:
                    q = p.copy()
                    q[cur] = 0.0
                    q /= q.sum()
                    cur[j] = int(rng.choice(E, p=q))
    m = np.zeros((T, E), dtype=np.float32)
    for t in range(T):
        m[t, sets[t]] = 1.0
    return m


def uniform_bytes(seed: int, n: int, *stream: int) -> np.ndarray:
    return _rng(seed, *stream).integers(0, 256, n, dtype=np.uint8)


def normal_f32(seed: int, shape, *stream: int) -> np.ndarray:
    return _rng(seed, *stream).standard_normal(shape, dtype=np.float32)


def bf16_bits(v: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns of float32 values via the library cast (RNE)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(v, dtype=np.float32)).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
