"""Pins of the oracle's MX activation quantiser (OCP Microscaling Formats (MX)
Specification v1.0 conversion: 32-element blocks, X = 2^(floor(log2 amax) - 2),
E2M1 round-half-to-even, saturation at 6)."""
import math

import numpy as np
import pytest

from oracle.formats import E2M1_TABLE
from oracle.mxquant import block_scale_byte, e2m1_code, mx_dequantize, mx_quantize, mx_round


def _block(vals):
    b = np.zeros((1, 32))
    b[0, :len(vals)] = vals
    return b


def test_grid_values_are_exact():
    # amax = 6 * 2^e gives X = 2^e, so every signed grid value times X is kept exactly
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -.5, -1, -1.5, -2, -3, -4, -6])
    for e in (-10, -1, 0, 3, 20):
        v = _block(grid * 2.0 ** e)
        c, s = mx_quantize(v)
        assert s[0, 0] == 127 + e
        assert np.array_equal(mx_dequantize(c, s, 32), v)


@pytest.mark.parametrize("m,code", [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
                                    (0.2499, 0), (0.2501, 1), (0.7499, 1), (5.0001, 7)])
def test_ties_go_to_the_even_code(m, code):
    # X = 1 (amax 4): each midpoint between grid values takes the code with mantissa bit 0
    v = _block([4.0, m, -m])
    c, s = mx_quantize(v)
    assert s[0, 0] == 127
    assert c[0, 0] >> 4 == code                     # element 1 (m), high nibble of byte 0
    assert c[0, 1] & 0xF == (code | 8 if code else 0)  # element 2 (-m), low nibble of byte 1


def test_saturation_and_scale_choice():
    # amax in [4, 8) -> X = 1 (byte 127): 7 and 7.9 saturate to 6
    for amax in (4.0, 5.0, 7.0, 7.9):
        c, s = mx_quantize(_block([amax]))
        assert s[0, 0] == 127
        assert E2M1_TABLE[c[0, 0] & 0xF] == min(6.0, {4.0: 4.0, 5.0: 4.0}.get(amax, 6.0))
    # amax 8 -> X = 2
    c, s = mx_quantize(_block([8.0, 1.0]))
    assert s[0, 0] == 128 and E2M1_TABLE[c[0, 0] & 0xF] == 4.0 and E2M1_TABLE[c[0, 0] >> 4] == 0.5


def test_zero_and_tiny_blocks():
    c, s = mx_quantize(np.zeros((2, 64)))
    assert not c.any() and not s.any()               # X = 2^-127, all codes +0
    assert block_scale_byte(2.0 ** -126) == 0        # floor(log2) - 2 + 127 < 0 clamps to 0
    assert block_scale_byte(2.0 ** -124) == 1
    assert block_scale_byte(2.0 ** 127) == 252
    assert e2m1_code(-0.1) == 0                      # rounds to zero: stored as +0


def test_brute_force_nearest_grid_point():
    # every element is the grid point nearest to v / X (searched over all 15 values);
    # among two equally near points, the one whose code is even
    rng = np.random.default_rng(5)
    v = rng.standard_normal((6, 256)) * np.exp(rng.uniform(-8, 8, (6, 1)))
    v[0, :32] = 0.0
    c, s = mx_quantize(v)
    d = mx_dequantize(c, s, 256)
    grid = [(E2M1_TABLE[code], code) for code in range(16) if code != 8]
    for r in range(6):
        for b in range(8):
            blk = v[r, 32 * b:32 * b + 32]
            amax = np.max(np.abs(blk))
            X = 2.0 ** (math.floor(math.log2(amax)) - 2) if amax > 0 else 2.0 ** -127
            for i in range(32):
                q = blk[i] / X
                dist = [(abs(q - g), code & 1, g) for g, code in grid]
                best = min(dist)
                cands = [g for dd, odd, g in dist if dd == best[0]]
                want = min(cands, key=lambda g: [code & 1 for gg, code in grid if gg == g][0])
                want = max(-6.0, min(6.0, want))
                assert d[r, 32 * b + i] == want * X


def test_round_trip_and_error_bound():
    rng = np.random.default_rng(9)
    v = rng.standard_normal((4, 128))
    r = mx_round(v)
    assert np.array_equal(mx_round(r), r)             # quantised values are fixed points
    for b in range(4):
        blk, rb = v[:, 32 * b:32 * b + 32], r[:, 32 * b:32 * b + 32]
        amax = np.max(np.abs(blk), axis=1, keepdims=True)
        # half the widest grid gap (2 between 4 and 6) in units of X <= amax / 4, so |err| <= amax / 4
        assert np.all(np.abs(rb - blk) <= amax / 4 + 1e-300)


def test_nibble_order():
    c, s = mx_quantize(_block([1.0, 2.0, 3.0, 4.0]))   # X = 1
    assert c[0, 0] == (4 << 4) | 2 and c[0, 1] == (6 << 4) | 5
