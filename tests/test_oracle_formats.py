"""Pins for the oracle's decoders and byte layouts (CPU only)."""
import math
import os

import numpy as np
import pytest
import torch

from oracle import formats as F
from synth import configs, gen

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLD, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_e2m1_table_matches_ocp_values():
    rows = _golden_lines("e2m1_ocp_mx.txt")
    assert len(rows) == 16
    for code_bits, val in rows:
        code = int(code_bits, 2)
        got = F.E2M1_TABLE[code]
        assert got == float(val)
        assert math.copysign(1.0, got) == math.copysign(1.0, float(val))  # -0.0 for code 8


def test_e4m3_table_matches_library_fp8_cast():
    lib = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = F.E4M3_TABLE
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(mine))
    assert nan.sum() == 2                       # S.1111.111 only
    assert np.array_equal(lib[~nan], mine[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(mine[~nan]))
    assert np.nanmax(mine) == 448.0
    assert F.E4M3_TABLE[1] == 2.0 ** -9         # smallest subnormal


def test_e8m0_values():
    assert F.E8M0_TABLE[127] == 1.0
    assert F.E8M0_TABLE[124] == 0.125
    assert F.E8M0_TABLE[128] == 2.0
    assert F.E8M0_TABLE[0] == 2.0 ** -127
    assert F.E8M0_TABLE[254] == 2.0 ** 127
    assert math.isnan(F.E8M0_TABLE[255])


def test_expert_byte_counts_printed_on_pages():
    rows = {r[0]: r for r in _golden_lines("expert_bytes.txt")}
    H, I = 4096, 2048
    assert F.fp4_expert_nbytes(H, I) == int(rows["fp4_expert"][3])
    assert F.int2_expert_nbytes(H, I) == float(rows["int2_expert_mib"][3]) * 2 ** 20
    total = 43 * 256 * F.int2_expert_nbytes(H, I)
    assert round(total / 1e9) == int(rows["int2_all_layers_gb"][3])
    assert 43 * 256 == int(rows["layer_expert_pairs"][3])
    # tiny workload: 3 * (128*256/2 + 128*256/32)
    assert F.fp4_expert_nbytes(256, 128) == 52224
    # shared expert, FP8 codes plus one fp32 scale per output row
    assert F.fp8_expert_nbytes(H, I) == 25198592


def test_generator_layout_agrees_with_oracle_layout():
    # The generator and the oracle each define the canonical layout; the
    # scale regions the oracle reads must hold only the generator's scale range.
    wl = configs.TINY
    blob = gen.fp4_expert(wl, 0, 3)
    lay, total = F.fp4_layout(wl.H, wl.I)
    assert blob.size == total == gen.fp4_expert_nbytes(wl.H, wl.I)
    names = list(lay)
    for i, m in enumerate(names):
        c, s, N, K = lay[m]
        end = lay[names[i + 1]][0] if i + 1 < len(names) else total
        sc = blob[s:end]
        assert sc.size == N * K // 32
        assert sc.min() >= wl.scale_lo and sc.max() <= wl.scale_hi
        codes = blob[c:s]
        # uniform codes: every nibble value appears
        assert len(np.unique(codes & 0xF)) == 16 and len(np.unique(codes >> 4)) == 16


def test_mxfp4_nibble_order_and_block_scale():
    # One row, K = 64: byte j holds elements 2j (low nibble) and 2j+1 (high).
    codes = np.zeros((1, 32), dtype=np.uint8)
    codes[0, 0] = 0x21          # element 0 -> code 1 (0.5), element 1 -> code 2 (1.0)
    codes[0, 16] = 0xF7         # element 32 -> 6.0, element 33 -> -6.0
    scales = np.array([[127, 129]], dtype=np.uint8)   # block 0 x1, block 1 x4
    W = F.decode_mxfp4(codes, scales, 1, 64)
    assert W[0, 0] == 0.5 and W[0, 1] == 1.0
    assert W[0, 32] == 24.0 and W[0, 33] == -24.0
    assert np.count_nonzero(W) == 4


def test_int2_bit_order_and_scale():
    # element 4j+q at bits 2q..2q+1; byte 0xE4 = codes (0,1,2,3) for elements 0..3
    codes = np.zeros((1, 8), dtype=np.uint8)
    codes[0, 0] = 0xE4
    codes[0, 1:] = 0x55         # all codes 1 -> level -0.5
    sc = np.array([[0x38]], dtype=np.uint8)   # E4M3 0x38 = 1.0
    W = F.decode_int2(codes, sc, 1, 32)
    assert list(W[0, :4]) == [-1.5, -0.5, 0.5, 1.5]
    assert np.all(W[0, 4:] == -0.5)


def test_fp8_row_scales():
    codes = np.array([[0x38, 0xB8], [0x40, 0x00]], dtype=np.uint8)   # 1, -1 / 2, 0
    rs = np.array([3.0, 0.5], dtype="<f4").view(np.uint8)
    W = F.decode_fp8_rows(codes, rs, 2, 2)
    assert W.tolist() == [[3.0, -3.0], [1.0, 0.0]]


def test_bf16_widening_exact():
    v = np.array([1.0, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    bits = gen.bf16_bits(v)
    back = F.bf16_to_f64(bits)
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(back, ref)


def test_splitmix64_backends_agree():
    base = gen.stream_base(7, 1, 2, 3)
    a = gen.counter_bytes(base, 1000)
    b = gen.counter_bytes(base, 1000, device="cpu").numpy()
    assert np.array_equal(a, b)
    ra = gen.counter_range_bytes(base, 999, 124, 128)
    rb = gen.counter_range_bytes(base, 999, 124, 128, device="cpu").numpy()
    assert np.array_equal(ra, rb)
    # published SplitMix64 first output for seed 0 (state 0 advanced by the gamma)
    assert gen.splitmix64_int(0) == 0xE220A8397B1DCDAF
