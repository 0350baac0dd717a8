"""Pins for the ladder, the expert MLP, the combine and the pair grouping (CPU only)."""
import math

import numpy as np
import pytest

from oracle import formats as F
from oracle.ladder import TAG_DROP, TAG_FP4, TAG_INT2, ladder_classify
from oracle.mlp import expert_mlp, moe_layer, rms_carry, silu
from oracle.permute import group_pairs
from oracle.slot_cache import FETCH, CapacityError, SlotCacheLRU
from synth import gen


# ------------------------------------------------------------------ ladder ----

def test_ladder_all_resident_keeps_everything():
    c4, c2 = SlotCacheLRU(8, 1, 16), SlotCacheLRU(8, 1, 16)
    ids = np.array([[0, 1, 2, 3, 4, 5]])
    c4.ensure(0, ids, 0, 6, FETCH)
    w = np.array([[0.3, 0.2, 0.2, 0.1, 0.1, 0.1]])
    slots, tags, wo, m4, m2, done = ladder_classify(c4, c2, 0, ids, w, 2, 4)
    assert (tags == TAG_FP4).all() and done == 1
    assert np.allclose(wo, w, atol=0) and m4 == ([], []) and m2 == ([], [])


def test_ladder_cold_pools_drop_tail_and_renormalise():
    c4, c2 = SlotCacheLRU(8, 1, 16), SlotCacheLRU(8, 1, 16)
    ids = np.array([[9, 8, 7, 6, 5, 4]])
    w = np.array([[0.4, 0.2, 0.15, 0.1, 0.1, 0.05]])
    slots, tags, wo, m4, m2, _ = ladder_classify(c4, c2, 0, ids, w, 2, 4)
    assert tags[0].tolist() == [TAG_FP4, TAG_FP4, TAG_INT2, TAG_INT2, TAG_DROP, TAG_DROP]
    assert m4[0] == [9, 8] and m2[0] == [7, 6]
    top4 = w[0, :4] / w[0, :4].sum()
    assert np.allclose(wo[0, :4], top4, atol=1e-15) and wo[0, 4:].tolist() == [0, 0]
    assert slots[0, 4:].tolist() == [-1, -1]


def test_ladder_residency_judged_after_earlier_passes():
    # token 0 fetches experts 1,2 in FP4 (pass i); token 1's rank-5 expert 1 and
    # rank-3 expert 2 then hit FP4; its rank-6 expert 3 hits the 2-bit copy that
    # token 0's rank-3 miss fetched in pass ii.
    c4, c2 = SlotCacheLRU(8, 1, 16), SlotCacheLRU(8, 1, 16)
    ids = np.array([[1, 2, 3, 10, 11, 12],
                    [13, 14, 2, 15, 1, 3]])
    w = np.full((2, 6), 1.0 / 6)
    slots, tags, wo, m4, m2, _ = ladder_classify(c4, c2, 0, ids, w, 2, 4)
    assert tags[1].tolist() == [TAG_FP4, TAG_FP4, TAG_FP4, TAG_INT2, TAG_FP4, TAG_INT2]
    assert tags[0].tolist() == [TAG_FP4, TAG_FP4, TAG_INT2, TAG_INT2, TAG_DROP, TAG_DROP]
    assert slots[1, 4] == slots[0, 0] and slots[1, 2] == slots[0, 1]
    assert slots[1, 5] == slots[0, 2]
    assert np.allclose(wo.sum(1), 1.0, atol=1e-15)


def test_ladder_capacity():
    c4, c2 = SlotCacheLRU(1, 1, 16), SlotCacheLRU(8, 1, 16)
    with pytest.raises(CapacityError):
        ladder_classify(c4, c2, 0, np.array([[1, 2, 3, 4, 5, 6]]), np.full((1, 6), 1 / 6), 2, 4)


def test_ladder_chunks_by_both_pools():
    c4, c2 = SlotCacheLRU(4, 1, 32), SlotCacheLRU(2, 1, 32)
    ids = np.array([[0, 1, 10, 11, 20, 21], [2, 3, 12, 13, 22, 23]])
    *_, done = ladder_classify(c4, c2, 0, ids, np.full((2, 6), 1 / 6), 2, 4)
    assert done == 1          # the 2-bit pool fits only token 0's ranks 3..4


# --------------------------------------------------------------------- mlp ----

def _loop_mlp(x, W):
    I, H = W["w1"].shape
    out = []
    for xr in x:
        h = []
        for n in range(I):
            g = sum(W["w1"][n, kk] * xr[kk] for kk in range(H))
            u = sum(W["w3"][n, kk] * xr[kk] for kk in range(H))
            h.append(g / (1.0 + math.exp(-g)) * u if g > -700 else 0.0 * u)
        out.append([sum(W["w2"][m, n] * h[n] for n in range(I)) for m in range(H)])
    return np.array(out)


def test_expert_mlp_matches_pure_python_loop():
    rng = np.random.default_rng(1)
    H, I = 64, 32
    blob = rng.integers(0, 256, F.fp4_expert_nbytes(H, I), dtype=np.uint8)
    lay, _ = F.fp4_layout(H, I)
    for m, (c, s, N, K) in lay.items():
        blob[s:s + N * K // 32] = rng.integers(124, 129, N * K // 32)
    W = F.decode_fp4_expert(blob, H, I)
    x = rng.standard_normal((3, H))
    assert np.allclose(expert_mlp(x, W), _loop_mlp(x, W), rtol=1e-12, atol=1e-9)


def _rank_one_expert(H, I, pattern, a_row, b_blk):
    """Canonical bytes whose decoded matrices are W[n, k] = v_k * 2^(a_n + b_{k//32})."""
    lay, total = F.fp4_layout(H, I)
    blob = np.zeros(total, dtype=np.uint8)
    for m, (c, s, N, K) in lay.items():
        codes = np.array([pattern[kk % len(pattern)] for kk in range(K)], dtype=np.uint8)
        packed = (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)
        blob[c:s] = np.tile(packed, N)
        sc = np.array([[127 + a_row[m][n] + b_blk[m][bb] for bb in range(K // 32)]
                       for n in range(N)], dtype=np.uint8)
        blob[s:s + N * K // 32] = sc.reshape(-1)
    return blob


def test_expert_mlp_rank_one_closed_form():
    H, I = 64, 96
    pattern = [1, 7, 10, 3, 12, 0, 5, 14, 2]      # asymmetric code pattern along K
    rng = np.random.default_rng(2)
    a_row = {m: rng.integers(-2, 3, N) for m, N in (("w1", I), ("w3", I), ("w2", H))}
    b_blk = {m: rng.integers(-2, 3, K // 32) for m, K in (("w1", H), ("w3", H), ("w2", I))}
    blob = _rank_one_expert(H, I, pattern, a_row, b_blk)
    W = F.decode_fp4_expert(blob, H, I)
    x = rng.standard_normal(H)
    v = lambda K: [F.e2m1_value(pattern[kk % len(pattern)]) for kk in range(K)]
    vH, vI = v(H), v(I)
    cg = sum(vH[kk] * 2.0 ** b_blk["w1"][kk // 32] * x[kk] for kk in range(H))
    cu = sum(vH[kk] * 2.0 ** b_blk["w3"][kk // 32] * x[kk] for kk in range(H))
    h = [0.0] * I
    for n in range(I):
        g = 2.0 ** a_row["w1"][n] * cg
        u = 2.0 ** a_row["w3"][n] * cu
        h[n] = g / (1.0 + math.exp(-g)) * u
    cd = sum(vI[n] * 2.0 ** b_blk["w2"][n // 32] * h[n] for n in range(I))
    want = np.array([2.0 ** a_row["w2"][m] * cd for m in range(H)])
    got = expert_mlp(x[None, :], W)[0]
    assert np.allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_silu_special_values():
    assert silu(np.array([0.0]))[0] == 0.0
    assert silu(np.array([-1000.0]))[0] == 0.0
    assert silu(np.array([1000.0]))[0] == 1000.0
    assert math.isclose(silu(np.array([1.0]))[0], 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)


def test_moe_layer_combine_invariants():
    rng = np.random.default_rng(3)
    H, I, T, k = 64, 32, 3, 2
    blob = _rank_one_expert(H, I, [2, 9, 4], {m: np.zeros(64, int) for m in ("w1", "w3", "w2")},
                            {m: np.zeros(4, int) for m in ("w1", "w3", "w2")})
    W = F.decode_fp4_expert(blob, H, I)
    x_bits = gen.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    ids = np.array([[0, 1], [1, 0], [2, 0]])
    w = np.array([[0.7, 0.3], [0.5, 0.5], [0.9, 0.1]])
    # identical experts: the weights sum to one, so y equals one expert's output
    y = moe_layer(x_bits, ids, w, lambda e, tag: W)
    x = F.bf16_to_f64(x_bits)
    assert np.allclose(y, expert_mlp(x, W), rtol=1e-12, atol=1e-9)
    # the shared expert adds with weight one
    ys = moe_layer(x_bits, ids, w, lambda e, tag: W, shared=W)
    assert np.allclose(ys, 2 * y, rtol=1e-12, atol=1e-9)
    # a dropped pair contributes nothing
    tags = np.zeros((T, k), dtype=int)
    tags[:, 1] = 2
    yd = moe_layer(x_bits, ids, np.stack([w[:, 0], w[:, 1]], 1), lambda e, tag: W, tags=tags)
    assert np.allclose(yd, w[:, :1] * expert_mlp(x, W), rtol=1e-12, atol=1e-9)


def test_rms_carry_unit_rms():
    y = np.array([[3.0, 4.0], [0.0, 0.0]])
    c = rms_carry(y, eps=0.0 + 1e-6)
    assert np.allclose(np.sqrt(np.mean(c[0] ** 2)), 1.0, atol=1e-6)
    assert np.all(c[1] == 0.0)


def test_rms_carry_eps_inside_the_root():
    # a row whose mean square equals eps: the divisor is sqrt(2 eps), so every
    # element becomes +-1/sqrt(2) (eps outside the root, or a sum in place of the
    # mean, would give ~1 or 1/2); rows are independent and signs are kept
    y = np.array([[1e-3, -1e-3], [30.0, -40.0]])
    c = rms_carry(y, eps=1e-6)
    assert np.allclose(c[0], [2 ** -0.5, -(2 ** -0.5)], rtol=1e-12)
    assert np.allclose(c[1], np.array([30.0, -40.0]) / np.sqrt(1250.0 + 1e-6), rtol=1e-12)
    # scale invariance far above eps
    assert np.allclose(rms_carry(7.0 * y[1:], eps=1e-6), c[1:], rtol=1e-9)


# ----------------------------------------------------------------- permute ----

def test_group_pairs_matches_buckets():
    rng = np.random.default_rng(4)
    ids = rng.integers(-1, 9, size=(20, 3))
    off, perm = group_pairs(ids, 9)
    flat = ids.reshape(-1)
    buckets = []
    for e in range(9):
        buckets += [p for p in range(flat.size) if flat[p] == e]
    assert list(perm) == buckets
    for e in range(9):
        assert off[e + 1] - off[e] == sum(1 for v in flat if v == e)
    assert off[-1] == sum(1 for v in flat if v >= 0)
