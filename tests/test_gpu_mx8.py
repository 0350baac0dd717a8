"""The block-scaled decode GEMM (tcgen05.mma.kind::mxf8f6f4: E2M1 weights as
stored, activations and h as two E4M3 terms with a power-of-two scale per 32
elements) against the oracle, and against the warp-level kernels it replaces.

Cases: groups of 1..48 rows (the hi and lo rows stack into one B operand of
up to 96 rows) and slots with more pairs than that, cut into groups of 48;
a generic shape (H = 1024, I = 512); the tiny shape, which the path does not
take (H, I not multiples of 512: the CUDA-core kernels run it); every token
of a full-size batch; FP8 shared expert on and off; run-to-run bit
equality.  Layer outputs within max |err| <= 2e-2 * RMS of the
oracle row.
"""
import numpy as np
import pytest
import torch

from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib
from tests.test_gpu_forward import Pools, _route

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _set(M, opt, value):
    return M.moe_set_option(opt, value)


@pytest.fixture
def mx8_on():
    M = load_lib()
    old_min = _set(M, M.MOE_OPT_MX8_MIN_TOKENS, 2)
    old_max = _set(M, M.MOE_OPT_MMA_MAX_TOKENS, 64)
    yield M
    _set(M, M.MOE_OPT_MX8_MIN_TOKENS, old_min)
    _set(M, M.MOE_OPT_MMA_MAX_TOKENS, old_max)


@pytest.mark.parametrize("T", [2, 5, 16, 33, 64])
def test_full_size_every_token(mx8_on, T):
    M = mx8_on
    wl = configs.DECODE
    P = Pools(M, wl, 20, shared=True)
    rng = np.random.default_rng(700 + T)
    slots, w = _route(rng, T, wl.k, 20)
    x = gen.activations(wl, 0, 40 + T, T)
    y, err = P.forward(x, slots, None, w)
    assert err == 0
    tokens = list(range(T)) if T <= 16 else sorted(set(range(0, T, 5)) | {T - 1})
    ref = P.reference(x, slots, None, w, tokens=tokens)
    assert bf16_rel_err(y[tokens], ref) <= TOL


@pytest.mark.parametrize("n_hot", [47, 48, 49, 64])
def test_groups_at_the_48_row_cut(mx8_on, n_hot):
    # slot 0 takes n_hot tokens: one group of 47 or 48 rows (N = 96), or a
    # group of 48 and one of 1 or 16; the rest spread over the other slots
    M = mx8_on
    wl = configs.scaled(configs.DECODE, H=1024, I=512)
    P = Pools(M, wl, 10, shared=True)
    rng = np.random.default_rng(n_hot)
    T, k = 64, 4
    slots = np.stack([1 + rng.permutation(9)[:k] for _ in range(T)])
    slots[:n_hot, 0] = 0
    w = rng.random((T, k)).astype(np.float32) + 0.05
    w /= w.sum(1, keepdims=True)
    x = gen.activations(wl, 0, 60, T)
    y, err = P.forward(x, slots, None, w)
    assert err == 0
    tokens = list(range(0, T, 3)) + [n_hot - 1, T - 1]
    ref = P.reference(x, slots, None, w, tokens=sorted(set(tokens)))
    assert bf16_rel_err(y[sorted(set(tokens))], ref) <= TOL


def test_slot_with_more_pairs_than_tokens(mx8_on):
    # a token's pairs may name one slot twice: slot 0 takes two pairs of every
    # token (128 or more pairs), cut into groups of 48 rows
    M = mx8_on
    wl = configs.scaled(configs.DECODE, H=1024, I=512)
    P = Pools(M, wl, 3, shared=False)
    rng = np.random.default_rng(5)
    T, k = 64, 4
    slots = np.zeros((T, k), dtype=np.int64)
    slots[:, 2] = rng.integers(1, 3, size=T)
    slots[:, 3] = rng.integers(0, 3, size=T)
    w = rng.random((T, k)).astype(np.float32) + 0.05
    w /= w.sum(1, keepdims=True)
    x = gen.activations(wl, 0, 61, T)
    y, err = P.forward(x, slots, None, w)
    assert err == 0
    tokens = [0, 1, 31, 62, 63]
    ref = P.reference(x, slots, None, w, tokens=tokens)
    assert bf16_rel_err(y[tokens], ref) <= TOL


@pytest.mark.parametrize("shared", [False, True])
def test_tiny_shape(mx8_on, shared):
    M = mx8_on
    wl = configs.TINY
    P = Pools(M, wl, wl.S, shared=shared)
    rng = np.random.default_rng(8)
    for T in (2, 4, 13, 64):
        slots, w = _route(rng, T, wl.k, wl.S)
        x = gen.activations(wl, 0, 70 + T, T)
        y, err = P.forward(x, slots, None, w)
        assert err == 0
        assert bf16_rel_err(y, P.reference(x, slots, None, w)) <= TOL


@pytest.mark.parametrize("T", [8, 64])
def test_repeatable_and_warp_mma_agree_with_oracle(mx8_on, T):
    M = mx8_on
    wl = configs.DECODE
    P = Pools(M, wl, 16, shared=True)
    rng = np.random.default_rng(900 + T)
    slots, w = _route(rng, T, wl.k, 16)
    x = gen.activations(wl, 0, 80, T)
    y1, e1 = P.forward(x, slots, None, w)
    y2, e2 = P.forward(x, slots, None, w)
    assert e1 == 0 and e2 == 0
    assert np.array_equal(y1, y2)
    _set(M, M.MOE_OPT_MX8_MIN_TOKENS, 0)
    y3, e3 = P.forward(x, slots, None, w)
    assert e3 == 0
    sample = list(range(T)) if T <= 8 else sorted({0, T // 2, T - 1})
    ref = P.reference(x, slots, None, w, tokens=sample)
    assert bf16_rel_err(y1[sample], ref) <= TOL
    assert bf16_rel_err(y3[sample], ref) <= TOL
