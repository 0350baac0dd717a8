"""Overlapped forward (resident experts' pairs first, missed experts' pairs
after the copies) vs the plain forward and the oracle.

Each pair's arithmetic does not depend on which other pairs share its work
item, so the overlapped call must reproduce moe_expert_forward bit for bit,
and both must stay within max |err| <= 2e-2 * RMS of the oracle row."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.mlp import moe_layer
from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib, pinned_fp4_bank
from tests.test_gpu_forward import Pools, _route

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _overlap(M, P, x_bits, slots, w, miss_slots, event=None, parts=None):
    T, k = slots.shape
    y = torch.empty((T, P.wl.H), dtype=torch.int16, device="cuda")
    ws = torch.empty(M.moe_expert_forward_overlap_workspace(P.views, T, k), dtype=torch.uint8, device="cuda")
    err = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    ms = torch.tensor(list(miss_slots) + [0], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([len(miss_slots)], dtype=torch.int32, device="cuda")
    args = (P.views, torch.from_numpy(x_bits.view(np.int16)).cuda(), torch.from_numpy(slots.astype(np.int32)).cuda(),
            torch.from_numpy(w.astype(np.float32)).cuda(), ms, cnt, len(miss_slots) + 1)
    if parts is None:
        M.moe_expert_forward_overlap(*args, event, y, ws, err)
    elif parts == "staged":
        M.moe_expert_forward_overlap_staged(*args, event, [event], y, ws, err)
    elif parts == "staged3":
        M.moe_expert_forward_overlap_staged(*args, event, [event] * 3, y, ws, err)
    else:
        M.moe_expert_forward_overlap_parts(*args, [event] * parts, y, ws, err)
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(err)


@pytest.mark.parametrize("T,nmiss", [(4, 3), (16, 0), (16, 5), (64, 9), (64, 64)])
def test_overlap_equals_forward_decode_shape(T, nmiss):
    # T = 4, 16: CUDA-core path; T = 64: grouped GEMM for the routed pairs
    M = load_lib()
    wl = configs.DECODE
    S = 64
    P = Pools(M, wl, S, shared=True)
    rng = np.random.default_rng(300 + T + nmiss)
    slots, w = _route(rng, T, wl.k, S)
    slots[0, 1] = -1                                  # a skipped pair
    misses = rng.choice(S, size=nmiss, replace=False) if nmiss < S else np.arange(S)
    x = gen.activations(wl, 0, 7, T)
    y0, e0 = P.forward(x, slots, None, w)
    y1, e1 = _overlap(M, P, x, slots, w, misses)
    assert e0 == 0 and e1 == 0
    assert np.array_equal(y0, y1)
    sample = sorted({0, T // 2, T - 1})
    assert bf16_rel_err(y1[sample], P.reference(x, slots, None, w, tokens=sample)) <= TOL


@pytest.mark.parametrize("T,nmiss,parts", [(64, 9, 2), (64, 9, 4), (64, 1, 3), (64, 64, 3), (16, 5, 2),
                                           (64, 0, 2), (64, 9, "staged"), (16, 5, "staged"), (64, 64, "staged"),
                                           (64, 9, "staged3"), (64, 1, "staged3"), (16, 5, "staged3")])
def test_overlap_parts_equal_forward(T, nmiss, parts):
    # misses split into parts as the part-wise copy divides the list (a part
    # may be empty); every pair is still computed exactly once
    M = load_lib()
    wl = configs.DECODE
    S = 64
    P = Pools(M, wl, S, shared=True)
    rng = np.random.default_rng(700 + T + nmiss + (parts if isinstance(parts, int) else 7))
    slots, w = _route(rng, T, wl.k, S)
    misses = rng.choice(S, size=nmiss, replace=False) if nmiss < S else rng.permutation(S)
    x = gen.activations(wl, 0, 9, T)
    y0, e0 = P.forward(x, slots, None, w)
    y1, e1 = _overlap(M, P, x, slots, w, misses, parts=parts)
    assert e0 == 0 and e1 == 0
    assert np.array_equal(y0, y1)


def test_overlap_parts_rejects_bad_count():
    M = load_lib()
    wl = configs.TINY
    P = Pools(M, wl, 4, shared=True)
    x = gen.activations(wl, 0, 1, 2)
    slots = np.array([[0, 1], [2, 3]])
    w = np.full((2, 2), 0.5, np.float32)
    for parts in (0, M.MOE_MAX_COPY_PARTS + 1):
        with pytest.raises(M.MoeError):
            _overlap(M, P, x, slots, w, [1], parts=parts)


def test_overlap_small_all_tokens_and_error_clearing():
    M = load_lib()
    wl = configs.scaled(configs.TINY, H=512, I=512, E=16)
    P = Pools(M, wl, 6, shared=True)
    rng = np.random.default_rng(21)
    T, k = 50, 6                                       # 300 pairs: grouped GEMM path
    slots = np.stack([rng.choice(6, size=k, replace=False) for _ in range(T)])
    w = rng.random((T, k)).astype(np.float32)
    x = gen.activations(wl, 0, 3, T)
    y, err = _overlap(M, P, x, slots, w, [2, 5])
    assert err == 0
    assert bf16_rel_err(y, P.reference(x, slots, None, w)) <= TOL
    bad = slots.copy()
    bad[3, 0] = 9                                      # slot >= pool size: flagged, pair skipped
    _, err = _overlap(M, P, x, bad, w, [2])
    assert err == M.MOE_ERR_INVALID
    _, err = _overlap(M, P, x, slots, w, [2])          # the next call starts clean
    assert err == 0


def test_forward_error_is_cleared_by_next_call():
    M = load_lib()
    wl = configs.TINY
    P = Pools(M, wl, 2)
    x = gen.activations(wl, 0, 1, 1)
    w = np.array([[0.5, 0.5]], np.float32)
    assert P.forward(x, np.array([[0, 5]]), None, w)[1] == M.MOE_ERR_INVALID
    assert P.forward(x, np.array([[0, 1]]), None, w)[1] == 0


def _decoder(bank_np, B, wl):
    memo = {}

    def f(e, tag):
        if e not in memo:
            memo[e] = F.decode_fp4_expert(bank_np[e * B:(e + 1) * B], wl.H, wl.I)
        return memo[e]
    return f


@pytest.mark.parametrize("wl,S,steps,full,parts", [
    (configs.TINY, 4, 6, True, 2),                                   # chunked
    (configs.scaled(configs.DECODE, T=4), 64, 4, False, 1),          # single chunk, CUDA-core path
    (configs.scaled(configs.DECODE, T=64), 40, 3, False, 1),         # chunked, grouped GEMM, staged copies
    (configs.scaled(configs.DECODE, T=64), 64, 3, False, (1, 2)),    # staged, down matrices in two parts
    (configs.scaled(configs.DECODE, T=64), 64, 3, False, (1, 3)),    # staged, down matrices in three parts
    (configs.scaled(configs.DECODE, T=64), 40, 3, False, 2),         # chunked, grouped GEMM, two parts
    (configs.scaled(configs.DECODE, T=64), 64, 3, False, 3),         # grouped GEMM, three copy parts
])
def test_layer_overlapped_copy(wl, S, steps, full, parts):
    M = load_lib()
    bank, B = pinned_fp4_bank(wl, (0,))
    slots = torch.empty(S * B, dtype=torch.uint8, device="cuda")
    cache = M.moe_cache(S, 1, wl.E, B, slots, bank)
    sh = torch.from_numpy(gen.shared_expert(wl, 0)).cuda() if wl.shared else None
    views = M.make_views(wl.H, wl.I, slots, S, None, 0, sh)
    cp, dp = parts if isinstance(parts, tuple) else (parts, 1)
    runner = M.DecodeLayerRunner(cache, views, wl.E, wl.k, wl.T, copy="device", overlap=True, copy_parts=cp,
                                 down_parts=dp)
    ref = SlotCacheLRU(S, 1, wl.E)
    dec = _decoder(bank.numpy(), B, wl)
    shw = F.decode_fp8_expert(gen.shared_expert(wl, 0), wl.H, wl.I) if wl.shared else None
    T = wl.T
    for step in range(steps):
        lg = gen.router_logits(wl, 0, step, T)
        x = gen.activations(wl, 0, step, T)
        y = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
        runner.run(0, torch.from_numpy(lg).cuda(), torch.from_numpy(x.view(np.int16)).cuda(), y)
        torch.cuda.synchronize()
        ids, w = router_topk(lg, wl.k)
        tb = 0
        while tb < T:
            _, _, _, tb = ref.ensure(0, ids, 0, wl.k, FETCH, tb)
        assert np.array_equal(cache.export()[0], ref.state()[0])
        rows = list(range(T)) if full else sorted({0, T // 3, T // 2 + 1, T - 1})
        r = moe_layer(x, ids, w, dec, shared=shw, tokens=None if full else rows)
        assert bf16_rel_err(y.cpu().numpy()[rows], r) <= TOL
    runner.check()
    assert runner.stats["misses"] > 0
    cache.close()
