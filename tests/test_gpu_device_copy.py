"""Device-driven miss copy and the enqueue-ahead layer mode vs the oracle.

moe_copy_missing_device must leave every listed slot byte-equal to its bank
expert; ensure in MOE_FETCH_MARK_REST mode must agree with the oracle's
ensure on the chunk it processes and mark the later tokens' entries -1; the
runner's copy="device" mode must give the same layer outputs and slot table
as the oracle, with and without capacity chunking.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.mlp import moe_layer
from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib, pinned_fp4_bank

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _cache(M, wl, S):
    bank, B = pinned_fp4_bank(wl, (0,))
    slots = torch.zeros(S * B, dtype=torch.uint8, device="cuda")
    return bank, B, slots, M.moe_cache(S, 1, wl.E, B, slots, bank)


def test_copy_missing_device_bytes():
    M = load_lib()
    wl = configs.scaled(configs.TINY, E=16)
    bank, B, slots, cache = _cache(M, wl, 8)
    keys = torch.tensor([3, 15, 0, 7, 99, 2], dtype=torch.int32, device="cuda")   # 99: out of range
    sl = torch.tensor([5, 0, 7, 2, 1, 9], dtype=torch.int32, device="cuda")       # 9: out of range
    cnt = torch.tensor([6], dtype=torch.int32, device="cuda")
    M.moe_copy_missing_device(cache, keys, sl, cnt)
    torch.cuda.synchronize()
    got = slots.cpu().numpy().reshape(8, B)
    b = bank.numpy().reshape(wl.E, B)
    for key, s in [(3, 5), (15, 0), (0, 7), (7, 2)]:
        assert np.array_equal(got[s], b[key])
    for s in (1, 3, 4, 6):
        assert not got[s].any()
    cnt.zero_()
    slots.zero_()
    M.moe_copy_missing_device(cache, keys, sl, cnt)     # empty list: nothing written
    torch.cuda.synchronize()
    assert not slots.cpu().numpy().any()
    cache.close()


@pytest.mark.parametrize("n", [0, 1, 2, 5, 7])
def test_copy_missing_device_parts(n):
    # part q of n_parts copies list entries [n q / n_parts, n (q + 1) / n_parts)
    M = load_lib()
    wl = configs.scaled(configs.TINY, E=16)
    bank, B, slots, cache = _cache(M, wl, 8)
    b = bank.numpy().reshape(wl.E, B)
    rng = np.random.default_rng(40 + n)
    keys_np = rng.choice(wl.E, size=n, replace=False).astype(np.int32)
    sl_np = rng.choice(8, size=n, replace=False).astype(np.int32)
    keys = torch.from_numpy(np.concatenate([keys_np, [0]]).astype(np.int32)).cuda()
    sl = torch.from_numpy(np.concatenate([sl_np, [0]]).astype(np.int32)).cuda()
    cnt = torch.tensor([n], dtype=torch.int32, device="cuda")
    for parts in (1, 2, 3, 4):
        for q in range(parts):
            slots.zero_()
            M.moe_copy_missing_device_part(cache, keys, sl, cnt, q, parts)
            torch.cuda.synchronize()
            got = slots.cpu().numpy().reshape(8, B)
            mine = set(range(n * q // parts, n * (q + 1) // parts))
            for i in range(n):
                if i in mine:
                    assert np.array_equal(got[sl_np[i]], b[keys_np[i]])
                else:
                    assert not got[sl_np[i]].any()
    for bad in ((0, 0), (1, 1), (0, M.MOE_MAX_COPY_PARTS + 1), (-1, 2)):
        with pytest.raises(M.MoeError):
            M.moe_copy_missing_device_part(cache, keys, sl, cnt, *bad)
    cache.close()


def test_copy_missing_device_range():
    # [b0, b1) of every listed expert; the rest of each slot untouched
    M = load_lib()
    wl = configs.scaled(configs.TINY, E=16)
    bank, B, slots, cache = _cache(M, wl, 8)
    b = bank.numpy().reshape(wl.E, B)
    keys = torch.tensor([3, 15, 0], dtype=torch.int32, device="cuda")
    sl = torch.tensor([5, 0, 7], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([3], dtype=torch.int32, device="cuda")
    gu = 2 * (wl.H * wl.I // 2 + wl.H * wl.I // 32)
    for b0, b1 in ((0, gu), (gu, B), (16, 48), (0, B)):
        slots.zero_()
        M.moe_copy_missing_device_range(cache, keys, sl, cnt, b0, b1)
        torch.cuda.synchronize()
        got = slots.cpu().numpy().reshape(8, B)
        for key, s in [(3, 5), (15, 0), (0, 7)]:
            assert np.array_equal(got[s, b0:b1], b[key, b0:b1])
            assert not got[s, :b0].any() and not got[s, b1:].any()
    for b0, b1 in ((0, 0), (8, 32), (0, B + 16), (32, 16)):
        with pytest.raises(M.MoeError):
            M.moe_copy_missing_device_range(cache, keys, sl, cnt, b0, b1)
    cache.close()


def test_copy_missing_device_full_size_expert():
    M = load_lib()
    wl = configs.scaled(configs.DECODE, E=4)
    bank, B = pinned_fp4_bank(wl, (0,))
    assert B == 13369344
    slots = torch.zeros(3 * B, dtype=torch.uint8, device="cuda")
    cache = M.moe_cache(3, 1, wl.E, B, slots, bank)
    keys = torch.tensor([2, 0, 3], dtype=torch.int32, device="cuda")
    sl = torch.tensor([1, 2, 0], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([3], dtype=torch.int32, device="cuda")
    M.moe_copy_missing_device(cache, keys, sl, cnt)
    torch.cuda.synchronize()
    bk = bank.cuda()
    for key, s in [(2, 1), (0, 2), (3, 0)]:
        assert torch.equal(slots[s * B:(s + 1) * B], bk[key * B:(key + 1) * B])
    cache.close()


def test_ensure_mark_rest_matches_oracle():
    M = load_lib()
    wl = configs.scaled(configs.TINY, E=32, k=4, T=24)
    S = 10
    bank, B, slots_mem, cache = _cache(M, wl, S)
    ref = SlotCacheLRU(S, 1, wl.E)
    m = min(S, wl.T * wl.k, wl.E)
    keys = torch.empty(m, dtype=torch.int32, device="cuda")
    sl = torch.empty(m, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    done = torch.empty(1, dtype=torch.int32, device="cuda")
    chunks = 0
    for step in range(4):
        ids, _ = router_topk(gen.router_logits(wl, 0, step), wl.k)
        ids_d = torch.from_numpy(ids.astype(np.int32)).cuda()
        out = torch.full_like(ids_d, 12345)
        tb = 0
        while tb < wl.T:
            M.moe_slot_ensure(cache, 0, ids_d, out, 0, wl.k, M.MOE_FETCH_MARK_REST, tb, keys, sl, cnt, done)
            torch.cuda.synchronize()
            r_slots, r_keys, r_sl, r_end = ref.ensure(0, ids, 0, wl.k, FETCH, tb)
            d = int(done.item())
            assert d == r_end
            n = int(cnt.item())
            assert n == len(r_keys)
            assert np.array_equal(keys.cpu().numpy()[:n], np.asarray(r_keys, dtype=np.int32))
            assert np.array_equal(sl.cpu().numpy()[:n], np.asarray(r_sl, dtype=np.int32))
            o = out.cpu().numpy()
            assert np.array_equal(o[tb:d], np.asarray(r_slots)[tb:d])
            assert (o[d:] == -1).all()
            tb = d
            chunks += 1
        assert np.array_equal(cache.export()[0], ref.state()[0])
    assert chunks > 4      # the trace needs capacity chunking
    cache.close()


def _decoder(bank_np, B, wl):
    memo = {}

    def f(e, tag):
        if e not in memo:
            memo[e] = F.decode_fp4_expert(bank_np[e * B:(e + 1) * B], wl.H, wl.I)
        return memo[e]
    return f


@pytest.mark.parametrize("wl,S,steps,full", [
    (configs.TINY, 4, 6, True),                                   # chunked, tiny
    (configs.scaled(configs.DECODE, T=16), 128, 4, False),        # single chunk by construction
    (configs.scaled(configs.DECODE, T=64), 40, 3, False),         # chunked, grouped-GEMM forward
])
def test_layer_device_copy(wl, S, steps, full):
    M = load_lib()
    bank, B = pinned_fp4_bank(wl, (0,))
    slots = torch.empty(S * B, dtype=torch.uint8, device="cuda")
    cache = M.moe_cache(S, 1, wl.E, B, slots, bank)
    sh = torch.from_numpy(gen.shared_expert(wl, 0)).cuda() if wl.shared else None
    views = M.make_views(wl.H, wl.I, slots, S, None, 0, sh)
    runner = M.DecodeLayerRunner(cache, views, wl.E, wl.k, wl.T, copy="device")
    ref = SlotCacheLRU(S, 1, wl.E)
    dec = _decoder(bank.numpy(), B, wl)
    shw = F.decode_fp8_expert(gen.shared_expert(wl, 0), wl.H, wl.I) if wl.shared else None
    T = wl.T
    ref_chunks = 0
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
            ref_chunks += 1
        assert np.array_equal(cache.export()[0], ref.state()[0])
        rows = list(range(T)) if full else sorted({0, T // 3, T // 2 + 1, T - 1})
        r = moe_layer(x, ids, w, dec, shared=shw, tokens=None if full else rows)
        assert bf16_rel_err(y.cpu().numpy()[rows], r) <= TOL
    runner.check()
    assert runner.stats["misses"] > 0
    assert runner.stats["chunks"] == ref_chunks
    if S < min(wl.E, T * wl.k):
        assert ref_chunks > steps        # the trace does split
    else:
        assert ref_chunks == steps
    cache.close()


def test_copy_missing_device_reports_bad_entries():
    # an entry naming no key or no slot is not copied and sets d_error; the
    # others are copied
    M = load_lib()
    S, L, E, B = 6, 1, 10, 4096
    slots = torch.zeros(S * B, dtype=torch.uint8, device="cuda")
    bank = torch.arange(L * E * B, dtype=torch.int64).remainder(253).to(torch.uint8).pin_memory()
    cache = M.moe_cache(S, L, E, B, slots, bank)
    keys = torch.tensor([3, E + 5, 7, 2], dtype=torch.int32, device="cuda")
    sl = torch.tensor([0, 1, S + 3, 4], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([4], dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_copy_missing_device(cache, keys, sl, cnt, d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == M.MOE_ERR_INVALID
    got = slots.cpu().numpy().reshape(S, B)
    ref = bank.numpy().reshape(L * E, B)
    assert np.array_equal(got[0], ref[3]) and np.array_equal(got[4], ref[2])
    assert not got[1].any()                       # the entry with key E + 5 was skipped
    err.zero_()
    M.moe_copy_missing_device(cache, keys[:1], sl[:1], torch.ones(1, dtype=torch.int32, device="cuda"),
                              d_error=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    cache.close()
