"""Slot-cache kernels vs the oracle: slots, miss lists, tokens_done and the LRU
state bit-exact, over seeded routing traces; copies and their rollback."""
import numpy as np
import pytest
import torch

from oracle.router import router_topk
from oracle.slot_cache import FETCH, LOOKUP, CapacityError, SlotCacheLRU
from synth import configs, gen
from tests.helpers import device_array, load_lib

pytestmark = pytest.mark.gpu


class Pair:
    """A GPU cache and the oracle cache driven with the same calls."""

    def __init__(self, M, S, L, E, B=16):
        self.M = M
        self.slots_mem = torch.zeros(S * B, dtype=torch.uint8, device="cuda")
        self.bank = torch.arange(L * E * B, dtype=torch.int64).remainder(251).to(torch.uint8).pin_memory()
        self.gpu = M.moe_cache(S, L, E, B, self.slots_mem, self.bank)
        self.ref = SlotCacheLRU(S, L, E)
        self.S, self.L, self.E, self.B = S, L, E, B
        self.info = torch.zeros(2 + 2 * S, dtype=torch.int32, device="cuda")

    def ensure(self, layer, ids_np, lo, hi, mode, tb, inplace=False):
        M = self.M
        ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).cuda()
        out = ids if inplace else ids.clone()
        S = self.S
        i = self.info
        M.moe_slot_ensure(self.gpu, layer, ids, out, lo, hi, mode, tb, i[2:2 + S], i[2 + S:], i[0:1], i[1:2])
        torch.cuda.synchronize()
        h = i.cpu().numpy()
        n, done = int(h[0]), int(h[1])
        try:
            rs, rk, rsl, rdone = self.ref.ensure(layer, ids_np, lo, hi, mode, tb)
        except CapacityError:
            assert n == -2 and done == tb
            return None
        assert n == len(rk), (n, len(rk))
        assert done == rdone
        assert list(h[2:2 + n]) == rk and list(h[2 + S:2 + S + n]) == rsl
        assert np.array_equal(out.cpu().numpy(), rs)
        return n, done, list(h[2:2 + n]), list(h[2 + S:2 + S + n])

    def check_state(self):
        key, stamp, clock = self.gpu.export()
        rkey, rstamp, rk2s, rclock = self.ref.state()
        assert np.array_equal(key, rkey)
        occ = key >= 0
        assert np.array_equal(stamp[occ], rstamp[occ])
        assert clock == rclock
        k2s = device_array(self.gpu.state_pointers()[2], self.L * self.E, "<i4")
        assert np.array_equal(k2s.cpu().numpy(), rk2s)


def _trace_ids(wl, layer, steps, T):
    return [router_topk(gen.router_logits(wl, layer, s, T), wl.k)[0] for s in range(steps)]


@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_decode_trace_bit_exact(T):
    M = load_lib()
    wl = configs.DECODE
    c = Pair(M, wl.S, 1, wl.E)
    for ids in _trace_ids(wl, 0, 24, T):
        tb = 0
        while tb < T:
            _, tb, _, _ = c.ensure(0, ids, 0, wl.k, FETCH, tb)
    c.check_state()


def test_tiny_chunking_and_hand_trace():
    M = load_lib()
    c = Pair(M, 4, 1, 8)
    ids = np.array([[0, 1], [2, 3], [4, 5], [0, 6]])
    n, done, keys, slots = c.ensure(0, ids, 0, 2, FETCH, 0)
    assert done == 2 and keys == [0, 1, 2, 3]
    n, done, keys, slots = c.ensure(0, ids, 0, 2, FETCH, 2)
    assert done == 4 and keys == [4, 5, 6] and slots == [1, 2, 3]
    c.check_state()
    wl = configs.TINY
    for ids in _trace_ids(wl, 0, 40, wl.T):
        tb = 0
        while tb < wl.T:
            _, tb, _, _ = c.ensure(0, ids, 0, wl.k, FETCH, tb)
    c.check_state()


def test_global_cache_multi_layer_inplace_lookup_and_rank_ranges():
    M = load_lib()
    wl = configs.scaled(configs.DECODE, zipf_s=1.1)
    c = Pair(M, 48, 3, wl.E)
    rng = np.random.default_rng(3)
    for step in range(30):
        layer = step % 3
        ids = router_topk(gen.router_logits(wl, layer, step, 8), wl.k)[0]
        if step % 5 == 4:
            ids = ids.copy()
            ids[rng.random(ids.shape) < 0.2] = -1      # skipped entries
        lo, hi = (0, wl.k) if step % 3 else (2, 6)
        mode = LOOKUP if step % 7 == 6 else FETCH
        tb = 0
        while tb < 8:
            r = c.ensure(layer, ids, lo, hi, mode, tb, inplace=(step % 2 == 0))
            tb = r[1]
    c.check_state()


def test_large_cache_eviction_paths():
    # more than 1024 eviction candidates: exercises the stamp binary search
    M = load_lib()
    E, L, S = 256, 20, 3000
    c = Pair(M, S, L, E)
    wl = configs.scaled(configs.DECODE)
    for step in range(40):
        layer = step % L
        ids = router_topk(gen.router_logits(wl, layer, step, 64), 8)[0]
        tb = 0
        while tb < 64:
            _, tb, _, _ = c.ensure(layer, ids, 0, 8, FETCH, tb)
    c.check_state()


def test_device_errors_leave_state_unchanged():
    M = load_lib()
    c = Pair(M, 2, 1, 8)
    c.ensure(0, np.array([[1, 2]]), 0, 2, FETCH, 0)
    before = c.gpu.export()
    # capacity: one token needs 3 slots
    r = c.ensure(0, np.array([[3, 4, 5]]), 0, 3, FETCH, 0)
    assert r is None
    # id >= E
    ids = torch.tensor([[9, 1]], dtype=torch.int32, device="cuda")
    i = c.info
    M.moe_slot_ensure(c.gpu, 0, ids, ids.clone(), 0, 2, FETCH, 0, i[2:4], i[4:6], i[0:1], i[1:2])
    torch.cuda.synchronize()
    assert int(i[0]) == -1
    after = c.gpu.export()
    assert np.array_equal(before[0], after[0]) and before[2] == after[2]
    with pytest.raises(M.MoeError):
        M.moe_slot_ensure(c.gpu, 1, ids, ids, 0, 2, FETCH, 0, i[2:4], i[4:6], i[0:1], i[1:2])


def test_copy_missing_and_rollback():
    M = load_lib()
    B = 64
    c = Pair(M, 4, 1, 8, B=B)
    n, done, keys, slots = c.ensure(0, np.array([[5, 3, 7]]), 0, 3, FETCH, 0)
    kh = np.array(keys, dtype=np.int32)
    sh = np.array(slots, dtype=np.int32)
    M.moe_copy_missing(c.gpu, kh, sh, n)
    torch.cuda.synchronize()
    mem = c.slots_mem.cpu().numpy()
    bank = c.bank.numpy()
    for kk, ss in zip(keys, slots):
        assert np.array_equal(mem[ss * B:(ss + 1) * B], bank[kk * B:(kk + 1) * B])
    # injected failure of the second copy: that slot and later ones become empty
    n, done, keys, slots = c.ensure(0, np.array([[0, 1, 2]]), 0, 3, FETCH, 0)
    M.moe_debug_fail_copy(c.gpu, 1)
    with pytest.raises(M.MoeError) as ei:
        M.moe_copy_missing(c.gpu, np.array(keys, np.int32), np.array(slots, np.int32), n)
    assert ei.value.status == M.MOE_ERR_CUDA
    torch.cuda.synchronize()
    key, _, _ = c.gpu.export()
    assert key[slots[0]] == keys[0]
    assert all(key[s] == -1 for s in slots[1:])
    c.ref.mark_empty(slots[1:])
    M.moe_debug_fail_copy(c.gpu, -1)
    c.ensure(0, np.array([[1, 2]]), 0, 2, FETCH, 0)   # the rolled-back experts miss again
    c.check_state()


def test_export_import_round_trip():
    M = load_lib()
    c = Pair(M, 8, 1, 16)
    c.ensure(0, np.array([[1, 2, 3], [4, 5, 6]]), 0, 3, FETCH, 0)
    key, stamp, clock = c.gpu.export()
    c.gpu.reset()
    torch.cuda.synchronize()
    c.gpu.import_(key, stamp, clock)
    c.check_state()
    bad = key.copy()
    bad[bad >= 0] = 1
    with pytest.raises(M.MoeError):
        c.gpu.import_(bad, stamp, clock)


def test_pageable_bank_rejected():
    M = load_lib()
    slots = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MoeError):
        M.moe_cache(4, 1, 8, 16, slots, torch.zeros(128, dtype=torch.uint8))
    with pytest.raises(M.MoeError):
        M.moe_cache(0, 1, 8, 16, slots, None)
