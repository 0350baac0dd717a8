"""Pins for the oracle slot cache: a hand-worked trace and an independent LRU (CPU only)."""
import os
from collections import OrderedDict

import numpy as np
import pytest

from oracle.slot_cache import FETCH, LOOKUP, CapacityError, SlotCacheLRU

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold():
    d = {}
    with open(os.path.join(GOLD, "lru_tiny_trace.txt")) as f:
        for ln in f:
            if ln.strip() and not ln.startswith("#"):
                p = ln.split()
                d[(p[0], p[1])] = p[2:]
    return d


def test_hand_worked_trace():
    g = _gold()
    ids = np.array([[0, 1], [2, 3], [4, 5], [0, 6]])
    c = SlotCacheLRU(4, 1, 8)
    s1, mk, ms, done = c.ensure(0, ids, 0, 2, FETCH, 0)
    assert done == int(g[("call1", "tokens_done")][0])
    assert list(s1[:2].reshape(-1)) == [int(v) for v in g[("call1", "slots")]]
    assert [f"{k}:{s}" for k, s in zip(mk, ms)] == g[("call1", "misses")]
    assert np.array_equal(s1[2:], ids[2:])            # untouched beyond the chunk
    s2, mk, ms, done = c.ensure(0, ids, 0, 2, FETCH, done)
    assert done == int(g[("call2", "tokens_done")][0])
    assert list(s2[2:].reshape(-1)) == [int(v) for v in g[("call2", "slots")]]
    assert [f"{k}:{s}" for k, s in zip(mk, ms)] == g[("call2", "misses")]
    key, stamp, _, clock = c.state()
    assert list(key) == [int(v) for v in g[("final", "slot_key")]]
    assert list(stamp) == [int(v) for v in g[("final", "stamps")]]
    assert clock == int(g[("final", "clock")][0])


class OrderedLRU:
    """Independent formulation: an ordered dict in recency order, with the
    call's resident working set protected from eviction while it is served."""

    def __init__(self, S):
        self.S = S
        self.od = OrderedDict()          # key -> slot, least recent first
        self.free = list(range(S))

    def call(self, keys_in_order):
        needed_resident = {k for k in keys_in_order if k in self.od}
        misses = []
        for key in keys_in_order:
            if key in self.od:
                self.od.move_to_end(key)
                continue
            if self.free:
                slot = min(self.free)
                self.free.remove(slot)
            else:
                victim = next(k for k in self.od if k not in needed_resident)
                slot = self.od.pop(victim)
            self.od[key] = slot
            misses.append((key, slot))
        return misses


def _first_appearance(ids, lo, hi, layer, E, t0, t1):
    seen, out = set(), []
    for t in range(t0, t1):
        for j in range(lo, hi):
            key = layer * E + int(ids[t, j])
            if ids[t, j] >= 0 and key not in seen:
                seen.add(key)
                out.append(key)
    return out


@pytest.mark.parametrize("S,E,k,T,L", [(4, 8, 2, 3, 1), (16, 64, 4, 8, 2), (64, 256, 8, 16, 3)])
def test_matches_ordered_dict_lru(S, E, k, T, L):
    rng = np.random.default_rng(S * 1000 + E)
    pop = np.exp(-1.1 * np.log(np.arange(1, E + 1)))
    pop /= pop.sum()
    c = SlotCacheLRU(S, L, E)
    ref = OrderedLRU(S)
    for step in range(60):
        layer = step % L
        ids = np.stack([rng.choice(E, size=k, replace=False, p=pop) for _ in range(T)])
        tb = 0
        while tb < T:
            slots, mk, ms, done = c.ensure(layer, ids, 0, k, FETCH, tb)
            # chunk end by brute force: longest prefix with distinct keys <= S
            best = tb
            for n in range(tb + 1, T + 1):
                if len(_first_appearance(ids, 0, k, layer, E, tb, n)) <= S:
                    best = n
            assert done == best
            keys = _first_appearance(ids, 0, k, layer, E, tb, done)
            assert list(zip(mk, ms)) == ref.call(keys)
            for t in range(tb, done):
                for j in range(k):
                    assert slots[t, j] == ref.od[layer * E + int(ids[t, j])]
            tb = done
        # the same residency and the same recency order
        skey, stamp, k2s, _ = c.state()
        resident = [int(x) for x in skey[np.argsort(stamp, kind="stable")] if x >= 0]
        resident_by_recency = [key for key in sorted(
            (int(x) for x in skey if x >= 0), key=lambda kk: stamp[c.key_to_slot[kk]])]
        assert resident_by_recency == list(ref.od.keys())
        assert sorted(resident) == sorted(ref.od.keys())
        for key, slot in ref.od.items():
            assert k2s[key] == slot


def test_lookup_hits_misses_and_no_eviction():
    c = SlotCacheLRU(3, 1, 10)
    c.ensure(0, np.array([[1, 2, 3]]), 0, 3, FETCH)
    before = c.state()[0].copy()
    out, mk, ms, done = c.ensure(0, np.array([[3, 9], [1, 4]]), 0, 2, LOOKUP)
    assert out.tolist() == [[2, -1], [0, -1]]
    assert mk == [] and ms == [] and done == 2
    assert np.array_equal(c.state()[0], before)
    # key 3 then key 1 were refreshed: key 2 (slot 1) is now the LRU victim
    out, mk, ms, _ = c.ensure(0, np.array([[7]]), 0, 1, FETCH)
    assert ms == [1] and out[0, 0] == 1


def test_rank_range_and_negative_ids_are_skipped():
    c = SlotCacheLRU(4, 1, 8)
    ids = np.array([[5, -1, 6], [7, 5, -1]])
    out, mk, ms, done = c.ensure(0, ids, 0, 2, FETCH)
    assert mk == [5, 7] and ms == [0, 1]
    assert out.tolist() == [[0, -1, 6], [1, 0, -1]]


def test_capacity_error_when_one_token_exceeds_slots():
    c = SlotCacheLRU(2, 1, 8)
    with pytest.raises(CapacityError):
        c.ensure(0, np.array([[0, 1, 2]]), 0, 3, FETCH)


def test_global_cache_across_layers():
    c = SlotCacheLRU(2, 2, 4)
    a, _, _, _ = c.ensure(0, np.array([[3]]), 0, 1, FETCH)
    b, mk, _, _ = c.ensure(1, np.array([[3]]), 0, 1, FETCH)
    assert mk == [1 * 4 + 3] and a[0, 0] != b[0, 0]


def test_rollback_marks_slots_empty():
    c = SlotCacheLRU(2, 1, 4)
    _, mk, ms, _ = c.ensure(0, np.array([[1, 2]]), 0, 2, FETCH)
    c.mark_empty(ms)
    assert list(c.state()[0]) == [-1, -1]
    _, mk2, _, _ = c.ensure(0, np.array([[1]]), 0, 1, FETCH)
    assert mk2 == [1]
