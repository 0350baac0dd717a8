"""Pins for the staging-ring oracle (CPU only): a hand-worked round-robin trace,
and the invariant that prefetching never changes the cache's own state."""
import numpy as np
import pytest

from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU, StagingRing
from synth import configs, gen


def test_hand_worked_ring():
    c = SlotCacheLRU(2, 1, 8)
    r = StagingRing(c, 3)
    c.ensure(0, np.array([[0, 1]]), 0, 2, FETCH, 0)          # keys 0, 1 resident in slots 0, 1
    # resident 1 skipped, duplicate 4 skipped, negative skipped
    assert r.prefetch(0, [1, 4, 5, 4, -1, 6]) == [(4, 2), (5, 3), (6, 4)]
    assert r.stage_key == [4, 5, 6] and r.pos == 3
    assert r.prefetch(0, [5, 7]) == [(7, 2)]                  # 5 already staged; 7 displaces 4 (ring pos 0)
    assert r.stage_key == [7, 5, 6]
    assert r.miss_source(5) == ("stage", 3) and r.miss_source(4) == ("bank", 4)
    _, mk, ms, _ = c.ensure(0, np.array([[5, 6]]), 0, 2, FETCH, 0)
    assert list(zip(mk, ms)) == [(5, 0), (6, 1)]              # LRU victims as without prefetch
    assert [r.miss_source(k) for k in mk] == [("stage", 3), ("stage", 4)]


def test_ring_wrap_within_one_call():
    # more new guesses than ring slots: a guess displaced by a later guess of the
    # same call is not copied (worked by hand: ring of 3, state [7, 5, 6], pos 4)
    c = SlotCacheLRU(2, 1, 8)
    r = StagingRing(c, 3)
    c.ensure(0, np.array([[0, 1]]), 0, 2, FETCH, 0)
    r.prefetch(0, [4, 5, 6])
    r.prefetch(0, [7])
    assert r.stage_key == [7, 5, 6] and r.pos == 4
    # 2 -> ring 1 (slot 3), 3 -> ring 2 (slot 4), 4 -> ring 0 (slot 2), 5 -> ring 1 (slot 3, displacing 2)
    assert r.prefetch(0, [2, 3, 4, 5]) == [(3, 4), (4, 2), (5, 3)]
    assert r.stage_key == [4, 5, 3] and r.pos == 8


@pytest.mark.parametrize("seed", [0, 1])
def test_prefetch_never_changes_cache_state(seed):
    wl = configs.scaled(configs.DECODE, T=4, seed=seed + 10)
    rng = np.random.default_rng(seed)
    a, b = SlotCacheLRU(12, 2, wl.E), SlotCacheLRU(12, 2, wl.E)
    ring = StagingRing(b, 5)
    for step in range(40):
        layer = step % 2
        ids = router_topk(gen.router_logits(wl, layer, step, 4), wl.k)[0]
        guesses = rng.integers(0, wl.E, size=10)
        ring.prefetch(1 - layer, guesses)
        tb = 0
        while tb < 4:
            ra = a.ensure(layer, ids, 0, wl.k, FETCH, tb)
            rb = b.ensure(layer, ids, 0, wl.k, FETCH, tb)
            assert np.array_equal(ra[0], rb[0]) and ra[1:] == rb[1:]
            tb = ra[3]
        for x, y in zip(a.state(), b.state()):
            assert np.array_equal(x, y)
        assert len(set(k for k in ring.stage_key if k >= 0)) == sum(1 for k in ring.stage_key if k >= 0)
