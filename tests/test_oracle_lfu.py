"""Pins for the LFU oracle slot cache (CPU only): a hand-worked trace, the exact
reduction to LRU, an independent eager-decay simulator, decay and saturation."""
import os

import numpy as np
import pytest

from oracle.slot_cache import FETCH, LOOKUP, SlotCacheLFU, SlotCacheLRU
from synth import configs, gen
from oracle.router import router_topk

GOLD = os.path.join(os.path.dirname(__file__), "golden", "lfu_tiny_trace.txt")


def _gold():
    d = {}
    for ln in open(GOLD):
        if ln.strip() and not ln.startswith("#"):
            p = ln.split()
            d[(p[0], p[1])] = p[2:]
    return d


def test_hand_worked_trace():
    g = _gold()
    c = SlotCacheLFU(2, 1, 4, decay_calls=4)
    for i, e in enumerate([0, 0, 0, 1, 2, 3]):
        _, mk, ms, done = c.ensure(0, np.array([[e]]), 0, 1, FETCH, 0)
        assert done == 1
        want = g[("misses", f"c{i}")]
        assert [f"{k}:{s}" for k, s in zip(mk, ms)] == ([] if want == ["-"] else want)
    key, stamp, _, clock = c.state()
    assert list(key) == [int(v) for v in g[("final", "slot_key")]]
    assert list(stamp) == [int(v) for v in g[("final", "stamps")]]
    assert clock == int(g[("final", "clock")][0])
    cnt, ep, calls = c.frequency_state()
    assert list(cnt) == [int(v) for v in g[("final", "count")]]
    assert list(ep) == [int(v) for v in g[("final", "count_epoch")]]
    assert calls == int(g[("final", "calls")][0])


def _zipf_calls(seed, n, T=6, k=3, E=12):
    wl = configs.scaled(configs.TINY, E=E, k=k, T=T, zipf_s=1.1, seed=seed)
    return [router_topk(gen.router_logits(wl, 0, s, T), k)[0] for s in range(n)]


@pytest.mark.parametrize("seed", [1, 2])
def test_reduces_to_lru_when_every_count_is_saturated(seed):
    # all counts at the cap and no decay within the trace: worth never differs,
    # so the order is the stamp order, exactly LRU's
    S, L, E = 5, 2, 12
    lfu = SlotCacheLFU(S, L, E, decay_calls=10 ** 9)
    lfu.seed(np.full(L * E, SlotCacheLFU.CAP))
    lru = SlotCacheLRU(S, L, E)
    for i, ids in enumerate(_zipf_calls(seed, 40, E=E)):
        layer, mode = i % L, (LOOKUP if i % 7 == 3 else FETCH)
        tb = 0
        while True:
            a = lfu.ensure(layer, ids, 0, ids.shape[1], mode, tb)
            b = lru.ensure(layer, ids, 0, ids.shape[1], mode, tb)
            assert np.array_equal(a[0], b[0]) and a[1:] == b[1:]
            tb = a[3]
            if tb >= ids.shape[0]:
                break
        for x, y in zip(lfu.state(), lru.state()):
            assert np.array_equal(x, y)


class EagerLFU:
    """Independent formulation: counts are halved eagerly at every epoch
    boundary, victims found by a linear scan; first-appearance order and
    chunking are recomputed here from scratch."""

    def __init__(self, S, L, E, decay):
        self.S, self.E, self.decay = S, E, decay
        self.slot_key = [-1] * S
        self.stamp = [0] * S
        self.cnt = [0] * (L * E)
        self.clock = 0
        self.calls = 0

    def call(self, layer, ids, tb):
        order, first = [], {}
        T, k = ids.shape
        for t in range(tb, T):
            for j in range(k):
                key = layer * self.E + int(ids[t, j])
                if key not in first:
                    first[key] = t
                    order.append(key)
        end, used = tb, 0
        for t in range(tb, T):
            n = sum(1 for key in order if first[key] == t)
            if used + n > self.S:
                break
            used += n
            end = t + 1
        chunk = [key for key in order if first[key] < end]
        where = {key: s for s, key in enumerate(self.slot_key) if key >= 0}
        pinned = {where[key] for key in chunk if key in where}
        misses = []
        for key in chunk:
            if key in where:
                continue
            free = [s for s in range(self.S) if self.slot_key[s] < 0]
            if free:
                v = free[0]
            else:
                best = None
                for s in range(self.S):
                    if s in pinned:
                        continue
                    cand = (self.cnt[self.slot_key[s]], self.stamp[s])
                    if best is None or cand < best[0]:
                        best = (cand, s)
                v = best[1]
            self.slot_key[v] = key
            where = {kk: s for s, kk in enumerate(self.slot_key) if kk >= 0}
            pinned.add(v)
            misses.append((key, v))
        for q, key in enumerate(chunk):
            self.stamp[where[key]] = self.clock + q
        self.clock += len(chunk)
        for key in chunk:
            self.cnt[key] = min(self.cnt[key] + 1, SlotCacheLFU.CAP)
        self.calls += 1
        if self.calls % self.decay == 0:           # entering a new epoch: halve everything now
            self.cnt = [c >> 1 for c in self.cnt]
        return misses, end


@pytest.mark.parametrize("seed,decay", [(3, 1), (4, 3), (5, 7)])
def test_matches_eager_decay_simulator(seed, decay):
    S, L, E = 6, 2, 12
    a = SlotCacheLFU(S, L, E, decay_calls=decay)
    b = EagerLFU(S, L, E, decay)
    for i, ids in enumerate(_zipf_calls(seed, 60, E=E)):
        layer, tb = i % L, 0
        while tb < ids.shape[0]:
            _, mk, ms, end = a.ensure(layer, ids, 0, ids.shape[1], FETCH, tb)
            mb, eb = b.call(layer, ids, tb)
            assert list(zip(mk, ms)) == mb and end == eb
            tb = end
        assert list(a.state()[0]) == b.slot_key
        worth = [a.worth(key) for key in range(L * E)]
        assert worth == b.cnt


def test_decay_closed_form_and_saturation():
    c = SlotCacheLFU(2, 1, 4, decay_calls=3)
    c.seed(np.array([1000, 5, 0, 7]))
    for n in range(1, 5):
        for _ in range(3):                         # three calls per epoch, on key 2 only
            c.ensure(0, np.array([[2]]), 0, 1, LOOKUP, 0)
        assert c.worth(0) == 1000 >> n and c.worth(1) == 5 >> n and c.worth(3) == 7 >> n
    d = SlotCacheLFU(1, 1, 2, decay_calls=10 ** 9)
    d.seed(np.array([SlotCacheLFU.CAP - 1, 0]))
    for _ in range(3):
        d.ensure(0, np.array([[0]]), 0, 1, FETCH, 0)
    assert d.worth(0) == SlotCacheLFU.CAP
