"""LFU eviction with frequency decay on the GPU vs the oracle: slots, miss lists,
tokens_done, the slot table and the frequency state bit-exact."""
import os

import numpy as np
import pytest
import torch

from oracle.router import router_topk
from oracle.slot_cache import FETCH, LOOKUP, SlotCacheLFU
from synth import configs, gen
from tests.helpers import load_lib
from tests.test_gpu_slot_cache import Pair

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden", "lfu_tiny_trace.txt")


class LfuPair(Pair):
    def __init__(self, M, S, L, E, decay, seed_counts=None):
        super().__init__(M, S, L, E)
        self.ref = SlotCacheLFU(S, L, E, decay)
        M.moe_cache_set_policy(self.gpu, M.MOE_EVICT_LFU, decay)
        if seed_counts is not None:
            self.ref.seed(seed_counts)
            M.moe_cache_seed_frequency(self.gpu, seed_counts)

    def check_freq(self):
        cnt, ep, calls = self.M.moe_cache_export_frequency(self.gpu)
        rc, re, rcalls = self.ref.frequency_state()
        assert calls == rcalls
        assert np.array_equal(cnt.astype(np.int64), rc)
        assert np.array_equal(ep.astype(np.int64), re)


def test_hand_worked_trace():
    M = load_lib()
    p = LfuPair(M, 2, 1, 4, decay=4)
    want = []
    for ln in open(GOLD):
        if ln.startswith("misses"):
            v = ln.split()[2]
            want.append([] if v == "-" else [tuple(int(x) for x in v.split(":"))])
    for e, w in zip([0, 0, 0, 1, 2, 3], want):
        n, done, mk, ms = p.ensure(0, np.array([[e]]), 0, 1, FETCH, 0)
        assert list(zip(mk, ms)) == w
    p.check_state()
    p.check_freq()
    assert list(p.gpu.export()[0]) == [3, 2]


def _seed_counts(wl, L, steps, T):
    # a routing trace disjoint from the one replayed: counts of each key's uses
    c = np.zeros(L * wl.E, dtype=np.int64)
    for layer in range(L):
        for s in range(1000, 1000 + steps):
            ids = router_topk(gen.router_logits(wl, layer, s, T), wl.k)[0]
            np.add.at(c, layer * wl.E + np.unique(ids), 1)
    return c


@pytest.mark.parametrize("decay", [1, 5, 1000])
def test_decode_trace_with_chunking_lookup_and_seed(decay):
    M = load_lib()
    wl = configs.scaled(configs.DECODE, T=16)
    L, S = 2, 48
    p = LfuPair(M, S, L, wl.E, decay, seed_counts=_seed_counts(wl, L, 6, 16))
    p.check_freq()
    for step in range(30):
        layer = step % L
        ids = router_topk(gen.router_logits(wl, layer, step, 16), wl.k)[0]
        mode = LOOKUP if step % 5 == 4 else FETCH
        tb = 0
        while tb < 16:
            r = p.ensure(layer, ids, 0, wl.k, mode, tb)
            tb = r[1]
        p.check_state()
        p.check_freq()


def test_large_cache_binary_search_path():
    # more than 1024 eviction candidates: the order-key binary search
    M = load_lib()
    E, L, S = 256, 20, 3000
    p = LfuPair(M, S, L, E, decay=3)
    wl = configs.scaled(configs.DECODE)
    for step in range(40):
        layer = step % L
        ids = router_topk(gen.router_logits(wl, layer, step, 64), 8)[0]
        tb = 0
        while tb < 64:
            tb = p.ensure(layer, ids, 0, 8, FETCH, tb)[1]
    p.check_state()
    p.check_freq()


def test_reset_clears_and_ladder_needs_lru():
    M = load_lib()
    p = LfuPair(M, 4, 1, 8, decay=2)
    p.ensure(0, np.array([[1, 2]]), 0, 2, FETCH, 0)
    p.gpu.reset()
    torch.cuda.synchronize()
    cnt, ep, calls = M.moe_cache_export_frequency(p.gpu)
    assert not cnt.any() and not ep.any() and calls == 0
    c2 = M.moe_cache(4, 1, 8, 16, torch.zeros(64, dtype=torch.uint8, device="cuda"))
    z = torch.zeros((1, 2), dtype=torch.int32, device="cuda")
    f = torch.zeros((1, 2), dtype=torch.float32, device="cuda")
    i8 = torch.zeros((1, 2), dtype=torch.int8, device="cuda")
    v = torch.zeros(8, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoeError):
        M.moe_ladder_classify(p.gpu, c2, 0, z, f, 1, 2, 0, z, i8, f, v[:2], v[2:4], v[4:5], v[5:6], v[6:7],
                              v[7:8], v[0:1])
    with pytest.raises(M.MoeError):
        M.moe_cache_set_policy(p.gpu, 7, 1)
    with pytest.raises(M.MoeError):
        M.moe_cache_set_policy(p.gpu, M.MOE_EVICT_LFU, 0)
