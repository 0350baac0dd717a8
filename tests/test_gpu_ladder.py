"""Ladder classifier vs the oracle over seeded routing traces: slots, tags,
miss lists, tokens_done and both pools' LRU state bit-exact; weights 1e-6."""
import numpy as np
import pytest
import torch

from oracle.ladder import ladder_classify
from oracle.router import router_topk
from oracle.slot_cache import CapacityError, SlotCacheLRU
from synth import configs, gen
from tests.helpers import load_lib

pytestmark = pytest.mark.gpu


class LadderPair:
    def __init__(self, M, S4, S2, L, E):
        self.M = M
        self.m4 = torch.zeros(S4 * 16, dtype=torch.uint8, device="cuda")
        self.m2 = torch.zeros(S2 * 16, dtype=torch.uint8, device="cuda")
        self.g4 = M.moe_cache(S4, L, E, 16, self.m4, None)
        self.g2 = M.moe_cache(S2, L, E, 16, self.m2, None)
        self.r4, self.r2 = SlotCacheLRU(S4, L, E), SlotCacheLRU(S2, L, E)
        self.S4, self.S2 = S4, S2
        self.info = torch.zeros(8 + 2 * S4 + 2 * S2, dtype=torch.int32, device="cuda")

    def step(self, layer, ids_np, w_np, a, b, tb):
        M, S4, S2, i = self.M, self.S4, self.S2, self.info
        T, k = ids_np.shape
        ids = torch.from_numpy(ids_np.astype(np.int32)).cuda()
        w = torch.from_numpy(w_np.astype(np.float32)).cuda()
        slots = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
        tags = torch.full((T, k), 9, dtype=torch.int8, device="cuda")
        wo = torch.zeros((T, k), dtype=torch.float32, device="cuda")
        o = 8
        M.moe_ladder_classify(self.g4, self.g2, layer, ids, w, a, b, tb, slots, tags, wo,
                              i[o:o + S4], i[o + S4:o + 2 * S4], i[0:1],
                              i[o + 2 * S4:o + 2 * S4 + S2], i[o + 2 * S4 + S2:], i[1:2], i[2:3])
        torch.cuda.synchronize()
        h = i.cpu().numpy()
        n4, n2, done = int(h[0]), int(h[1]), int(h[2])
        try:
            rs, rt, rw, (k4, s4), (k2, s2), rdone = ladder_classify(
                self.r4, self.r2, layer, ids_np, w_np.astype(np.float32).astype(np.float64), a, b, tb)
        except CapacityError:
            assert n4 == -2 and n2 == -2 and done == tb
            return tb
        assert done == rdone and n4 == len(k4) and n2 == len(k2)
        assert list(h[o:o + n4]) == k4 and list(h[o + S4:o + S4 + n4]) == s4
        assert list(h[o + 2 * S4:o + 2 * S4 + n2]) == k2
        assert list(h[o + 2 * S4 + S2:o + 2 * S4 + S2 + n2]) == s2
        sl, tg, ww = slots.cpu().numpy(), tags.cpu().numpy(), wo.cpu().numpy()
        assert np.array_equal(sl[tb:done], rs[tb:done])
        assert np.array_equal(tg[tb:done], rt[tb:done])
        assert np.max(np.abs(ww[tb:done] - rw[tb:done])) <= 1e-6
        assert np.all(sl[done:] == -7) and np.all(tg[done:] == 9)
        return done

    def check_state(self):
        for g, r in ((self.g4, self.r4), (self.g2, self.r2)):
            key, stamp, clock = g.export()
            rkey, rstamp, _, rclock = r.state()
            assert np.array_equal(key, rkey) and clock == rclock
            assert np.array_equal(stamp[key >= 0], rstamp[key >= 0])


def test_ladder_trace_matches_oracle():
    M = load_lib()
    wl = configs.LADDER
    p = LadderPair(M, wl.S, wl.S2, 1, wl.E)
    a, b = wl.ladder
    for step in range(40):
        ids, w = router_topk(gen.router_logits(wl, 0, step), wl.k)
        tb = 0
        while tb < wl.T:
            tb = p.step(0, ids, w.astype(np.float32), a, b, tb)
    p.check_state()


def test_ladder_small_pools_chunk_and_multi_layer():
    M = load_lib()
    wl = configs.scaled(configs.LADDER, T=12)
    p = LadderPair(M, 9, 7, 2, wl.E)
    for step in range(30):
        layer = step % 2
        ids, w = router_topk(gen.router_logits(wl, layer, step), wl.k)
        tb = 0
        while tb < wl.T:
            tb = p.step(layer, ids, w.astype(np.float32), 2, 4, tb)
    p.check_state()


@pytest.mark.parametrize("a,b", [(1, 1), (1, 6), (6, 6), (3, 5)])
def test_ladder_other_rungs(a, b):
    M = load_lib()
    wl = configs.scaled(configs.LADDER, T=16)
    p = LadderPair(M, 40, 40, 1, wl.E)
    for step in range(12):
        ids, w = router_topk(gen.router_logits(wl, 0, step), wl.k)
        tb = 0
        while tb < wl.T:
            tb = p.step(0, ids, w.astype(np.float32), a, b, tb)
    p.check_state()


def test_ladder_capacity_error():
    M = load_lib()
    p = LadderPair(M, 1, 8, 1, 16)
    ids = np.array([[1, 2, 3, 4, 5, 6]])
    p.step(0, ids, np.full((1, 6), 1 / 6), 2, 4, 0)
