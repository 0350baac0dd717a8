"""Staging ring on the GPU vs the oracle: ring state and copy lists bit-exact,
the cache state untouched by prefetching, promotion served from the staging
slot, and layer outputs identical with and without prefetching."""
import numpy as np
import pytest
import torch

from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU, StagingRing
from synth import configs, gen
from tests.helpers import load_lib, pinned_fp4_bank

pytestmark = pytest.mark.gpu


class StagedPair:
    def __init__(self, M, S, R, L, E, B=16):
        self.M, self.S, self.R, self.L, self.E, self.B = M, S, R, L, E, B
        self.slots_mem = torch.zeros((S + R) * B, dtype=torch.uint8, device="cuda")
        self.bank = torch.arange(L * E * B, dtype=torch.int64).remainder(251).to(torch.uint8).pin_memory()
        self.gpu = M.moe_cache(S, L, E, B, self.slots_mem, self.bank)
        M.moe_cache_set_staging(self.gpu, R)
        self.ref = SlotCacheLRU(S, L, E)
        self.ring = StagingRing(self.ref, R)
        self.lk = torch.zeros(64, dtype=torch.int32, device="cuda")
        self.ls = torch.zeros(64, dtype=torch.int32, device="cuda")
        self.lc = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.info = torch.zeros(2 + 2 * S, dtype=torch.int32, device="cuda")

    def prefetch(self, layer, experts):
        M = self.M
        d = torch.tensor(list(experts), dtype=torch.int32, device="cuda")
        M.moe_prefetch(self.gpu, layer, d, self.lk, self.ls, self.lc)
        M.moe_copy_missing_device(self.gpu, self.lk, self.ls, self.lc)
        torch.cuda.synchronize()
        n = int(self.lc.item())
        got = list(zip(self.lk.cpu().tolist()[:n], self.ls.cpu().tolist()[:n]))
        assert got == self.ring.prefetch(layer, experts)
        key, pos = M.moe_cache_export_staging(self.gpu)
        assert list(key) == self.ring.stage_key and pos == self.ring.pos

    def ensure(self, layer, ids):
        M, S, i = self.M, self.S, self.info
        d = torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()
        out = d.clone()
        tb = 0
        while tb < ids.shape[0]:
            M.moe_slot_ensure(self.gpu, layer, d, out, 0, ids.shape[1], M.MOE_FETCH, tb, i[2:2 + S], i[2 + S:],
                              i[0:1], i[1:2])
            srcs = []
            torch.cuda.synchronize()
            h = i.cpu().numpy()
            n, done = int(h[0]), int(h[1])
            rs, rk, rsl, rdone = self.ref.ensure(layer, ids, 0, ids.shape[1], FETCH, tb)
            assert (n, done) == (len(rk), rdone)
            assert list(h[2:2 + n]) == rk and list(h[2 + S:2 + S + n]) == rsl
            srcs = [self.ring.miss_source(k) for k in rk]
            M.moe_copy_missing_device(self.gpu, i[2:2 + S], i[2 + S:], i[0:1])
            torch.cuda.synchronize()
            tb = done
        return list(zip(rk, rsl)), srcs


def test_ring_state_lists_and_unchanged_cache():
    M = load_lib()
    wl = configs.scaled(configs.DECODE, T=4)
    p = StagedPair(M, 12, 5, 2, wl.E)
    plain = SlotCacheLRU(12, 2, wl.E)
    rng = np.random.default_rng(3)
    for step in range(30):
        layer = step % 2
        ids = router_topk(gen.router_logits(wl, layer, step, 4), wl.k)[0]
        p.prefetch(1 - layer, list(rng.integers(-1, wl.E, size=9)))
        p.ensure(layer, ids)
        tb = 0
        while tb < 4:
            tb = plain.ensure(layer, ids, 0, wl.k, FETCH, tb)[3]
        key, stamp, clock = p.gpu.export()
        assert np.array_equal(key, plain.state()[0]) and clock == plain.state()[3]
        # every occupied slot, staged or cached, holds its key's bank bytes
        mem = p.slots_mem.cpu().numpy().reshape(-1, p.B)
        bank = p.bank.numpy().reshape(-1, p.B)
        for s_, kk in enumerate(list(key) + list(M.moe_cache_export_staging(p.gpu)[0])):
            if kk >= 0:
                assert np.array_equal(mem[s_], bank[kk])
    bad = torch.tensor([1, wl.E], dtype=torch.int32, device="cuda")
    M.moe_prefetch(p.gpu, 0, bad, p.lk, p.ls, p.lc)
    torch.cuda.synchronize()
    assert int(p.lc.item()) == -M.MOE_ERR_INVALID


def test_promotion_copies_from_the_staging_slot():
    # change the bank row after staging: a promotion from the staging slot keeps
    # the staged bytes, a copy from the bank would bring the changed ones
    M = load_lib()
    p = StagedPair(M, 2, 2, 1, 8)
    p.ensure(0, np.array([[0, 1]]))
    p.prefetch(0, [5])
    staged = p.bank[5 * p.B:6 * p.B].clone()
    p.bank[5 * p.B:6 * p.B] = 7
    misses, srcs = p.ensure(0, np.array([[5, 0]]))
    assert misses == [(5, 1)] and srcs == [("stage", 2)]
    assert torch.equal(p.slots_mem[1 * p.B:2 * p.B].cpu(), staged)
    misses, srcs = p.ensure(0, np.array([[6, 7]]))          # not staged: from the bank
    assert srcs == [("bank", 6), ("bank", 7)]


@pytest.mark.parametrize("T,overlap,sync", [(4, False, True), (64, True, True), (64, True, False),
                                             (4, False, False)])
def test_layer_outputs_identical_with_prefetch(T, overlap, sync):
    # sync=False enqueues every step back to back: a step's prefetch copy is
    # still running on the side stream when the next step assigns new ring
    # slots, so the assignment must wait for it
    M = load_lib()
    wl = configs.scaled(configs.DECODE, T=T)
    S, R = 48, 12
    bank, B = pinned_fp4_bank(wl, (0,))
    outs = []
    for use_pf in (False, True):
        slots = torch.empty((S + R) * B, dtype=torch.uint8, device="cuda")
        cache = M.moe_cache(S, 1, wl.E, B, slots, bank)
        if use_pf:
            M.moe_cache_set_staging(cache, R)
        sh = torch.from_numpy(gen.shared_expert(wl, 0)).cuda()
        views = M.make_views(wl.H, wl.I, slots, S, None, 0, sh)
        runner = M.DecodeLayerRunner(cache, views, wl.E, wl.k, T, copy="device", overlap=overlap)
        ys = []
        for step in range(5):
            lg = gen.router_logits(wl, 0, step, T)
            x = gen.activations(wl, 0, step, T)
            nxt = router_topk(gen.router_logits(wl, 0, step + 1, T), wl.k)[0]
            # half of the next step's experts; unsynchronised steps stage a full
            # ring of guesses so that the copy is long
            guess = np.unique(nxt)[::2] if sync else np.unique(np.concatenate([nxt.ravel(), np.arange(R) * 7]))
            pf = (0, torch.from_numpy(guess.astype(np.int32)).cuda()) if use_pf else None
            y = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
            runner.run(0, torch.from_numpy(lg).cuda(), torch.from_numpy(x.view(np.int16)).cuda(), y, prefetch=pf)
            if sync:
                torch.cuda.synchronize()
            ys.append(y)
        torch.cuda.synchronize()
        ys = [y.cpu().numpy() for y in ys]
        runner.check()
        outs.append((ys, cache.export()[0], runner.stats["misses"]))
        cache.close()
    for a, b in zip(outs[0][0], outs[1][0]):
        assert np.array_equal(a, b)
    assert np.array_equal(outs[0][1], outs[1][1]) and outs[0][2] == outs[1][2]
