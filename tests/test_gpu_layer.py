"""Whole layer through the host runner (router, ensure, one sync, miss copies
on a side stream, forward) vs the oracle over seeded traces."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.ladder import ladder_classify
from oracle.mlp import moe_layer
from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib, pinned_fp4_bank

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _setup(M, wl, layers=(0,), S=None, shared=False, assume_resident=False):
    bank, B = pinned_fp4_bank(wl, layers)
    S = wl.S if S is None else S
    slots = torch.empty(S * B, dtype=torch.uint8, device="cuda")
    cache = M.moe_cache(S, len(layers), wl.E, B, slots, bank)
    sh = torch.from_numpy(gen.shared_expert(wl, 0)).cuda() if shared else None
    views = M.make_views(wl.H, wl.I, slots, S, None, 0, sh)
    runner = M.DecodeLayerRunner(cache, views, wl.E, wl.k, wl.T, assume_resident=assume_resident)
    return bank, B, cache, runner, sh


def _decoder(bank_np, B, wl, layer_index=0):
    memo = {}

    def f(e, tag):
        if e not in memo:
            o = (layer_index * wl.E + e) * B
            memo[e] = F.decode_fp4_expert(bank_np[o:o + B], wl.H, wl.I)
        return memo[e]
    return f


def test_layer_tiny_trace():
    M = load_lib()
    wl = configs.TINY
    bank, B, cache, runner, _ = _setup(M, wl)
    ref = SlotCacheLRU(wl.S, 1, wl.E)
    dec = _decoder(bank.numpy(), B, wl)
    for step in range(wl.steps):
        lg = gen.router_logits(wl, 0, step)
        x = gen.activations(wl, 0, step)
        y = torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda")
        runner.run(0, torch.from_numpy(lg).cuda(), torch.from_numpy(x.view(np.int16)).cuda(), y)
        torch.cuda.synchronize()
        ids, w = router_topk(lg, wl.k)
        tb = 0
        while tb < wl.T:
            _, _, _, tb = ref.ensure(0, ids, 0, wl.k, FETCH, tb)
        assert bf16_rel_err(y.cpu().numpy(), moe_layer(x, ids, w, dec)) <= TOL
        assert np.array_equal(cache.export()[0], ref.state()[0])
    assert runner.stats["chunks"] > runner.stats["calls"]     # capacity splits happened


@pytest.mark.parametrize("T", [1, 16])
def test_layer_decode_trace_sampled(T):
    M = load_lib()
    wl = configs.scaled(configs.DECODE, T=T)
    bank, B, cache, runner, sh = _setup(M, wl, shared=True)
    ref = SlotCacheLRU(wl.S, 1, wl.E)
    dec = _decoder(bank.numpy(), B, wl)
    shw = F.decode_fp8_expert(gen.shared_expert(wl, 0), wl.H, wl.I)
    for step in range(6):
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
        if step in (0, 5):
            sample = [0, T - 1]
            r = moe_layer(x, ids, w, dec, shared=shw, tokens=sample)
            assert bf16_rel_err(y.cpu().numpy()[sample], r) <= TOL
    assert runner.stats["misses"] > 0


def test_layer_ladder_trace():
    M = load_lib()
    wl = configs.scaled(configs.LADDER, H=256, I=128, T=8, S=20, S2=30)
    bank4, B4 = pinned_fp4_bank(wl, (0,))
    B2 = M.moe_int2_expert_bytes(wl.H, wl.I)
    bank2 = torch.empty(wl.E * B2, dtype=torch.uint8, pin_memory=True)
    for e in range(wl.E):
        bank2[e * B2:(e + 1) * B2] = torch.from_numpy(gen.int2_expert(wl, 0, e))
    s4 = torch.empty(wl.S * B4, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(wl.S2 * B2, dtype=torch.uint8, device="cuda")
    c4 = M.moe_cache(wl.S, 1, wl.E, B4, s4, bank4)
    c2 = M.moe_cache(wl.S2, 1, wl.E, B2, s2, bank2)
    views = M.make_views(wl.H, wl.I, s4, wl.S, s2, wl.S2, None)
    runner = M.DecodeLayerRunner(c4, views, wl.E, wl.k, wl.T, int2_cache=c2, ladder=wl.ladder)
    r4, r2 = SlotCacheLRU(wl.S, 1, wl.E), SlotCacheLRU(wl.S2, 1, wl.E)
    b4, b2 = bank4.numpy(), bank2.numpy()

    def dec(e, tag):
        if tag == 0:
            return F.decode_fp4_expert(b4[e * B4:(e + 1) * B4], wl.H, wl.I)
        return F.decode_int2_expert(b2[e * B2:(e + 1) * B2], wl.H, wl.I)

    for step in range(10):
        lg = gen.router_logits(wl, 0, step)
        x = gen.activations(wl, 0, step)
        y = torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda")
        runner.run(0, torch.from_numpy(lg).cuda(), torch.from_numpy(x.view(np.int16)).cuda(), y)
        torch.cuda.synchronize()
        ids, w = router_topk(lg, wl.k)
        w32 = w.astype(np.float32).astype(np.float64)
        tb = 0
        tags = np.full(ids.shape, 2)
        wout = np.zeros(ids.shape)
        while tb < wl.T:
            _, tg, wo, _, _, end = ladder_classify(r4, r2, 0, ids, w32, *wl.ladder, tb)
            tags[tb:end], wout[tb:end] = tg[tb:end], wo[tb:end]
            tb = end
        ref = moe_layer(x, np.where(tags == 2, -1, ids), wout, dec, tags=tags)
        assert bf16_rel_err(y.cpu().numpy(), ref) <= TOL
        assert np.array_equal(c4.export()[0], r4.state()[0])
        assert np.array_equal(c2.export()[0], r2.state()[0])


def test_stack_all_resident_no_sync():
    M = load_lib()
    wl = configs.scaled(configs.STACK, H=256, I=128, E=16, k=4, T=4, layers=3, S=48)
    layers = (0, 1, 2)
    bank, B, cache, runner, _ = _setup(M, wl, layers=layers, S=48, assume_resident=True)
    # populate: every key resident (slot = key), as after a warm-up pass
    slots_mem = runner.views._keep[0]
    slots_mem.copy_(bank.cuda())
    cache.import_(np.arange(48, dtype=np.int32), np.arange(48, dtype=np.uint64), 48)
    x = gen.activations(wl, 0, 0)
    xin = torch.from_numpy(x.view(np.int16)).cuda()
    for layer in layers:
        lg = gen.router_logits(wl, layer, 0)
        y = torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda")
        runner.run(layer, torch.from_numpy(lg).cuda(), xin, y)
        torch.cuda.synchronize()
        ids, w = router_topk(lg, wl.k)
        xin_np = xin.cpu().numpy().view(np.uint16)
        r = moe_layer(xin_np, ids, w, _decoder(bank.numpy(), B, wl, layer))
        assert bf16_rel_err(y.cpu().numpy(), r) <= TOL
        nxt = torch.empty_like(y)
        M.moe_rms_carry(y, 1e-6, nxt)
        xin = nxt
    assert runner.stats["misses"] == 0


def test_layer_ladder_device_copy():
    # the ladder chunk fits both pools by construction (T*a <= S4, T*(b-a) <= S2):
    # classify, both pools' copies by kernels and the forward run with no host wait
    M = load_lib()
    wl = configs.scaled(configs.LADDER, H=256, I=128, T=8, S=20, S2=30)
    bank4, B4 = pinned_fp4_bank(wl, (0,))
    B2 = M.moe_int2_expert_bytes(wl.H, wl.I)
    bank2 = torch.empty(wl.E * B2, dtype=torch.uint8, pin_memory=True)
    for e in range(wl.E):
        bank2[e * B2:(e + 1) * B2] = torch.from_numpy(gen.int2_expert(wl, 0, e))
    s4 = torch.empty(wl.S * B4, dtype=torch.uint8, device="cuda")
    s2 = torch.empty(wl.S2 * B2, dtype=torch.uint8, device="cuda")
    c4 = M.moe_cache(wl.S, 1, wl.E, B4, s4, bank4)
    c2 = M.moe_cache(wl.S2, 1, wl.E, B2, s2, bank2)
    views = M.make_views(wl.H, wl.I, s4, wl.S, s2, wl.S2, None)
    runner = M.DecodeLayerRunner(c4, views, wl.E, wl.k, wl.T, int2_cache=c2, ladder=wl.ladder, copy="device")
    assert runner._ladder_single_chunk(wl.T)
    r4, r2 = SlotCacheLRU(wl.S, 1, wl.E), SlotCacheLRU(wl.S2, 1, wl.E)
    b4, b2 = bank4.numpy(), bank2.numpy()

    def dec(e, tag):
        if tag == 0:
            return F.decode_fp4_expert(b4[e * B4:(e + 1) * B4], wl.H, wl.I)
        return F.decode_int2_expert(b2[e * B2:(e + 1) * B2], wl.H, wl.I)

    for step in range(10):
        lg = gen.router_logits(wl, 0, step)
        x = gen.activations(wl, 0, step)
        y = torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda")
        runner.run(0, torch.from_numpy(lg).cuda(), torch.from_numpy(x.view(np.int16)).cuda(), y)
        torch.cuda.synchronize()
        ids, w = router_topk(lg, wl.k)
        w32 = w.astype(np.float32).astype(np.float64)
        _, tg, wo, _, _, end = ladder_classify(r4, r2, 0, ids, w32, *wl.ladder, 0)
        assert end == wl.T
        ref = moe_layer(x, np.where(tg == 2, -1, ids), wo, dec, tags=tg)
        assert bf16_rel_err(y.cpu().numpy(), ref) <= TOL
        assert np.array_equal(c4.export()[0], r4.state()[0])
        assert np.array_equal(c2.export()[0], r2.state()[0])
    runner.check()
    assert runner.stats["misses"] > 0 and runner.stats["chunks"] == runner.stats["calls"]


def test_stack_full_size_sample_4_layers_x_4_steps():
    # the 43-layer stack workload at full size (H=4096, I=2048, E=256, top-8
    # plus the FP8 shared expert, T=16, 70% step-to-step reuse): a seeded
    # sample of 4 of its layers and 4 of its 64 steps, every expert of the
    # sampled layers resident; each step carries x from layer to layer on the
    # GPU (moe_rms_carry) and each layer is checked against the oracle from
    # the GPU's own bf16 input to that layer, on two sampled tokens
    M = load_lib()
    wl = configs.STACK
    H, I, E, k, T = wl.H, wl.I, wl.E, wl.k, wl.T
    rng = np.random.default_rng(wl.seed)
    layers = sorted(int(v) for v in rng.choice(wl.layers, size=4, replace=False))
    steps = sorted(int(v) for v in rng.choice(wl.steps, size=4, replace=False))
    B = M.moe_fp4_expert_bytes(H, I)
    S = len(layers) * E
    pool = torch.empty(S * B, dtype=torch.uint8, device="cuda")
    for li, layer in enumerate(layers):
        for e in range(E):
            key = li * E + e
            pool[key * B:(key + 1) * B] = gen.fp4_expert(wl, layer, e, device="cuda")
    cache = M.moe_cache(S, len(layers), E, B, pool, None)
    cache.import_(np.arange(S, dtype=np.int32), np.arange(S, dtype=np.uint64), S)
    shared_np = [gen.shared_expert(wl, layer) for layer in layers]
    shared = [torch.from_numpy(b).cuda() for b in shared_np]
    runners = [M.DecodeLayerRunner(cache, M.make_views(H, I, pool, S, None, 0, shared[li]), E, k, T,
                                   assume_resident=True) for li in range(len(layers))]
    record = {}      # (layer index, step) -> (x bits, logits, y bits)
    for step in steps:
        x = torch.from_numpy(gen.activations(wl, 0, step).view(np.int16)).cuda()
        for li, layer in enumerate(layers):
            lg = gen.router_logits(wl, layer, step)
            y = torch.empty((T, H), dtype=torch.int16, device="cuda")
            runners[li].run(li, torch.from_numpy(lg).cuda(), x, y)
            record[(li, step)] = (x.cpu().numpy().view(np.uint16), lg, y)
            nxt = torch.empty_like(y)
            M.moe_rms_carry(y, 1e-6, nxt)
            x = nxt
    torch.cuda.synchronize()
    for r in runners:
        r.check()
    assert all(r.stats["misses"] == 0 for r in runners)
    for li, layer in enumerate(layers):
        memo = {}      # decoded experts kept in float32 (exact for these scales) across the steps

        def dec(e, tag, layer=layer, memo=memo):
            if e not in memo:
                memo[e] = {m: v.astype(np.float32) for m, v in
                           F.decode_fp4_expert(gen.fp4_expert(wl, layer, e), H, I).items()}
            return {m: v.astype(np.float64) for m, v in memo[e].items()}
        shw = F.decode_fp8_expert(shared_np[li], H, I)
        for step in steps:
            xb, lg, y = record[(li, step)]
            ids, w = router_topk(lg, k)
            # the same two tokens at every step: their experts recur (70% reuse)
            tokens = sorted(int(v) for v in np.random.default_rng(1000 + layer).choice(T, 2, replace=False))
            ref = moe_layer(xb, ids, w, dec, shared=shw, tokens=tokens)
            assert bf16_rel_err(y.cpu().numpy()[tokens], ref) <= TOL, (layer, step)
    cache.close()
