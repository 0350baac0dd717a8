"""Layer steps replayed as CUDA graphs give the same outputs, slot tables and
miss counts as the same steps run eagerly (and so as the oracle)."""
import numpy as np
import pytest
import torch

from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU
from synth import configs, gen
from tests.helpers import load_lib, pinned_fp4_bank

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 4])
def test_graph_replay_equals_eager(T):
    M = load_lib()
    wl = configs.scaled(configs.DECODE, T=T)
    S = 64
    bank, B = pinned_fp4_bank(wl, (0,))
    sh = torch.from_numpy(gen.shared_expert(wl, 0)).cuda()
    runs = []
    for graph in (False, True):
        slots = torch.empty(S * B, dtype=torch.uint8, device="cuda")
        cache = M.moe_cache(S, 1, wl.E, B, slots, bank)
        views = M.make_views(wl.H, wl.I, slots, S, None, 0, sh)
        runner = M.DecodeLayerRunner(cache, views, wl.E, wl.k, T, copy="device", graph=graph)
        ys, tables = [], []
        for step in range(8):
            lg = torch.from_numpy(gen.router_logits(wl, 0, step, T)).cuda()
            x = torch.from_numpy(gen.activations(wl, 0, step, T).view(np.int16)).cuda()
            y = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
            runner.run(0, lg, x, y)
            torch.cuda.synchronize()
            ys.append(y.cpu().numpy())
            tables.append(cache.export()[0].copy())
        runner.check()
        runs.append((ys, tables, runner.stats["misses"], len(runner.graphs)))
        cache.close()
    assert runs[0][3] == 0 and runs[1][3] == 1          # one graph, replayed for steps 1..7
    for a, b in zip(runs[0][0], runs[1][0]):
        assert np.array_equal(a, b)
    for a, b in zip(runs[0][1], runs[1][1]):
        assert np.array_equal(a, b)
    assert runs[0][2] == runs[1][2] > 0
    # and the slot tables follow the oracle
    ref = SlotCacheLRU(S, 1, wl.E)
    for step in range(8):
        ids = router_topk(gen.router_logits(wl, 0, step, T), wl.k)[0]
        ref.ensure(0, ids, 0, wl.k, FETCH, 0)
        assert np.array_equal(runs[1][1][step], ref.state()[0])
