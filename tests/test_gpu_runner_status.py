"""The host runner's status plumbing: an expert forward's error word reaches the
host through the status read-back of the next call (or `synchronize`), in every
copy mode, and the runner works on a stream other than the current one.

The failure is made on the host: the test writes an error code into the
forward's error word, as a failing forward would, and checks that the runner
raises it.  Nothing faults or waits on the GPU."""
import numpy as np
import pytest
import torch

from oracle.mlp import moe_layer
from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib, pinned_fp4_bank
from tests.test_gpu_layer import _decoder

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _runner(M, wl, S, copy):
    bank, B = pinned_fp4_bank(wl)
    slots = torch.empty(S * B, dtype=torch.uint8, device="cuda")
    cache = M.moe_cache(S, 1, wl.E, B, slots, bank)
    views = M.make_views(wl.H, wl.I, slots, S)
    return bank, B, cache, M.DecodeLayerRunner(cache, views, wl.E, wl.k, wl.T, copy=copy)


def _step(wl, step):
    lg = torch.from_numpy(gen.router_logits(wl, 0, step)).cuda()
    x = torch.from_numpy(gen.activations(wl, 0, step).view(np.int16)).cuda()
    return lg, x, torch.empty((wl.T, wl.H), dtype=torch.int16, device="cuda")


def test_device_copy_single_chunk_reports_forward_error_one_call_late():
    M = load_lib()
    wl = configs.TINY
    _, _, cache, r = _runner(M, wl, wl.E, "device")          # E slots: one chunk by construction
    r.run(0, *_step(wl, 0))
    r.synchronize()                                          # clean so far
    r.err.fill_(M.MOE_ERR_TIMEOUT)                           # as a forward that gave up would leave it
    r.run(0, *_step(wl, 1))                                  # reads call 1's status: clean
    with pytest.raises(M.MoeError) as ei:
        r.run(0, *_step(wl, 2))                              # reads call 2's status: the error word
    assert ei.value.status == M.MOE_ERR_TIMEOUT
    r.synchronize()                                          # call 2's own forward cleared it
    r.err.fill_(M.MOE_ERR_INVALID)
    with pytest.raises(M.MoeError) as ei:
        r.synchronize()
    assert ei.value.status == M.MOE_ERR_INVALID
    cache.close()


@pytest.mark.parametrize("copy", ["engine", "device"])
def test_multi_chunk_reads_forward_error_with_the_chunk_status(copy):
    M = load_lib()
    wl = configs.TINY                                        # 4 slots < 8 experts: several chunks
    _, _, cache, r = _runner(M, wl, wl.S, copy)
    r.run(0, *_step(wl, 0))
    r.synchronize()
    r.err.fill_(M.MOE_ERR_TIMEOUT)
    with pytest.raises(M.MoeError) as ei:
        r.run(0, *_step(wl, 1))                              # the first chunk's read-back carries it
    assert ei.value.status == M.MOE_ERR_TIMEOUT
    cache.close()


@pytest.mark.parametrize("copy", ["engine", "device"])
def test_runner_on_a_side_stream_matches_oracle(copy):
    M = load_lib()
    wl = configs.TINY
    bank, B, cache, r = _runner(M, wl, wl.S, copy)
    ref = SlotCacheLRU(wl.S, 1, wl.E)
    dec = _decoder(bank.numpy(), B, wl)
    s = torch.cuda.Stream()
    for step in range(wl.steps):
        lg, x, y = _step(wl, step)
        s.wait_stream(torch.cuda.current_stream())
        r.run(0, lg, x, y, stream=s)
        r.synchronize(stream=s)
        ids, w = router_topk(gen.router_logits(wl, 0, step), wl.k)
        tb = 0
        while tb < wl.T:
            _, _, _, tb = ref.ensure(0, ids, 0, wl.k, FETCH, tb)
        assert bf16_rel_err(y.cpu().numpy(), moe_layer(gen.activations(wl, 0, step), ids, w, dec)) <= TOL
        assert np.array_equal(cache.export()[0], ref.state()[0])
    cache.close()
