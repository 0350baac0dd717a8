"""Bank priming leaves the bank and the cache unchanged; the profile timeline
orders its records and spans both streams of an overlapped step."""
import numpy as np
import pytest
import torch

from synth import configs
from tests.helpers import load_lib, pinned_fp4_bank

pytestmark = pytest.mark.gpu


def test_prime_bank_reads_only():
    M = load_lib()
    wl = configs.scaled(configs.TINY, E=16)
    bank, B = pinned_fp4_bank(wl, (0,))
    before = bank.clone()
    slots = torch.zeros(4 * B, dtype=torch.uint8, device="cuda")
    cache = M.moe_cache(4, 1, wl.E, B, slots, bank)
    state0 = cache.export()
    M.moe_cache_prime_bank(cache)
    torch.cuda.synchronize()
    assert torch.equal(bank, before)
    assert not slots.any()
    for a, b in zip(state0, cache.export()):
        assert np.array_equal(a, b)
    cache.prime_bank()                      # the wrapper primes once per cache
    assert cache.primed
    cache.close()
    no_bank = M.moe_cache(4, 1, wl.E, B, slots, None)
    with pytest.raises(M.MoeError):
        M.moe_cache_prime_bank(no_bank)
    no_bank.close()


def test_profile_timeline_records():
    M = load_lib()
    logits = torch.randn((8, 64), device="cuda")
    M.moe_profile_enable(True)
    try:
        M.moe_router_topk(logits, 4)
        M.moe_router_topk(logits, 4)
        torch.cuda.synchronize()
        tl = M.moe_profile_timeline()
    finally:
        M.moe_profile_enable(False)
    assert [r[0] for r in tl] == [M.MOE_K_ROUTER, M.MOE_K_ROUTER]
    assert tl[0][1] == 0.0
    for kid, a, b in tl:
        assert 0.0 <= a <= b
    assert tl[1][1] >= tl[0][2] - 1e-3       # same stream: the second starts after the first ends
    assert M.moe_profile_timeline() == []    # disabling clears nothing, enabling clears: empty when off
