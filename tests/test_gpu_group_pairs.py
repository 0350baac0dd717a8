"""Pair grouping vs the oracle (bit-exact, stable order)."""
import numpy as np
import pytest
import torch

from oracle.permute import group_pairs
from oracle.router import router_topk
from synth import configs, gen
from tests.helpers import load_lib

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,k,E", [(4, 2, 8), (64, 8, 256), (8192, 6, 256), (1, 1, 1), (333, 5, 40)])
def test_group_pairs_matches_oracle(T, k, E):
    M = load_lib()
    rng = np.random.default_rng(T + E)
    ids = rng.integers(-1, E, size=(T, k)).astype(np.int32)
    off, perm, err = M.moe_group_pairs(torch.from_numpy(ids).cuda(), E)
    torch.cuda.synchronize()
    roff, rperm = group_pairs(ids, E)
    assert int(err) == 0
    assert np.array_equal(off.cpu().numpy(), roff)
    assert np.array_equal(perm.cpu().numpy()[:roff[-1]], rperm)


def test_group_pairs_prefill_routing():
    M = load_lib()
    wl = configs.PREFILL
    ids = router_topk(gen.router_logits(wl, 0, 0), wl.k)[0]
    off, perm, err = M.moe_group_pairs(torch.from_numpy(ids).cuda(), wl.E)
    roff, rperm = group_pairs(ids, wl.E)
    assert np.array_equal(off.cpu().numpy(), roff) and np.array_equal(perm.cpu().numpy(), rperm)
    counts = np.diff(roff)
    assert 120 < counts.mean() < 260   # near-uniform ~192 pairs per expert


def test_group_pairs_bad_id():
    M = load_lib()
    off, perm, err = M.moe_group_pairs(torch.tensor([[0, 9]], dtype=torch.int32, device="cuda"), 4)
    torch.cuda.synchronize()
    assert int(err) == M.MOE_ERR_INVALID
