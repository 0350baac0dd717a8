"""Router kernel vs the oracle: ids bit-exact, weights within 1e-6."""
import numpy as np
import pytest
import torch

from oracle.router import router_topk
from synth import configs, gen
from tests.helpers import load_lib

pytestmark = pytest.mark.gpu


def _run(M, lg, k, renorm=True):
    ids, w = M.moe_router_topk(torch.from_numpy(lg).cuda(), k, renorm)
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T,E,k", [(4, 8, 2), (1, 256, 8), (64, 256, 8), (1000, 256, 6),
                                   (37, 100, 5), (3, 2048, 32), (5, 32, 32), (9, 1, 1), (33, 300, 7)])
def test_router_matches_oracle(T, E, k):
    M = load_lib()
    rng = np.random.default_rng(T * 7 + E)
    lg = (rng.standard_normal((T, E)) * 2).astype(np.float32)
    ids, w = _run(M, lg, k)
    rid, rw = router_topk(lg, k)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= 1e-6


def test_router_ties_go_to_lower_id():
    M = load_lib()
    rng = np.random.default_rng(1)
    lg = rng.integers(-3, 4, size=(200, 64)).astype(np.float32)
    ids, w = _run(M, lg, 8)
    rid, rw = router_topk(lg, 8)
    assert np.array_equal(ids, rid)
    assert np.max(np.abs(w - rw)) <= 1e-6


def test_router_no_renorm():
    M = load_lib()
    lg = np.random.default_rng(2).standard_normal((16, 256)).astype(np.float32)
    ids, w = _run(M, lg, 8, renorm=False)
    rid, rw = router_topk(lg, 8, renorm=False)
    assert np.array_equal(ids, rid) and np.max(np.abs(w - rw)) <= 1e-6


def test_router_decode_trace_zipf():
    M = load_lib()
    wl = configs.DECODE
    for step in range(4):
        lg = gen.router_logits(wl, 0, step, 64)
        ids, w = _run(M, lg, wl.k)
        rid, rw = router_topk(lg, wl.k)
        assert np.array_equal(ids, rid) and np.max(np.abs(w - rw)) <= 1e-6


def test_router_empty_and_invalid():
    M = load_lib()
    ids, w = M.moe_router_topk(torch.empty((0, 8), device="cuda"), 2)
    assert ids.shape == (0, 2)
    with pytest.raises(M.MoeError):
        M.moe_router_topk(torch.zeros((2, 8), device="cuda"), 9)
