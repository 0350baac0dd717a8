"""Pins for the oracle router: brute force on tiny inputs and closed forms (CPU only)."""
import itertools

import numpy as np
import pytest
from scipy.special import softmax

from oracle.router import router_topk


def _brute_topk(row, k):
    E = len(row)
    best = None
    for sub in itertools.combinations(range(E), k):
        key = sorted((-float(row[e]), e) for e in sub)
        if best is None or key < best:
            best = key
    return [e for _, e in best]


@pytest.mark.parametrize("E,k", [(4, 1), (6, 2), (8, 2), (8, 3), (10, 4), (7, 7)])
def test_topk_matches_subset_enumeration(E, k):
    rng = np.random.default_rng(100 + E * 10 + k)
    for trial in range(30):
        if trial % 3 == 0:      # many ties: tie rule must pick lower ids
            lg = rng.integers(-2, 3, size=(3, E)).astype(np.float32)
        else:
            lg = rng.standard_normal((3, E)).astype(np.float32)
        ids, w = router_topk(lg, k)
        for t in range(3):
            assert list(ids[t]) == _brute_topk(lg[t], k)


def test_weights_sum_to_one_and_match_softmax_of_kept():
    rng = np.random.default_rng(5)
    lg = (rng.standard_normal((16, 256)) * 3).astype(np.float32)
    ids, w = router_topk(lg, 8)
    assert np.all(np.abs(w.sum(1) - 1.0) <= 1e-12)
    assert np.all(w > 0)
    for t in range(16):
        kept = lg[t, ids[t]].astype(np.float64)
        assert np.allclose(w[t], softmax(kept), rtol=0, atol=1e-15)
        # weights are non-increasing along rank
        assert np.all(np.diff(w[t]) <= 1e-15)


def test_no_renorm_gives_full_softmax_probabilities():
    rng = np.random.default_rng(6)
    lg = rng.standard_normal((4, 32)).astype(np.float32)
    ids, w = router_topk(lg, 4, renorm=False)
    for t in range(4):
        p = softmax(lg[t].astype(np.float64))
        assert np.allclose(w[t], p[ids[t]], rtol=0, atol=1e-15)


def test_k_equals_E_is_full_softmax_in_sorted_order():
    lg = np.array([[0.5, -1.0, 2.0, 0.5]], dtype=np.float32)
    ids, w = router_topk(lg, 4)
    assert list(ids[0]) == [2, 0, 3, 1]
    assert np.allclose(w[0], softmax(lg[0].astype(np.float64))[[2, 0, 3, 1]], atol=1e-15)


def test_selection_uses_fp32_logits_exactly():
    # two logits one fp32 ulp apart: the larger wins even though exp() of both may round equal
    a = np.float32(1.0)
    b = np.nextafter(a, np.float32(2.0))
    lg = np.array([[a, b, -5.0]], dtype=np.float32)
    ids, _ = router_topk(lg, 1)
    assert ids[0, 0] == 1


def test_rejects_non_finite():
    with pytest.raises(ValueError):
        router_topk(np.array([[0.0, np.nan]], dtype=np.float32), 1)
