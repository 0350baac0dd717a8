"""Grouped-GEMM (tcgen05) prefill path vs the oracle: outputs within
max |err| <= 2e-2 * RMS of the oracle row."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.mlp import moe_layer
from oracle.router import router_topk
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _pool(M, wl, S):
    B = M.moe_fp4_expert_bytes(wl.H, wl.I)
    experts = [(11 * s + 5) % wl.E for s in range(S)]
    pool = torch.empty(S * B, dtype=torch.uint8, device="cuda")
    for s, e in enumerate(experts):
        pool[s * B:(s + 1) * B] = gen.fp4_expert(wl, 0, e, device="cuda")
    memo = {}

    def weights(slot, tag):
        if slot not in memo:
            memo[slot] = F.decode_fp4_expert(gen.fp4_expert(wl, 0, experts[slot]), wl.H, wl.I)
        return memo[slot]
    return pool, M.make_views(wl.H, wl.I, pool, S), weights


def _run(M, views, x, slots, w, entry="prefill"):
    T, k = slots.shape
    xs = torch.from_numpy(x.view(np.int16)).cuda()
    sl = torch.from_numpy(slots.astype(np.int32)).cuda()
    ww = torch.from_numpy(w.astype(np.float32)).cuda()
    y = torch.empty((T, views.H), dtype=torch.int16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    if entry == "prefill":
        ws = torch.empty(M.moe_expert_prefill_workspace(views, T, k), dtype=torch.uint8, device="cuda")
        M.moe_expert_prefill(views, xs, sl, ww, y, ws, err)
    else:
        ws = torch.empty(M.moe_expert_forward_workspace(views, T, k), dtype=torch.uint8, device="cuda")
        M.moe_expert_forward(views, xs, sl, None, ww, y, ws, err)
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(err)


def test_prefill_small_all_tokens_multi_item_and_ragged():
    M = load_lib()
    wl = configs.scaled(configs.PREFILL, H=512, I=512, E=16)
    S = 12
    pool, views, weights = _pool(M, wl, S)
    rng = np.random.default_rng(1)
    T, k = 300, 6
    slots = np.stack([rng.choice(S, size=k, replace=False) for _ in range(T)])
    slots[:, 0] = 3                  # one slot with 300 rows: two items of 256 + 44
    for t in range(T):                # keep ids distinct per token
        row = slots[t]
        for j in range(1, k):
            if row[j] == 3:
                row[j] = [s for s in range(S) if s not in row][0]
    slots[7, 2] = -1                  # a skipped pair
    w = rng.random((T, k)).astype(np.float32)
    x = gen.activations(wl, 0, 0, T)
    y, err = _run(M, views, x, slots, w)
    assert err == 0
    ref = moe_layer(x, slots, w.astype(np.float64), weights)
    assert bf16_rel_err(y, ref) <= TOL


def test_prefill_full_size_via_forward_dispatch_sampled():
    M = load_lib()
    wl = configs.PREFILL
    S = 64
    pool, views, weights = _pool(M, wl, S)
    T = 700                           # 4200 pairs: above the decode-plan limit
    ids, w = router_topk(gen.router_logits(wl, 0, 0, T), wl.k)
    slots = ids % S
    for t in range(T):                # distinct slots per token
        seen = set()
        for j in range(wl.k):
            while slots[t, j] in seen:
                slots[t, j] = (slots[t, j] + 1) % S
            seen.add(slots[t, j])
    x = gen.activations(wl, 0, 0, T)
    y, err = _run(M, views, x, slots, w.astype(np.float32), entry="forward")
    assert err == 0
    sample = [0, 351, 699]
    ref = moe_layer(x, slots, w.astype(np.float32).astype(np.float64), weights, tokens=sample)
    assert bf16_rel_err(y[sample], ref) <= TOL


@pytest.mark.parametrize("T", [64, 100])
def test_prefill_matches_decode_path(T):
    # the two expert paths agree on the same call (both within the oracle
    # tolerance); T = 64 takes the deep-ring GEMM shape, T = 100 the wide one
    M = load_lib()
    wl = configs.scaled(configs.PREFILL, H=512, I=1024, E=16)
    S = 8
    pool, views, weights = _pool(M, wl, S)
    rng = np.random.default_rng(5)
    k = 4
    slots = np.stack([rng.choice(S, size=k, replace=False) for _ in range(T)])
    w = rng.random((T, k)).astype(np.float32)
    x = gen.activations(wl, 0, 1, T)
    y1, e1 = _run(M, views, x, slots, w, "prefill")
    y2, e2 = _run(M, views, x, slots, w, "forward")
    assert e1 == 0 and e2 == 0
    ref = moe_layer(x, slots, w.astype(np.float64), weights)
    assert bf16_rel_err(y1, ref) <= TOL and bf16_rel_err(y2, ref) <= TOL


def test_grouped_gemm_item_sizes_at_the_shape_limit():
    # decode-sized call through the grouped GEMM: one slot routed from all 64
    # tokens (an item of exactly 64 rows), one from at least 33, the rest ragged
    M = load_lib()
    wl = configs.scaled(configs.PREFILL, H=1024, I=512, E=16)
    S = 10
    pool, views, weights = _pool(M, wl, S)
    rng = np.random.default_rng(9)
    T, k = 64, 6
    slots = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        rest = [s for s in range(S) if s != 3 and (t >= 33 or s != 5)]
        picks = list(rng.choice(rest, size=k - (1 if t >= 33 else 2), replace=False))
        slots[t] = [3] + ([] if t >= 33 else [5]) + picks
    w = rng.random((T, k)).astype(np.float32)
    x = gen.activations(wl, 0, 2, T)
    y, err = _run(M, views, x, slots, w, "forward")
    assert err == 0
    ref = moe_layer(x, slots, w.astype(np.float64), weights)
    assert bf16_rel_err(y, ref) <= TOL


def test_prefill_rejects_unsupported():
    M = load_lib()
    wl = configs.scaled(configs.TINY)
    pool, views, _ = _pool(M, wl, 2)
    with pytest.raises(M.MoeError):
        _run(M, views, gen.activations(wl, 0, 0, 2), np.array([[0, 1], [1, 0]]),
             np.full((2, 2), 0.5, np.float32))
