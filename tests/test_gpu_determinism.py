"""Identical calls must give bit-identical outputs: the grouped-GEMM pipeline
at the full prefill size and the decode forward, repeated.  Races between the
pipeline's producers and consumers show up here as run-to-run differences,
which sampled-row parity against the oracle can miss."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.mlp import moe_layer
from oracle.router import router_topk
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib
from tests.test_gpu_forward import Pools, _route

pytestmark = pytest.mark.gpu


def test_prefill_full_size_repeatable_and_oracle_rows():
    # the full prefill workload (T = 8192, top-6, all 256 experts resident):
    # four identical calls give identical bits, and sampled rows match the
    # oracle -- the first and last tokens and a token of the largest and of
    # the smallest expert group (items of 256 rows at K = H and K = I)
    M = load_lib()
    wl = configs.PREFILL
    H, I, E = wl.H, wl.I, wl.E
    B = M.moe_fp4_expert_bytes(H, I)
    pool = torch.empty(E * B, dtype=torch.uint8, device="cuda")
    for e in range(E):
        pool[e * B:(e + 1) * B] = gen.fp4_expert(wl, 0, e, device="cuda")
    views = M.make_views(H, I, pool, E)
    ids, w = router_topk(gen.router_logits(wl, 0, 0), wl.k)
    sl = torch.from_numpy(ids.astype(np.int32)).cuda()
    ww = torch.from_numpy(w.astype(np.float32)).cuda()
    x = torch.from_numpy(gen.activations(wl, 0, 0).view(np.int16)).cuda()
    ws = torch.empty(M.moe_expert_prefill_workspace(views, wl.T, wl.k), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(4):
        y = torch.empty((wl.T, H), dtype=torch.int16, device="cuda")
        M.moe_expert_prefill(views, x, sl, ww, y, ws, err)
        torch.cuda.synchronize()
        assert int(err) == 0
        outs.append(y)
    for y in outs[1:]:
        assert torch.equal(y, outs[0])
    counts = np.bincount(ids.ravel(), minlength=E)
    big, small = int(np.argmax(counts)), int(np.argmin(np.where(counts > 0, counts, 1 << 30)))
    sample = sorted({0, wl.T - 1, int(np.nonzero((ids == big).any(1))[0][0]),
                     int(np.nonzero((ids == small).any(1))[0][-1])})
    xb = gen.activations(wl, 0, 0)
    ref = moe_layer(xb, ids, w.astype(np.float32).astype(np.float64),
                    lambda e, tag: F.decode_fp4_expert(gen.fp4_expert(wl, 0, e), H, I), tokens=sample)
    got = outs[0].cpu().numpy()[sample]
    assert bf16_rel_err(got, ref) <= 2e-2


@pytest.mark.parametrize("T", [1, 2, 16, 64])
def test_decode_forward_repeatable(T):
    M = load_lib()
    wl = configs.DECODE
    P = Pools(M, wl, 64, shared=True)
    rng = np.random.default_rng(900 + T)
    slots, w = _route(rng, T, wl.k, 64)
    x = gen.activations(wl, 0, 2, T)
    first = None
    for _ in range(6):
        y, err = P.forward(x, slots, None, w)
        assert err == 0
        if first is None:
            first = y
        assert np.array_equal(y, first)
