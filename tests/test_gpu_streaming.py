"""Whole-layer streaming prefill: each streamed layer gives bit-identical
outputs to the grouped-GEMM prefill on the same layer resident, and matches the
oracle (max |err| <= 2e-2 * RMS of the oracle row)."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.mlp import moe_layer
from oracle.router import router_topk
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib, pinned_fp4_bank

pytestmark = pytest.mark.gpu
TOL = 2e-2


def test_streamed_layers_match_resident_prefill_and_oracle():
    M = load_lib()
    wl = configs.scaled(configs.PREFILL, H=512, I=512, E=16, k=4, T=96)
    layers = (0, 1, 2)
    bank, B = pinned_fp4_bank(wl, layers)
    st = M.PrefillStreamer(bank, len(layers), wl.E, wl.H, wl.I, wl.k, wl.T)
    st.begin(0)
    T = wl.T
    for layer in layers:
        lg = gen.router_logits(wl, layer, 0, T)
        x = gen.activations(wl, layer, 0, T)
        xd = torch.from_numpy(x.view(np.int16)).cuda()
        y = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
        st.run_layer(layer, torch.from_numpy(lg).cuda(), xd, y)
        st.synchronize()                       # raises if the grouped GEMM reported a failure
        assert int(st.err) == 0
        # the same layer resident in a pool of its own, through moe_expert_prefill
        pool = bank[layer * wl.E * B:(layer + 1) * wl.E * B].cuda()
        views = M.make_views(wl.H, wl.I, pool, wl.E)
        ids, w = router_topk(lg, wl.k)
        assert np.array_equal(st.ids[:T].cpu().numpy(), ids)     # same routing as the oracle
        y2 = torch.empty_like(y)
        ws = torch.empty(M.moe_expert_prefill_workspace(views, T, wl.k), dtype=torch.uint8, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        M.moe_expert_prefill(views, xd, st.ids[:T].clone(), st.w[:T].clone(), y2, ws, err)
        torch.cuda.synchronize()
        assert torch.equal(y, y2)
        b = bank.numpy()

        def dec(e, tag):
            o = (layer * wl.E + e) * B
            return F.decode_fp4_expert(b[o:o + B], wl.H, wl.I)
        ref = moe_layer(x, ids, w.astype(np.float32).astype(np.float64), dec)
        assert bf16_rel_err(y.cpu().numpy(), ref) <= TOL


def test_copy_layer_rejects_pageable_bank():
    M = load_lib()
    buf = torch.empty(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MoeError):
        M.moe_copy_layer(torch.zeros(256, dtype=torch.uint8), 0, 4, 16, buf)
