"""The allocation-free forward entry point (for callers that cannot allocate
device memory: it uses the library's fixed device scratch) gives the same
result as moe_expert_forward with a caller workspace, bit for bit, on two calls in
a row.
Runs last so that a failure here leaves every other test already run."""
import numpy as np
import pytest
import torch

from synth import configs, gen
from tests.helpers import load_lib

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_forward_two_calls():
    M = load_lib()
    wl = configs.DECODE
    H, I, S = wl.H, wl.I, 16
    B = M.moe_fp4_expert_bytes(H, I)
    pool = torch.empty(S * B, dtype=torch.uint8, device="cuda")
    for s in range(S):
        pool[s * B:(s + 1) * B] = gen.fp4_expert(wl, 0, 3 * s + 1, device="cuda")
    shared = torch.from_numpy(gen.shared_expert(wl, 0)).cuda()
    views = M.make_views(H, I, pool, S, None, 0, shared)
    rng = np.random.default_rng(21)
    for call, T in enumerate((64, 5)):
        slots = torch.from_numpy(np.stack([rng.choice(S, size=wl.k, replace=False) for _ in range(T)])
                                 .astype(np.int32)).cuda()
        w = torch.from_numpy(rng.random((T, wl.k)).astype(np.float32)).cuda()
        x = torch.from_numpy(gen.activations(wl, 0, 40 + call, T).view(np.int16)).cuda()
        ws = torch.empty(M.moe_expert_forward_workspace(views, T, wl.k), dtype=torch.uint8, device="cuda")
        err_ref = torch.zeros(1, dtype=torch.int32, device="cuda")
        err_na = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        y_ref = torch.empty((T, H), dtype=torch.int16, device="cuda")
        y_na = torch.empty((T, H), dtype=torch.int16, device="cuda")
        M.moe_expert_forward(views, x, slots, None, w, y_ref, ws, err_ref)
        M.moe_expert_forward_noalloc(views, x, slots, None, w, y_na, err_na)
        torch.cuda.synchronize()
        assert int(err_ref) == 0 and int(err_na) == 0
        # the same kernels on the same inputs: bit-identical, so leftover scratch
        # contents from the first call cannot leak into the second call's output
        assert torch.equal(y_na, y_ref)


def test_noalloc_rejects_oversize():
    M = load_lib()
    wl = configs.DECODE
    S = 2
    B = M.moe_fp4_expert_bytes(wl.H, wl.I)
    pool = torch.zeros(S * B, dtype=torch.uint8, device="cuda")
    views = M.make_views(wl.H, wl.I, pool, S)
    T = 512                       # 4096 pairs: needs far more than the fixed scratch
    slots = torch.zeros((T, 8), dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoeError) as ei:
        M.moe_expert_forward_noalloc(views, torch.zeros((T, wl.H), dtype=torch.int16, device="cuda"), slots,
                                     None, torch.zeros((T, 8), device="cuda"),
                                     torch.empty((T, wl.H), dtype=torch.int16, device="cuda"))
    assert ei.value.status == M.MOE_ERR_INVALID
