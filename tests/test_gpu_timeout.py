"""Failure detection on the GPU without a fault: a bounded device-side wait
that nothing satisfies gives up, reports MOE_ERR_TIMEOUT, and the context
stays usable."""
import time

import numpy as np
import pytest
import torch

from tests.helpers import load_lib

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    M = load_lib()
    status = torch.full((1,), 7, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    M.moe_debug_timeout_probe(20_000_000, status)      # 20 ms
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status) == M.MOE_ERR_TIMEOUT
    assert dt < 1.0
    # the context still runs kernels
    lg = torch.from_numpy(np.arange(8, dtype=np.float32)[None, :]).cuda()
    ids, w = M.moe_router_topk(lg, 2)
    torch.cuda.synchronize()
    assert ids.cpu().tolist() == [[7, 6]]


def test_probe_rejects_bad_limits():
    M = load_lib()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(M.MoeError):
        M.moe_debug_timeout_probe(0, status)
