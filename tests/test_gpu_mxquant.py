"""A-quantised (MXFP4 activations) prefill mode: the device quantiser bit-exact
against the oracle's OCP MX rule, and the grouped-GEMM prefill in that mode
within max |err| <= 2e-2 * RMS of the oracle row computed with the same
quantisation of x and of its own fp64 h."""
import numpy as np
import pytest
import torch

from oracle.mlp import moe_layer
from oracle.mxquant import mx_quantize, mx_round
from oracle.router import router_topk
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib
from tests.test_gpu_prefill import _pool

pytestmark = pytest.mark.gpu
TOL = 2e-2


def _bf16_bits(v):
    """fp64 -> bf16 bits (round to nearest even), as uint16."""
    f = np.asarray(v, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def _bits_to_f64(b):
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_quantiser_bit_exact():
    M = load_lib()
    rng = np.random.default_rng(3)
    rows, K = 40, 256
    v = rng.standard_normal((rows, K)) * np.exp(rng.uniform(-20, 20, (rows, 1)))
    v[0, :32] = 0.0                                          # zero block
    v[1, :32] = 0.0
    v[1, 0] = 4.0                                           # X = 1: every midpoint, both signs
    v[1, 1:15] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0]
    v[2, :32] = 7.9                                         # saturation
    v[3, :32] = -0.0                                        # negative zeros
    v[4, :32] = 2.0 ** -130                                 # subnormal block (clamped scale)
    v[5, :32] = rng.standard_normal(32) * 1e37              # near the top of the range
    b = _bf16_bits(v)
    b[6, 5] = 0x8000                                        # -0 inside a normal block
    ref_codes, ref_scales = mx_quantize(_bits_to_f64(b))
    x = torch.from_numpy(b.view(np.int16)).cuda()
    codes = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((rows, K // 32), dtype=torch.uint8, device="cuda")
    M.moe_mx_quantize(x, codes, scales)
    torch.cuda.synchronize()
    assert np.array_equal(scales.cpu().numpy(), ref_scales)
    assert np.array_equal(codes.cpu().numpy(), ref_codes)


def test_quantiser_rejects_bad_sizes():
    M = load_lib()
    x = torch.zeros((2, 48), dtype=torch.int16, device="cuda")
    with pytest.raises(M.MoeError):
        M.moe_mx_quantize(x, torch.empty(48, dtype=torch.uint8, device="cuda"),
                          torch.empty(4, dtype=torch.uint8, device="cuda"))


def _prefill(M, views, x, slots, w, mode):
    T, k = slots.shape
    y = torch.empty((T, views.H), dtype=torch.int16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(M.moe_expert_prefill_workspace(views, T, k), dtype=torch.uint8, device="cuda")
    M.moe_expert_prefill_prec(views, torch.from_numpy(x.view(np.int16)).cuda(),
                              torch.from_numpy(slots.astype(np.int32)).cuda(),
                              torch.from_numpy(w.astype(np.float32)).cuda(), mode, y, ws, err)
    torch.cuda.synchronize()
    return y.cpu().numpy(), int(err)


def test_prefill_mxfp4_mode_small_all_tokens():
    M = load_lib()
    wl = configs.scaled(configs.PREFILL, H=512, I=512, E=16)
    S = 12
    pool, views, weights = _pool(M, wl, S)
    rng = np.random.default_rng(11)
    T, k = 300, 6
    slots = np.stack([rng.choice(S, size=k, replace=False) for _ in range(T)])
    w = rng.random((T, k)).astype(np.float32)
    x = gen.activations(wl, 0, 2, T)
    y, err = _prefill(M, views, x, slots, w, M.MOE_PREC_A_MXFP4)
    assert err == 0
    ref = moe_layer(x, slots, w.astype(np.float64), weights, quant=mx_round)
    assert bf16_rel_err(y, ref) <= TOL
    # the mode changes the result (it is not the W4A16 path)
    y16, _ = _prefill(M, views, x, slots, w, M.MOE_PREC_W4A16)
    assert not np.array_equal(y, y16)
    with pytest.raises(M.MoeError):
        _prefill(M, views, x, slots, w, 7)


def test_prefill_mxfp4_mode_full_size_sampled():
    M = load_lib()
    wl = configs.PREFILL
    S = 64
    pool, views, weights = _pool(M, wl, S)
    T = 700
    ids, w = router_topk(gen.router_logits(wl, 0, 1, T), wl.k)
    slots = ids % S
    for t in range(T):
        seen = set()
        for j in range(wl.k):
            while slots[t, j] in seen:
                slots[t, j] = (slots[t, j] + 1) % S
            seen.add(int(slots[t, j]))
    x = gen.activations(wl, 0, 1, T)
    y, err = _prefill(M, views, x, slots, w, M.MOE_PREC_A_MXFP4)
    assert err == 0
    rows = [0, 1, 350, 699]
    ref = moe_layer(x, slots, w.astype(np.float64), weights, tokens=rows, quant=mx_round)
    assert bf16_rel_err(y[rows], ref) <= TOL


def test_fp4_mma_peak_probe():
    # back-to-back kind::mxf4 MMAs: a dense block-scaled FP4 rate well above the
    # bf16 tensor rate of the same GPU
    M = load_lib()
    tf = M.moe_fp4_mma_peak(1024)
    assert 2000.0 < tf < 30000.0
    with pytest.raises(M.MoeError):
        M.moe_fp4_mma_peak(100)
