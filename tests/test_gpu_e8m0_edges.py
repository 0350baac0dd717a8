"""E8M0 block scales at the ends of their range, mixed within one weight tile.

The generated workloads draw scales from 124..128 only, which leaves two
paths unexercised: the grouped GEMM's bf16-operand branch (a tile whose scales
do not all lie where scaled E2M1 values are exact fp16 numbers) and the fp32
block scaling of the decode kernels at extreme exponents (2^-127 .. 2^127,
including the subnormal scale byte 0).  Here scale bytes 0, 1, 100, 150, 253
and 254 are written into the first rows of every matrix of one expert, next to
the generated 124..128 ones.  Checked: the decoded weights bit-exact, and the
decode forward (T = 1, 4, 64) and the grouped-GEMM prefill within
2e-2 * RMS of the oracle row.  Blocks with scale 253 or 254 get zero codes
in the experts run through the MLP, so that every product stays within fp32
(6 * 2^127 alone exceeds it); the dequantisation check keeps their codes.

Every row of every matrix gets each edge value in the same number of blocks
(blocks 0 .. 11 of the row).  A row of w2 scales one output feature, so edge
scales in some rows only would make a few features ~2^23 times the rest; the
bf16 rounding of the output alone would then exceed 2e-2 of the row's RMS.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.mlp import moe_layer
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib

pytestmark = pytest.mark.gpu
TOL = 2e-2
EDGES = (0, 1, 100, 150, 253, 254)


def edge_expert(wl, expert, zero_huge):
    """Generated expert bytes with edge scale bytes in every row of each matrix:
    block b < 12 of row n gets EDGES[(n + b) % 6] (each edge value twice per
    row); the other blocks keep their generated 124..128 scales."""
    blob = gen.fp4_expert(wl, 0, expert).copy()
    lay, _ = F.fp4_layout(wl.H, wl.I)
    for m in F.MATRICES:
        c, s, N, K = lay[m]
        nb = K // 32
        codes = blob[c:s].reshape(N, K // 2)
        sc = blob[s:s + N * nb].reshape(N, nb)
        n = np.arange(N)[:, None]
        b = np.arange(12)[None, :]
        sc[:, :12] = np.asarray(EDGES, dtype=np.uint8)[(n + b) % 6]
        if zero_huge:
            big = sc[:, :12] >= 253
            codes[:, :192].reshape(N, 12, 16)[big] = 0
    return blob


def _pool(M, wl, blobs):
    B = M.moe_fp4_expert_bytes(wl.H, wl.I)
    pool = torch.empty(len(blobs) * B, dtype=torch.uint8, device="cuda")
    for s, b in enumerate(blobs):
        pool[s * B:(s + 1) * B] = torch.from_numpy(b).cuda()
    return pool


def test_dequant_edge_scales_bit_exact():
    M = load_lib()
    wl = configs.DECODE
    blob = edge_expert(wl, 5, zero_huge=False)
    pool = _pool(M, wl, [blob])
    views = M.make_views(wl.H, wl.I, pool, 1)
    ref = F.decode_fp4_expert(blob, wl.H, wl.I)
    for mi, m in enumerate(F.MATRICES):
        N, K = F.matrix_shape(m, wl.H, wl.I)
        out = torch.empty((N, K), dtype=torch.float32, device="cuda")
        M.moe_dequant_debug(views, M.MOE_POOL_FP4, 0, mi, out)
        torch.cuda.synchronize()
        with np.errstate(over="ignore"):
            want = ref[m].astype(np.float32)       # 2 * 2^127 and above are inf in fp32
        assert np.array_equal(out.cpu().numpy().view(np.uint32), want.view(np.uint32)), m


def _mlp_setup(M, wl, n_slots):
    # slot 0 and slot 2 hold edge-scale experts, the others generated ones
    blobs = [edge_expert(wl, 7, True) if s in (0, 2) else gen.fp4_expert(wl, 0, 11 + s) for s in range(n_slots)]
    pool = _pool(M, wl, blobs)
    dec = {s: F.decode_fp4_expert(b, wl.H, wl.I) for s, b in enumerate(blobs)}
    return pool, (lambda e, tag: dec[e])


@pytest.mark.parametrize("T", [1, 4, 64])
def test_forward_edge_scales(T):
    M = load_lib()
    wl = configs.DECODE
    S = 6
    pool, weights = _mlp_setup(M, wl, S)
    shared_np = gen.shared_expert(wl, 0)
    views = M.make_views(wl.H, wl.I, pool, S, None, 0, torch.from_numpy(shared_np).cuda())
    rng = np.random.default_rng(500 + T)
    k = wl.k
    kk = min(k, S)
    slots = np.empty((T, kk), dtype=np.int32)
    for t in range(T):
        # every token routes to an edge-scale expert first, and to no slot twice
        e = 0 if t % 2 == 0 else 2
        order = [int(v) for v in rng.permutation(S) if v != e]
        slots[t] = [e] + order[:kk - 1]
    w = rng.random((T, kk)).astype(np.float32) + 0.05
    w /= w.sum(1, keepdims=True)
    x = gen.activations(wl, 0, 77, T)
    y = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
    ws = torch.empty(M.moe_expert_forward_workspace(views, T, kk), dtype=torch.uint8, device="cuda")
    err = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    M.moe_expert_forward(views, torch.from_numpy(x.view(np.int16)).cuda(), torch.from_numpy(slots).cuda(), None,
                         torch.from_numpy(w).cuda(), y, ws, err)
    torch.cuda.synchronize()
    assert int(err) == 0
    sample = sorted({0, T - 1, T // 2})
    ref = moe_layer(x, slots, w.astype(np.float64), weights, shared=F.decode_fp8_expert(shared_np, wl.H, wl.I),
                    tokens=sample)
    assert bf16_rel_err(y.cpu().numpy()[sample], ref) <= TOL


def test_prefill_edge_scales():
    M = load_lib()
    wl = configs.PREFILL
    S = 4
    pool, weights = _mlp_setup(M, wl, S)
    views = M.make_views(wl.H, wl.I, pool, S)
    T, k = 400, 3               # ~300 rows per slot: items of 256 rows and ragged tails
    rng = np.random.default_rng(9)
    slots = np.stack([rng.permutation(S)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32) + 0.05
    w /= w.sum(1, keepdims=True)
    x = gen.activations(wl, 0, 78, T)
    y = torch.empty((T, wl.H), dtype=torch.int16, device="cuda")
    ws = torch.empty(M.moe_expert_prefill_workspace(views, T, k), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_expert_prefill(views, torch.from_numpy(x.view(np.int16)).cuda(), torch.from_numpy(slots).cuda(),
                         torch.from_numpy(w).cuda(), y, ws, err)
    torch.cuda.synchronize()
    assert int(err) == 0
    sample = [0, 1, 2, 150, T - 2, T - 1]
    ref = moe_layer(x, slots, w.astype(np.float64), weights, tokens=sample)
    assert bf16_rel_err(y.cpu().numpy()[sample], ref) <= TOL
