"""Expert forward (gate/up + SwiGLU, down, combine with the shared expert) and the
dequant hook vs the oracle.  Dequantised weights bit-exact; layer outputs within
max |err| <= 2e-2 * RMS of the oracle row."""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle.mlp import moe_layer
from synth import configs, gen
from tests.helpers import bf16_rel_err, load_lib

pytestmark = pytest.mark.gpu
TOL = 2e-2


class Pools:
    """Device pools whose slot s holds a known generated expert, plus decoders."""

    def __init__(self, M, wl, n4, n2=0, shared=False, layer=0):
        self.M, self.wl = M, wl
        H, I = wl.H, wl.I
        self.B4 = M.moe_fp4_expert_bytes(H, I)
        self.B2 = M.moe_int2_expert_bytes(H, I)
        self.e4 = [(7 * s + 3) % wl.E for s in range(n4)]
        self.e2 = [(5 * s + 1) % wl.E for s in range(n2)]
        self.fp4 = torch.empty(max(n4, 1) * self.B4, dtype=torch.uint8, device="cuda")
        for s, e in enumerate(self.e4):
            self.fp4[s * self.B4:(s + 1) * self.B4] = gen.fp4_expert(wl, layer, e, device="cuda")
        self.int2 = None
        if n2:
            self.int2 = torch.empty(n2 * self.B2, dtype=torch.uint8, device="cuda")
            for s, e in enumerate(self.e2):
                self.int2[s * self.B2:(s + 1) * self.B2] = torch.from_numpy(gen.int2_expert(wl, layer, e)).cuda()
        self.shared_np = gen.shared_expert(wl, layer) if shared else None
        self.shared = torch.from_numpy(self.shared_np).cuda() if shared else None
        self.views = M.make_views(H, I, self.fp4, n4, self.int2, n2, self.shared)
        self.layer = layer
        self._cache = {}

    def weights(self, slot, tag):
        key = (slot, tag)
        if key not in self._cache:
            wl = self.wl
            if tag == 0:
                blob = gen.fp4_expert(wl, self.layer, self.e4[slot])
                self._cache[key] = F.decode_fp4_expert(blob, wl.H, wl.I)
            else:
                blob = gen.int2_expert(wl, self.layer, self.e2[slot])
                self._cache[key] = F.decode_int2_expert(blob, wl.H, wl.I)
        return self._cache[key]

    def shared_weights(self):
        return F.decode_fp8_expert(self.shared_np, self.wl.H, self.wl.I) if self.shared is not None else None

    def forward(self, x_bits, slots, tags, w):
        M = self.M
        T, k = slots.shape
        y = torch.empty((T, self.wl.H), dtype=torch.int16, device="cuda")
        ws = torch.empty(M.moe_expert_forward_workspace(self.views, T, k), dtype=torch.uint8, device="cuda")
        err = torch.full((1,), -5, dtype=torch.int32, device="cuda")
        M.moe_expert_forward(self.views, torch.from_numpy(x_bits.view(np.int16)).cuda(),
                             torch.from_numpy(slots.astype(np.int32)).cuda(),
                             None if tags is None else torch.from_numpy(tags.astype(np.int8)).cuda(),
                             torch.from_numpy(w.astype(np.float32)).cuda(), y, ws, err)
        torch.cuda.synchronize()
        return y.cpu().numpy(), int(err)

    def reference(self, x_bits, slots, tags, w, tokens=None):
        return moe_layer(x_bits, slots, w.astype(np.float32).astype(np.float64), self.weights,
                         shared=self.shared_weights(), tags=tags, tokens=tokens)


def _route(rng, T, k, n, skew=True):
    p = 1.0 / np.arange(1, n + 1) ** (1.1 if skew else 0.0)
    p /= p.sum()
    slots = np.stack([rng.choice(n, size=k, replace=False, p=p) for _ in range(T)])
    w = rng.random((T, k)) + 0.05
    return slots, (w / w.sum(1, keepdims=True)).astype(np.float32)


@pytest.mark.parametrize("pool,matrix", [(0, 0), (0, 1), (0, 2), (1, 0), (1, 2), (2, 0), (2, 2)])
def test_dequant_bit_exact_tiny(pool, matrix):
    M = load_lib()
    wl = configs.scaled(configs.TINY, H=256, I=128)
    P = Pools(M, wl, 2, 2, shared=True)
    N, K = F.matrix_shape(F.MATRICES[matrix], wl.H, wl.I)
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    M.moe_dequant_debug(P.views, pool, 1 if pool < 2 else 0, matrix, out)
    torch.cuda.synchronize()
    if pool == 2:
        ref = P.shared_weights()[F.MATRICES[matrix]]
    else:
        ref = P.weights(1, pool)[F.MATRICES[matrix]]
    got = out.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), ref.astype(np.float32).view(np.uint32))


def test_dequant_bit_exact_full_size_slot():
    M = load_lib()
    wl = configs.DECODE
    P = Pools(M, wl, 1, 1, shared=True)
    for pool in (0, 1, 2):
        for matrix in (0, 2):
            N, K = F.matrix_shape(F.MATRICES[matrix], wl.H, wl.I)
            out = torch.empty((N, K), dtype=torch.float32, device="cuda")
            M.moe_dequant_debug(P.views, pool, 0, matrix, out)
            torch.cuda.synchronize()
            ref = (P.shared_weights() if pool == 2 else P.weights(0, pool))[F.MATRICES[matrix]]
            assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("shared", [False, True])
def test_forward_tiny_all_tokens(shared):
    M = load_lib()
    wl = configs.TINY
    P = Pools(M, wl, wl.S, shared=shared)
    rng = np.random.default_rng(11)
    for T in (1, 4, 13):
        slots, w = _route(rng, T, wl.k, wl.S)
        x = gen.activations(wl, 0, T, T)
        y, err = P.forward(x, slots, None, w)
        assert err == 0
        assert bf16_rel_err(y, P.reference(x, slots, None, w)) <= TOL


def test_forward_generic_shape_many_tokens_per_slot_ladder_tags():
    # H, I not the specialised sizes; > 8 tokens on one slot (several groups);
    # FP4 / 2-bit / dropped pairs; a token with every pair dropped; negative slots
    M = load_lib()
    wl = configs.scaled(configs.TINY, H=512, I=256, E=16)
    P = Pools(M, wl, 6, 5, shared=True)
    rng = np.random.default_rng(12)
    T, k = 37, 4
    slots = rng.integers(0, 5, size=(T, k))
    slots[:20, 0] = 2
    tags = rng.integers(0, 3, size=(T, k))
    tags[5] = 2
    slots[7, 1] = -1
    w = rng.random((T, k)).astype(np.float32)
    x = gen.activations(wl, 0, 99, T)
    y, err = P.forward(x, slots, tags, w)
    assert err == 0
    ref = P.reference(x, np.where(tags == 2, -1, slots), tags, w)
    assert bf16_rel_err(y, ref) <= TOL


def test_forward_reports_bad_slot():
    M = load_lib()
    wl = configs.TINY
    P = Pools(M, wl, 2)
    slots = np.array([[0, 5]])
    y, err = P.forward(gen.activations(wl, 0, 1, 1), slots, None, np.array([[0.5, 0.5]], np.float32))
    assert err == M.MOE_ERR_INVALID


@pytest.mark.parametrize("T", [1, 2, 4, 16, 64])
def test_forward_decode_full_size_sampled(T):
    M = load_lib()
    wl = configs.DECODE
    P = Pools(M, wl, wl.S, shared=True)
    rng = np.random.default_rng(100 + T)
    slots, w = _route(rng, T, wl.k, wl.S)
    x = gen.activations(wl, 0, 5, T)
    y, err = P.forward(x, slots, None, w)
    assert err == 0
    sample = sorted(set([0, T - 1, T // 2]))
    ref = P.reference(x, slots, None, w, tokens=sample)
    assert bf16_rel_err(y[sample], ref) <= TOL


def test_forward_ladder_full_size_sampled():
    M = load_lib()
    wl = configs.LADDER
    P = Pools(M, wl, 12, 12)
    rng = np.random.default_rng(7)
    T, k = wl.T, wl.k
    slots, w = _route(rng, T, k, 12)
    tags = np.zeros((T, k), dtype=np.int64)
    tags[:, 2:4] = rng.integers(0, 2, size=(T, 2))
    tags[:, 4:] = rng.choice([0, 1, 2], size=(T, 2))
    x = gen.activations(wl, 0, 3, T)
    y, err = P.forward(x, slots, tags, w)
    assert err == 0
    sample = [0, 17, 31]
    ref = P.reference(x, np.where(tags == 2, -1, slots), tags, w, tokens=sample)
    assert bf16_rel_err(y[sample], ref) <= TOL


def test_rms_carry():
    M = load_lib()
    rng = np.random.default_rng(3)
    y = (rng.standard_normal((5, 4096)) * 1e5).astype(np.float32)
    yb = gen.bf16_bits(y)
    out = torch.empty((5, 4096), dtype=torch.int16, device="cuda")
    M.moe_rms_carry(torch.from_numpy(yb.view(np.int16)).cuda(), 1e-6, out)
    torch.cuda.synchronize()
    from oracle.mlp import rms_carry
    ref = rms_carry(F.bf16_to_f64(yb))
    got = F.bf16_to_f64(out.cpu().numpy().view(np.uint16))
    assert np.max(np.abs(got - ref) / np.abs(ref).clip(1e-30)) <= 2 ** -8


@pytest.mark.parametrize("T", [4, 16, 64])
def test_decode_paths_both_match_oracle(T):
    # the warp-MMA kernels (the default up to 64 tokens) and, with them switched
    # off, the CUDA-core GEMV (below 256 pairs) or the tcgen05 grouped GEMM
    M = load_lib()
    wl = configs.DECODE
    P = Pools(M, wl, 24, shared=True)
    rng = np.random.default_rng(300 + T)
    slots, w = _route(rng, T, wl.k, 24)
    x = gen.activations(wl, 0, 8, T)
    sample = sorted(set([0, T - 1, T // 3]))
    ref = P.reference(x, slots, None, w, tokens=sample)
    old = M.moe_set_option(M.MOE_OPT_MMA_MAX_TOKENS, 64)
    try:
        y_mma, err = P.forward(x, slots, None, w)
        assert err == 0
        M.moe_set_option(M.MOE_OPT_MMA_MAX_TOKENS, 0)
        y_other, err = P.forward(x, slots, None, w)
        assert err == 0
    finally:
        M.moe_set_option(M.MOE_OPT_MMA_MAX_TOKENS, old)
    assert bf16_rel_err(y_mma[sample], ref) <= TOL
    assert bf16_rel_err(y_other[sample], ref) <= TOL
    with pytest.raises(M.MoeError):
        M.moe_set_option(M.MOE_OPT_MMA_MAX_TOKENS, -1)
