"""SwiGLU expert MLP and the router-weighted combine with the shared expert, in fp64.

"Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
cache actually does" (the routed experts' grouped GEMM over w1/w2/w3) and
"An elephant through a straw", section "Rig, model & methodology" (256
routed experts, top-6, plus one shared expert per layer; DeepSeek-V3
lineage).  Per (token, expert) pair: h = SiLU(W1 x) * (W3 x) with
SiLU(z) = z / (1 + e^-z), o = W2 h.  Layer output:
y_t = sum_j w_{t,j} o_{t,j} + shared(x_t), the shared expert being the same
SwiGLU MLP with weight 1.

Reading for carrying a stack of layers: the next layer's input is the bf16
rounding of y / sqrt(mean(y^2) + 1e-6) per token (a weightless RMSNorm that
stands in for the model's pre-MoE norm).
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_to_f64


def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_mlp(x: np.ndarray, W: dict, quant=None) -> np.ndarray:
    """x fp64 [n, H]; W = {'w1': [I,H], 'w3': [I,H], 'w2': [H,I]} fp64 -> [n, H].

    ``quant`` (e.g. ``mxquant.mx_round``) is applied to x and to h before
    their products when the activations are quantised."""
    if quant is not None:
        x = quant(x)
    g = x @ W["w1"].T
    u = x @ W["w3"].T
    h = silu(g) * u
    if quant is not None:
        h = quant(h)
    return h @ W["w2"].T


def moe_layer(x_bits: np.ndarray, ids: np.ndarray, w: np.ndarray, expert_weights,
              shared: dict | None = None, tags: np.ndarray | None = None,
              tokens=None, quant=None) -> np.ndarray:
    """y fp64 [len(tokens), H].

    ``expert_weights(expert, tag) -> W`` decodes a routed expert (tag 0 FP4,
    1 the 2-bit copy); pairs with tag 2 (dropped) or a negative id are skipped.
    ``quant``: activation quantiser of the routed experts' x and h (None: W4A16).
    """
    x = bf16_to_f64(x_bits)
    T, k = ids.shape
    tokens = list(range(T)) if tokens is None else list(tokens)
    H = x.shape[1]
    # per-pair outputs, grouped by (expert, tag) only to decode each expert once
    groups = {}
    for t in tokens:
        for j in range(k):
            tag = 0 if tags is None else int(tags[t, j])
            if ids[t, j] < 0 or tag == 2:
                continue
            groups.setdefault((int(ids[t, j]), tag), []).append((t, j))
    o = {}
    for (e, tag), pairs in groups.items():
        W = expert_weights(e, tag)
        out = expert_mlp(x[[t for t, _ in pairs]], W, quant)
        for (t, j), row in zip(pairs, out):
            o[(t, j)] = row
    y = np.zeros((len(tokens), H), dtype=np.float64)
    for r, t in enumerate(tokens):
        for j in range(k):
            if (t, j) in o:
                y[r] += w[t, j] * o[(t, j)]
        if shared is not None:
            y[r] += expert_mlp(x[t:t + 1], shared)[0]
    return y


def rms_carry(y: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    """fp64 y / sqrt(mean(y^2) + eps) per row (the next layer's input before bf16 rounding)."""
    y = np.asarray(y, dtype=np.float64)
    return y / np.sqrt(np.mean(y * y, axis=1, keepdims=True) + eps)
