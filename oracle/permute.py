"""Grouping of (token, rank) pairs by expert for the grouped GEMM.

"Running DeepSeek-V4-Flash across four free GPUs", section "All four workers
die, but only on prompts over 32 tokens": past T * top_k >= num_experts a
prefill chunk touches most of the layer, and the experts run as one grouped
GEMM over all tokens routed to each.  Plain definition: the flat pair index
p = t * k + j of every pair with a non-negative id, stably sorted by id;
offsets[e] is the first position of expert e (offsets has E + 1 entries).
"""
from __future__ import annotations

import numpy as np


def group_pairs(ids: np.ndarray, E: int):
    flat = np.asarray(ids, dtype=np.int64).reshape(-1)
    valid = np.nonzero(flat >= 0)[0]
    if np.any(flat[valid] >= E):
        raise ValueError("id >= E")
    order = valid[np.argsort(flat[valid], kind="stable")]
    counts = np.bincount(flat[valid], minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    return offsets, order.astype(np.int64)
