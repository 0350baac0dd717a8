"""Router: softmax over the E expert logits, keep the top_k, renormalise.

"Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
cache actually does": each decode step the router picks its top_k experts per
layer.  "An elephant through a straw", section "Not all six experts matter
equally": the router emits one weight per selected expert; survivors are
renormalised.  Selection is on the fp32 logits (softmax is monotone), ties go
to the lower expert id; weights are p_id / sum of kept p, p = softmax in fp64.
"""
from __future__ import annotations

import numpy as np


def router_topk(logits: np.ndarray, k: int, renorm: bool = True):
    """ids int32 [T, k] sorted by (logit descending, id ascending); weights fp64 [T, k]."""
    lg = np.asarray(logits, dtype=np.float32)
    if lg.ndim != 2:
        raise ValueError("logits must be [T, E]")
    T, E = lg.shape
    if not (1 <= k <= E):
        raise ValueError("need 1 <= k <= E")
    if not np.all(np.isfinite(lg)):
        raise ValueError("non-finite router logit")
    ids = np.empty((T, k), dtype=np.int32)
    w = np.empty((T, k), dtype=np.float64)
    eidx = np.arange(E)
    for t in range(T):
        # lexsort: last key is primary -> primary = -logit (fp32 exact), secondary = id
        order = np.lexsort((eidx, -lg[t].astype(np.float64)))
        sel = order[:k]
        ids[t] = sel
        z = lg[t].astype(np.float64)
        p = np.exp(z - z.max())
        p /= p.sum()
        kept = p[sel]
        w[t] = kept / kept.sum() if renorm else kept
    return ids, w
