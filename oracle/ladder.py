"""The (a, b) precision ladder over an FP4 pool and a 2-bit-copy pool.

"An elephant through a straw", section "Not all six experts matter equally":
precision follows the router's ranking.  Ranks 1..a always use FP4 and are
fetched if missing; ranks a+1..b use FP4 when resident and the 2-bit copy
otherwise; ranks below b are used if resident (in either pool) and dropped
if not; the survivors' weights are renormalised.

Readings where the page is silent: the passes run over the whole token chunk
in this order -- (i) FP4 FETCH of ranks 1..a; (ii) FP4 LOOKUP of ranks
a+1..b, then 2-bit FETCH of those still unresolved; (iii) for the remaining
ranks FP4 LOOKUP, then 2-bit LOOKUP, then drop.  Residency is judged after
the earlier passes' fetches.  The chunk is the longest token prefix whose
distinct rank-1..a experts fit the FP4 pool and whose distinct rank-a+1..b
experts fit the 2-bit pool.
"""
from __future__ import annotations

import numpy as np

from .slot_cache import FETCH, LOOKUP, CapacityError, SlotCacheLRU

TAG_FP4 = 0
TAG_INT2 = 1
TAG_DROP = 2


def _chunk_end(ids, token_begin, lo, hi, cap):
    seen = set()
    end = token_begin
    for t in range(token_begin, ids.shape[0]):
        new = {int(e) for e in ids[t, lo:hi] if e >= 0} - seen
        if len(seen) + len(new) > cap:
            break
        seen |= new
        end = t + 1
    return end


def ladder_classify(c4: SlotCacheLRU, c2: SlotCacheLRU, layer: int, ids, w, a: int, b: int,
                    token_begin: int = 0):
    """Returns (slots, tags, w_out, (keys4, slots4), (keys2, slots2), tokens_done)."""
    ids = np.asarray(ids)
    w = np.asarray(w, dtype=np.float64)
    T, k = ids.shape
    if not (1 <= a <= b <= k):
        raise ValueError("need 1 <= a <= b <= k")
    end = min(_chunk_end(ids, token_begin, 0, a, c4.S), _chunk_end(ids, token_begin, a, b, c2.S))
    if end == token_begin and token_begin < T:
        raise CapacityError("one token needs more experts than a pool has slots")
    sub = ids[:end]

    s4, mk4, ms4, e1 = c4.ensure(layer, sub, 0, a, FETCH, token_begin)
    assert e1 == end
    l4, _, _, _ = c4.ensure(layer, sub, a, b, LOOKUP, token_begin)
    need2 = sub.copy()
    need2[l4 >= 0] = -1
    s2, mk2, ms2, e2 = c2.ensure(layer, need2, a, b, FETCH, token_begin)
    assert e2 == end
    l4b, _, _, _ = c4.ensure(layer, sub, b, k, LOOKUP, token_begin)
    need2b = sub.copy()
    need2b[l4b >= 0] = -1
    l2b, _, _, _ = c2.ensure(layer, need2b, b, k, LOOKUP, token_begin)

    slots = np.full((T, k), -1, dtype=np.int64)
    tags = np.full((T, k), TAG_DROP, dtype=np.int64)
    w_out = np.zeros((T, k), dtype=np.float64)
    for t in range(token_begin, end):
        for j in range(k):
            if j < a:
                slots[t, j], tags[t, j] = s4[t, j], TAG_FP4
            elif j < b:
                if l4[t, j] >= 0:
                    slots[t, j], tags[t, j] = l4[t, j], TAG_FP4
                else:
                    slots[t, j], tags[t, j] = s2[t, j], TAG_INT2
            else:
                if l4b[t, j] >= 0:
                    slots[t, j], tags[t, j] = l4b[t, j], TAG_FP4
                elif l2b[t, j] >= 0:
                    slots[t, j], tags[t, j] = l2b[t, j], TAG_INT2
        keep = tags[t] != TAG_DROP
        w_out[t] = np.where(keep, w[t], 0.0) / np.sum(w[t][keep])
    return slots, tags, w_out, (mk4, ms4), (mk2, ms2), end
