"""One routed MoE layer served from the expert-slot cache, driven from the host.

The per-layer sequence is the pages': router, ensure_experts (ids remapped to
slots on the device), exactly one host synchronisation to read the miss list
("An elephant through a straw", section "43 graphs, 43 syncs"), the misses
copied from the pinned bank on a side stream ("Running DeepSeek-V4-Flash
across four free GPUs", section "What the expert cache actually does"), then
the grouped expert MLP.  When a token chunk needs more distinct experts than
there are slots, ensure reports how far it got and the sequence repeats for
the rest.  All arithmetic runs in the library's kernels; this file only
sequences calls and owns buffers.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib as L


class DecodeLayerRunner:
    """Buffers and streams for running layers of one model shape on one cache."""

    def __init__(self, cache: L.moe_cache, views: L.moe_expert_views, E: int, k: int,
                 T_max: int, device=None, int2_cache: Optional[L.moe_cache] = None,
                 ladder=None, assume_resident: bool = False):
        self.cache, self.views, self.E, self.k, self.T_max = cache, views, E, k, T_max
        self.dev = torch.device(device or "cuda")
        self.c2, self.ladder = int2_cache, ladder
        dev = self.dev
        P = T_max * k
        self.ids = torch.empty((T_max, k), dtype=torch.int32, device=dev)
        self.w = torch.empty((T_max, k), dtype=torch.float32, device=dev)
        self.slots = torch.empty((T_max, k), dtype=torch.int32, device=dev)
        self.tags = torch.empty((T_max, k), dtype=torch.int8, device=dev)
        self.w2 = torch.empty((T_max, k), dtype=torch.float32, device=dev)
        m4 = min(cache.S, P, E)
        m2 = min(int2_cache.S, P, E) if int2_cache is not None else 0
        self.m4, self.m2 = m4, m2
        # [count4, done, count2, pad, keys4[m4], slots4[m4], keys2[m2], slots2[m2]]
        n = 4 + 2 * m4 + 2 * m2
        self.info = torch.zeros(n, dtype=torch.int32, device=dev)
        self.info_h = torch.zeros(n, dtype=torch.int32, pin_memory=True)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = torch.empty(L.moe_expert_forward_workspace(views, T_max, k), dtype=torch.uint8,
                              device=dev)
        self.copy_stream = torch.cuda.Stream(device=dev)
        self.ready = torch.cuda.Event()
        self.done = torch.cuda.Event()
        self.assume_resident = assume_resident
        if assume_resident and cache.S < cache.L * cache.E:
            raise ValueError("assume_resident needs a cache with a slot for every key")
        self.stats = {"misses": 0, "hits_pairs": 0, "calls": 0, "bytes_copied": 0, "chunks": 0}

    def _views(self, t):
        i = self.info
        m4, m2 = self.m4, self.m2
        return dict(count4=i[0:1], done=i[1:2], count2=i[2:3], keys4=i[4:4 + m4],
                    slots4=i[4 + m4:4 + 2 * m4], keys2=i[4 + 2 * m4:4 + 2 * m4 + m2],
                    slots2=i[4 + 2 * m4 + m2:4 + 2 * m4 + 2 * m2])

    def run(self, layer_id: int, logits, x, y, stream=None):
        """y[T, H] (bf16 bits) = the MoE layer applied to x[T, H] with router logits [T, E]."""
        T = logits.shape[0]
        assert T <= self.T_max
        stream = stream or torch.cuda.current_stream(self.dev)
        k = self.k
        ids, w, slots = self.ids[:T], self.w[:T], self.slots[:T]
        L.moe_router_topk(logits, k, True, ids, w, stream)
        v = self._views(T)
        tb = 0
        self.stats["calls"] += 1
        while tb < T:
            if self.ladder is None:
                L.moe_slot_ensure(self.cache, layer_id, ids, slots, 0, k, L.MOE_FETCH, tb,
                                  v["keys4"], v["slots4"], v["count4"], v["done"], stream)
                tags, wuse = None, w
            else:
                a, b = self.ladder
                L.moe_ladder_classify(self.cache, self.c2, layer_id, ids, w, a, b, tb, slots,
                                      self.tags[:T], self.w2[:T], v["keys4"], v["slots4"],
                                      v["count4"], v["keys2"], v["slots2"], v["count2"], v["done"],
                                      stream)
                tags, wuse = self.tags[:T], self.w2[:T]
            if self.assume_resident and self.ladder is None:
                done = T
            else:
                self.info_h.copy_(self.info, non_blocking=True)
                stream.synchronize()
                h = self.info_h
                n4, done = int(h[0]), int(h[1])
                n2 = int(h[2]) if self.ladder is not None else 0
                if n4 < 0 or n2 < 0:
                    code = -min(n4, n2)
                    raise L.MoeError(code, "slot ensure failed on the device "
                                     f"(token_begin={tb})")
                if n4 or n2:
                    self.ready.record(stream)
                    m4 = self.m4
                    if n4:
                        L.moe_copy_missing(self.cache, h[4:4 + m4], h[4 + m4:4 + 2 * m4], n4,
                                           self.copy_stream, self.ready, None)
                    if n2:
                        o = 4 + 2 * m4
                        L.moe_copy_missing(self.c2, h[o:o + self.m2], h[o + self.m2:o + 2 * self.m2],
                                           n2, self.copy_stream, self.ready, None)
                    self.done.record(self.copy_stream)
                    stream.wait_event(self.done)
                    self.stats["misses"] += n4 + n2
                    self.stats["bytes_copied"] += n4 * self.cache.B + (n2 * self.c2.B if n2 else 0)
            self.stats["chunks"] += 1
            L.moe_expert_forward(self.views, x[tb:done], slots[tb:done],
                                 None if tags is None else tags[tb:done], wuse[tb:done], y[tb:done],
                                 self.ws, self.err, stream)
            tb = done
        return y
