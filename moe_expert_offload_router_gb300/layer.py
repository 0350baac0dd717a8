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

With ``copy="device"`` the misses are instead copied by a kernel that reads
the miss list on the device (``moe_copy_missing_device``), so router, ensure,
copy and forward are enqueued back to back.  Ensure runs in the mode that
marks tokens past its chunk as skipped, the forward is enqueued for every
remaining token, and the host reads ``tokens_done`` afterwards, while the GPU
works; a second chunk (if any) then recomputes the rows it owns.  When the
batch cannot need more distinct experts than there are slots
(``min(E, T*k) <= S``) there is a single chunk by construction and the host
does not wait at all: the status of each layer is checked on the next call
(or by :meth:`check`).

An expert forward reports a failure (a slot out of range, a pipeline wait that
gave up) through an error word on the device.  The runner keeps that word in
its status block, so the read-back that follows the next ensure brings it to
the host with the ensure status: `run` raises a forward's failure one call
later, and :meth:`synchronize` raises the last call's.

With ``graph=True`` (device copy, no ladder) a layer step whose batch is one
chunk by construction is captured once as a CUDA graph (router, ensure,
status read-back, copies, forward) and replayed on static buffers, which
removes the per-launch host cost of small batches.

With ``overlap=True`` (device copy only) the copy kernel runs on a side stream
with a small grid while ``moe_expert_forward_overlap`` computes the pairs of
resident experts and the shared expert; only the pairs of missed experts wait
for the copies.  ``overlap="auto"`` does so from 256 pairs per call.

The precision ladder takes ``copy="device"`` too: when a batch cannot need more
distinct experts of either rank range than its pool has slots, classify, the
copies of both pools and the forward are enqueued without a host wait.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import _lib as L


class DecodeLayerRunner:
    """Buffers and streams for running layers of one model shape on one cache.

    ``run(layer_id, logits, x, y)`` performs one layer step: router, slot
    ensure, miss copies, expert MLP and combine.

    * ``copy``: "engine" (one host read of the miss list, then copy-engine
      copies) or "device" (a kernel copies the misses straight from the miss
      list on the device; no host wait when the batch is one chunk).
    * ``overlap`` (device copies): True, False or "auto" (from
      OVERLAP_MIN_PAIRS pairs): pairs of resident experts compute while the
      misses are copied.  With ``copy_parts`` 1 the copies are staged: every
      miss's gate/up matrices first, then its down matrices in ``down_parts``
      parts of the miss list; ``copy_parts`` > 1 instead splits the miss list
      into that many parts, each with its own pass.
    * ``copy_ctas``: the copy kernel's grid (each CTA keeps an SM from the
      grouped GEMM).
    * ``graph``: replay single-chunk device-copy steps as CUDA graphs.
    * ``assume_resident``: every key has its slot (a cache of L * E slots);
      no copies, no host waits.
    * ``int2_cache`` and ``ladder`` = (a, b): the precision ladder.
    """

    # overlap="auto" overlaps copies and compute from this many pairs per call:
    # below it the second forward pass costs more than the short copies hide
    OVERLAP_MIN_PAIRS = 256

    def __init__(self, cache: L.moe_cache, views: L.moe_expert_views, E: int, k: int,
                 T_max: int, device=None, int2_cache: Optional[L.moe_cache] = None,
                 ladder=None, assume_resident: bool = False, copy: str = "engine",
                 overlap=False, copy_ctas: int = 32, graph: bool = False, copy_parts: int = 1,
                 down_parts: int = 1):
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
        # [count4, done, count2, err, keys4[m4], slots4[m4], keys2[m2], slots2[m2]]
        n = 4 + 2 * m4 + 2 * m2
        self.info = torch.zeros(n, dtype=torch.int32, device=dev)
        self.info_h = torch.zeros(n, dtype=torch.int32, pin_memory=True)
        # the forward's error word sits in the status block: every status read-back
        # (taken after ensure, before the next forward clears it) carries the
        # previous forward's status to the host at no extra cost
        self.err = self.info[3:4]
        self.ws = torch.empty(L.moe_expert_forward_workspace(views, T_max, k), dtype=torch.uint8,
                              device=dev)
        # high priority: a copy launched while the compute stream's GEMM still has
        # CTAs waiting for SMs gets the next free SMs instead of queueing behind them
        self.copy_stream = torch.cuda.Stream(device=dev, priority=-1)
        self.ready = torch.cuda.Event()
        self.done = torch.cuda.Event()
        if copy not in ("engine", "device"):
            raise ValueError("copy must be 'engine' or 'device'")
        if copy == "device" and ladder is not None and overlap:
            raise ValueError("the ladder takes copy='device' without overlap")
        self.copy = copy
        if overlap not in (False, True, "auto"):
            raise ValueError("overlap must be False, True or 'auto'")
        if overlap and copy != "device":
            raise ValueError("overlap needs copy='device'")
        self.overlap, self.copy_ctas = overlap, copy_ctas
        if not 1 <= copy_parts <= L.MOE_MAX_COPY_PARTS:
            raise ValueError(f"copy_parts must be in [1, {L.MOE_MAX_COPY_PARTS}]")
        self.copy_parts = copy_parts
        self.part_done = [torch.cuda.Event() for _ in range(copy_parts)]
        self.gu_done = torch.cuda.Event()
        if not 1 <= down_parts <= L.MOE_MAX_COPY_PARTS:
            raise ValueError(f"down_parts must be in [1, {L.MOE_MAX_COPY_PARTS}]")
        self.down_done = [torch.cuda.Event() for _ in range(down_parts)]
        # bytes of one FP4 matrix (codes + E8M0 scales); w1 and w3 come first in an expert
        self.gu_half = views.H * views.I // 2 + views.H * views.I // 32
        self.ws_ov = (torch.empty(L.moe_expert_forward_overlap_workspace(views, T_max, k), dtype=torch.uint8,
                                  device=dev) if overlap else None)
        self.status_h = torch.zeros(4, dtype=torch.int32, pin_memory=True)
        self.status_ev = torch.cuda.Event()
        self.pending = None   # (layer_id, T) whose status is still to be read
        # staging-ring prefetch (moe_cache_set_staging on the cache)
        npf = 4096
        self.pf_key = torch.empty(npf, dtype=torch.int32, device=dev)
        self.pf_slot = torch.empty(npf, dtype=torch.int32, device=dev)
        self.pf_cnt = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pf_ready = torch.cuda.Event()
        self.pf_done = torch.cuda.Event()
        self.pf_pending = False
        if copy == "device" and not assume_resident:
            # the first GPU read of a bank page is slow: translate every page now
            for c in (cache, int2_cache):
                if c is not None:
                    c.prime_bank()
        # CUDA graphs of whole single-chunk device-copy layer steps, per (layer, T)
        self.graph = graph
        self.graphs = {}
        self._capturing = False
        self.assume_resident = assume_resident
        if assume_resident and cache.S < cache.L * cache.E:
            raise ValueError("assume_resident needs a cache with a slot for every key")
        self._vcache = None   # views into self.info, built on first use
        self.stats = {"misses": 0, "hits_pairs": 0, "calls": 0, "bytes_copied": 0, "chunks": 0}

    def _views(self, t):
        if self._vcache is not None:
            return self._vcache
        i = self.info
        m4, m2 = self.m4, self.m2
        self._vcache = dict(count4=i[0:1], done=i[1:2], count2=i[2:3], keys4=i[4:4 + m4],
                    slots4=i[4 + m4:4 + 2 * m4], keys2=i[4 + 2 * m4:4 + 2 * m4 + m2],
                    slots2=i[4 + 2 * m4 + m2:4 + 2 * m4 + 2 * m2])
        return self._vcache

    def prefetch(self, layer_id: int, d_experts, stream=None):
        """Stages predicted experts of `layer_id` (device int32 ids) in the cache's
        ring: the assignment runs on `stream` after everything enqueued there,
        the copies on the side stream after the copies already queued on it."""
        stream = stream or torch.cuda.current_stream(self.dev)
        # the previous prefetch's copy kernel (side stream) still reads the key /
        # slot lists and its ring slots: the assignment that rewrites them waits
        self._wait_prefetch(stream)
        L.moe_prefetch(self.cache, layer_id, d_experts, self.pf_key, self.pf_slot, self.pf_cnt, stream)
        self.pf_ready.record(stream)
        self.copy_stream.wait_event(self.pf_ready)
        L.moe_copy_missing_device(self.cache, self.pf_key, self.pf_slot, self.pf_cnt, self.copy_stream,
                                  self.copy_ctas)
        self.pf_done.record(self.copy_stream)
        self.pf_pending = True

    def _wait_prefetch(self, stream):
        # a staged expert promoted by a copy on `stream` must have landed
        if self.pf_pending:
            stream.wait_event(self.pf_done)

    @staticmethod
    def _forward_status(e: int):
        # the error word a read-back carries is that of the forward enqueued before it
        if e != L.MOE_OK:
            raise L.MoeError(e, "an earlier expert forward reported a failure on the device")

    def check(self):
        """Reads the status of the last device-mode layer whose check was deferred
        (and with it the error word of the forward enqueued before that layer)."""
        if self.pending is None:
            return
        layer_id, T = self.pending
        self.pending = None
        self.status_ev.synchronize()
        n4, done = int(self.status_h[0]), int(self.status_h[1])
        n2 = int(self.status_h[2]) if self.ladder is not None else 0
        self._forward_status(int(self.status_h[3]))
        if n4 < 0 or n2 < 0:
            raise L.MoeError(-min(n4, n2), f"slot ensure failed on the device (layer {layer_id})")
        self.stats["misses"] += n4 + n2
        self.stats["bytes_copied"] += n4 * self.cache.B + (n2 * self.c2.B if n2 else 0)
        if done != T:
            raise L.MoeError(L.MOE_ERR_CAPACITY, f"layer {layer_id}: single chunk expected, got {done}/{T}")

    def _run_device(self, layer_id, T, ids, w, slots, x, y, stream, prefetch=None):
        v = self._views(T)
        k = self.k
        single = min(self.E, T * k) <= self.cache.S
        tb = 0
        while tb < T:
            L.moe_slot_ensure(self.cache, layer_id, ids, slots, 0, k, L.MOE_FETCH_MARK_REST, tb,
                              v["keys4"], v["slots4"], v["count4"], v["done"], stream)
            overlap = self.overlap is True or (self.overlap == "auto" and T * k >= self.OVERLAP_MIN_PAIRS)
            if overlap:
                # copies on the side stream, in parts, launched first: they are
                # the step's critical path
                self.ready.record(stream)
                self.copy_stream.wait_event(self.ready)
                if self.copy_parts == 1:
                    # every miss's gate/up matrices first, then their down
                    # matrices in parts of the miss list
                    gu = 2 * self.gu_half
                    L.moe_copy_missing_device_range(self.cache, v["keys4"], v["slots4"], v["count4"], 0, gu,
                                                    self.copy_stream, self.copy_ctas)
                    self.gu_done.record(self.copy_stream)
                    nd = len(self.down_done)
                    for q, ev in enumerate(self.down_done):
                        L.moe_copy_missing_device_slice(self.cache, v["keys4"], v["slots4"], v["count4"], q, nd,
                                                        gu, self.cache.B, self.copy_stream, self.copy_ctas)
                        ev.record(self.copy_stream)
                else:
                    for q, ev in enumerate(self.part_done):
                        L.moe_copy_missing_device_part(self.cache, v["keys4"], v["slots4"], v["count4"], q,
                                                       self.copy_parts, self.copy_stream, self.copy_ctas)
                        ev.record(self.copy_stream)
            with torch.cuda.stream(stream):
                self.status_h.copy_(self.info[0:4], non_blocking=True)
            if not self._capturing:      # a replayed graph records it after the replay
                self.status_ev.record(stream)
            self.stats["chunks"] += 1
            if overlap:
                # resident experts' pairs compute meanwhile, then each part's
                # pairs once it has landed
                if prefetch is not None:   # after this chunk's own copies on the side stream
                    self.prefetch(*prefetch, stream=stream)
                    prefetch = None
                if self.copy_parts == 1:
                    L.moe_expert_forward_overlap_staged(self.views, x[tb:T], slots[tb:T], w[tb:T], v["slots4"],
                                                        v["count4"], self.m4, self.gu_done, self.down_done,
                                                        y[tb:T], self.ws_ov, self.err, stream)
                else:
                    L.moe_expert_forward_overlap_parts(self.views, x[tb:T], slots[tb:T], w[tb:T], v["slots4"],
                                                       v["count4"], self.m4, self.part_done, y[tb:T], self.ws_ov,
                                                       self.err, stream)
            else:
                self._wait_prefetch(stream)
                L.moe_copy_missing_device(self.cache, v["keys4"], v["slots4"], v["count4"], stream)
                if prefetch is not None:
                    self.prefetch(*prefetch, stream=stream)
                    prefetch = None
                L.moe_expert_forward(self.views, x[tb:T], slots[tb:T], None, w[tb:T], y[tb:T], self.ws,
                                     self.err, stream)
            if single:
                self.pending = (layer_id, T)
                return y
            self.status_ev.synchronize()
            n4, done = int(self.status_h[0]), int(self.status_h[1])
            self._forward_status(int(self.status_h[3]))
            if n4 < 0:
                raise L.MoeError(-n4, f"slot ensure failed on the device (token_begin={tb})")
            self.stats["misses"] += n4
            self.stats["bytes_copied"] += n4 * self.cache.B
            tb = done
        return y

    def _ladder_single_chunk(self, T):
        a, b = self.ladder
        return (min(self.E, T * a) <= self.cache.S and min(self.E, T * (b - a)) <= self.c2.S)

    def _run_device_ladder(self, layer_id, T, ids, w, slots, x, y, stream):
        """Ladder chunk that fits both pools by construction: classify, both
        pools' misses copied by kernels, forward; no host wait."""
        v = self._views(T)
        a, b = self.ladder
        tags, wuse = self.tags[:T], self.w2[:T]
        L.moe_ladder_classify(self.cache, self.c2, layer_id, ids, w, a, b, 0, slots, tags, wuse, v["keys4"],
                              v["slots4"], v["count4"], v["keys2"], v["slots2"], v["count2"], v["done"], stream)
        with torch.cuda.stream(stream):
            self.status_h.copy_(self.info[0:4], non_blocking=True)
        self.status_ev.record(stream)
        self._wait_prefetch(stream)
        L.moe_copy_missing_device(self.cache, v["keys4"], v["slots4"], v["count4"], stream)
        L.moe_copy_missing_device(self.c2, v["keys2"], v["slots2"], v["count2"], stream)
        self.stats["chunks"] += 1
        L.moe_expert_forward(self.views, x, slots, tags, wuse, y, self.ws, self.err, stream)
        self.pending = (layer_id, T)
        return y

    def _graph_ok(self, T, prefetch):
        return (self.graph and self.copy == "device" and self.ladder is None and not self.assume_resident
                and prefetch is None and min(self.E, T * self.k) <= self.cache.S and not L.moe_profile_active())

    def _replay(self, layer_id, logits, x, y, stream):
        """Whole layer step as one CUDA graph: router, ensure, status read-back,
        device copies and the forward, replayed on static input and output buffers."""
        T = logits.shape[0]
        key = (layer_id, T)
        if key not in self.graphs:
            return False
        g, lg, xb, yb = self.graphs[key]
        with torch.cuda.stream(stream):
            lg.copy_(logits, non_blocking=True)
            xb.copy_(x, non_blocking=True)
            g.replay()
            y.copy_(yb, non_blocking=True)
        self.status_ev.record(stream)
        self.pending = (layer_id, T)
        self.stats["calls"] += 1
        self.stats["chunks"] += 1
        return True

    def _capture(self, layer_id, T):
        g = torch.cuda.CUDAGraph()
        H = self.views.H
        lg = torch.empty((T, self.E), dtype=torch.float32, device=self.dev)
        xb = torch.empty((T, H), dtype=torch.int16, device=self.dev)
        yb = torch.empty((T, H), dtype=torch.int16, device=self.dev)
        calls, chunks = self.stats["calls"], self.stats["chunks"]
        self._capturing = True
        try:
            with torch.cuda.graph(g):
                s = torch.cuda.current_stream(self.dev)
                ids, w, slots = self.ids[:T], self.w[:T], self.slots[:T]
                L.moe_router_topk(lg, self.k, True, ids, w, s)
                self._run_device(layer_id, T, ids, w, slots, xb, yb, s)
        finally:
            self._capturing = False
            self.pending = None
            self.stats["calls"], self.stats["chunks"] = calls, chunks
        self.graphs[(layer_id, T)] = (g, lg, xb, yb)

    def synchronize(self, stream=None):
        """Waits for the work enqueued on `stream` and raises what the device
        reported: a deferred ensure status or an expert forward's error word
        (`run` reads each of those one call late, without waiting)."""
        stream = stream or torch.cuda.current_stream(self.dev)
        stream.synchronize()
        self.check()
        with torch.cuda.stream(stream):
            e = int(self.err.item())
        self._forward_status(e)

    def run(self, layer_id: int, logits, x, y, stream=None, prefetch=None):
        """y[T, H] (bf16 bits) = the MoE layer applied to x[T, H] with router logits [T, E].

        prefetch=(layer, d_experts): predicted experts to stage once this layer's
        own miss copies are queued (device-copy mode; the cache needs a ring)."""
        T = logits.shape[0]
        assert T <= self.T_max
        stream = stream or torch.cuda.current_stream(self.dev)
        k = self.k
        self.check()
        if self._graph_ok(T, prefetch):
            if self._replay(layer_id, logits, x, y, stream):
                return y
            # first call of this (layer, T): run it eagerly below, then capture the
            # step for the next calls (capturing executes nothing)
            capture_after = True
        else:
            capture_after = False
        ids, w, slots = self.ids[:T], self.w[:T], self.slots[:T]
        L.moe_router_topk(logits, k, True, ids, w, stream)
        if self.copy == "device" and not self.assume_resident:
            if self.ladder is None:
                self.stats["calls"] += 1
                out = self._run_device(layer_id, T, ids, w, slots, x, y, stream, prefetch)
                if capture_after:
                    torch.cuda.synchronize(self.dev)
                    pending = self.pending
                    self._capture(layer_id, T)
                    self.pending = pending
                return out
            if self._ladder_single_chunk(T):
                self.stats["calls"] += 1
                return self._run_device_ladder(layer_id, T, ids, w, slots, x, y, stream)
        if prefetch is not None:
            raise ValueError("prefetch needs copy='device' (the copy engine copies from the bank)")
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
                with torch.cuda.stream(stream):   # ordered after this call's ensure
                    self.info_h.copy_(self.info, non_blocking=True)
                stream.synchronize()
                h = self.info_h
                n4, done = int(h[0]), int(h[1])
                n2 = int(h[2]) if self.ladder is not None else 0
                self._forward_status(int(h[3]))
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


class PrefillStreamer:
    """Whole-layer streaming prefill with two layer buffers.

    Past the crossover T * top_k >= E a prefill chunk touches most of a layer's
    experts, so the layer is streamed whole ("Running DeepSeek-V4-Flash across
    four free GPUs", section "What the expert cache actually does") into one of
    two device buffers of E experts each (section "Step 7": with overlap, two
    full expert-layer buffers): while layer l computes from one buffer, layer
    l + 1 streams into the other on the copy engine.  Each layer: router top-k
    (the expert id is the buffer slot), wait for the layer's copy, grouped-GEMM
    prefill; the buffer is then refilled with layer l + 2.
    """

    def __init__(self, h_bank, num_layers: int, E: int, H: int, I: int, k: int, T_max: int, device=None):
        self.bank, self.L, self.E, self.H, self.I, self.k = h_bank, num_layers, E, H, I, k
        self.dev = torch.device(device or "cuda")
        self.B = L.moe_fp4_expert_bytes(H, I)
        self.bufs = [torch.empty(E * self.B, dtype=torch.uint8, device=self.dev) for _ in range(2)]
        self.views = [L.make_views(H, I, b, E) for b in self.bufs]
        self.ids = torch.empty((T_max, k), dtype=torch.int32, device=self.dev)
        self.w = torch.empty((T_max, k), dtype=torch.float32, device=self.dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.ws = torch.empty(L.moe_expert_prefill_workspace(self.views[0], T_max, k), dtype=torch.uint8,
                              device=self.dev)
        self.copy_stream = torch.cuda.Stream(device=self.dev)
        self.loaded = [torch.cuda.Event(), torch.cuda.Event()]
        self.freed = [torch.cuda.Event(), torch.cuda.Event()]
        self.layer_in = [-1, -1]

    def _load(self, layer: int, stream):
        b = layer % 2
        self.freed[b].record(stream)               # the last compute reading this buffer is enqueued
        self.copy_stream.wait_event(self.freed[b])
        L.moe_copy_layer(self.bank, layer, self.E, self.B, self.bufs[b], self.copy_stream)
        self.loaded[b].record(self.copy_stream)
        self.layer_in[b] = layer

    def begin(self, first_layer: int = 0, stream=None):
        """Starts streaming the first two layers."""
        stream = stream or torch.cuda.current_stream(self.dev)
        for layer in range(first_layer, min(first_layer + 2, self.L)):
            self._load(layer, stream)

    def synchronize(self, stream=None):
        """Waits for the work enqueued on `stream` and raises the error word of
        the last layer's grouped GEMM (each call clears it first)."""
        stream = stream or torch.cuda.current_stream(self.dev)
        stream.synchronize()
        with torch.cuda.stream(stream):
            e = int(self.err.item())
        if e != L.MOE_OK:
            raise L.MoeError(e, "the streamed prefill's grouped GEMM reported a failure on the device")

    def run_layer(self, layer: int, logits, x, y, stream=None):
        """y[T, H] = the MoE layer `layer` on x[T, H] with router logits [T, E]."""
        stream = stream or torch.cuda.current_stream(self.dev)
        b = layer % 2
        if self.layer_in[b] != layer:
            self._load(layer, stream)
        T = logits.shape[0]
        ids, w = self.ids[:T], self.w[:T]
        L.moe_router_topk(logits, self.k, True, ids, w, stream)
        stream.wait_event(self.loaded[b])
        L.moe_expert_prefill(self.views[b], x, ids, w, y, self.ws, self.err, stream)
        if layer + 2 < self.L:
            self._load(layer + 2, stream)
        return y
