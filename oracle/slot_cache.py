"""The GPU expert-slot cache: ensure_experts remap with LRU eviction.

"Running DeepSeek-V4-Flash across four free GPUs", section "What the expert
cache actually does": a fixed number of expert slots live in VRAM; each step
the router's expert ids are remapped in place onto slots, only the misses are
copied from pinned host RAM, eviction is LRU, and the cache is global across
layers (keyed here by layer * E + expert).  Section "moe_cache_size=128 is
too small" (the engine refuses a cache smaller than one layer's experts).

Readings where the pages are silent:

* Within one call the distinct keys are taken in first-appearance order
  (token-major, then rank).  All hits are marked first, so a miss never
  evicts an expert the same call needs.  Each distinct key gets stamp
  clock + (its first-appearance index); the clock then advances by the
  number of distinct keys.  Misses, in first-appearance order, take empty
  slots by ascending index, then untouched slots by ascending stamp.
* LOOKUP mode never evicts: hits refresh their stamp, misses map to -1 and
  emit nothing.
* Capacity: FETCH handles the longest prefix of tokens (from token_begin)
  whose distinct keys fit in the S slots and reports where it stopped
  (tokens_done); a single token needing more than S slots is an error.
* Entries holding a negative id are skipped and left as they are.
"""
from __future__ import annotations

import numpy as np

FETCH = 0
LOOKUP = 1


class CapacityError(Exception):
    pass


class SlotCacheLRU:
    def __init__(self, num_slots: int, num_layers: int, num_experts: int):
        if num_slots < 1 or num_layers < 1 or num_experts < 1:
            raise ValueError("num_slots, num_layers, num_experts must be >= 1")
        self.S, self.L, self.E = num_slots, num_layers, num_experts
        self.slot_key = [-1] * num_slots
        self.slot_stamp = [0] * num_slots
        self.key_to_slot = [-1] * (num_layers * num_experts)
        self.clock = 0

    # -- state, for bit-exact comparison --------------------------------------------
    def state(self):
        return (np.array(self.slot_key, dtype=np.int64),
                np.array(self.slot_stamp, dtype=np.uint64),
                np.array(self.key_to_slot, dtype=np.int64),
                self.clock)

    def ensure(self, layer: int, ids, rank_lo: int, rank_hi: int, mode: int,
               token_begin: int = 0):
        """Returns (slots [T,k] int64, miss_keys, miss_slots, tokens_done)."""
        ids = np.asarray(ids)
        if ids.ndim != 2:
            raise ValueError("ids must be [T, k]")
        T, k = ids.shape
        if not (0 <= layer < self.L):
            raise ValueError("layer out of range")
        if not (0 <= rank_lo <= rank_hi <= k):
            raise ValueError("bad rank range")
        if mode not in (FETCH, LOOKUP):
            raise ValueError("bad mode")
        if token_begin < 0:
            raise ValueError("token_begin < 0")
        if np.any(ids >= self.E):
            raise ValueError("expert id >= E")
        out = ids.astype(np.int64).copy()
        base = layer * self.E

        first_tok = {}
        order = []
        for t in range(token_begin, T):
            for j in range(rank_lo, rank_hi):
                e = int(ids[t, j])
                if e < 0:
                    continue
                key = base + e
                if key not in first_tok:
                    first_tok[key] = t
                    order.append(key)

        if mode == FETCH:
            end = token_begin
            count = 0
            new_per_tok = {}
            for key in order:
                new_per_tok[first_tok[key]] = new_per_tok.get(first_tok[key], 0) + 1
            for t in range(token_begin, T):
                add = new_per_tok.get(t, 0)
                if count + add > self.S:
                    break
                count += add
                end = t + 1
            if end == token_begin and token_begin < T:
                raise CapacityError("one token needs more experts than there are slots")
        else:
            end = max(T, token_begin)
        chunk = [key for key in order if first_tok[key] < end]
        D = len(chunk)

        miss_keys, miss_slots = [], []
        if mode == FETCH:
            pinned = {self.key_to_slot[key] for key in chunk if self.key_to_slot[key] >= 0}
            misses = [key for key in chunk if self.key_to_slot[key] < 0]
            empties = [s for s in range(self.S) if self.slot_key[s] < 0]
            untouched = sorted((self._evict_order(s), s) for s in range(self.S)
                               if self.slot_key[s] >= 0 and s not in pinned)
            victims = empties[:len(misses)]
            victims += [s for _, s in untouched[:len(misses) - len(victims)]]
            assert len(victims) == len(misses)
            for key, v in zip(misses, victims):
                old = self.slot_key[v]
                if old >= 0:
                    self.key_to_slot[old] = -1
                self.slot_key[v] = key
                self.key_to_slot[key] = v
                miss_keys.append(key)
                miss_slots.append(v)
        for q, key in enumerate(chunk):
            s = self.key_to_slot[key]
            if s >= 0:
                self.slot_stamp[s] = self.clock + q
        self.clock += D
        self._after_call(chunk)

        for t in range(token_begin, end):
            for j in range(rank_lo, rank_hi):
                e = int(ids[t, j])
                if e < 0:
                    continue
                out[t, j] = self.key_to_slot[base + e]
        return out, miss_keys, miss_slots, end

    # -- eviction policy hooks ---------------------------------------------------
    def _evict_order(self, s):
        """Sort key of an occupied, unneeded slot among eviction candidates."""
        return self.slot_stamp[s]

    def _after_call(self, chunk):
        pass

    def mark_empty(self, slots):
        """Roll back: the given slots hold nothing (their copy did not land)."""
        for s in slots:
            key = self.slot_key[s]
            if key >= 0:
                self.key_to_slot[key] = -1
            self.slot_key[s] = -1


class SlotCacheLFU(SlotCacheLRU):
    """The same slot cache with LFU eviction and frequency decay.

    "An elephant through a straw", section "Rig, model & methodology": the
    best configuration evicts by LFU with frequency decay, seeded from a
    routing trace.  The pages give no more; the readings here are:

    * every key (layer * E + expert) has an integer count; each ensure call
      adds 1 to the count of every distinct key it handles (hits and misses,
      FETCH and LOOKUP), capped at CAP;
    * decay halves every count once per decay_calls ensure calls: the epoch of
      a call is calls // decay_calls (calls counts the ensure calls that
      returned), and a count last written in epoch e0 is worth
      count >> min(31, epoch - e0) in epoch `epoch`;
    * misses take empty slots by ascending index, then the untouched slots
      with the lowest worth, ties by the older stamp (stamps are unique), so
      with equal counts the order is exactly LRU's;
    * seed(counts) sets every key's count (capped) in the current epoch.
    """

    CAP = (1 << 20) - 1

    def __init__(self, num_slots: int, num_layers: int, num_experts: int, decay_calls: int):
        super().__init__(num_slots, num_layers, num_experts)
        if decay_calls < 1:
            raise ValueError("decay_calls must be >= 1")
        self.decay_calls = decay_calls
        self.count = [0] * (num_layers * num_experts)
        self.count_epoch = [0] * (num_layers * num_experts)
        self.calls = 0

    def epoch(self):
        return self.calls // self.decay_calls

    def worth(self, key):
        return self.count[key] >> min(31, self.epoch() - self.count_epoch[key])

    def seed(self, counts):
        counts = np.asarray(counts)
        if counts.shape != (self.L * self.E,) or np.any(counts < 0):
            raise ValueError("counts must be L*E non-negative integers")
        e = self.epoch()
        for key, c in enumerate(counts):
            self.count[key] = min(int(c), self.CAP)
            self.count_epoch[key] = e

    def frequency_state(self):
        return (np.array(self.count, dtype=np.int64), np.array(self.count_epoch, dtype=np.int64), self.calls)

    def _evict_order(self, s):
        return (self.worth(self.slot_key[s]), self.slot_stamp[s])

    def _after_call(self, chunk):
        e = self.epoch()
        for key in chunk:
            self.count[key] = min(self.worth(key) + 1, self.CAP)
            self.count_epoch[key] = e
        self.calls += 1


class StagingRing:
    """Staging ring for predicted experts, beside a slot cache.

    "An elephant through a straw", section "Guessing the router two layers
    ahead": predicted experts are copied into a small round-robin region
    appended to the same slot buffer, so a guess never evicts a resident
    expert; a wrong guess is overwritten by a later prediction, a right one is
    already in GPU memory when the router asks for it.  Readings:

    * the ring has R slots, numbered S .. S+R-1 in the slot buffer;
    * prefetch(layer, experts) takes the predicted experts in order, skips
      negative ids, ids already seen in this call, keys resident in the cache
      and keys already staged; each remaining key takes ring position
      pos % R (pos then advances), displacing the key staged there; the call
      returns the (key, slot) copy list, without the guesses that a later
      guess of the same call displaced (only the last R assignments);
    * the cache's own state is never changed by prefetching; when ensure
      later lists a staged key as a miss, the miss is filled from its staging
      slot instead of the host bank (same bytes), and the key stays staged.
    """

    def __init__(self, cache: SlotCacheLRU, num_stage: int):
        if num_stage < 1:
            raise ValueError("num_stage must be >= 1")
        self.c = cache
        self.R = num_stage
        self.stage_key = [-1] * num_stage
        self.pos = 0

    def staged_slot(self, key):
        for j, kk in enumerate(self.stage_key):
            if kk == key:
                return self.c.S + j
        return -1

    def prefetch(self, layer: int, experts):
        c = self.c
        if not (0 <= layer < c.L):
            raise ValueError("layer out of range")
        out, seen = [], set()
        for e in experts:
            e = int(e)
            if e < 0 or e in seen:
                continue
            if e >= c.E:
                raise ValueError("expert id >= E")
            seen.add(e)
            key = layer * c.E + e
            if c.key_to_slot[key] >= 0 or self.staged_slot(key) >= 0:
                continue
            j = self.pos % self.R
            self.pos += 1
            self.stage_key[j] = key
            out.append((key, c.S + j))
        return out[-self.R:]

    def miss_source(self, key):
        """Where a miss of `key` is copied from: ('stage', slot) or ('bank', key)."""
        s = self.staged_slot(key)
        return ("stage", s) if s >= 0 else ("bank", key)
