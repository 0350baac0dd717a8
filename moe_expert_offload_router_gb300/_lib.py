"""ctypes binding of libmoe_gb300.so: one Python function per C entry point,
same names, argument marshalling only (torch tensors -> raw pointers, torch
streams/events -> handles).  Every computation runs in the library's kernels;
if the library is not built this module raises on import."""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK, MOE_ERR_INVALID, MOE_ERR_CAPACITY, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_NOMEM = range(6)
MOE_FETCH, MOE_LOOKUP, MOE_FETCH_MARK_REST = 0, 1, 2
MOE_EVICT_LRU, MOE_EVICT_LFU = 0, 1
MOE_TAG_FP4, MOE_TAG_INT2, MOE_TAG_DROP = 0, 1, 2
MOE_POOL_FP4, MOE_POOL_INT2, MOE_POOL_SHARED = 0, 1, 2
MOE_W1, MOE_W3, MOE_W2 = 0, 1, 2
(MOE_K_ROUTER, MOE_K_ENSURE, MOE_K_LADDER, MOE_K_GROUP, MOE_K_PLAN, MOE_K_GATEUP, MOE_K_DOWN,
 MOE_K_COMBINE, MOE_K_CARRY, MOE_K_GEMM_GATEUP, MOE_K_GEMM_DOWN, MOE_K_COPY, MOE_K_COUNT) = range(13)
KERNEL_NAMES = ["router", "ensure", "ladder", "group_pairs", "plan", "gateup", "down", "combine",
                "rms_carry", "gemm_gateup", "gemm_down", "copy_device"]
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_CAPACITY", 3: "MOE_ERR_CUDA",
                4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_NOMEM"}


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run moe_expert_offload_router_gb300.build.build()")
_lib = C.CDLL(LIB_PATH)

vp, i32, sz, f32, u64 = C.c_void_p, C.c_int, C.c_size_t, C.c_float, C.c_uint64
P_i32, P_u64 = C.POINTER(C.c_int32), C.POINTER(C.c_uint64)


class moe_expert_views(C.Structure):
    _fields_ = [("H", i32), ("I", i32), ("fp4_slots", vp), ("fp4_num_slots", i32),
                ("int2_slots", vp), ("int2_num_slots", i32), ("shared", vp)]


_SIGS = {
    "moe_last_error": (C.c_char_p, []),
    "moe_version": (i32, []),
    "moe_fp4_expert_bytes": (sz, [i32, i32]),
    "moe_int2_expert_bytes": (sz, [i32, i32]),
    "moe_fp8_expert_bytes": (sz, [i32, i32]),
    "moe_router_topk": (i32, [vp, i32, i32, i32, i32, vp, vp, vp]),
    "moe_cache_create": (i32, [i32, i32, i32, sz, vp, vp, C.POINTER(vp)]),
    "moe_cache_destroy": (i32, [vp]),
    "moe_cache_reset": (i32, [vp, vp]),
    "moe_cache_state": (i32, [vp, C.POINTER(vp), C.POINTER(vp), C.POINTER(vp), C.POINTER(vp)]),
    "moe_cache_export": (i32, [vp, vp, vp, vp]),
    "moe_cache_import": (i32, [vp, vp, vp, u64]),
    "moe_slot_ensure": (i32, [vp, i32, vp, vp, i32, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp]),
    "moe_copy_missing": (i32, [vp, vp, vp, i32, vp, vp, vp]),
    "moe_debug_fail_copy": (i32, [vp, i32]),
    "moe_copy_layer": (i32, [vp, i32, i32, sz, vp, vp]),
    "moe_copy_missing_device": (i32, [vp, vp, vp, vp, i32, vp, vp]),
    "moe_copy_missing_device_part": (i32, [vp, vp, vp, vp, i32, i32, i32, vp, vp]),
    "moe_cache_prime_bank": (i32, [vp, vp]),
    "moe_copy_missing_device_range": (i32, [vp, vp, vp, vp, sz, sz, i32, vp, vp]),
    "moe_copy_missing_device_slice": (i32, [vp, vp, vp, vp, i32, i32, sz, sz, i32, vp, vp]),
    "moe_cache_set_policy": (i32, [vp, i32, i32]),
    "moe_cache_seed_frequency": (i32, [vp, vp]),
    "moe_cache_export_frequency": (i32, [vp, vp, vp, vp]),
    "moe_cache_set_staging": (i32, [vp, i32]),
    "moe_prefetch": (i32, [vp, i32, vp, i32, vp, vp, vp, vp]),
    "moe_cache_export_staging": (i32, [vp, vp, vp]),
    "moe_ladder_classify": (i32, [vp, vp, i32, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp,
                                  vp, vp, vp, vp, vp, vp, vp, vp]),
    "moe_group_pairs": (i32, [vp, i32, i32, i32, vp, vp, vp, vp]),
    "moe_expert_forward_workspace": (sz, [C.POINTER(moe_expert_views), i32, i32]),
    "moe_expert_forward": (i32, [C.POINTER(moe_expert_views), vp, i32, i32, vp, vp, vp, vp, vp,
                                 sz, vp, vp]),
    "moe_dequant_debug": (i32, [C.POINTER(moe_expert_views), i32, i32, i32, vp, vp]),
    "moe_set_option": (i32, [i32, i32, vp]),
    "moe_fp4_mma_peak": (i32, [i32, vp, vp]),
    "moe_expert_forward_overlap_workspace": (sz, [C.POINTER(moe_expert_views), i32, i32]),
    "moe_expert_forward_overlap": (i32, [C.POINTER(moe_expert_views), vp, i32, i32, vp, vp, vp, vp, i32, vp,
                                         vp, vp, sz, vp, vp]),
    "moe_expert_forward_overlap_staged": (i32, [C.POINTER(moe_expert_views), vp, i32, i32, vp, vp, vp, vp, i32,
                                                vp, i32, vp, vp, vp, sz, vp, vp]),
    "moe_expert_forward_overlap_parts": (i32, [C.POINTER(moe_expert_views), vp, i32, i32, vp, vp, vp, vp, i32,
                                               i32, vp, vp, vp, sz, vp, vp]),
    "moe_expert_forward_noalloc": (i32, [C.POINTER(moe_expert_views), vp, i32, i32, vp, vp, vp, vp, vp, vp]),
    "moe_expert_prefill_workspace": (sz, [C.POINTER(moe_expert_views), i32, i32]),
    "moe_expert_prefill": (i32, [C.POINTER(moe_expert_views), vp, i32, i32, vp, vp, vp, vp, sz, vp, vp]),
    "moe_expert_prefill_prec": (i32, [C.POINTER(moe_expert_views), vp, i32, i32, vp, vp, i32, vp, vp, sz, vp,
                                      vp]),
    "moe_mx_quantize": (i32, [vp, i32, i32, vp, vp, vp]),
    "moe_rms_carry": (i32, [vp, i32, i32, f32, vp, vp]),
    "moe_selftest": (i32, []),
    "moe_debug_timeout_probe": (i32, [C.c_int64, vp, vp]),
    "moe_profile_enable": (i32, [i32]),
    "moe_profile_query": (i32, [i32, C.POINTER(C.c_double), C.POINTER(C.c_int)]),
    "moe_profile_timeline": (i32, [i32, C.c_void_p, C.c_void_p, C.c_void_p, C.POINTER(C.c_int)]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args


def raw():
    """The ctypes library handle."""
    return _lib


def _check(status: int):
    if status != MOE_OK:
        raise MoeError(status, _lib.moe_last_error().decode(errors="replace"))


def _p(t):
    """Raw data pointer of a tensor (or None).  The library reads every array
    as dense row-major memory, so a strided view is refused here rather than
    read as if it were dense."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(t.shape)} and strides {t.stride()} is not contiguous")
    return t.data_ptr()


def _s(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _e(event):
    if event is None:
        return None
    return event.cuda_event


def moe_version() -> int:
    return _lib.moe_version()


def moe_fp4_expert_bytes(H: int, I: int) -> int:
    return _lib.moe_fp4_expert_bytes(H, I)


def moe_int2_expert_bytes(H: int, I: int) -> int:
    return _lib.moe_int2_expert_bytes(H, I)


def moe_fp8_expert_bytes(H: int, I: int) -> int:
    return _lib.moe_fp8_expert_bytes(H, I)


def moe_router_topk(logits, k: int, renorm: bool = True, topk_ids=None, topk_w=None, stream=None):
    T, E = logits.shape
    dev = logits.device
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    _check(_lib.moe_router_topk(_p(logits), T, E, k, int(bool(renorm)), _p(topk_ids), _p(topk_w),
                                _s(stream)))
    return topk_ids, topk_w


class moe_cache:
    """Owner of one library slot cache (moe_cache_create / moe_cache_destroy)."""

    def __init__(self, num_slots: int, num_layers: int, num_experts: int, expert_bytes: int,
                 d_slots, h_bank=None):
        h = vp()
        _check(_lib.moe_cache_create(num_slots, num_layers, num_experts, expert_bytes, _p(d_slots),
                                     _p(h_bank), C.byref(h)))
        self.handle = h
        self.S, self.L, self.E, self.B = num_slots, num_layers, num_experts, expert_bytes
        self.R = 0
        self._keep = (d_slots, h_bank)
        self.has_bank = h_bank is not None
        self.primed = False

    def prime_bank(self, stream=None):
        """moe_cache_prime_bank once per cache (later calls do nothing)."""
        if self.has_bank and not self.primed:
            moe_cache_prime_bank(self, stream)
            self.primed = True

    def close(self):
        if self.handle:
            _check(_lib.moe_cache_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def reset(self, stream=None):
        _check(_lib.moe_cache_reset(self.handle, _s(stream)))

    def export(self):
        import numpy as np
        key = np.empty(self.S, dtype=np.int32)
        stamp = np.empty(self.S, dtype=np.uint64)
        clock = np.empty(1, dtype=np.uint64)
        _check(_lib.moe_cache_export(self.handle, key.ctypes.data, stamp.ctypes.data, clock.ctypes.data))
        return key, stamp, int(clock[0])

    def import_(self, key, stamp, clock: int):
        import numpy as np
        key = np.ascontiguousarray(key, dtype=np.int32)
        stamp = np.ascontiguousarray(stamp, dtype=np.uint64)
        _check(_lib.moe_cache_import(self.handle, key.ctypes.data, stamp.ctypes.data, clock))

    def state_pointers(self):
        a, b, c, d = vp(), vp(), vp(), vp()
        _check(_lib.moe_cache_state(self.handle, C.byref(a), C.byref(b), C.byref(c), C.byref(d)))
        return a.value, b.value, c.value, d.value


def moe_cache_set_policy(cache: moe_cache, policy: int, decay_calls: int = 1):
    _check(_lib.moe_cache_set_policy(cache.handle, policy, decay_calls))


def moe_cache_seed_frequency(cache: moe_cache, counts):
    """counts: host array of L*E non-negative integers (key = layer * E + expert)."""
    import numpy as np
    c = np.ascontiguousarray(np.minimum(np.asarray(counts, dtype=np.int64), 2 ** 32 - 1), dtype=np.uint32)
    if c.shape != (cache.L * cache.E,):
        raise ValueError("counts must have L*E entries")
    _check(_lib.moe_cache_seed_frequency(cache.handle, c.ctypes.data))


def moe_cache_export_frequency(cache: moe_cache):
    """(counts [L*E] uint32, epochs [L*E] uint32, calls) of the LFU state."""
    import numpy as np
    n = cache.L * cache.E
    cnt = np.empty(n, dtype=np.uint32)
    ep = np.empty(n, dtype=np.uint32)
    calls = np.empty(1, dtype=np.uint64)
    _check(_lib.moe_cache_export_frequency(cache.handle, cnt.ctypes.data, ep.ctypes.data, calls.ctypes.data))
    return cnt, ep, int(calls[0])


def moe_cache_set_staging(cache: moe_cache, num_stage: int):
    _check(_lib.moe_cache_set_staging(cache.handle, num_stage))
    cache.R = num_stage


def moe_prefetch(cache: moe_cache, layer_id: int, d_experts, d_list_key, d_list_slot, d_list_count, stream=None):
    n = d_experts.numel()
    _check(_lib.moe_prefetch(cache.handle, layer_id, _p(d_experts), n, _p(d_list_key), _p(d_list_slot),
                             _p(d_list_count), _s(stream)))


def moe_cache_export_staging(cache: moe_cache):
    """(stage_key [R] int32, next ring position)."""
    import numpy as np
    key = np.empty(cache.R, dtype=np.int32)
    pos = np.empty(1, dtype=np.uint32)
    _check(_lib.moe_cache_export_staging(cache.handle, key.ctypes.data, pos.ctypes.data))
    return key, int(pos[0])


def moe_slot_ensure(cache: moe_cache, layer_id: int, ids, slots_out, rank_lo: int, rank_hi: int,
                    mode: int, token_begin: int, d_miss_key, d_miss_slot, d_miss_count,
                    d_tokens_done, stream=None):
    T, k = ids.shape
    _check(_lib.moe_slot_ensure(cache.handle, layer_id, _p(ids), _p(slots_out), T, k, rank_lo, rank_hi,
                                mode, token_begin, _p(d_miss_key), _p(d_miss_slot), _p(d_miss_count),
                                _p(d_tokens_done), _s(stream)))


def moe_copy_missing(cache: moe_cache, h_miss_key, h_miss_slot, n_miss: int, copy_stream=None,
                     ready=None, done=None):
    """h_miss_key / h_miss_slot: host int32 arrays (numpy or CPU tensors)."""
    def hp(a):
        if a is None:
            return None
        if hasattr(a, "data_ptr"):
            return _p(a)
        if not a.flags["C_CONTIGUOUS"]:
            raise ValueError("host miss arrays must be contiguous")
        return a.ctypes.data
    _check(_lib.moe_copy_missing(cache.handle, hp(h_miss_key), hp(h_miss_slot), n_miss,
                                 _s(copy_stream), _e(ready), _e(done)))


def moe_copy_missing_device(cache: moe_cache, d_miss_key, d_miss_slot, d_miss_count, stream=None,
                            max_ctas: int = 0, d_error=None):
    _check(_lib.moe_copy_missing_device(cache.handle, _p(d_miss_key), _p(d_miss_slot), _p(d_miss_count),
                                        max_ctas, _p(d_error), _s(stream)))


MOE_MAX_COPY_PARTS = 4


def moe_copy_missing_device_range(cache: moe_cache, d_miss_key, d_miss_slot, d_miss_count, byte_begin: int,
                                  byte_end: int, stream=None, max_ctas: int = 0, d_error=None):
    _check(_lib.moe_copy_missing_device_range(cache.handle, _p(d_miss_key), _p(d_miss_slot), _p(d_miss_count),
                                              byte_begin, byte_end, max_ctas, _p(d_error), _s(stream)))


def moe_copy_missing_device_slice(cache: moe_cache, d_miss_key, d_miss_slot, d_miss_count, part: int, n_parts: int,
                                  byte_begin: int, byte_end: int, stream=None, max_ctas: int = 0,
                                  d_error=None):
    _check(_lib.moe_copy_missing_device_slice(cache.handle, _p(d_miss_key), _p(d_miss_slot), _p(d_miss_count),
                                              part, n_parts, byte_begin, byte_end, max_ctas, _p(d_error),
                                              _s(stream)))


def moe_cache_prime_bank(cache: moe_cache, stream=None):
    """Reads one word of every 4 KB page of the cache's pinned bank from the GPU
    (address translations warmed before the first miss copy)."""
    _check(_lib.moe_cache_prime_bank(cache.handle, _s(stream)))


def moe_copy_missing_device_part(cache: moe_cache, d_miss_key, d_miss_slot, d_miss_count, part: int,
                                 n_parts: int, stream=None, max_ctas: int = 0, d_error=None):
    _check(_lib.moe_copy_missing_device_part(cache.handle, _p(d_miss_key), _p(d_miss_slot), _p(d_miss_count),
                                             part, n_parts, max_ctas, _p(d_error), _s(stream)))


def moe_copy_layer(h_bank, layer_id: int, num_experts: int, expert_bytes: int, d_buf, stream=None):
    _check(_lib.moe_copy_layer(_p(h_bank), layer_id, num_experts, expert_bytes, _p(d_buf), _s(stream)))


def moe_debug_fail_copy(cache: moe_cache, index: int):
    _check(_lib.moe_debug_fail_copy(cache.handle, index))


def moe_ladder_classify(c4: moe_cache, c2: moe_cache, layer_id: int, ids, w, a: int, b: int,
                        token_begin: int, slots_out, tags_out, w_out, miss4_key, miss4_slot,
                        miss4_count, miss2_key, miss2_slot, miss2_count, tokens_done, stream=None):
    T, k = ids.shape
    _check(_lib.moe_ladder_classify(c4.handle, c2.handle, layer_id, _p(ids), _p(w), T, k, a, b,
                                    token_begin, _p(slots_out), _p(tags_out), _p(w_out),
                                    _p(miss4_key), _p(miss4_slot), _p(miss4_count), _p(miss2_key),
                                    _p(miss2_slot), _p(miss2_count), _p(tokens_done), _s(stream)))


def moe_group_pairs(ids, E: int, offsets=None, perm=None, d_error=None, stream=None):
    T, k = ids.shape
    dev = ids.device
    if offsets is None:
        offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    if perm is None:
        perm = torch.empty(T * k, dtype=torch.int32, device=dev)
    if d_error is None:
        d_error = torch.empty(1, dtype=torch.int32, device=dev)
    _check(_lib.moe_group_pairs(_p(ids), T, k, E, _p(offsets), _p(perm), _p(d_error), _s(stream)))
    return offsets, perm, d_error


def make_views(H: int, I: int, fp4_slots=None, fp4_num_slots: int = 0, int2_slots=None,
               int2_num_slots: int = 0, shared=None) -> moe_expert_views:
    v = moe_expert_views(H, I, _p(fp4_slots), fp4_num_slots, _p(int2_slots), int2_num_slots, _p(shared))
    v._keep = (fp4_slots, int2_slots, shared)
    return v


def moe_expert_forward_workspace(views: moe_expert_views, T: int, k: int) -> int:
    return _lib.moe_expert_forward_workspace(C.byref(views), T, k)


def moe_expert_forward(views: moe_expert_views, x, slots, tags, w, y, workspace, d_error=None,
                       stream=None):
    T, k = slots.shape
    _check(_lib.moe_expert_forward(C.byref(views), _p(x), T, k, _p(slots), _p(tags), _p(w), _p(y),
                                   _p(workspace), workspace.numel() * workspace.element_size(),
                                   _p(d_error), _s(stream)))


def moe_expert_forward_overlap_workspace(views: moe_expert_views, T: int, k: int) -> int:
    return _lib.moe_expert_forward_overlap_workspace(C.byref(views), T, k)


def moe_expert_forward_overlap(views: moe_expert_views, x, slots, w, d_miss_slot, d_miss_count, max_miss: int,
                               copies_done, y, workspace, d_error=None, stream=None):
    T, k = slots.shape
    _check(_lib.moe_expert_forward_overlap(C.byref(views), _p(x), T, k, _p(slots), _p(w), _p(d_miss_slot),
                                           _p(d_miss_count), max_miss, _e(copies_done), _p(y), _p(workspace),
                                           workspace.numel() * workspace.element_size(), _p(d_error),
                                           _s(stream)))


def moe_expert_forward_overlap_staged(views: moe_expert_views, x, slots, w, d_miss_slot, d_miss_count,
                                      max_miss: int, gateup_ready, down_ready, y, workspace, d_error=None,
                                      stream=None):
    """down_ready: one event (or None) per part of the miss list's down matrices, in part order."""
    T, k = slots.shape
    n = len(down_ready)
    evs = (C.c_void_p * max(n, 1))(*[_e(e) for e in down_ready])
    _check(_lib.moe_expert_forward_overlap_staged(C.byref(views), _p(x), T, k, _p(slots), _p(w), _p(d_miss_slot),
                                                  _p(d_miss_count), max_miss, _e(gateup_ready), n,
                                                  C.addressof(evs), _p(y), _p(workspace),
                                                  workspace.numel() * workspace.element_size(), _p(d_error),
                                                  _s(stream)))


def moe_expert_forward_overlap_parts(views: moe_expert_views, x, slots, w, d_miss_slot, d_miss_count,
                                     max_miss: int, parts_done, y, workspace, d_error=None, stream=None):
    """parts_done: one event (or None) per part of the miss list, in part order."""
    T, k = slots.shape
    n = len(parts_done)
    evs = (C.c_void_p * max(n, 1))(*[_e(e) for e in parts_done])
    _check(_lib.moe_expert_forward_overlap_parts(C.byref(views), _p(x), T, k, _p(slots), _p(w), _p(d_miss_slot),
                                                 _p(d_miss_count), max_miss, n, C.addressof(evs), _p(y),
                                                 _p(workspace), workspace.numel() * workspace.element_size(),
                                                 _p(d_error), _s(stream)))


def moe_expert_forward_noalloc(views: moe_expert_views, x, slots, tags, w, y, d_error=None, stream=None):
    """moe_expert_forward with the library's fixed device scratch instead of a workspace."""
    T, k = slots.shape
    _check(_lib.moe_expert_forward_noalloc(C.byref(views), _p(x), T, k, _p(slots), _p(tags), _p(w), _p(y),
                                           _p(d_error), _s(stream)))


def moe_expert_prefill_workspace(views: moe_expert_views, T: int, k: int) -> int:
    return _lib.moe_expert_prefill_workspace(C.byref(views), T, k)


def moe_expert_prefill(views: moe_expert_views, x, slots, w, y, workspace, d_error, stream=None):
    T, k = slots.shape
    _check(_lib.moe_expert_prefill(C.byref(views), _p(x), T, k, _p(slots), _p(w), _p(y), _p(workspace),
                                   workspace.numel() * workspace.element_size(), _p(d_error), _s(stream)))


MOE_PREC_W4A16, MOE_PREC_A_MXFP4 = 0, 1


def moe_expert_prefill_prec(views: moe_expert_views, x, slots, w, prec_mode: int, y, workspace, d_error,
                            stream=None):
    T, k = slots.shape
    _check(_lib.moe_expert_prefill_prec(C.byref(views), _p(x), T, k, _p(slots), _p(w), prec_mode, _p(y),
                                        _p(workspace), workspace.numel() * workspace.element_size(), _p(d_error),
                                        _s(stream)))


def moe_mx_quantize(x, codes, scales, stream=None):
    """x device bf16 bits [rows, K] -> codes uint8 [rows, K/2], scales uint8 [rows, K/32]."""
    rows, K = x.shape
    _check(_lib.moe_mx_quantize(_p(x), rows, K, _p(codes), _p(scales), _s(stream)))


MOE_OPT_MMA_MAX_TOKENS = 0
MOE_OPT_MX8_MIN_TOKENS = 1


def moe_set_option(option: int, value: int) -> int:
    """Sets a process-wide tuning option; returns its previous value."""
    old = C.c_int(0)
    _check(_lib.moe_set_option(option, value, C.byref(old)))
    return old.value


def moe_fp4_mma_peak(iters: int = 4096, stream=None) -> float:
    """Dense block-scaled FP4 tensor rate of this GPU (TFLOP/s), measured."""
    v = C.c_double(0.0)
    _check(_lib.moe_fp4_mma_peak(iters, C.byref(v), _s(stream)))
    return v.value


def moe_dequant_debug(views: moe_expert_views, pool: int, slot: int, matrix: int, out, stream=None):
    _check(_lib.moe_dequant_debug(C.byref(views), pool, slot, matrix, _p(out), _s(stream)))


def moe_rms_carry(y, eps: float, x_next, stream=None):
    T, H = y.shape
    _check(_lib.moe_rms_carry(_p(y), T, H, eps, _p(x_next), _s(stream)))


def moe_debug_timeout_probe(limit_ns: int, d_status, stream=None):
    _check(_lib.moe_debug_timeout_probe(limit_ns, _p(d_status), _s(stream)))


def moe_selftest():
    _check(_lib.moe_selftest())


_PROFILING = [False]


def moe_profile_enable(enable: bool = True):
    _check(_lib.moe_profile_enable(int(bool(enable))))
    _PROFILING[0] = bool(enable)


def moe_profile_active() -> bool:
    """Whether moe_profile_enable(True) is in effect (kernel timing events are recorded)."""
    return _PROFILING[0]


def moe_profile_query(kernel: int):
    """(total milliseconds, launches) recorded for one kernel id since profiling was enabled."""
    ms, n = C.c_double(), C.c_int()
    _check(_lib.moe_profile_query(kernel, C.byref(ms), C.byref(n)))
    return ms.value, n.value


def moe_profile_timeline():
    """Every record since profiling was enabled, in recording order, as a list of
    (kernel id, start ms, stop ms) relative to the first record's start."""
    n = C.c_int()
    z = (C.c_int32 * 1)(), (C.c_double * 1)(), (C.c_double * 1)()
    _check(_lib.moe_profile_timeline(0, C.addressof(z[0]), C.addressof(z[1]), C.addressof(z[2]), C.byref(n)))
    m = max(n.value, 1)
    k, t0, t1 = (C.c_int32 * m)(), (C.c_double * m)(), (C.c_double * m)()
    _check(_lib.moe_profile_timeline(m, C.addressof(k), C.addressof(t0), C.addressof(t1), C.byref(n)))
    return [(int(k[i]), float(t0[i]), float(t1[i])) for i in range(min(m, n.value))]
