"""Argument checks of the C ABI that return before any device work (CPU only):
each bad call returns MOE_ERR_INVALID and leaves a message in moe_last_error."""
import ctypes as C

import pytest

MOE_ERR_INVALID = 1


@pytest.fixture(scope="module")
def lib():
    from moe_expert_offload_router_gb300 import build
    L = C.CDLL(build.build())
    L.moe_last_error.restype = C.c_char_p
    return L


def _invalid(L, rc):
    assert rc == MOE_ERR_INVALID
    assert L.moe_last_error()


def test_mx_quantize_needs_k_multiple_of_32(lib):
    _invalid(lib, lib.moe_mx_quantize(None, 2, 48, None, None, None))
    _invalid(lib, lib.moe_mx_quantize(None, -1, 32, None, None, None))
    assert lib.moe_mx_quantize(None, 0, 64, None, None, None) == 0     # nothing to do


def test_copy_entry_points_need_a_cache(lib):
    _invalid(lib, lib.moe_copy_missing_device(None, None, None, None, 0, None, None))
    _invalid(lib, lib.moe_copy_missing_device_part(None, None, None, None, 0, 2, 0, None, None))
    _invalid(lib, lib.moe_copy_missing_device_range(None, None, None, None, C.c_size_t(0), C.c_size_t(16), 0,
                                                    None, None))
    _invalid(lib, lib.moe_copy_missing_device_slice(None, None, None, None, 0, 1, C.c_size_t(0), C.c_size_t(16),
                                                    0, None, None))
    _invalid(lib, lib.moe_cache_prime_bank(None, None))


def test_overlap_entry_points_check_their_part_counts(lib):
    ev = (C.c_void_p * 1)()
    for n in (0, 5):
        _invalid(lib, lib.moe_expert_forward_overlap_parts(None, None, 1, 1, None, None, None, None, 1, n, ev,
                                                           None, None, C.c_size_t(0), None, None))
        _invalid(lib, lib.moe_expert_forward_overlap_staged(None, None, 1, 1, None, None, None, None, 1, None, n,
                                                            ev, None, None, C.c_size_t(0), None, None))


def test_prefill_prec_checks(lib):
    _invalid(lib, lib.moe_expert_prefill_prec(None, None, 1, 1, None, None, 0, None, None, C.c_size_t(0), None,
                                              None))

    class Views(C.Structure):
        _fields_ = [("H", C.c_int), ("I", C.c_int), ("fp4_slots", C.c_void_p), ("fp4_num_slots", C.c_int),
                    ("int2_slots", C.c_void_p), ("int2_num_slots", C.c_int), ("shared", C.c_void_p)]
    v = Views(512, 512, None, 1, None, 0, None)
    _invalid(lib, lib.moe_expert_prefill_prec(C.byref(v), None, 1, 1, None, None, 7, None, None, C.c_size_t(0),
                                              None, None))


def test_profile_timeline_host_side(lib):
    n = C.c_int(-1)
    _invalid(lib, lib.moe_profile_timeline(-1, None, None, None, C.byref(n)))
    assert lib.moe_profile_enable(0) == 0
    k, a, b = (C.c_int32 * 1)(), (C.c_double * 1)(), (C.c_double * 1)()
    assert lib.moe_profile_timeline(1, k, a, b, C.byref(n)) == 0 and n.value == 0


def test_binding_refuses_strided_views():
    # the binding hands raw pointers to a library that reads dense rows: a
    # transposed or sliced-along-columns view is refused before any call
    import numpy as np
    import torch
    from moe_expert_offload_router_gb300 import _lib as B
    with pytest.raises(ValueError, match="not contiguous"):
        B.moe_router_topk(torch.zeros((8, 4)).t(), 2)
    with pytest.raises(ValueError, match="not contiguous"):
        B.moe_rms_carry(torch.zeros((4, 64), dtype=torch.int16)[:, ::2], 1e-6,
                        torch.zeros((4, 32), dtype=torch.int16))
    keys = np.zeros((4, 2), dtype=np.int32)[:, 0]
    no_cache = B.moe_cache.__new__(B.moe_cache)
    no_cache.handle = None
    with pytest.raises(ValueError, match="contiguous"):
        B.moe_copy_missing(no_cache, keys, keys, 1)
