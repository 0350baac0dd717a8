"""Routed MoE layer over a GPU expert-slot cache, for one GB300 (sm_103a).

The compute path is the C-ABI library ``libmoe_gb300.so`` (see
``include/moe_gb300.h``); this package is its ctypes binding plus a host-side
layer runner.  Importing it fails if the library has not been built: there is
no fallback path.
"""
from ._lib import *  # noqa: F401,F403
from ._lib import MoeError, moe_cache, make_views, raw  # noqa: F401
from .layer import DecodeLayerRunner  # noqa: F401
