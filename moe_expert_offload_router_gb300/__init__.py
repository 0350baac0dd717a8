"""Routed MoE layer over a GPU expert-slot cache, for one GB300 (sm_103a).

The compute path is the C-ABI library ``libmoe_gb300.so`` (see
``include/moe_gb300.h``); this package is its ctypes binding plus a host-side
layer runner.  The binding loads on first use of any of its names and raises
if the library has not been built (``moe_expert_offload_router_gb300.build``):
there is no fallback path.
"""
import importlib

_SUBMODULES = ("build", "layer", "_lib")


def __getattr__(name):
    if name in _SUBMODULES or name.startswith("__"):
        raise AttributeError(name)   # the import system then loads the submodule
    if name in ("DecodeLayerRunner", "PrefillStreamer"):
        return getattr(importlib.import_module(__name__ + ".layer"), name)
    lib = importlib.import_module(__name__ + "._lib")
    try:
        return getattr(lib, name)
    except AttributeError:
        raise AttributeError(f"module {__name__!r} has no attribute {name!r}") from None
