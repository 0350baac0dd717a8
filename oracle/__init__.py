"""CPU oracle for the routed MoE layer over a GPU expert-slot cache.

TEST INFRASTRUCTURE ONLY.  Plain, slow, fp64 (NumPy) statements of what the
path computes, written from the pages' description of the method.  Only the
test suite, the package's smoke check and the benchmark's CPU-baseline leg may
import it; the library and its Python binding never do, and share no code
with it.

Functions and what pins each one (see the ``-m "not gpu"`` tests):

* ``formats``    - E2M1 / E8M0 / E4M3 / 2-bit decoders by table; expert byte
                   sizes.  Pinned by OCP-spec values, the library fp8 cast,
                   and the byte counts the pages print.
* ``router``     - softmax, top-k (ties to lower id), renormalise.  Pinned by
                   brute-force subset enumeration and closed forms.
* ``slot_cache`` - LRU slot cache with miss list and capacity chunking.
                   Pinned by an independent ordered-dict LRU and a hand-worked
                   trace.
* ``ladder``     - the (a, b) precision ladder.  Pinned by hand-built cases.
* ``mlp``        - SwiGLU expert MLP and the weighted combine with the shared
                   expert.  Pinned by a pure-Python loop and rank-one closed
                   forms.
* ``permute``    - grouping of (token, rank) pairs by expert.  Pinned by a
                   brute-force bucket construction.
* ``mxquant``    - OCP MX quantisation of activations to MXFP4 (the
                   A-quantised prefill mode).  Pinned by hand-worked blocks
                   (grid values, every tie, saturation, zero and tiny blocks)
                   and a brute-force nearest-grid-point search.
* Model quality of the ladder and of the 2-bit level values: parity
  unpinned (needs trained weights and text).
"""
from . import formats, router, slot_cache, ladder, mlp, permute, mxquant  # noqa: F401
