"""The five synthetic MoE-layer workloads, as plain data.

Shapes follow the pages' model: DeepSeek-V4-Flash with 256 routed experts per
layer, hidden size 4096 and expert intermediate size 2048 ("Running
DeepSeek-V4-Flash across four free GPUs", section "The model"; "An elephant
through a straw", section "Rig, model & methodology").  Nothing here computes
any part of the MoE layer; these are sizes, seeds and knobs for the input
generator in :mod:`synth.gen`.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional, Tuple


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    E: int                      # routed experts per layer
    k: int                      # router top_k
    H: int                      # hidden size
    I: int                      # expert intermediate size
    T: int                      # tokens per step (decode batch / prefill length)
    S: int                      # FP4 slot-cache slots (one pool shared by all layers)
    layers: int = 1
    steps: int = 1
    shared: bool = False        # one FP8 E4M3 shared expert with per-row fp32 scale
    zipf_s: Optional[float] = None   # log-Zipf popularity bias exponent (None = no bias)
    ladder: Optional[Tuple[int, int]] = None  # (a, b) precision ladder
    S2: int = 0                 # slots of the 2-bit copy pool (ladder only)
    reuse: Optional[float] = None    # step-to-step expert reuse probability
    reuse_boost: float = 8.0    # logit boost given to a reused expert
    T_sweep: Tuple[int, ...] = field(default_factory=tuple)
    scale_lo: int = 124         # E8M0 biased exponent range of the FP4 block scales
    scale_hi: int = 128


TINY = Workload(name="tiny", seed=0, E=8, k=2, H=256, I=128, T=4, S=4, steps=6)

DECODE = Workload(name="decode", seed=1, E=256, k=8, H=4096, I=2048, T=64, S=64,
                  steps=256, shared=True, zipf_s=1.1, T_sweep=(1, 4, 16, 64))

PREFILL = Workload(name="prefill", seed=2, E=256, k=6, H=4096, I=2048, T=8192, S=256)

LADDER = Workload(name="ladder", seed=3, E=256, k=6, H=4096, I=2048, T=32, S=96,
                  steps=128, zipf_s=1.1, ladder=(2, 4), S2=192)

STACK = Workload(name="stack", seed=4, E=256, k=8, H=4096, I=2048, T=16, S=43 * 256,
                 layers=43, steps=64, shared=True, zipf_s=1.1, reuse=0.7)

WORKLOADS = {w.name: w for w in (TINY, DECODE, PREFILL, LADDER, STACK)}


def scaled(w: Workload, **over) -> Workload:
    """A copy of ``w`` with some fields replaced (small variants for tests)."""
    d = dict(w.__dict__)
    d.update(over)
    return Workload(**d)
