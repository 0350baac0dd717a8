"""A CPU model of the grouped GEMM kernel's mbarrier protocol (expert_prefill.cu).

The kernel's warp roles share three rings of shared-memory stages, each guarded
by mbarriers that are waited on by phase parity:

* raw ring (kRing slots): the raw producer TMA-loads a K step's FP4/FP8 codes
  into slot ks % kRing once the slot's previous step has been converted
  (rawe), and the load's completion arrives on rawf;
* operand ring (kStages slots): converter group ks % 3 turns the codes into
  16-bit A tiles in slot ks % kStages once the MMA has drained that slot
  (empty) and arrives on full; the B producer's activation load arrives on
  full too;
* the MMA warp waits on full and commits each K step to empty, and the last
  commit to done, which the epilogue waits on.

A parity wait for phase n is exact only while the barrier has completed n or
n + 1 phases: with n - 1 it passes too early, with n + 2 or more it never
passes.  TMA completions can land in any order; MMA commits complete in
issue order (a commit tracks every earlier MMA).  The model runs every role as
a generator over random and adversarial interleavings and fails on a wait
that is not exact or on a deadlock.  The shapes (kRing, kStages) and the
guard condition are read from the kernel source, so that the model follows
it.
"""
import pathlib
import random
import re

import pytest

SRC = pathlib.Path(__file__).resolve().parents[1] / "moe_expert_offload_router_gb300" / "csrc" / "expert_prefill.cu"


def _shapes():
    s = SRC.read_text()
    groups = int(re.search(r"constexpr int kPfConvGroups = (\d+);", s).group(1))
    shapes = {m.group(1): (int(m.group(3)), int(m.group(4)))
              for m in re.finditer(r"using (Pf\w+) = PfCfg<(\d+), (\d+), (\d+)>;", s)}
    guard = re.search(r"constexpr bool kRawGuard = (.*);", s).group(1)
    return groups, shapes, guard


GROUPS, SHAPES, GUARD = _shapes()


class _Bar:
    def __init__(self, name, count):
        self.name, self.count, self.pend, self.done = name, count, 0, 0

    def arrive(self):
        self.pend += 1
        assert self.pend <= self.count, f"over-arrival on {self.name}"
        if self.pend == self.count:
            self.pend, self.done = 0, self.done + 1


class ProtocolError(Exception):
    pass


def run_model(nk, stages, ring, guard, seed, strategy, groups=GROUPS):
    """One CTA's K loop; raises ProtocolError on an inexact wait or a deadlock."""
    rng = random.Random(seed)
    full = [_Bar(f"full{s}", 2) for s in range(stages)]   # the converting group + the B load
    empty = [_Bar(f"empty{s}", 1) for s in range(stages)]
    rawf = [_Bar(f"rawf{s}", 1) for s in range(ring)]
    rawe = [_Bar(f"rawe{s}", 1) for s in range(ring)]
    done = _Bar("done", 1)
    tma, commits = [], []

    def raw_producer():
        for rk in range(nk):
            rs, rr = rk % ring, rk // ring
            if rr > 0:
                yield rawe[rs], rr - 1
            tma.append(rawf[rs])

    def b_producer():
        for ks in range(nk):
            s, r = ks % stages, ks // stages
            if r > 0:
                yield empty[s], r - 1
            tma.append(full[s])

    def mma():
        for ks in range(nk):
            s, r = ks % stages, ks // stages
            yield full[s], r
            commits.append(empty[s])
        commits.append(done)

    def converter(cg):
        for ks in range(cg, nk, groups):
            rs, rr, s, rnd = ks % ring, ks // ring, ks % stages, ks // stages
            if guard and rr > 0:
                yield rawe[rs], rr - 1
            yield rawf[rs], rr
            if rnd > 0:
                yield empty[s], rnd - 1
            full[s].arrive()
            rawe[rs].arrive()
        yield done, 0

    roles = {"raw": raw_producer(), "b": b_producer(), "mma": mma()}
    roles.update({f"conv{c}": converter(c) for c in range(groups)})
    waits = {}
    for k in list(roles):
        try:
            waits[k] = next(roles[k])
        except StopIteration:
            del roles[k]
    victim = rng.choice(sorted(roles) + ["tma0"])

    while roles or tma or commits:
        runnable = []
        for k in roles:
            bar, n = waits[k]
            if bar.done >= n + 2:
                raise ProtocolError(f"{k}: {bar.name} phase {n} aliased ({bar.done} completed)")
            if bar.done == n - 1:
                raise ProtocolError(f"{k}: {bar.name} phase {n} would pass early ({bar.done} completed)")
            if bar.done == n + 1:
                runnable.append(k)
        opts = runnable + (["tma"] if tma else []) + (["commit"] if commits else [])
        if not opts:
            raise ProtocolError("deadlock: " + ", ".join(f"{k} on {waits[k][0].name}" for k in roles))
        if strategy == "starve":
            pref = [o for o in opts if o != victim and not (o == "tma" and victim == "tma0" and len(tma) == 1)]
            pick = rng.choice(pref or opts)
        else:
            pick = rng.choice(opts)
        if pick == "commit":
            commits.pop(0).arrive()
        elif pick == "tma":
            if strategy == "lifo":
                i = len(tma) - 1
            elif strategy == "starve" and victim == "tma0" and len(tma) > 1:
                i = rng.randrange(1, len(tma))
            else:
                i = rng.randrange(len(tma))
            tma.pop(i).arrive()
        else:
            try:
                waits[pick] = next(roles[pick])
            except StopIteration:
                del roles[pick]


def _kernel_guard(ring, stages):
    expr = GUARD.replace("kRing", str(ring)).replace("C::kStages", str(stages)).replace(
        "kPfConvGroups", str(GROUPS)).replace("&&", " and ").replace("!=", " != ")
    assert re.fullmatch(r"[\d\s%<>=!+and]+", expr), GUARD
    return bool(eval(expr))


def _rings():
    # the FP4 kernels use kRaw slots; the FP8 shared-expert shape takes twice
    # the bytes per K step in half as many
    return [(name, stages, raw) for name, (raw, stages) in SHAPES.items() if name != "PfShared"] + \
           [("PfShared", SHAPES["PfShared"][1], SHAPES["PfShared"][0] // 2)]


def test_source_shapes_found():
    assert GROUPS == 3
    assert set(SHAPES) == {"PfBig", "PfSmall", "PfShared"}


@pytest.mark.parametrize("name,stages,ring", _rings())
@pytest.mark.parametrize("nk", [1, 2, 3, 4, 5, 7, 32, 64])
def test_every_wait_is_exact(name, stages, ring, nk):
    guard = _kernel_guard(ring, stages)
    for seed in range(6 if nk <= 8 else 2):
        for strategy in ("uniform", "lifo", "starve"):
            run_model(nk, stages, ring, guard, seed, strategy)


def test_model_catches_an_unguarded_short_ring():
    # a raw ring shorter than kStages + groups and not a multiple of the group
    # count lets a group reach a slot before its previous fill has landed
    stages, ring = 3, 4
    assert _kernel_guard(ring, stages)
    hits = 0
    for seed in range(20):
        try:
            run_model(32, stages, ring, False, seed, "lifo")
        except ProtocolError as e:
            assert "rawf" in str(e) and "early" in str(e)
            hits += 1
    assert hits > 0
    for seed in range(20):
        run_model(32, stages, ring, True, seed, "lifo")


@pytest.mark.parametrize("stages,ring", [(3, 4), (3, 6)])
def test_four_converter_groups_lap_a_three_stage_operand_ring(stages, ring):
    # A 20-warp variant of the kernel (four converter groups) faulted the GPU on
    # the wide shape (three operand stages).  The model shows why: with four
    # groups over three stages a stage is filled by a different group each
    # round, so a fast group reaches its next step on a stage while the group
    # of the round in between has not filled it yet; its parity wait on that
    # stage's "empty" barrier passes a round early, it overwrites operands the
    # MMA has not read and arrives on "full" in the wrong phase.  With three
    # groups (each group always fills the same stage) every wait is exact.
    hits = 0
    for nk in (8, 32, 64):
        for seed in range(10):
            for strategy in ("uniform", "starve"):
                try:
                    run_model(nk, stages, ring, ring % 4 != 0 and ring < stages + 4, seed, strategy, groups=4)
                except ProtocolError as e:
                    assert "empty" in str(e) and "early" in str(e)
                    hits += 1
    assert hits > 0
    for nk in (8, 32, 64):
        for seed in range(4):
            run_model(nk, stages, ring, _kernel_guard(ring, stages), seed, "starve", groups=3)


@pytest.mark.parametrize("stages,ring", [(4, 4), (4, 8)])
def test_four_converter_groups_with_four_stages_are_exact(stages, ring):
    # as many operand stages as groups: each group owns its stage again
    for nk in (1, 5, 32, 64):
        for seed in range(4):
            for strategy in ("uniform", "lifo", "starve"):
                run_model(nk, stages, ring, ring % 4 != 0 and ring < stages + 4, seed, strategy, groups=4)
