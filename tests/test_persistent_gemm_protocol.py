"""A CPU model of the barrier protocol of the two persistent block-scaled GEMM
kernels: the decode GEMM (`mx8_gemm_kernel`, decode_mx8.cu) and the FP4
prefill GEMM (`mxf4_gemm_kernel`, expert_prefill.cu).

Both kernels run one CTA as warp roles that share, through mbarriers waited on
by phase parity:

* an item queue (kQueue entries): the TMA thread publishes each work index it
  draws (qfull), every consumer warp reads it and arrives on qempty;
* a ring of shared-memory operand stages (kStages): the TMA thread waits for
  the stage's previous MMAs (empty), arrives on full with the stage's byte
  count, and the TMA copies complete the bytes in any order; the scale-factor
  warps write the stage's scale factors to tensor memory and arrive on full;
* scale-factor slots in tensor memory: one per stage in the decode GEMM, two
  for three stages in the prefill GEMM (a store waits for the MMAs of the
  stage two back);
* the accumulators: the MMA warp waits until the epilogue warps have read
  the previous item's (acce) and commits the item's last MMAs to accf;
* a shared buffer guarded by warp-group syncs: the decode GEMM's two buffers
  of B scale rows (the next item's copied while the current item's MMAs
  drain), the prefill GEMM's staged h rows (written between two syncs, then
  stored to global memory by every epilogue warp).

The model runs every role as a generator over random and adversarial
interleavings of the roles, the TMA completions and the MMA commits (which
complete in issue order).  It fails on a parity wait that is not exact (one
that would pass a phase early, or wait on an aliased phase), an arrival
outside its phase, a deadlock, or a read or write of shared data that races:
an operand stage or scale-factor slot overwritten while an MMA reads it, an
MMA that reads a stage or slot not yet filled for its step, accumulators read
before the item's MMAs complete or overwritten before the epilogue has read
them, a queue entry read stale, a buffer row read before it was written or
after it was rewritten.  The ring depths, queue length, scale-factor slots and
warp counts are read from the kernel sources, so that the model follows them.
"""
import pathlib
import random
import re

import pytest

CSRC = pathlib.Path(__file__).resolve().parents[1] / "moe_expert_offload_router_gb300" / "csrc"


def _const(src, name):
    return int(re.search(rf"constexpr int {name} = (\d+);", src).group(1))


def _params():
    mx8 = (CSRC / "decode_mx8.cu").read_text()
    pf = (CSRC / "expert_prefill.cu").read_text()
    dec = dict(stages=_const(mx8, "kM8Stages"), queue=_const(mx8, "kM8Queue"), sf_slots=_const(mx8, "kM8Stages"),
               sf_warps=_const(mx8, "kM8Threads") // 32 - 2, epi_warps=_const(mx8, "kM8Threads") // 32 - 2)
    threads = _const(pf, "kMxThreads")
    pre = dict(stages=_const(pf, "kMxStages"), queue=_const(pf, "kMxQueue"), sf_slots=_const(pf, "kMxSfSlots"),
               sf_warps=4, epi_warps=threads // 32 - 4)
    # the structure the model follows, checked in the source text
    assert "mbar_init(&full[s], 1 + 4)" in mx8 and "mbar_init(&full[s], 1 + 4)" in pf
    assert "mbar_init(&qempty[j], 1 + 4)" in mx8 and "mbar_init(&qempty[j], 1 + kMxEpiWarps)" in pf
    assert "mbar_init(acce, 4)" in mx8 and "mbar_init(acce, kMxEpiWarps)" in pf
    assert "const int p = (int)gs - kMxSfSlots;" in pf
    return dec, pre


DECODE, PREFILL = _params()


class ProtocolError(Exception):
    pass


class _Bar:
    """An mbarrier: `count` arrivals and a transaction byte count per phase."""

    def __init__(self, name, count):
        self.name, self.count, self.pend, self.tx, self.done = name, count, 0, 0, 0

    def _check_phase(self, phase, what):
        if phase != self.done:
            raise ProtocolError(f"{what} on {self.name} for phase {phase} while phase {self.done} is open")

    def arrive(self, phase, tx=0):
        self._check_phase(phase, "arrival")
        self.pend += 1
        self.tx += tx
        if self.pend > self.count:
            raise ProtocolError(f"over-arrival on {self.name}")
        self._complete()

    def complete_tx(self, phase, n):
        self._check_phase(phase, "transaction bytes")
        self.tx -= n
        self._complete()

    def _complete(self):
        if self.pend == self.count and self.tx == 0:
            self.pend, self.done = 0, self.done + 1


STEP = None   # a role yields STEP for a scheduling point with no wait


def run_model(kind, p, runs, nk, seed, strategy, ntma=3, mutate=None):
    """One CTA of `kind` ("decode": either launch of the decode GEMM;
    "prefill_gateup" or "prefill_down": the FP4 prefill GEMM's two launches)
    over the items `runs` (True for an item the kernel computes, False for
    one every role skips)."""
    rng = random.Random(seed)
    S, Q, SF, NW, NE = p["stages"], p["queue"], p["sf_slots"], p["sf_warps"], p["epi_warps"]
    full = [_Bar(f"full{s}", 1 + NW) for s in range(S)]
    empty = [_Bar(f"empty{s}", 1) for s in range(S)]
    accf, acce, drain = _Bar("accf", 1), _Bar("acce", NE), _Bar("drain", 1)
    qfull = [_Bar(f"qfull{j}", 1) for j in range(Q)]
    qempty = [_Bar(f"qempty{j}", 1 + NE) for j in range(Q)]
    gsync = _Bar("group_sync", NW if kind == "decode" else NE)
    seq = list(range(len(runs))) + [-1]
    itq = [None] * Q
    tma, commits = [], []
    # shared data: what each stage / scale slot / buffer share holds, and readers in flight
    landed = [(None, 0)] * S               # (global step, TMA copies landed)
    stage_reads = [0] * S                   # MMAs issued on the stage, not yet complete
    sf = [[None] * NW for _ in range(SF)]   # global step whose scales each warp's quadrant holds
    sf_reads = [0] * SF
    acc = {"item": None, "done": 0, "reads": {}}
    bufs = [[None] * NW for _ in range(2)]  # decode: item whose B scale rows each warp's share holds
    hrows = [None] * NE                     # prefill: item whose h rows each epilogue warp has staged
    pending_reads = [0] * NE

    def check(cond, msg):
        if not cond:
            raise ProtocolError(msg)

    def next_item(qi):
        j, r = qi % Q, qi // Q
        yield qfull[j], r
        check(itq[j] is not None and itq[j][0] == qi, f"queue entry {j} read stale for publication {qi}")
        qempty[j].arrive(r)
        return itq[j][1]

    def producer():
        q, gs = 0, 0

        def publish(v):
            nonlocal q
            j, r = q % Q, q // Q
            if r > 0:
                yield qempty[j], r - 1
            itq[j] = (q, v)
            qfull[j].arrive(r)
            q += 1

        yield from publish(seq[0])
        for n in range(len(runs)):
            if runs[n]:
                for _ in range(nk):
                    s, r = gs % S, gs // S
                    if r > 0:
                        yield empty[s], r - 1
                    full[s].arrive(r, tx=ntma)
                    tma.extend((s, r, gs) for _ in range(ntma))
                    gs += 1
            yield from publish(seq[n + 1])

    def mma():
        gs, i, qi = 0, 0, 0
        while True:
            v = yield from next_item(qi)
            qi += 1
            if v < 0:
                break
            if not runs[v]:
                continue
            if i > 0 and mutate != "mma_skips_acce":
                yield acce, i - 1
            for ks in range(nk):
                s, r = gs % S, gs // S
                yield full[s], r
                check(landed[s] == (gs, ntma), f"MMA of step {gs} reads stage {s} holding {landed[s]}")
                slot = gs % SF
                check(all(x == gs for x in sf[slot]), f"MMA of step {gs} reads scale slot {slot} holding {sf[slot]}")
                if ks == 0:
                    check(i == 0 or acc["reads"].get(i - 1, 0) == NE,
                          f"item {i}'s first MMA overwrites accumulators the epilogue has not read")
                    acc.update(item=i, done=0)
                stage_reads[s] += 1
                sf_reads[slot] += 1
                commits.append(("stage", s, r, slot, i))
                gs += 1
            commits.append(("accf", i, None, None, i))
            i += 1
        commits.append(("drain", 0, None, None, None))
        yield drain, 0

    def store_scales(w, gs, reading_buf=None, item=None):
        """The scale-factor warp w's store for global step gs (a generator)."""
        s, r = gs % S, gs // S
        if kind == "decode":
            if r > 0:
                yield empty[s], r - 1
        else:
            back = gs - SF
            if back >= 0 and mutate != "prefill_sf_skips_wait":
                yield empty[back % S], back // S
        if reading_buf is not None:
            check(all(x == item for x in bufs[reading_buf]),
                  f"warp {w} reads B scale buffer {reading_buf} holding {bufs[reading_buf]} for item {item}")
        slot = gs % SF
        check(sf_reads[slot] == 0, f"warp {w} overwrites scale slot {slot} while an MMA reads it")
        sf[slot][w] = gs
        yield STEP
        full[s].arrive(r)

    def epilogue_read(w, i):
        check(acc["item"] == i and acc["done"] == nk, f"warp {w} reads item {i}'s accumulators in state {acc}")
        acc["reads"][i] = acc["reads"].get(i, 0) + 1

    def group_sync(state):
        gsync.arrive(state["n"])
        yield gsync, state["n"]
        state["n"] += 1

    def decode_warp(w):
        gs, i, qi = 0, 0, 0
        sync = {"n": 0}

        def take_run():
            nonlocal qi
            while True:
                v = yield from next_item(qi)
                qi += 1
                if v < 0 or runs[v]:
                    return v

        def copy_b(item, b):
            bufs[b][w] = item

        it = yield from take_run()
        buf = 0
        if it >= 0:
            copy_b(it, 0)
            if mutate != "decode_skips_copy_sync":
                yield from group_sync(sync)
        while it >= 0:
            for _ in range(nk):
                yield from store_scales(w, gs, buf, it)
                gs += 1
            nit = yield from take_run()
            if nit >= 0:
                yield STEP
                copy_b(nit, buf ^ 1)
                if mutate != "decode_skips_copy_sync":
                    yield from group_sync(sync)
            yield accf, i
            epilogue_read(w, i)
            yield STEP
            acce.arrive(i)
            i += 1
            it, buf = nit, buf ^ 1

    def prefill_warp(w):
        gs, i, qi = 0, 0, 0
        sync = {"n": 0}
        while True:
            v = yield from next_item(qi)
            qi += 1
            if v < 0:
                break
            if not runs[v]:
                continue
            if w < NW:
                for _ in range(nk):
                    yield from store_scales(w, gs)
                    gs += 1
            yield accf, i
            if kind == "prefill_down":
                # down: fp32 rows straight from the accumulators to global memory
                epilogue_read(w, i)
                yield STEP
                acce.arrive(i)
                i += 1
                continue
            if mutate != "prefill_skips_first_sync":
                yield from group_sync(sync)      # the previous item's rows have left
            check(not any(pending_reads), f"warp {w} rewrites staged h rows another warp has not stored yet")
            epilogue_read(w, i)
            hrows[w] = i
            yield STEP
            acce.arrive(i)
            yield from group_sync(sync)
            check(all(x == i for x in hrows), f"warp {w} stores h rows {hrows} for item {i}")
            pending_reads[w] = 1
            yield STEP
            check(all(x == i for x in hrows), f"staged h rows rewritten under warp {w}'s stores for item {i}")
            pending_reads[w] = 0
            i += 1

    roles = {"producer": producer(), "mma": mma()}
    for w in range(NW if kind == "decode" else NE):
        roles[f"w{w}"] = decode_warp(w) if kind == "decode" else prefill_warp(w)
    waits = {}
    for k in list(roles):
        try:
            waits[k] = next(roles[k])
        except StopIteration:
            del roles[k]
    victim = rng.choice(sorted(roles))

    while roles or tma or commits:
        runnable = []
        for k in roles:
            if waits[k] is STEP:
                runnable.append(k)
                continue
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
            pick = rng.choice([o for o in opts if o != victim] or opts)
        elif strategy == "copies_last":
            pick = rng.choice([o for o in opts if o not in ("tma", "commit")] or opts)
        else:
            pick = rng.choice(opts)
        if pick == "commit":
            what, a, r, slot, i = commits.pop(0)
            if what == "stage":
                stage_reads[a] -= 1
                sf_reads[slot] -= 1
                check(acc["item"] == i, f"an MMA of item {i} completes into the accumulators of item {acc['item']}")
                acc["done"] += 1
                empty[a].arrive(r)
            elif what == "accf":
                accf.arrive(a)
            else:
                drain.arrive(0)
        elif pick == "tma":
            s, r, gs = tma.pop(len(tma) - 1 if strategy == "lifo" else rng.randrange(len(tma)))
            check(stage_reads[s] == 0, f"TMA of step {gs} lands in stage {s} while an MMA reads it")
            prev_gs, n = landed[s]
            landed[s] = (gs, n + 1 if prev_gs == gs else 1)
            full[s].complete_tx(r, 1)
        else:
            try:
                waits[pick] = next(roles[pick])
            except StopIteration:
                del roles[pick]
    check(accf.done == sum(runs) and acce.done == sum(runs), "every computed item completes once")


ITEM_LISTS = [
    [True],
    [True, True, True],
    [True, False, True, True, False],
    [False, True],
    [False, False],
    [True] * 7,
]
STRATEGIES = ("uniform", "lifo", "starve", "copies_last")


def test_source_parameters_found():
    assert DECODE["stages"] == 2 and DECODE["sf_warps"] == 4 and DECODE["epi_warps"] == 4
    assert PREFILL["stages"] == 3 and PREFILL["sf_slots"] == 2 and PREFILL["epi_warps"] == 12
    assert DECODE["queue"] >= 2 and PREFILL["queue"] >= 2


@pytest.mark.parametrize("kind,p", [("decode", DECODE), ("prefill_gateup", PREFILL), ("prefill_down", PREFILL)])
@pytest.mark.parametrize("nk", [1, 2, 3, 4, 5, 8])
def test_every_wait_exact_and_no_race(kind, p, nk):
    for runs in ITEM_LISTS:
        for seed in range(3):
            for strategy in STRATEGIES:
                run_model(kind, p, runs, nk, seed, strategy)


@pytest.mark.parametrize("kind,p", [("decode", DECODE), ("prefill_gateup", PREFILL), ("prefill_down", PREFILL)])
def test_shorter_queue_and_deeper_ring_stay_exact(kind, p):
    # the protocol does not depend on the kernels' particular depths
    for q in (1, 2, 3):
        for stages in (2, 3, 4):
            sf = stages if kind == "decode" else PREFILL["sf_slots"]
            pp = dict(p, queue=q, stages=stages, sf_slots=sf)
            for seed in range(3):
                for strategy in STRATEGIES:
                    run_model(kind, pp, [True, False, True, True], 5, seed, strategy)


def _hits(kind, p, mutate, expect):
    hits = 0
    for runs in ITEM_LISTS[1:]:
        for nk in (1, 3, 5):
            for seed in range(6):
                for strategy in STRATEGIES:
                    try:
                        run_model(kind, p, runs, nk, seed, strategy, mutate=mutate)
                    except ProtocolError as e:
                        assert any(x in str(e) for x in expect), str(e)
                        hits += 1
    return hits


def test_model_catches_an_mma_that_skips_the_accumulator_release():
    # in the prefill GEMM's down launch eight of the twelve epilogue warps
    # store no scale factors and meet no other warp, so only the release
    # barrier keeps the next item's MMAs off the accumulators they still read
    assert _hits("prefill_down", PREFILL, "mma_skips_acce", ["acc", "deadlock"]) > 0


@pytest.mark.parametrize("kind,p", [("decode", DECODE), ("prefill_gateup", PREFILL)])
def test_release_is_also_implied_where_the_scale_warps_follow_every_read(kind, p):
    # the next item's first MMA waits for the scale-factor warps' first stores.
    # In the decode GEMM those four warps are the epilogue warps and store only
    # after their own epilogue; in the prefill GEMM's gate/up launch they store
    # only after the sync that follows every epilogue warp's accumulator reads
    # (the h staging).  Either way the release barrier is a second guard there.
    assert _hits(kind, p, "mma_skips_acce", ["acc", "deadlock"]) == 0


def test_model_catches_a_scale_store_that_skips_its_wait():
    # two scale slots for three stages: a store must wait for the MMAs of the
    # step two back, or it overwrites scale factors an MMA is reading
    assert _hits("prefill_down", PREFILL, "prefill_sf_skips_wait", ["scale slot", "full"]) > 0


def test_model_catches_a_b_scale_copy_without_its_sync():
    assert _hits("decode", DECODE, "decode_skips_copy_sync", ["B scale buffer"]) > 0


def test_model_catches_h_staging_without_its_first_sync():
    assert _hits("prefill_gateup", PREFILL, "prefill_skips_first_sync", ["h rows", "group_sync"]) > 0
