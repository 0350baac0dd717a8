#!/usr/bin/env python
"""Benchmark of the routed MoE decode layer served from the GPU expert-slot cache.

Workload (default): the V4-Flash-shaped decode layer -- H=4096, I=2048, E=256
routed MXFP4 experts (13,369,344 B each), top_k=8, one FP8 shared expert, a
64-slot cache backed by a pinned host bank of all 256 experts, bf16 N(0,1)
activations, fp32 N(0,1) router logits plus a log-Zipf(1.1) popularity bias,
run over a seeded routing trace.  One step = one layer call on one trace step:
router, ensure_experts, the one host sync, the misses copied from the pinned
bank, the grouped expert MLP with the shared expert and combine.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s + HBM GB/s (decode); FP4 TFLOPS vs peak (prefill)"
UNIT = "tokens/s"


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    # decode steps copy experts over the host link; in some processes the first
    # ~15 steps after setup ran up to 2x slower before settling, so the default
    # warm-up covers that transient
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--T", type=int, default=64, help="decode batch of the headline line")
    p.add_argument("--sweep", default="1,4,16,64", help="decode batches also measured (comma list, '' for none)")
    p.add_argument("--cpu-sample-tokens", type=int, default=12,
                   help="tokens of the decode workload the oracle is timed on (about 10 s of host time)")
    p.add_argument("--workload", default="decode", choices=["decode", "prefill", "ladder", "stack", "forward"],
                   help="forward: the decode layer's compute alone (router, ensure, expert MLP) on all 256 "
                        "experts resident, no copies and no CPU baseline (a small case for profiling)")
    p.add_argument("--copy", default="device", choices=["engine", "device"],
                   help="miss copies: copy engine after one host sync, or a kernel reading the miss list")
    p.add_argument("--prefill-experts", type=int, default=0,
                   help="prefill workload with this many experts (all resident), for profiling a smaller case")
    p.add_argument("--prefill-tokens", type=int, default=0, help="prefill workload with this many tokens")
    p.add_argument("--stream-layers", type=int, default=0,
                   help="prefill: stream this many layers whole from the pinned bank (nothing resident)")
    p.add_argument("--evict", default="lru", choices=["lru", "lfu"],
                   help="decode: slot eviction policy (lfu: counts seeded from a disjoint stretch of the trace)")
    p.add_argument("--lfu-decay", type=int, default=64, help="decode, lfu: ensure calls per count halving")
    p.add_argument("--prefetch", type=int, default=0,
                   help="decode: staging-ring slots for predicted experts of the next step (0 = off)")
    p.add_argument("--pf-recall", type=float, default=0.75,
                   help="decode prefetch: share of the next step's experts the synthetic predictor includes")
    p.add_argument("--no-overlap", action="store_true",
                   help="device copy: run the forward after the copies instead of beside them")
    p.add_argument("--window-start", type=int, default=128,
                   help="decode: first trace step of the timed window; the steps before it are replayed untimed "
                        "(the warm-up steps are the last of them), so the window sits at the trace's steady state")
    p.add_argument("--extras", default="prefill,ladder,stack",
                   help="decode: other workloads measured in the same run and reported under their own keys "
                        "(comma list of prefill, ladder, stack; '' for none)")
    p.add_argument("--mma-max-tokens", type=int, default=None,
                   help="decode batches of 2 up to this many tokens take the tensor-core decode kernels (library "
                        "default if omitted; 0 = never)")
    p.add_argument("--mx8-min-tokens", type=int, default=None,
                   help="of those, batches from this many tokens take the block-scaled tcgen05 GEMM, the others "
                        "the warp-MMA kernels (library default if omitted; 0 = never)")
    return p.parse_args()


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# DRAM bytes (read + write) of one launch of a kernel from an ncu capture of
# the same workload (profiles/), with the algorithmic bytes of that same
# launch: a bench line scales the ratio to its own launches.  An entry is
# removed when its kernel changes.
NCU_TRAFFIC = {
    ("mx8_gemm_kernel (gate/up)", "decode"): {
        "dram_bytes": 503_437_056 + 5_178_112, "algorithmic_bytes": 505_278_464,
        "capture": "ncu dram__bytes_read/write.sum of mx8_gemm_kernel gate/up, bench.py --workload forward --T 64 "
                   "(trace step 3: 54 experts + shared), profiles/mx8_gemm_kernel_decode_forward_T64.md"},
    ("mxf4_gemm_kernel (gate/up)", "prefill"): {
        "dram_bytes": 597_576_704 + 12_771_584, "algorithmic_bytes": 610_533_376,
        "capture": "ncu dram__bytes_read/write.sum of mxf4_gemm_kernel gate/up, bench.py --workload prefill "
                   "--prefill-experts 64 --prefill-tokens 2048, profiles/mxf4_gemm_kernel_prefill_E64_T2048.md"},
    ("prefill_gemm_kernel (gate/up)", "prefill"): {
        "dram_bytes": 676_065_280 + 45_294_592, "algorithmic_bytes": 721_420_288,
        "capture": "ncu dram__bytes_read/write.sum of prefill_gemm_kernel gate/up, bench.py --workload prefill "
                   "--prefill-experts 64 --prefill-tokens 2048, profiles/prefill_gemm_kernel_prefill_E64_T2048.md"},
}


def apply_options(M, args):
    """Sets the library's decode-path options from the command line; returns
    (mma_max, mx8_min) as they stand."""
    if args.mma_max_tokens is not None:
        M.moe_set_option(M.MOE_OPT_MMA_MAX_TOKENS, args.mma_max_tokens)
    if getattr(args, "mx8_min_tokens", None) is not None:
        M.moe_set_option(M.MOE_OPT_MX8_MIN_TOKENS, args.mx8_min_tokens)
    mma_max = M.moe_set_option(M.MOE_OPT_MMA_MAX_TOKENS, 0)
    M.moe_set_option(M.MOE_OPT_MMA_MAX_TOKENS, mma_max)
    mx8_min = M.moe_set_option(M.MOE_OPT_MX8_MIN_TOKENS, 0)
    M.moe_set_option(M.MOE_OPT_MX8_MIN_TOKENS, mx8_min)
    return mma_max, mx8_min


def gateup_kernel(T, mma_max, mx8_min):
    """Name of the kernel that runs a decode batch's gate/up (below the grouped-GEMM size)."""
    if 2 <= T <= mma_max:
        return "mx8_gemm_kernel (gate/up)" if 0 < mx8_min <= T else "mma_gateup_kernel"
    return "gateup_kernel"


def gateup_io_bytes(kernel, T, k, H, I):
    """Activation and h bytes one gate/up launch moves for a batch of T tokens
    (k pairs each, plus the shared expert's T rows): bf16 x and fp32 h for the
    CUDA-core and warp-MMA kernels; E4M3 hi/lo rows with a scale byte per 32
    elements, read and written, for the block-scaled GEMM."""
    rows = T * k + T
    if kernel.startswith("mx8"):
        return rows * (2 * H + H // 32) + rows * (2 * I + I // 32)
    return T * H * 2 + rows * I * 4


DTYPE_MX8 = ("e2m1/e8m0 weights x e4m3 hi+lo activations (tcgen05.mma.kind::mxf8f6f4), fp32 accumulate")
DTYPE_MMA = "e2m1/e8m0 weights, fp16 products, fp32 accumulate"


def ncu_traffic(kernel, workload, bytes_per_launch):
    t = NCU_TRAFFIC.get((kernel, workload))
    return (t["dram_bytes"] / t["algorithmic_bytes"] * bytes_per_launch, t["capture"]) if t else (None, None)


def roofline_hbm(kernel, achieved, bytes_per_launch, ms_per_launch, peak, peak_kind, note, workload=None):
    traffic, src = ncu_traffic(kernel, workload, bytes_per_launch)
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
            "traffic": traffic, "traffic_source": src,
            "kernel": kernel, "peak_kind": peak_kind + " (copy bandwidth)",
            "bytes_per_launch": bytes_per_launch, "ms_per_launch": ms_per_launch, "note": note}


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "200"],
                                      stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(timeout=5)
        except Exception:
            self.p.kill()
        self.f.flush()
        rows = []
        with open(self.f.name) as fh:
            for ln in fh:
                parts = [x.strip() for x in ln.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.f.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample of the workload
# ----------------------------------------------------------------------------

_CPU_SNIPPET = r"""
import json, sys, time
sys.path.insert(0, {root!r})
import numpy as np
from oracle import formats as F
from oracle.mlp import moe_layer
from oracle.router import router_topk
from oracle.slot_cache import FETCH, SlotCacheLRU
from synth import configs, gen
wl = configs.scaled(configs.DECODE, T={T})
shared_bytes = gen.shared_expert(wl, 0)
t0 = time.perf_counter()
cache = SlotCacheLRU(wl.S, 1, wl.E)
shw = F.decode_fp8_expert(shared_bytes, wl.H, wl.I)
tokens = 0
step_seconds = []
for step in range({warm} + {steps}):
    if step == {warm}:
        t0, tokens = time.perf_counter(), 0
    ts = time.perf_counter()
    lg = gen.router_logits(wl, 0, step, wl.T)
    x = gen.activations(wl, 0, step, wl.T)
    ids, w = router_topk(lg, wl.k)
    tb = 0
    while tb < wl.T:
        _, _, _, tb = cache.ensure(0, ids, 0, wl.k, FETCH, tb)
    y = moe_layer(x, ids, w, lambda e, tag: F.decode_fp4_expert(gen.fp4_expert(wl, 0, e), wl.H, wl.I),
                  shared=shw)
    tokens += wl.T
    step_seconds.append(time.perf_counter() - ts)
dt = time.perf_counter() - t0
print(json.dumps({{"tokens": tokens, "seconds": dt, "step_seconds": step_seconds[{warm}:]}}))
"""


def aggregate(ms_local: float, tokens_local: int, world: int, device=None):
    """Whole-job numbers for N independent replicas: the step time is the max
    over ranks, the throughput counts every rank's tokens."""
    ms = ms_local
    if world > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([ms_local], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, world * tokens_local / (ms / 1e3)


def _run_oracle(T: int, steps: int, threads: int, warm: int = 0):
    """The oracle over `warm` untimed and `steps` timed decode trace steps of
    T tokens, in a child process with `threads` BLAS/OpenMP threads: its
    record ({"tokens", "seconds", "step_seconds"}) or the error's last line."""
    n = str(threads)
    env = dict(os.environ, OMP_NUM_THREADS=n, OPENBLAS_NUM_THREADS=n, MKL_NUM_THREADS=n)
    code = _CPU_SNIPPET.format(root=ROOT, T=T, steps=steps, warm=warm)
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return "failed: " + (r.stderr.strip().splitlines()[-1][:200] if r.stderr.strip() else "no output")
    return json.loads(r.stdout.strip().splitlines()[-1])


def cpu_baseline(T: int, steps: int = 1, threads: int = 1):
    """The oracle timed on the host cores: `threads` BLAS/OpenMP threads."""
    d = _run_oracle(T, steps, threads)
    if isinstance(d, str):
        return {"value": None, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": d}
    how = "single-threaded" if threads == 1 else f"{threads} threads"
    return {"value": d["tokens"] / d["seconds"], "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{steps} trace step(s) x {T} tokens of the decode workload (fp64 NumPy, "
                      f"weights regenerated and decoded per expert), {d['seconds']:.1f} s {how}"}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def decode_line(args):
    """The decode workload's contract line (rank 0; None elsewhere)."""
    import numpy as np
    import torch
    import torch.distributed as dist

    from moe_expert_offload_router_gb300 import build as B
    B.build()
    import moe_expert_offload_router_gb300 as M
    from synth import configs, gen

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    apply_options(M, args)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    base = configs.DECODE
    Ts = sorted({args.T} | {int(t) for t in args.sweep.split(",") if t.strip()})
    Tmax = max(Ts)
    H, I, E, k, S = base.H, base.I, base.E, base.k, base.S
    Bx = M.moe_fp4_expert_bytes(H, I)
    # pinned bank of all 256 experts, generated on the device by the seeded counter generator
    bank = torch.empty(E * Bx, dtype=torch.uint8, pin_memory=True)
    for e in range(E):
        bank[e * Bx:(e + 1) * Bx].copy_(gen.fp4_expert(base, 0, e, device=dev))
    slots = torch.empty((S + args.prefetch) * Bx, dtype=torch.uint8, device=dev)
    shared = torch.from_numpy(gen.shared_expert(base, 0)).to(dev)
    cache = M.moe_cache(S, 1, E, Bx, slots, bank)
    if args.prefetch:
        M.moe_cache_set_staging(cache, args.prefetch)
    views = M.make_views(H, I, slots, S, None, 0, shared)
    if args.evict == "lfu":
        # seed: how often each expert was routed over 64 steps of the trace that the timed steps do not replay
        seed = np.zeros(E, dtype=np.int64)
        for st in range(1000, 1064):
            ids_s = np.argsort(-gen.router_logits(configs.scaled(base, T=Tmax), 0, st, Tmax), axis=1, kind="stable")
            np.add.at(seed, np.unique(ids_s[:, :k]), 1)
        M.moe_cache_set_policy(cache, M.MOE_EVICT_LFU, args.lfu_decay)
        lfu_seed = seed
    else:
        lfu_seed = None
    overlap = "auto" if args.copy == "device" and not args.no_overlap else False
    runner = M.DecodeLayerRunner(cache, views, E, k, Tmax, dev, copy=args.copy, overlap=overlap)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)     # > 129 MB L2
    hbm_peak, peak_kind = _peaks()

    def link_probe():
        """Copy-engine bandwidth from the pinned bank to the device (one
        cudaMemcpyAsync of 128 MB, median of 5 after one untimed), the
        reference that host_link_gbs is reported against; None if it fails."""
        try:
            n = min(128 << 20, bank.numel(), flush.numel())
            src, dst = bank[:n], flush[:n]
            rates = []
            for _ in range(6):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                dst.copy_(src, non_blocking=True)
                b.record(stream)
                b.synchronize()
                rates.append(n / (a.elapsed_time(b) / 1e3) / 1e9)
            return statistics.median(rates[1:])
        except Exception:
            return None
    stream = torch.cuda.current_stream(dev)
    mma_max, mx8_min = apply_options(M, args)
    # trace steps: [0, start - warmup) replayed untimed from an empty cache, then
    # [start - warmup, start) as warm-up, then the timed window [start, start + steps)
    start = max(args.window_start, args.warmup)
    n_steps = start + args.steps
    first_warm = start - args.warmup

    def inputs(T):
        wl = configs.scaled(base, T=T)
        lg_np = [gen.router_logits(wl, 0, s % base.steps, T) for s in range(n_steps + 1)]
        lg = [torch.from_numpy(v).to(dev) for v in lg_np[:n_steps]]
        xs = [torch.from_numpy(gen.activations(wl, 0, s % base.steps, T).view(np.int16)).to(dev)
              for s in range(n_steps)]
        return lg, xs, predictions(lg_np)

    def predictions(lg_np):
        """Synthetic predictor (the pages' trained predictor is out of scope): for
        step s, each expert that step s+1 routes to is included with probability
        pf_recall, plus a quarter as many experts it does not route to."""
        if not args.prefetch:
            return None
        rng = np.random.default_rng(17)
        out = []
        for s in range(n_steps):
            nxt = np.unique(np.argsort(-lg_np[s + 1], axis=1, kind="stable")[:, :k])
            keep = nxt[rng.random(nxt.size) < args.pf_recall]
            others = np.setdiff1d(np.arange(E), nxt)
            fp = rng.choice(others, size=max(1, keep.size // 4), replace=False)
            guess = rng.permutation(np.concatenate([keep, fp])).astype(np.int32)
            out.append((0, torch.from_numpy(guess).to(dev)))
        return out

    gu_expert = 2 * (I * H // 2 + I * H // 32)             # w1 + w3 bytes of one FP4 expert
    gu_shared = 2 * (I * H + I * 4)                          # w1 + w3 of the FP8 shared expert
    layer_shared = M.moe_fp8_expert_bytes(H, I)

    def measure(T):
        lg, xs, pf = inputs(T)
        y = torch.empty((T, H), dtype=torch.int16, device=dev)

        def fresh():
            cache.reset()
            torch.cuda.synchronize()
            if lfu_seed is not None:
                M.moe_cache_seed_frequency(cache, lfu_seed)
            for s in range(start):      # replay, then warm-up: the cache reaches the window's state
                runner.run(0, lg[s], xs[s], y, prefetch=pf[s] if pf else None)
            torch.cuda.synchronize()
            runner.check()

        # timed pass: no per-kernel events inside the timed steps
        fresh()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        misses0, bytes0 = runner.stats["misses"], runner.stats["bytes_copied"]
        ids_seen = []
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            s = start + i
            flush.zero_()
            ev[i][0].record(stream)
            runner.run(0, lg[s], xs[s], y, prefetch=pf[s] if pf else None)
            ev[i][1].record(stream)
            ids_seen.append(runner.ids[:T].clone())
        torch.cuda.synchronize()
        runner.check()
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
        step_ms = [a.elapsed_time(b) for a, b in ev]
        misses = runner.stats["misses"] - misses0
        copied = runner.stats["bytes_copied"] - bytes0
        # accounting: distinct experts per step
        gu_name = gateup_kernel(T, mma_max, mx8_min)
        acct_gu_bytes, acct_layer_bytes, acct_gemm_bytes = 0, 0, 0
        distinct = 0
        for ids in ids_seen:
            d = int(torch.unique(ids).numel())
            distinct += d
            acct_gemm_bytes += d * gu_expert + T * H * 2 + T * k * I * 2
            acct_gu_bytes += gu_shared + d * gu_expert + gateup_io_bytes(gu_name, T, k, H, I)
            acct_layer_bytes += d * Bx + layer_shared + 2 * T * H * 2
        # profiled pass: the same steps again from the same cache state, each
        # kernel bracketed by the library's events (for the breakdown only)
        fresh()
        M.moe_profile_enable(True)
        for i in range(args.steps):
            s = start + i
            flush.zero_()
            runner.run(0, lg[s], xs[s], y, prefetch=pf[s] if pf else None)
        torch.cuda.synchronize()
        runner.check()
        kt = {M.KERNEL_NAMES[kid]: M.moe_profile_query(kid) for kid in range(M.MOE_K_COUNT)}
        M.moe_profile_enable(False)
        ms, tps = aggregate(sum(step_ms) / len(step_ms), T, world, dev)
        gu_ms, gu_n = kt["gateup"]
        gg_ms, gg_n = kt["gemm_gateup"]
        if gg_n and gg_ms >= gu_ms:   # the tcgen05 grouped GEMM dominates this batch size
            dom, dms, dn, dbytes = "prefill_gemm_kernel (gate/up)", gg_ms, gg_n, acct_gemm_bytes
        else:
            # the routed experts' bytes count only where this kernel computed them
            dbytes = acct_gu_bytes if not gg_n else acct_gu_bytes - acct_gemm_bytes + T * H * 2
            dom, dms, dn = gu_name, gu_ms, gu_n
        gu_ms, gu_n, acct_gu_bytes = dms, dn, dbytes
        compute_ms = sum(v[0] for n, v in kt.items() if n != "copy_device") / args.steps
        return {
            "dominant": dom,
            "T": T, "ms_per_step": ms, "tokens_per_s": tps,
            "kernel_sum_tokens_per_s": T / (compute_ms / 1e3),
            "layer_gbs": acct_layer_bytes / args.steps / (ms / 1e3) / 1e9,
            "gateup_ms": gu_ms / max(gu_n, 1), "gateup_launches": gu_n,
            "gateup_gbs": (acct_gu_bytes / max(gu_n, 1)) / (gu_ms / max(gu_n, 1) / 1e3) / 1e9,
            "gateup_bytes_per_launch": acct_gu_bytes / max(gu_n, 1),
            "misses_per_step": misses / args.steps,
            # distinct experts of a step found resident (capacity chunks that re-fetch count as misses)
            "hit_rate": 1.0 - misses / max(distinct, 1),
            "host_link_gbs": (copied / args.steps / (kt["copy_device"][0] / args.steps / 1e3)
                              / 1e9 if kt["copy_device"][1] else None),
            "h2d_gb_per_step": copied / args.steps / 1e9,
            "kernel_ms": {n: round(v[0] / args.steps, 4) for n, v in kt.items() if v[1]},
            "launches": sum(v[1] for v in kt.values()),
            "wall_s": wall,
        }

    def measure_e2e(T):
        """Same steps through the public API with host buffers: inputs copied in
        from pinned memory and the output read back, every step."""
        lg, xs, pf = inputs(T)
        h_lg = {s: lg[s].cpu().pin_memory() for s in range(first_warm, n_steps)}
        h_x = {s: xs[s].cpu().pin_memory() for s in range(first_warm, n_steps)}
        d_lg = torch.empty_like(lg[0])
        d_x = torch.empty_like(xs[0])
        y = torch.empty((T, H), dtype=torch.int16, device=dev)
        h_y = torch.empty((T, H), dtype=torch.int16, pin_memory=True)
        cache.reset()
        torch.cuda.synchronize()
        if lfu_seed is not None:
            M.moe_cache_seed_frequency(cache, lfu_seed)
        for s in range(first_warm):          # untimed replay to the window's cache state
            runner.run(0, lg[s], xs[s], y, prefetch=pf[s] if pf else None)
        for s in range(first_warm, start):
            d_lg.copy_(h_lg[s], non_blocking=True)
            d_x.copy_(h_x[s], non_blocking=True)
            runner.run(0, d_lg, d_x, y, prefetch=pf[s] if pf else None)
            h_y.copy_(y, non_blocking=True)
        torch.cuda.synchronize()
        tot = 0.0
        for i in range(args.steps):
            s = start + i
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            d_lg.copy_(h_lg[s], non_blocking=True)
            d_x.copy_(h_x[s], non_blocking=True)
            runner.run(0, d_lg, d_x, y, prefetch=pf[s] if pf else None)
            h_y.copy_(y, non_blocking=True)
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        ms = tot / args.steps
        return {"value": world * T / (ms / 1e3), "unit": UNIT,
                "h2d_bytes_per_step": T * E * 4 + T * H * 2, "d2h_bytes_per_step": T * H * 2}

    def measure_compute_only(T):
        """Router + ensure + forward with every expert resident (a 256-slot pool
        filled from the bank, no copies): the compute-only step of the same trace."""
        full = torch.empty(E * Bx, dtype=torch.uint8, device=dev)
        full.copy_(bank)
        fcache = M.moe_cache(E, 1, E, Bx, full, None)
        fcache.import_(np.arange(E, dtype=np.int32), np.arange(E, dtype=np.uint64), E)
        fviews = M.make_views(H, I, full, E, None, 0, shared)
        frunner = M.DecodeLayerRunner(fcache, fviews, E, k, T, dev, assume_resident=True)
        lg, xs, _ = inputs(T)
        y = torch.empty((T, H), dtype=torch.int16, device=dev)
        for s in range(first_warm, start):
            frunner.run(0, lg[s], xs[s], y)
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        seen = []
        for i in range(args.steps):
            s = start + i
            flush.zero_()
            ev[i][0].record(stream)
            frunner.run(0, lg[s], xs[s], y)
            ev[i][1].record(stream)
            seen.append(frunner.ids[:T].clone())
        torch.cuda.synchronize()
        ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
        # the same steps again with the library's per-kernel events: the
        # dominant kernel's launch time (kept out of the step timing above)
        M.moe_profile_enable(True)
        for i in range(args.steps):
            s = start + i
            flush.zero_()
            frunner.run(0, lg[s], xs[s], y)
        torch.cuda.synchronize()
        kt = {M.KERNEL_NAMES[kid]: M.moe_profile_query(kid) for kid in range(M.MOE_K_COUNT)}
        M.moe_profile_enable(False)
        fcache.close()
        del full
        dsum = [int(torch.unique(ids).numel()) for ids in seen]
        nbytes = sum(d * Bx + layer_shared + 2 * T * H * 2 for d in dsum)
        gbs = nbytes / args.steps / (ms / 1e3) / 1e9
        # gate/up launch: the routed experts' w1/w3 (or only the shared expert's when
        # the tcgen05 grouped GEMM took the routed pairs), x and h
        gg_ms, gg_n = kt["gemm_gateup"]
        gu_ms, gu_n = kt["gateup"]
        P = T * k
        if gg_n:
            kname, kms, kn = "prefill_gemm_kernel (gate/up)", gg_ms, gg_n
            kbytes = sum(d * gu_expert + T * H * 2 + P * I * 2 for d in dsum) / kn
        else:
            kname = gateup_kernel(T, mma_max, mx8_min)
            kms, kn = gu_ms, gu_n
            kbytes = sum(d * gu_expert + gu_shared + gateup_io_bytes(kname, T, k, H, I) for d in dsum) / kn
        kgbs = kbytes / (kms / kn / 1e3) / 1e9
        return {"ms_per_step": ms, "tokens_per_s": T / (ms / 1e3), "layer_hbm_gbs": gbs,
                "frac_of_hbm": gbs / hbm_peak, "kernel": kname, "kernel_ms_per_launch": kms / kn,
                "kernel_bytes_per_launch": kbytes, "kernel_gbs": kgbs,
                "kernel_ms_per_step": {n: round(v[0] / args.steps, 4) for n, v in kt.items() if v[1]},
                "note": "router + ensure + forward, all 256 experts resident, same trace steps, L2 flushed"}

    def measure_trace(T):
        """Misses over the whole seeded trace (every step from an empty cache), beside
        the timed window's figures."""
        wl = configs.scaled(base, T=T)
        y = torch.empty((T, H), dtype=torch.int16, device=dev)
        cache.reset()
        torch.cuda.synchronize()
        if lfu_seed is not None:
            M.moe_cache_seed_frequency(cache, lfu_seed)
        m0 = runner.stats["misses"]
        distinct = 0
        for s in range(base.steps):
            lg_s = torch.from_numpy(gen.router_logits(wl, 0, s, T)).to(dev)
            x_s = torch.from_numpy(gen.activations(wl, 0, s, T).view(np.int16)).to(dev)
            runner.run(0, lg_s, x_s, y)
            distinct += int(torch.unique(runner.ids[:T]).numel())
        torch.cuda.synchronize()
        runner.check()
        misses = runner.stats["misses"] - m0
        return {"steps": base.steps, "misses_per_step": misses / base.steps,
                "hit_rate": 1.0 - misses / max(distinct, 1)}

    def measure_graph(T):
        """The same steps with each layer step replayed as one CUDA graph (batches
        that are one chunk by construction); no per-kernel profiling."""
        grunner = M.DecodeLayerRunner(cache, views, E, k, T, dev, copy=args.copy, graph=True)
        cache.reset()
        torch.cuda.synchronize()
        if lfu_seed is not None:
            M.moe_cache_seed_frequency(cache, lfu_seed)
        lg, xs, _ = inputs(T)
        y = torch.empty((T, H), dtype=torch.int16, device=dev)
        for s in range(start):
            grunner.run(0, lg[s], xs[s], y)
        torch.cuda.synchronize()
        grunner.check()
        tot = 0.0
        for i in range(args.steps):
            s = start + i
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            grunner.run(0, lg[s], xs[s], y)
            b.record(stream)
            b.synchronize()
            tot += a.elapsed_time(b)
        grunner.check()
        ms = tot / args.steps
        return {"graph_ms_per_step": ms, "graph_tokens_per_s": T / (ms / 1e3)}

    clocks = Clocks(local)
    results = {}
    clocks.start()
    for T in Ts:
        results[T] = measure(T)
    ck = clocks.stop()
    if args.copy == "device" and not args.prefetch:
        for T in Ts:
            if min(E, T * k) <= S:
                results[T].update(measure_graph(T))
    head = results[args.T]
    compute_only = measure_compute_only(args.T)
    e2e = measure_e2e(args.T)
    trace = measure_trace(args.T)
    link_gbs = link_probe() if args.copy == "device" else None
    cpu = cpu_baseline(args.cpu_sample_tokens) if (rank == 0 and world == 1) else None
    cpu_all = (cpu_baseline(args.cpu_sample_tokens, threads=os.cpu_count() or 1)
               if (rank == 0 and world == 1) else None)
    if rank == 0:
        line = {
            "metric": METRIC, "value": head["tokens_per_s"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": DTYPE_MX8 if gateup_kernel(args.T, mma_max, mx8_min).startswith("mx8") else DTYPE_MMA,
            "data": "synthetic (seeded generator; no checkpoint weights)",
            "config": {"workload": f"decode layer H=4096 I=2048 E=256 top_k=8 + FP8 shared, 64-slot cache over a pinned "
                                   f"256-expert bank, Zipf(1.1) routing trace, T={args.T}",
                       "T": args.T, "copy": args.copy, "overlap": overlap,
                       "prefetch": (f"{args.prefetch} staging slots, synthetic predictor of the next step "
                                    f"(recall {args.pf_recall})") if args.prefetch else None,
                       "evict": args.evict if args.evict == "lru" else f"lfu (decay every {args.lfu_decay} calls, "
                                                                        "seeded from 64 other trace steps)",
                       "parallelism": "replicas" if world > 1 else "single GPU",
                       "l2": "flushed (256 MB write) before every timed step"},
            "roofline": roofline_hbm(compute_only["kernel"], compute_only["kernel_gbs"],
                                     compute_only["kernel_bytes_per_launch"], compute_only["kernel_ms_per_launch"],
                                     hbm_peak, peak_kind,
                                     "dominant kernel of the decode layer's compute (all experts resident, the "
                                     "timed window's steps, one launch per step); inside the copy-bound step it "
                                     "runs as two passes beside the copy kernel: see roofline_in_step",
                                     workload="decode"),
            "roofline_in_step": {"kernel": head["dominant"], "achieved": head["gateup_gbs"],
                                 "frac": head["gateup_gbs"] / hbm_peak, "unit": "GB/s",
                                 "bytes_per_launch": head["gateup_bytes_per_launch"],
                                 "ms_per_launch": head["gateup_ms"], "launches": head["gateup_launches"]},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": e2e,
            "gpu_launches": head["launches"],
            "clocks": ck,
            "compute_only": compute_only,
            "kernel_sum_tokens_per_s": head["kernel_sum_tokens_per_s"],
            "layer_gbs": head["layer_gbs"],
            "misses_per_step": head["misses_per_step"],
            "h2d_gb_per_step": head["h2d_gb_per_step"],
            "host_link_gbs": head["host_link_gbs"],
            "host_link_probe_gbs": link_gbs,
            "host_link_frac_of_probe": (head["host_link_gbs"] / link_gbs
                                        if head["host_link_gbs"] and link_gbs else None),
            "hit_rate": head["hit_rate"],
            "trace_window": {"timed_steps": [start, start + args.steps], "warmup_steps": [first_warm, start],
                             "replayed_untimed": [0, first_warm], "full_trace": trace},
            "kernel_ms_per_step": head["kernel_ms"],
            "sweep": {str(T): {kk: (round(v, 4) if isinstance(v, float) else v) for kk, v in r.items()
                               if kk not in ("kernel_ms",)} for T, r in results.items()},
        }
        return line
    return None


def run_ours(args):
    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    line = decode_line(args)
    torch.cuda.empty_cache()
    # the other workloads, each under its own key (single GPU, rank 0 only)
    if rank == 0 and world == 1:
        for name in [w.strip() for w in args.extras.split(",") if w.strip()]:
            line[name] = other_entry(args, name)
            torch.cuda.empty_cache()
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def _tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (cuBLAS bf16 burst)"
    except Exception:
        return 1900.0, "fallback"


# Oracle timings of the other workloads on bounded samples (fp64 NumPy, one host
# core): the prefill's first tokens, one ladder step of a few tokens from empty
# pools, one token of one stack layer.
_CPU_OTHER = {
    "prefill": r"""
wl = configs.PREFILL
ids, w = router_topk(gen.router_logits(wl, 0, 0), wl.k)
x = gen.activations(wl, 0, 0)
t0 = time.perf_counter()
moe_layer(x, ids, w, lambda e, tag: F.decode_fp4_expert(gen.fp4_expert(wl, 0, e), wl.H, wl.I),
          tokens=list(range(NTOK)))
dt = time.perf_counter() - t0
print(json.dumps({"tokens": NTOK, "seconds": dt}))
""",
    "ladder": r"""
wl = configs.scaled(configs.LADDER, T=NTOK)
lg = gen.router_logits(wl, 0, 0, NTOK)
x = gen.activations(wl, 0, 0, NTOK)
t0 = time.perf_counter()
ids, w = router_topk(lg, wl.k)
c4, c2 = SlotCacheLRU(wl.S, 1, wl.E), SlotCacheLRU(wl.S2, 1, wl.E)
_, tags, wout, _, _, end = ladder_classify(c4, c2, 0, ids, w, *wl.ladder, 0)
def dec(e, tag):
    if tag == 0:
        return F.decode_fp4_expert(gen.fp4_expert(wl, 0, e), wl.H, wl.I)
    return F.decode_int2_expert(gen.int2_expert(wl, 0, e), wl.H, wl.I)
moe_layer(x, np.where(tags == 2, -1, ids), wout, dec, tags=tags, tokens=list(range(end)))
dt = time.perf_counter() - t0
print(json.dumps({"tokens": end, "seconds": dt}))
""",
    "stack": r"""
wl = configs.STACK
lg = gen.router_logits(wl, 0, 0)
x = gen.activations(wl, 0, 0)
t0 = time.perf_counter()
ids, w = router_topk(lg, wl.k)
shw = F.decode_fp8_expert(gen.shared_expert(wl, 0), wl.H, wl.I)
moe_layer(x, ids, w, lambda e, tag: F.decode_fp4_expert(gen.fp4_expert(wl, 0, e), wl.H, wl.I), shared=shw,
          tokens=list(range(NTOK)))
dt = time.perf_counter() - t0
print(json.dumps({"tokens": NTOK, "seconds": dt}))
""",
}
_CPU_HEAD = r"""
import json, sys, time
sys.path.insert(0, ROOT)
import numpy as np
from oracle import formats as F
from oracle.ladder import ladder_classify
from oracle.mlp import moe_layer
from oracle.router import router_topk
from oracle.slot_cache import SlotCacheLRU
from synth import configs, gen
"""


def cpu_baseline_other(name: str, ntok: int):
    """The oracle on a bounded sample of workload `name`, single-threaded."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = _CPU_HEAD.replace("ROOT", repr(ROOT)) + _CPU_OTHER[name].replace("NTOK", str(ntok))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": "failed: " + (r.stderr.strip().splitlines()[-1][:200] if r.stderr else "")}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    what = {"prefill": f"the first {d['tokens']} tokens of the prefill batch (their experts decoded)",
            "ladder": f"one ladder step of {d['tokens']} tokens from empty pools (classify + MLP)",
            "stack": f"{d['tokens']} token(s) of one stack layer with the shared expert"}[name]
    out = {"value": d["tokens"] / d["seconds"], "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": f"{what}, fp64 NumPy, {d['seconds']:.1f} s single-threaded"}
    if name == "stack":
        # the line's unit is tokens per 43-layer step: the oracle's per-layer rate / 43
        out["value"] = d["tokens"] / d["seconds"] / configs_layers()
        out["sample"] += " (tokens/s of one layer divided by the 43 layers of a step)"
    return out


def configs_layers():
    from synth import configs
    return configs.STACK.layers


def other_entry(args, name):
    """Prefill grouped GEMM, precision-ladder decode, or the 43-layer stack: one
    contract-shaped entry (timed steps, per-kernel breakdown, roofline, oracle
    baseline)."""
    import numpy as np
    import torch

    from moe_expert_offload_router_gb300 import build as B
    B.build()
    import moe_expert_offload_router_gb300 as M
    from synth import configs, gen

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    mma_max, mx8_min = apply_options(M, args)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    hbm_peak, hbm_kind = _peaks()
    out = {"metric": METRIC, "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "data": "synthetic (seeded generator; no checkpoint weights)"}
    clocks = Clocks(0)

    def timed(step_fn, n):
        ev = []
        for i in range(n):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            step_fn(i)
            b.record(stream)
            ev.append((a, b))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / n

    def profiled(step_fn, n):
        """Per-kernel totals of n more steps run with the library's kernel events
        on (kept out of the timed steps)."""
        M.moe_profile_enable(True)
        for i in range(n):
            flush.zero_()
            step_fn(i)
        torch.cuda.synchronize()
        kt = {M.KERNEL_NAMES[kid]: M.moe_profile_query(kid) for kid in range(M.MOE_K_COUNT)}
        M.moe_profile_enable(False)
        return kt

    wl = {"prefill": configs.PREFILL, "ladder": configs.LADDER, "stack": configs.STACK}[name]
    if name == "prefill" and (args.prefill_experts or args.prefill_tokens):
        e = args.prefill_experts or wl.E
        wl = configs.scaled(wl, E=e, S=e, T=args.prefill_tokens or wl.T)
    H, I, E, k, T = wl.H, wl.I, wl.E, wl.k, wl.T
    Bx = M.moe_fp4_expert_bytes(H, I)
    gu4 = 2 * (I * H // 2 + I * H // 32)     # w1 + w3 bytes of an FP4 expert
    if name == "prefill" and args.stream_layers > 0:
        # whole-layer streaming: every layer's experts cross the host link each pass
        nl = args.stream_layers
        bank = torch.empty(nl * E * Bx, dtype=torch.uint8, pin_memory=True)
        for layer in range(nl):
            for e in range(E):
                o = (layer * E + e) * Bx
                bank[o:o + Bx].copy_(gen.fp4_expert(wl, layer, e, device=dev))
        st = M.PrefillStreamer(bank, nl, E, H, I, k, T, dev)
        lg = [torch.from_numpy(gen.router_logits(wl, layer, 0, T)).to(dev) for layer in range(nl)]
        xs = [torch.from_numpy(gen.activations(wl, layer, 0, T).view(np.int16)).to(dev) for layer in range(nl)]
        y = torch.empty((T, H), dtype=torch.int16, device=dev)

        def one_pass(_):
            st.begin(0)
            for layer in range(nl):
                st.run_layer(layer, lg[layer], xs[layer], y)
        for _ in range(args.warmup):
            one_pass(0)
        torch.cuda.synchronize()
        clocks.start()
        ms = timed(one_pass, args.steps)
        ck = clocks.stop()
        kt = profiled(one_pass, args.steps)
        per_layer = ms / nl
        out.update({"value": T / (per_layer / 1e3), "unit": UNIT, "ms_per_step": ms, "clocks": ck,
                    "gpu_launches": sum(v[1] for v in kt.values()),
                    "kernel_ms_per_step": {nm: round(v[0] / args.steps, 4) for nm, v in kt.items() if v[1]},
                    "dtype": "bf16 MMA (fp32 accumulate) on exactly decoded MXFP4 weights",
                    "config": {"workload": f"whole-layer streaming prefill: {nl} layers x (E={E} MXFP4 experts, "
                                           f"H={H} I={I} top_k={k}), T={T} per layer, every layer streamed from "
                                           "the pinned bank through two layer buffers", "T": T, "layers": nl},
                    "ms_per_layer": per_layer,
                    "host_link_gbs": E * Bx / (per_layer / 1e3) / 1e9,
                    "roofline": None})
        return out
    if name in ("prefill", "ladder"):
        bank = torch.empty(E * Bx, dtype=torch.uint8, pin_memory=True)
        for e in range(E):
            bank[e * Bx:(e + 1) * Bx].copy_(gen.fp4_expert(wl, 0, e, device=dev))
        slots = torch.empty(wl.S * Bx, dtype=torch.uint8, device=dev)
        cache = M.moe_cache(wl.S, 1, E, Bx, slots, bank)
        c2, s2 = None, None
        if name == "ladder":
            B2 = M.moe_int2_expert_bytes(H, I)
            bank2 = torch.empty(E * B2, dtype=torch.uint8, pin_memory=True)
            for e in range(E):
                bank2[e * B2:(e + 1) * B2] = torch.from_numpy(gen.int2_expert(wl, 0, e))
            s2 = torch.empty(wl.S2 * B2, dtype=torch.uint8, device=dev)
            c2 = M.moe_cache(wl.S2, 1, E, B2, s2, bank2)
        views = M.make_views(H, I, slots, wl.S, s2, wl.S2 if s2 is not None else 0, None)
        runner = M.DecodeLayerRunner(cache, views, E, k, T, dev, int2_cache=c2, ladder=wl.ladder,
                                     copy=args.copy)
        # ladder: steady state as in the decode workload (untimed replay of the
        # steps before the window); prefill: one batch, all experts resident
        nsteps = max(wl.steps, 1)
        start = min(max(args.window_start, args.warmup), max(nsteps - args.steps, args.warmup)) \
            if name == "ladder" else args.warmup
        n = start + args.steps
        lg = [torch.from_numpy(gen.router_logits(wl, 0, s % nsteps, T)).to(dev) for s in range(n)]
        xs = [torch.from_numpy(gen.activations(wl, 0, s % nsteps, T).view(np.int16)).to(dev) for s in range(n)]
        y = torch.empty((T, H), dtype=torch.int16, device=dev)

        def fresh():
            cache.reset()
            if c2 is not None:
                c2.reset()
            torch.cuda.synchronize()
            for s in range(start):
                runner.run(0, lg[s], xs[s], y)
            torch.cuda.synchronize()
            runner.check()

        fresh()
        m0 = runner.stats["misses"]
        seen = []

        def step(i):
            runner.run(0, lg[start + i], xs[start + i], y)
            seen.append((runner.slots[:T].clone(), runner.tags[:T].clone()) if name == "ladder" else None)
        clocks.start()
        ms = timed(step, args.steps)
        ck = clocks.stop()
        runner.check()
        m1 = runner.stats["misses"]
        fresh()
        kt = profiled(lambda i: runner.run(0, lg[start + i], xs[start + i], y), args.steps)
        runner.check()
        out.update({"value": T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "clocks": ck,
                    "gpu_launches": sum(v[1] for v in kt.values()),
                    "kernel_ms_per_step": {nm: round(v[0] / args.steps, 4) for nm, v in kt.items() if v[1]},
                    "misses_per_step": (m1 - m0) / args.steps})
        if name == "prefill":
            P = T * k
            gu_ms = kt["gemm_gateup"][0] / max(kt["gemm_gateup"][1], 1)
            dn_ms = kt["gemm_down"][0] / max(kt["gemm_down"][1], 1)
            gu_tf = 4.0 * P * H * I / (gu_ms / 1e3) / 1e12
            peak, kind = _tensor_peak()
            floor_ms = 3 * E * (H * I // 2 + H * I // 32) / (hbm_peak * 1e6)
            out["dtype"] = "bf16/fp16 MMA (fp32 accumulate) on exactly decoded MXFP4 weights (W4A16)"
            out["config"] = {"workload": f"prefill grouped GEMM H=4096 I=2048 E={E} top_k=6 T={T}, all {E} "
                                         "experts resident, W4A16", "T": T}
            out["grouped_gemm_tflops"] = 6.0 * P * H * I / ((gu_ms + dn_ms) / 1e3) / 1e12
            gu_bytes = E * gu4 + P * H * 2 + P * I * 2
            traffic, src = ncu_traffic("prefill_gemm_kernel (gate/up)", "prefill", gu_bytes)
            out["roofline"] = {"bound": "tensor", "achieved": gu_tf, "peak": peak, "unit": "TFLOP/s",
                               "frac": gu_tf / peak, "traffic": traffic, "traffic_source": src,
                               "bytes_per_launch": gu_bytes, "kernel": "prefill_gemm_kernel (gate/up)",
                               "peak_kind": kind, "ms_per_launch": gu_ms, "flops_per_launch": 4.0 * P * H * I,
                               "hbm_floor_ms_weights": floor_ms,
                               "step_frac_of_hbm_floor": floor_ms / ms}
            out["cpu_baseline"] = cpu_baseline_other("prefill", 3)
            # the A-quantised mode on the block-scaled FP4 MMA, on the same batch
            # (the runner's slots and router weights of its last step)
            sl, ww = runner.slots[:T].clone(), runner.w[:T].clone()
            ws_mx = torch.empty(M.moe_expert_prefill_workspace(views, T, k), dtype=torch.uint8, device=dev)
            err = torch.zeros(1, dtype=torch.int32, device=dev)

            def mx_step(i):
                M.moe_expert_prefill_prec(views, xs[start], sl, ww, M.MOE_PREC_A_MXFP4, y, ws_mx, err)
            for _ in range(args.warmup):
                mx_step(0)
            torch.cuda.synchronize()
            ms_mx = timed(mx_step, args.steps)
            kmx = profiled(mx_step, args.steps)
            if int(err.item()) != 0:
                raise RuntimeError(f"A-quantised prefill reported status {int(err.item())}")
            fp4_peak = M.moe_fp4_mma_peak(4096)
            mgu = kmx["gemm_gateup"][0] / max(kmx["gemm_gateup"][1], 1)
            mdn = kmx["gemm_down"][0] / max(kmx["gemm_down"][1], 1)
            mgu_tf = 4.0 * P * H * I / (mgu / 1e3) / 1e12
            mdn_tf = 2.0 * P * H * I / (mdn / 1e3) / 1e12
            out["a_mxfp4"] = {
                "ms_per_step": ms_mx, "tokens_per_s": T / (ms_mx / 1e3),
                "note": "activations x and h quantised to MXFP4 (OCP MX, blocks of 32) and multiplied on "
                        "tcgen05.mma.kind::mxf4.block_scale; the expert forward only (the batch's slots given)",
                "kernel_ms_per_step": {nm: round(v[0] / args.steps, 4) for nm, v in kmx.items() if v[1]},
                "gemm_gateup_tflops": mgu_tf, "gemm_down_tflops": mdn_tf,
                "grouped_gemm_tflops": 6.0 * P * H * I / ((mgu + mdn) / 1e3) / 1e12,
                "fp4_peak_tflops": fp4_peak,
                "fp4_peak_kind": "measured in this run: back-to-back kind::mxf4 MMAs (M=128, N=256, K=64) from "
                                 "shared memory on every SM (moe_fp4_mma_peak)",
                "step_frac_of_hbm_floor": floor_ms / ms_mx,
            }
            # algorithmic bytes of the launch: the experts' w1 + w3 codes and scales,
            # x's MXFP4 codes and scales read, h's written
            mx_bytes = E * gu4 + P * (H // 2 + H // 32) + P * (I // 2 + I // 32)
            mx_traffic, mx_src = ncu_traffic("mxf4_gemm_kernel (gate/up)", "prefill", mx_bytes)
            out["roofline_fp4"] = {"bound": "tensor", "achieved": mgu_tf, "peak": fp4_peak, "unit": "TFLOP/s",
                                   "frac": mgu_tf / fp4_peak, "traffic": mx_traffic, "traffic_source": mx_src,
                                   "bytes_per_launch": mx_bytes,
                                   "kernel": "mxf4_gemm_kernel (gate/up)", "peak_kind": out["a_mxfp4"]["fp4_peak_kind"],
                                   "ms_per_launch": mgu, "flops_per_launch": 4.0 * P * H * I}
        else:
            # touched bytes of the timed steps: each pool's distinct slots of kept pairs
            B2 = M.moe_int2_expert_bytes(H, I)
            gu2 = 2 * (I * H // 4 + I * H // 32)
            lay_b, gu_b = 0, 0
            kname = gateup_kernel(T, mma_max, mx8_min)
            for sl, tg in seen:
                sl, tg = sl.cpu().numpy(), tg.cpu().numpy()
                d4 = len(np.unique(sl[(tg == 0) & (sl >= 0)]))
                d2 = len(np.unique(sl[(tg == 1) & (sl >= 0)]))
                lay_b += d4 * Bx + d2 * B2 + 2 * T * H * 2
                gu_b += d4 * gu4 + d2 * gu2 + gateup_io_bytes(kname, T, k, H, I)
            gu_ms, gu_n = kt["gateup"]
            gu_bytes = gu_b / max(gu_n, 1)
            gu_gbs = gu_bytes / (gu_ms / max(gu_n, 1) / 1e3) / 1e9
            out["dtype"] = ("FP4 pairs: " + (DTYPE_MX8 if kname.startswith("mx8") else DTYPE_MMA) +
                            "; 2-bit pairs: e4m3-scaled 2-bit weights, fp16 products, fp32 accumulate")
            out["config"] = {"workload": "ladder (2,4) decode H=4096 I=2048 E=256 top_k=6 T=32, 96 FP4 + "
                                         "192 2-bit slots, Zipf(1.1) trace", "T": T,
                             "timed_steps": [start, start + args.steps]}
            out["layer_gbs"] = lay_b / args.steps / (ms / 1e3) / 1e9
            # every launch of the gate/up scope (the warp-MMA kernel for the FP4
            # pairs and the CUDA-core kernel for the 2-bit ones share it)
            out["roofline"] = roofline_hbm(f"gateup ({kname} + gateup_kernel)", gu_gbs, gu_bytes,
                                           gu_ms / max(gu_n, 1), hbm_peak, hbm_kind,
                                           "the gate/up kernels of the ladder's steps: touched FP4 and 2-bit "
                                           "experts' w1/w3, x and h")
            out["cpu_baseline"] = cpu_baseline_other("ladder", 4)
        return out
    # 43-layer stack, every expert resident, no host sync per layer
    L = wl.layers
    S = L * E
    pool = torch.empty(S * Bx, dtype=torch.uint8, device=dev)
    for layer in range(L):
        for e in range(E):
            key = layer * E + e
            pool[key * Bx:(key + 1) * Bx] = gen.fp4_expert(wl, layer, e, device=dev)
    cache = M.moe_cache(S, L, E, Bx, pool, None)
    cache.import_(np.arange(S, dtype=np.int32), np.arange(S, dtype=np.uint64), S)
    shared = [torch.from_numpy(gen.shared_expert(wl, layer)).to(dev) for layer in range(L)]
    views = [M.make_views(H, I, pool, S, None, 0, shared[layer]) for layer in range(L)]
    runners = [M.DecodeLayerRunner(cache, views[layer], E, k, T, dev, assume_resident=True)
               for layer in range(L)]
    for r in runners[1:]:
        r.ws = runners[0].ws
    n = args.warmup + args.steps
    lg = [[torch.from_numpy(gen.router_logits(wl, layer, s % wl.steps, T)).to(dev) for layer in range(L)]
          for s in range(n)]
    x0 = torch.from_numpy(gen.activations(wl, 0, 0, T).view(np.int16)).to(dev)
    ya = torch.empty((T, H), dtype=torch.int16, device=dev)
    xb = torch.empty((T, H), dtype=torch.int16, device=dev)

    def step(s):
        x = x0
        for layer in range(L):
            runners[layer].run(layer, lg[s][layer], x, ya)
            M.moe_rms_carry(ya, 1e-6, xb)
            x = xb

    for s in range(args.warmup):
        step(s)
    torch.cuda.synchronize()
    clocks.start()
    ms = timed(lambda i: step(args.warmup + i), args.steps)
    ck = clocks.stop()
    kt = profiled(lambda i: step(args.warmup + i), args.steps)
    # touched bytes per step: distinct experts per layer
    tb, gub = 0, 0
    kname = gateup_kernel(T, mma_max, mx8_min)
    fp8 = M.moe_fp8_expert_bytes(H, I)
    gu8 = 2 * (I * H + I * 4)
    for s in range(args.warmup, n):
        for layer in range(L):
            ids, _ = M.moe_router_topk(lg[s][layer], k)
            d = int(torch.unique(ids).numel())
            tb += d * Bx + fp8
            gub += d * gu4 + gu8 + gateup_io_bytes(kname, T, k, H, I)
    gbs = tb / args.steps / (ms / 1e3) / 1e9
    gu_ms, gu_n = kt["gateup"]
    gu_bytes = gub / max(gu_n, 1)
    gu_gbs = gu_bytes / (gu_ms / max(gu_n, 1) / 1e3) / 1e9
    out.update({"value": T / (ms / 1e3), "unit": UNIT, "ms_per_step": ms, "clocks": ck,
                "dtype": DTYPE_MX8 if kname.startswith("mx8") else DTYPE_MMA,
                "config": {"workload": "43-layer stack decode, 256 FP4 experts + FP8 shared per layer, all "
                                       "resident (148 GB), T=16, 70% step-to-step reuse", "T": T, "layers": L},
                "stack_hbm_gbs": gbs, "hbm_frac_of_step": gbs / hbm_peak,
                "gpu_launches": sum(v[1] for v in kt.values()),
                "kernel_ms_per_step": {nm: round(v[0] / args.steps, 4) for nm, v in kt.items() if v[1]},
                "roofline": roofline_hbm(kname, gu_gbs,
                                         gu_bytes, gu_ms / max(gu_n, 1), hbm_peak, hbm_kind,
                                         "gate/up kernel of each layer: touched experts' w1/w3, the shared "
                                         "expert's, x and h"),
                "cpu_baseline": cpu_baseline_other("stack", 1)})
    del pool
    return out


def run_other(args):
    print(json.dumps(other_entry(args, args.workload)))


def run_forward(args):
    """Router + ensure + expert forward of the decode layer at T = args.T with every
    expert resident (3.4 GB on the device), L2 flushed between steps."""
    import numpy as np
    import torch

    from moe_expert_offload_router_gb300 import build as B
    B.build()
    import moe_expert_offload_router_gb300 as M
    from synth import configs, gen

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    apply_options(M, args)
    wl = configs.scaled(configs.DECODE, T=args.T)
    H, I, E, k, T = wl.H, wl.I, wl.E, wl.k, wl.T
    Bx = M.moe_fp4_expert_bytes(H, I)
    pool = torch.empty(E * Bx, dtype=torch.uint8, device=dev)
    for e in range(E):
        pool[e * Bx:(e + 1) * Bx] = gen.fp4_expert(wl, 0, e, device=dev)
    cache = M.moe_cache(E, 1, E, Bx, pool, None)
    cache.import_(np.arange(E, dtype=np.int32), np.arange(E, dtype=np.uint64), E)
    shared = torch.from_numpy(gen.shared_expert(wl, 0)).to(dev)
    views = M.make_views(H, I, pool, E, None, 0, shared)
    runner = M.DecodeLayerRunner(cache, views, E, k, T, dev, assume_resident=True)
    n = args.warmup + args.steps
    lg = [torch.from_numpy(gen.router_logits(wl, 0, s % wl.steps, T)).to(dev) for s in range(n)]
    xs = [torch.from_numpy(gen.activations(wl, 0, s % wl.steps, T).view(np.int16)).to(dev) for s in range(n)]
    y = torch.empty((T, H), dtype=torch.int16, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for s in range(args.warmup):
        runner.run(0, lg[s], xs[s], y)
    torch.cuda.synchronize()
    ev, seen = [], []
    for i in range(args.steps):
        s = args.warmup + i
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        runner.run(0, lg[s], xs[s], y)
        b.record(stream)
        ev.append((a, b))
        seen.append(runner.ids[:T].clone())
    torch.cuda.synchronize()
    ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    nbytes = sum(int(torch.unique(ids).numel()) * Bx + M.moe_fp8_expert_bytes(H, I) + 2 * T * H * 2 for ids in seen)
    gbs = nbytes / args.steps / (ms / 1e3) / 1e9
    hbm_peak, _ = _peaks()
    cache.close()
    print(json.dumps({"metric": METRIC, "value": T / (ms / 1e3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
                      "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                      "vs_baseline": None, "data": "synthetic (seeded generator; no checkpoint weights)",
                      "config": {"workload": f"decode layer compute alone (router, ensure, expert MLP), all {E} "
                                             f"experts resident, T={T}", "T": T},
                      "layer_hbm_gbs": gbs, "frac_of_hbm": gbs / hbm_peak}))


def run_reference(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # every step is a bounded sample of the decode workload: T tokens of one
    # trace step (one or two, so that the --warmup + --steps run stays within
    # a few minutes of host time: ~0.5-1 s per token-step)
    K, W = max(1, args.steps), max(0, args.warmup)
    T = max(1, min(args.cpu_sample_tokens, 2 if K + W <= 60 else 1))
    d = _run_oracle(T, K, 1, warm=W)
    if isinstance(d, str):
        print(json.dumps({"impl": "reference", "unavailable": d}))
        return
    per = d["step_seconds"]
    ms = 1e3 * sum(per) / len(per)
    value = T / (ms / 1e3)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
        "config": {"workload": f"decode layer H=4096 I=2048 E=256 top_k=8 + FP8 shared, 64-slot cache, "
                               f"Zipf(1.1) routing trace, bounded sample of T={T} tokens per step"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"{W} untimed + {K} timed trace steps x {T} tokens, single-threaded fp64 NumPy"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


if __name__ == "__main__":
    a = _args()
    if a.impl == "reference":
        run_reference(a)
    elif a.workload == "decode":
        run_ours(a)
    elif a.workload == "forward":
        run_forward(a)
    else:
        run_other(a)
