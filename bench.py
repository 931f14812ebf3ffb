#!/usr/bin/env python
"""Benchmark of DARTree supertree builds on one GB300 (or N replicas).

A step is one full build: D batched head calls (state step, fused corrected
logits + log-softmax + top-K, row merge, top-W select) and the deferred
Top-B + mask, over seeded synthetic inputs of the chosen workload.  Prints
one JSON line (rank 0).

  python bench.py [--config q8b] [--steps K] [--warmup W] [--gpus N]
  python bench.py --impl reference ...    # the CPU oracle, timed as stated
  python bench.py --variant markov|base|bestfirst ...   # a build variant

The default line is the depth-wise DARTree build; --variant measures one of
the build variants (Markov correction head, base-logit candidates, the
sequential best-first baseline) on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

_ROOT = os.path.dirname(os.path.abspath(__file__))
if _ROOT not in sys.path:
    sys.path.insert(0, _ROOT)

from speculative_decoding_draft_06_gb300 import inputs as I  # noqa: E402

DEFAULT_CONFIG = "q8b"
FALLBACK_HBM_GBS = 6800.0
ROWS_MIN = 64  # head calls with this many rows run k_head_rows (the library's default)
KERNEL_SOURCES = ("speculative_decoding_draft_06_gb300/csrc/head_tc.cu",
                  "speculative_decoding_draft_06_gb300/csrc/epilogue.cuh",
                  "speculative_decoding_draft_06_gb300/csrc/ptx.cuh",
                  "speculative_decoding_draft_06_gb300/csrc/common.cuh",
                  "speculative_decoding_draft_06_gb300/csrc/head_rows.cu")


def parse_args(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("dartree", "reference"), default="dartree")
    ap.add_argument("--config", choices=sorted(I.CONFIGS), default=DEFAULT_CONFIG)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--profile-head", type=int, default=0, metavar="N",
                    help="profiling aid: run N head calls (fused logits + log-softmax + "
                         "top-K) of the workload's widest depth and exit")
    ap.add_argument("--vocab", type=int, default=0,
                    help="override V (profiling aid for small ncu captures)")
    ap.add_argument("--variant", choices=sorted(VARIANTS), default="dartree")
    ap.add_argument("--wout-layout", choices=("auto", "blocks", "rows"), default="auto",
                    help="layout of the output projection in HBM (bf16): blocks of 128 x 64 "
                         "(converted once before timing), row-major, or auto: blocks where "
                         "the head calls stream it, rows where the base-logit candidates "
                         "gather whole rows of it")
    return ap.parse_args(argv)


def prepare_wout(ctx, dev: dict, bf16: bool, layout: str, variant: str = "dartree") -> str:
    """Puts the output projection in the layout the context will read:
    converted once, before any timing (the weights do not change between
    builds).  auto: the blocked layout, except for the base-logit candidate
    variants, whose K gathered rows per head row are contiguous only
    row-major (measured: 2757 vs 2620 builds/s).  Returns the layout used."""
    from speculative_decoding_draft_06_gb300 import dartree as dtl
    if layout == "auto":
        layout = "rows" if VARIANTS.get(variant, {}).get("candidates") == "base" else "blocks"
    if not bf16 or layout == "rows":
        return "rows"
    if not dev.get("wout_blocked"):
        dev["Wout"] = dtl.block_weights(dev["Wout"])
        dev["wout_blocked"] = True
    ctx.set_weight_layout("blocks")
    return "blocks of 128 x 64 (converted once before timing)"


# build variants: options of DARTree.build
VARIANTS = {
    "dartree": {},
    "markov": {"head": "markov"},
    "base": {"candidates": "base"},
    "markov-base": {"head": "markov", "candidates": "base"},
    "bestfirst": {"expansion": "bestfirst"},
    "verify": {},    # the default build followed by the verification consumer
}


# ------------------------------------------------------------- bookkeeping

def build_bytes(w: I.Workload, variant: str = "dartree") -> float:
    """Algorithmic bytes of one build: D output projections, D-1 state
    matrices, the gathered embedding rows and all base logits (per variant:
    no state matrix for the Markov head; K gathered Wout rows per request
    instead of the projection for base candidates; B head calls of one row
    per request for best-first)."""
    wb = 2 if w.bf16 else 4
    rows = w.head_rows()
    opt = VARIANTS[variant]
    if opt.get("expansion") == "bestfirst":
        return (w.B * (w.V * w.H * wb + w.R * w.V * 4 + w.R * w.H * wb)
                + (w.B - 1) * (w.H * w.H * wb + 2 * w.R * w.H * wb))
    state = 0 if opt.get("head") == "markov" else (w.D - 1) * w.H * w.H * wb
    gathered = sum(rows[1:]) * w.H * wb
    if opt.get("candidates") == "base":
        return (w.D * (w.R * w.K * w.H * wb + max(rows) * w.H * wb) + state + gathered
                + w.R * w.D * w.V * 4)
    return w.D * w.V * w.H * wb + state + gathered + w.R * w.D * w.V * 4


def kernel_bytes_per_launch(w: I.Workload, variant: str, kind: str) -> float | None:
    """Algorithmic bytes of one launch of kernel kind `kind` (averaged over a
    build's launches of that kind), or None where no byte count bounds it."""
    wb = 2 if w.bf16 else 4
    opt = VARIANTS[variant]
    rows = [w.R] * w.B if opt.get("expansion") == "bestfirst" else w.head_rows()
    if kind == "head":
        if opt.get("candidates") == "base":
            per = [w.R * w.K * w.H * wb + m * w.H * wb + w.R * w.K * 4 for m in rows]
        else:
            per = [w.V * w.H * wb + w.R * w.V * 4 + m * w.H * wb for m in rows]
            if not w.bf16 and not opt and w.H % 4 == 0 and f32_head_fits(w.H, w.K):
                # fp32 head calls of at most 16 rows with a next depth also
                # stream A (the folded state contraction)
                per = [b + (w.H * w.H * 4 if m <= 16 and d < w.D else 0)
                       for d, (b, m) in enumerate(zip(per, rows), start=1)]
        return sum(per) / len(per)
    if kind == "state":
        # parent states in, the tokens' embedding rows, new states out (+ A)
        per = [3 * m * w.H * wb + (0 if opt.get("head") == "markov" else w.H * w.H * wb)
               for m in rows[1:]]
        return sum(per) / len(per) if per else None
    if kind == "candidates":
        return w.R * w.D * w.V * 4
    return None


def kernels_per_build(w: I.Workload, variant: str = "dartree", sms: int = 152) -> int:
    opt = VARIANTS[variant]
    # a bf16 state step splits its contraction over the SMs and then runs a
    # finish kernel; the Markov head's step is one kernel
    tiles = -(-w.H // 128)
    state = 2 if (w.bf16 and opt.get("head") != "markov" and sms // tiles > 1) else 1
    if opt.get("expansion") == "bestfirst":      # root, init, B x (head, merge, step), states
        return 2 + 3 * w.B + (w.B - 1) * state
    base = 1 if opt.get("candidates") == "base" else 0
    # fp32 head calls of at most 16 rows (k_head_f32) also compute the next
    # state contraction, and their selection finishes the step: no launch
    folded = 0
    if not w.bf16 and not opt and w.H % 4 == 0 and f32_head_fits(w.H, w.K):
        folded = sum(1 for m in w.head_rows()[:-1] if m <= 16)
    # root, head + merge/select, states, prune
    return 1 + base + w.D * 2 + (w.D - 1 - folded) * state + 1


def f32_head_fits(H: int, K: int) -> bool:
    """Shared memory of k_head_f32 (head rows, two tile-sum buffers, the
    16-row epilogue) within its 200 KB."""
    ld = -(-H // 256) * 256
    epi = 16 * K * 8 + 2 * 16 * 132 * 4 + 4 * 16 * 8 + 4 * 32 * 8
    return 16 * ld * 4 + 2 * 128 * 17 * 4 + epi <= 200 * 1024


def _code_only(text: str) -> str:
    """The source without comments and layout: the hash follows code only."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(_ROOT, f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> tuple[float, str]:
    p = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(config: str) -> float | None:
    """DRAM bytes per head-call launch from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(_ROOT, "profiles", f"head_logits_{config}.md")
    try:
        txt = open(p).read()
    except OSError:
        return None
    vals = {}
    for line in txt.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("kernel_source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


def aggregate(ms_local: float, world: int) -> float:
    """Max of the per-rank step time over all ranks (torch.distributed)."""
    if world <= 1:
        return ms_local
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_local], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_max: float, world: int, requests: int) -> float:
    """Whole-job builds/s: every rank builds `requests` trees per step and the
    step time is the slowest rank's (weak scaling, no data-path collective)."""
    return world * requests * 1e3 / ms_max


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "0").split(",")[0] or "0"
        self.idx = vis
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}",
                                       "--format=csv,noheader,nounits", "-lms", "200",
                                       "-i", self.idx],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                      text=True)
        except OSError:
            self.p = None

    def stop(self) -> dict | None:
        if self.p is None:
            return None
        self.p.terminate()
        try:
            out, _ = self.p.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.p.kill()
            out, _ = self.p.communicate()
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- CPU oracle

def host_info() -> dict:
    """Host cores and CPU model of the machine the oracle is timed on."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    return {"host_cores": os.cpu_count(), "cpu_model": model}


class PinnedCore:
    """Runs the enclosed oracle work on one core (the calling thread's
    affinity), restoring the previous affinity afterwards."""

    def __init__(self):
        self.core = None
        self.prev = None

    def __enter__(self):
        try:
            self.prev = os.sched_getaffinity(0)
            self.core = max(self.prev)           # the last allowed core
            os.sched_setaffinity(0, {self.core})
        except (AttributeError, OSError):
            self.core = None
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            try:
                os.sched_setaffinity(0, self.prev)
            except OSError:
                pass
        return False


def oracle_sample(w: I.Workload, inp: dict, budget_s: float, request: int = 0,
                  variant: str = "dartree") -> dict:
    """Time the CPU oracle on a bounded sample of one request's build.

    Returns the measured seconds, the fraction of one build the sample
    covers and builds/s = fraction / seconds.  The sample is the whole build
    when it fits in budget_s (then nothing is extrapolated), else the first
    depths of the build (fraction = their head rows over the build's: the
    dominant cost is one V x H fp64 pass per head row), else one head row
    restricted to a vocabulary slice.  Best-first: a build with fewer calls.
    Base candidates: the first depths of the variant's own oracle build."""
    import oracle
    opt = VARIANTS[variant]
    markov = opt.get("head") == "markov"
    if opt.get("candidates") == "base":
        d_s, t = 0, 0.0
        while d_s < w.D and t * (d_s + 1) / max(1, d_s) <= budget_s:
            d_s += 1
            t0 = time.perf_counter()
            oracle.build_tree(inp, request, d_s, w.W, w.K, w.bf16, markov=markov,
                              cand_base=True)
            t = time.perf_counter() - t0
        frac = d_s / w.D
        return {"seconds": t, "fraction": frac, "builds_per_s": frac / t,
                "extrapolated": d_s < w.D,
                "sample": (f"oracle (fp64, 1 thread), base-candidate build of depths 1..{d_s} "
                           f"of {w.D} of request {request} ({t:.2f} s)")}
    if opt.get("expansion") == "bestfirst":
        rows = [1] * w.B
    else:
        rows = [m // w.R for m in w.head_rows()]   # head rows per request per depth
    total_rows = sum(rows)
    s0 = inp["state0"][request]
    vs = min(w.V, 4096)
    t0 = time.perf_counter()
    oracle.logits_row(inp["z"][request, 0, :vs], inp["Wout"][:vs], s0, w.bf16)
    t_row = (time.perf_counter() - t0) * w.V / vs  # estimated cost of one full row
    if t_row > budget_s:
        vs = max(256, min(w.V, int(w.V * budget_s / t_row)))
        t0 = time.perf_counter()
        oracle.logits_row(inp["z"][request, 0, :vs], inp["Wout"][:vs], s0, w.bf16)
        t = time.perf_counter() - t0
        frac = vs / w.V / total_rows
        return {"seconds": t, "fraction": frac, "builds_per_s": frac / t, "extrapolated": True,
                "sample": (f"oracle (fp64, 1 thread): one head row over {vs} of {w.V} "
                           f"vocabulary entries ({t:.2f} s) = {frac:.2e} of a build of "
                           f"{total_rows} head rows")}
    if opt.get("expansion") == "bestfirst":
        n = max(1, min(w.B, int(budget_s / t_row)))
        t0 = time.perf_counter()
        o = oracle.bestfirst(inp, request, w.D, w.K, n, w.beta, w.bf16, markov=markov)
        t = time.perf_counter() - t0
        frac = o["calls"] / w.B
        return {"seconds": t, "fraction": frac, "builds_per_s": frac / t,
                "extrapolated": n < w.B,
                "sample": (f"oracle (fp64, 1 thread): best-first build with budget {n} of "
                           f"{w.B}, request {request} ({o['calls']} head calls, {t:.1f} s)")}
    d_s, acc = 1, rows[0]
    while d_s < w.D and (acc + rows[d_s]) * t_row <= budget_s:
        acc += rows[d_s]
        d_s += 1
    t0 = time.perf_counter()
    if d_s == w.D:
        oracle.build_request(inp, request, w.D, w.W, w.K, w.B, w.beta, w.bf16)
    else:
        oracle.build_tree(inp, request, d_s, w.W, w.K, w.bf16, markov=markov)
    t = time.perf_counter() - t0
    frac = acc / total_rows
    whole = d_s == w.D
    return {"seconds": t, "fraction": frac, "builds_per_s": frac / t, "extrapolated": not whole,
            "sample": (f"oracle (fp64, 1 thread): the whole build of request {request} incl. "
                       f"Top-B and mask ({t:.2f} s)" if whole else
                       f"oracle (fp64, 1 thread) on depths 1..{d_s} of {w.D} of request "
                       f"{request} ({acc} of {total_rows} head rows, {t:.1f} s)")}


def cpu_baseline(w: I.Workload, inp: dict, budget_s: float, variant: str) -> dict:
    """The oracle on one pinned host core: a bounded sample of this workload,
    plus (for other workloads) one whole tiny build timed directly."""
    info = host_info()
    with PinnedCore() as pc:
        s = oracle_sample(w, inp, budget_s, variant=variant)
        direct = None
        if w.name != "tiny" or s["extrapolated"]:
            import oracle
            t = I.CONFIGS["tiny"]
            ti = I.make_inputs(t)
            t0 = time.perf_counter()
            oracle.build_request(ti, 0, t.D, t.W, t.K, t.B, t.beta, t.bf16)
            sec = time.perf_counter() - t0
            direct = {"workload": "tiny", "seconds": sec, "builds_per_s": 1.0 / sec}
    return {"value": s["builds_per_s"], "unit": "builds/s", "cores": 1, "kind": "oracle",
            "sample": s["sample"], "extrapolated": s["extrapolated"],
            "sample_seconds": s["seconds"], "sample_build_fraction": s["fraction"],
            "pinned_core": pc.core, **info, "direct_full_build": direct}


# -------------------------------------------------------------- reference arm

def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = I.CONFIGS[args.config]
    inp = I.make_inputs(w)
    budget = max(0.5, 150.0 / max(1, args.steps + args.warmup))
    info = host_info()
    with PinnedCore() as pc:
        for _ in range(args.warmup):
            oracle_sample(w, inp, budget, variant=args.variant)
        vals = [oracle_sample(w, inp, budget, variant=args.variant) for _ in range(args.steps)]
    sec = sum(v["seconds"] for v in vals)
    frac = sum(v["fraction"] for v in vals)
    value = frac / sec                   # builds of work done per second of oracle time
    line = {
        "impl": "reference", "metric": "supertree builds/s", "value": value,
        "unit": "builds/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec / len(vals) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w), "variant": args.variant,
        "step": (f"a bounded sample of the workload: {frac / len(vals):.3g} of one build per "
                 f"step (measured seconds; value = build fraction / seconds)"),
        "cpu_baseline": {"value": value, "unit": "builds/s", "cores": 1, "kind": "oracle",
                         "sample": vals[-1]["sample"],
                         "extrapolated": any(v["extrapolated"] for v in vals),
                         "pinned_core": pc.core, **info},
        "e2e": {"value": value, "unit": "builds/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(w: I.Workload) -> dict:
    return {"workload": (f"{w.name}: V={w.V} H={w.H} D={w.D} W={w.W} K={w.K} B={w.B} "
                         f"beta={w.beta} R={w.R} {'bf16' if w.bf16 else 'fp32'} weights"),
            "R": w.R, "V": w.V, "H": w.H, "D": w.D, "W": w.W, "K": w.K, "B": w.B,
            "beta": w.beta, "weights": "bf16" if w.bf16 else "fp32",
            "l2": ("inputs larger than L2: the output projection is streamed from HBM once per "
                   "head call" if w.V * w.H * (2 if w.bf16 else 4) > 129e6 else
                   "L2-resident (weights fit in L2); no flush between steps")}


# -------------------------------------------------------------- GPU arm

def run_gpu(args) -> None:
    import torch

    from speculative_decoding_draft_06_gb300 import dartree as dtl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    w = I.CONFIGS[args.config]
    if world > 1:   # replicas: every rank builds its own requests
        w = w.replace(seed=w.seed + 7919 * rank)
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    ctx = dtl.DARTree(w.V, w.H, max_D=w.D, max_W=w.W, max_K=w.K, max_B=w.B,
                      max_requests=w.R, bf16=w.bf16)
    layout = prepare_wout(ctx, dev, w.bf16, args.wout_layout, args.variant)
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    opt = VARIANTS[args.variant]
    kw = dict(D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta, out=out, stream=stream, **opt)
    args_t = (dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"])

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # warm-up, then the timed region (device events on the build stream)
    for _ in range(max(3, args.warmup)):
        ctx.build(*args_t, **kw)
    ctx.sync(stream)
    barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        ctx.build(*args_t, **kw)
    e1.record(stream)
    e1.synchronize()
    clock_info = clocks.stop()
    ctx.sync(stream)
    torch.cuda.synchronize()
    barrier()
    ms_local = e0.elapsed_time(e1) / args.steps
    ms = aggregate(ms_local, world)
    value = job_value(ms, world, w.R)

    # per-kernel durations (events around each launch, same stream)
    ctx.set_timing(True)
    ctx.reset_timing()
    for _ in range(min(args.steps, 50)):
        ctx.build(*args_t, **kw)
        ctx.sync(stream)
    kt = ctx.timing()
    ctx.set_timing(False)
    # the dominant kernel: the head call of the default build; for a variant
    # the kind with the most device time among those with a byte count
    kind = "head"
    if args.variant != "dartree":
        kind = max((k for k in ("head", "state", "candidates")
                    if kernel_bytes_per_launch(w, args.variant, k) and kt[k][1]),
                   key=lambda k: kt[k][0])
    k_ms, k_n = kt[kind]
    head_avg_ms = k_ms / max(1, k_n)
    peak, peak_kind = measured_peaks()
    bytes_launch = kernel_bytes_per_launch(w, args.variant, kind)
    achieved = bytes_launch / (head_avg_ms * 1e-3) / 1e9
    traffic = profiled_traffic(args.config) if args.variant == "dartree" else None
    traffic_source = (f"ncu dram__bytes_read.sum + dram__bytes_write.sum per head launch, "
                      f"profiles/head_logits_{args.config}.md @ kernel_source_hash "
                      f"{kernel_source_hash()}" if traffic is not None else
                      "none: no ncu capture on the current kernel sources for this workload")
    big = [m for m in w.head_rows() if m >= ROWS_MIN]
    kernel_name = {
        "head": ("k_cand_logits (candidate logits)" if opt.get("candidates") == "base" else
                 ("k_head_f32 (fp32 head call, at most 16 rows: 16 dot-product warps, 4 epilogue "
                  "warps; also the next state contraction)"
                  if not w.bf16 and max(w.head_rows()) <= 16 and w.H % 4 == 0
                  and f32_head_fits(w.H, w.K) else "k_head_simt (fp32 head call)")
                 if not w.bf16 else
                 "k_head_tc (head call: Wout stream, fused log-softmax + top-K)" if not big else
                 f"k_head_rows (head call, {max(big)} head rows on the MMA M side: Wout stream, "
                 f"fused log-softmax + top-K; calls with fewer than {ROWS_MIN} rows: k_head_tc)"),
        "state": ("k_state_markov" if opt.get("head") == "markov" else
                  "k_head_tc + k_state_finish (state step: A stream, split-K, finish)"),
        "candidates": "k_base_topk (top-K of the base logits)"}[kind]

    # the same head launches against the tensor roofline (their flops are
    # fixed by the head rows: a few at 16 rows, at the ridge at 256)
    tensor_line = None
    fl = head_flops_per_launch(w, args.variant) if kind == "head" else None
    if fl:
        tpk, tpk_kind = measured_bf16_tflops(sustained=True)
        ach = fl / (head_avg_ms * 1e-3) / 1e12
        tensor_line = {"achieved": ach, "peak": tpk, "unit": "TFLOP/s", "frac": ach / tpk,
                       "peak_source": f"{tpk_kind} (sustained dense bf16)",
                       "flops_per_launch": fl}

    # a projection that fits in L2 is re-read from L2 by every head call: its
    # HBM fraction bounds nothing, so the line also gives the fraction of an
    # L2-resident copy measured here (two 24 MB buffers, events)
    l2_line = None
    w_bytes = w.V * w.H * (2 if w.bf16 else 4)
    if kind == "head" and w_bytes <= 64e6:
        a = torch.empty(6 << 20, dtype=torch.float32, device="cuda")
        b = torch.empty_like(a)
        for _ in range(20):
            b.copy_(a)
        torch.cuda.synchronize()
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record()
        for _ in range(200):
            b.copy_(a)
        c1.record()
        c1.synchronize()
        l2_gbs = 2 * a.numel() * 4 * 200 / (c0.elapsed_time(c1) * 1e-3) / 1e9
        l2_line = {"achieved": achieved, "peak": l2_gbs, "unit": "GB/s", "frac": achieved / l2_gbs,
                   "peak_source": "measured in this run: copy of a 24 MB fp32 buffer (L2-resident), "
                                  "read + write bytes",
                   "note": (f"the {w_bytes / 1e6:.1f} MB projection stays in L2 between head "
                            "calls; the call is latency-bound (a short chain of load rounds "
                            "and the fused epilogue), not bound by a pipe")}
        del a, b

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and args.variant != "dartree":
        # host inputs -> device, build, tree -> host, through the public API
        zh = torch.from_numpy(inp["z"]).pin_memory()
        sh = torch.from_numpy(inp["state0"]).pin_memory()
        oh = ctx.alloc_tree(w.R, w.B, device="cpu", pin=True)

        def step_host():
            with torch.cuda.stream(stream):
                dev["z"].copy_(zh, non_blocking=True)
                dev["state0"].copy_(sh, non_blocking=True)
                ctx.build(*args_t, **kw)
                for k in oh:
                    oh[k].copy_(out[k], non_blocking=True)
            ctx.sync(stream)
        for _ in range(max(3, args.warmup)):
            step_host()
        barrier()
        n_e2e = max(5, min(args.steps, 100))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            step_host()
        t_e2e = aggregate((time.perf_counter() - t0) / n_e2e * 1e3, world)
        e2e = {"value": world * w.R * 1e3 / t_e2e, "unit": "builds/s",
               "h2d_bytes_per_step": int(zh.numel() * 4 + sh.numel() * 4),
               "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in oh.values())),
               "ms_per_step": t_e2e}
    elif not args.no_e2e:
        zh = torch.from_numpy(inp["z"]).pin_memory()
        sh = torch.from_numpy(inp["state0"]).pin_memory()
        oh = ctx.alloc_tree(w.R, w.B, device="cpu", pin=True)
        for _ in range(max(3, args.warmup)):
            ctx.build_host(zh, sh, dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W, K=w.K, B=w.B,
                           beta=w.beta, out_host=oh, stream=stream)
        barrier()
        n_e2e = max(5, min(args.steps, 100))
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            ctx.build_host(zh, sh, dev["A"], dev["E"], dev["Wout"], D=w.D, W=w.W, K=w.K,
                           B=w.B, beta=w.beta, out_host=oh, stream=stream)
        t_e2e = (time.perf_counter() - t0) / n_e2e * 1e3
        t_e2e = aggregate(t_e2e, world)
        e2e = {"value": world * w.R * 1e3 / t_e2e, "unit": "builds/s",
               "h2d_bytes_per_step": int(zh.numel() * 4 + sh.numel() * 4),
               "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in oh.values())),
               "ms_per_step": t_e2e}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, inp, args.cpu_budget, args.variant)

    if rank == 0:
        line = {
            "metric": "supertree builds/s", "value": value, "unit": "builds/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.bf16 else "f32", "data": "synthetic",
            "config": dict(workload_config(w), wout_layout=layout),
            "variant": args.variant,
            "head_calls_per_build": ctx.head_calls(),
            "nodes_scored_per_s": (value / w.R * w.candidates_per_build()
                                   if args.variant != "bestfirst" else None),
            "path_GBps_per_gpu": build_bytes(w, args.variant) * (value / world / w.R) / 1e9,
            "roofline": {"bound": "hbm", "kernel": kernel_name,
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_source": peak_kind,
                         "traffic": traffic, "traffic_source": traffic_source,
                         "bytes_per_launch": bytes_launch, "launch_ms": head_avg_ms},
            "tensor": tensor_line,
            "l2": l2_line,
            "kernel_ms_per_build": {k: v[0] / max(1, min(args.steps, 50)) for k, v in kt.items()},
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": kernels_per_build(w, args.variant) * args.steps,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def measured_bf16_tflops(sustained: bool = False) -> tuple[float, str]:
    """Measured dense bf16 peak: the burst figure for a kernel timed alone,
    the sustained one for a kernel timed inside a long step."""
    p = os.path.join(_ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(p) as f:
            return float(json.load(f)[key]), "measured"
    except (OSError, KeyError, ValueError):
        return (1700.0 if sustained else 1900.0), "fallback"


def head_flops_per_launch(w: I.Workload, variant: str) -> float | None:
    """Tensor flops of one head call (2 M V H), averaged over a build's calls;
    None where the head call is not a dense contraction over the vocabulary."""
    opt = VARIANTS[variant]
    if opt.get("candidates") == "base" or not w.bf16:
        return None
    rows = [w.R] * w.B if opt.get("expansion") == "bestfirst" else w.head_rows()
    return sum(2.0 * m * w.V * w.H for m in rows) / len(rows)


def run_verify(args) -> None:
    """A step = one default build, then the verification consumer on its
    tree: tree attention of a synthetic target layer (Qwen3-8B attention
    shape, 2048 prefix positions) with the build's mask, the target's greedy
    token per row through an output projection [V, 4096] (the head-call
    kernel, K = 1, zero base logits; the stand-in projection is the head's
    Wout), and the longest accepted prefix.  One GPU (replicas as run_gpu)."""
    import numpy as np
    import torch

    from speculative_decoding_draft_06_gb300 import dartree as dtl

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    w = I.CONFIGS[args.config]
    if world > 1:
        w = w.replace(seed=w.seed + 7919 * rank)
    vs = I.VerifyShape()
    inp = I.make_inputs(w)
    dev = dtl.weights_to_device(inp, w.bf16)
    xv = I.make_verify_inputs(w.R, w.B, vs)
    xd = {k: torch.from_numpy(v.view(np.int16)).cuda() for k, v in xv.items()}
    Kc, VTc = dtl.kv_cache(xd["Kp"], xd["Vp"], xd["Kt"], xd["Vt"])
    ctx = dtl.DARTree(w.V, w.H, max_D=w.D, max_W=w.W, max_K=w.K, max_B=w.B,
                      max_requests=w.R, bf16=w.bf16)
    H2 = vs.Hq * vs.dh
    rows = w.R * (w.B + 1)
    tgt = dtl.DARTree(w.V, H2, max_D=1, max_W=rows, max_K=1, max_B=1, bf16=True)
    layout = prepare_wout(ctx, dev, w.bf16, args.wout_layout)
    if layout != "rows":
        tgt.set_weight_layout("blocks")
    U = dev["Wout"] if H2 == w.H else None
    if U is None:
        raise SystemExit("verify: the stand-in projection needs H == Hq * dh")
    zero = torch.zeros(w.V, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    out = ctx.alloc_tree(w.R, w.B)
    kw = dict(D=w.D, W=w.W, K=w.K, B=w.B, beta=w.beta, out=out, stream=stream)
    args_t = (dev["z"], dev["state0"], dev["A"], dev["E"], dev["Wout"])
    ev = {}

    def step(timed: bool = False):
        ctx.build(*args_t, **kw)
        with torch.cuda.stream(stream):
            if timed:
                ev["a0"].record(stream)
            att = dtl.tree_attention(xd["Q"], Kc, VTc, out["mask"], Lp=vs.Lp, stream=stream)
            if timed:
                ev["a1"].record(stream)
            S = att["O16"].view(rows, H2)
            r = tgt.head_topk(S, zero, U, K=1, rows_per_req=rows, stream=stream)
            if timed:
                ev["p1"].record(stream)
            pred = r["tok"].view(w.R, w.B + 1)
            acc = dtl.accept(out["parent"], out["token"], out["n_out"], pred, max_len=w.D,
                             stream=stream)
        return acc

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    e1.synchronize()
    clock_info = clocks.stop()
    ctx.sync(stream)
    ms = aggregate(e0.elapsed_time(e1) / args.steps, world)
    # the attention and projection launches alone (events on the same stream)
    ev = {k: torch.cuda.Event(enable_timing=True) for k in ("a0", "a1", "p1")}
    n_t = min(args.steps, 20)
    t_att = t_proj = 0.0
    for _ in range(n_t):
        acc = step(timed=True)
        stream.synchronize()
        t_att += ev["a0"].elapsed_time(ev["a1"])
        t_proj += ev["a1"].elapsed_time(ev["p1"])
    t_att /= n_t
    t_proj /= n_t
    # the attention alone, back to back: 20 launches captured in a CUDA graph
    # and replayed (no launch latency or host time between them)
    n_bb, n_rep = 20, 5
    g_att = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_att, stream=stream):
        for _ in range(n_bb):
            dtl.tree_attention(xd["Q"], Kc, VTc, out["mask"], Lp=vs.Lp)
    with torch.cuda.stream(stream):
        for _ in range(2):
            g_att.replay()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_rep):
            g_att.replay()
        e1.record(stream)
    e1.synchronize()
    t_att_bb = e0.elapsed_time(e1) / (n_bb * n_rep)
    acc_len = acc["len"].cpu().numpy()
    depth = out["depth"].cpu().numpy()
    n_out = out["n_out"].cpu().numpy()
    # attention flops: QK and PV, 2 * 2 * dh per visible (row, key) pair
    vis = sum(vs.Hq * ((w.B + 1) * vs.Lp + int(depth[r, :n_out[r]].sum())) for r in range(w.R))
    att_flops = 4.0 * vs.dh * vis
    tfl, tfl_kind = measured_bf16_tflops()
    proj_bytes = w.V * H2 * 2 + w.V * 4 + rows * H2 * 2
    peak, peak_kind = measured_peaks()
    if rank == 0:
        value = world * w.R * 1e3 / ms
        line = {
            "metric": "supertree builds + verifications/s", "value": value,
            "unit": "verified builds/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "variant": "verify",
            "config": dict(workload_config(w), wout_layout=layout, verify=(
                f"target layer: prefix {vs.Lp}, {vs.Hq} query heads, {vs.Hkv} kv heads, head "
                f"dim {vs.dh}; projection [V, {H2}] (the head's Wout as stand-in)")),
            "roofline": {"bound": "hbm", "kernel": (
                             "k_head_rows" if rows >= ROWS_MIN else "k_head_tc") +
                         f" (target output projection, {rows} rows, K=1)", "achieved": proj_bytes / (t_proj * 1e-3) / 1e9,
                         "peak": peak, "unit": "GB/s",
                         "frac": proj_bytes / (t_proj * 1e-3) / 1e9 / peak,
                         "peak_source": peak_kind, "traffic": None,
                         "bytes_per_launch": proj_bytes, "launch_ms": t_proj},
            "attention": {"kernel": "k_tree_attention (tcgen05, S and O in TMEM, online softmax, key split)",
                          "bound": "tensor", "launch_ms": t_att,
                          "achieved": att_flops / (t_att * 1e-3) / 1e12, "peak": tfl,
                          "unit": "TFLOP/s", "frac": att_flops / (t_att * 1e-3) / 1e12 / tfl,
                          "peak_source": tfl_kind, "flops_per_launch": att_flops,
                          "launch_ms_back_to_back": t_att_bb,
                          "achieved_back_to_back": att_flops / (t_att_bb * 1e-3) / 1e12},
            "accept_len_mean": float(acc_len.mean()),
            "cpu_baseline": None, "e2e": None,
            "gpu_launches": (kernels_per_build(w) + 4) * args.steps,
            "clocks": clock_info,
        }
        print(json.dumps(line), flush=True)
    tgt.close()
    ctx.close()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_profile_head(args) -> None:
    """N head calls on one stream, for ncu captures of k_head_tc on a case
    that still streams its weights from HBM but holds only a few GB."""
    import numpy as np
    import torch

    from speculative_decoding_draft_06_gb300 import dartree as dtl
    torch.cuda.set_device(0)
    w = I.CONFIGS[args.config]
    if args.vocab:
        w = w.replace(V=args.vocab)
    M = max(w.head_rows())
    inp = I.make_inputs(w.replace(D=1))
    dev = dtl.weights_to_device(inp, w.bf16)
    g = np.random.default_rng(1)
    S = np.tanh(g.standard_normal((M, w.H))).astype(np.float32)
    S = torch.from_numpy(I.to_bf16_bits(S)).view(torch.int16).cuda() if w.bf16 else \
        torch.from_numpy(S).cuda()
    ctx = dtl.DARTree(w.V, w.H, max_D=1, max_W=w.W, max_K=w.K, max_B=w.B, max_requests=w.R,
                      bf16=w.bf16)
    prepare_wout(ctx, dev, w.bf16, args.wout_layout)
    z = dev["z"][:, 0].contiguous()
    for _ in range(args.profile_head):
        ctx.head_topk(S, z, dev["Wout"], K=w.K, rows_per_req=M // w.R, z_req_stride=w.V)
    ctx.sync()
    print(json.dumps({"profile_head": args.profile_head, "V": w.V, "H": w.H, "M": M,
                      "K": w.K}), flush=True)
    ctx.close()


def main(argv=None):
    args = parse_args(argv)
    if args.profile_head:
        run_profile_head(args)
        return
    if args.impl == "reference":
        run_reference(args)
    elif args.variant == "verify":
        run_verify(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
