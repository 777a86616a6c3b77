"""Benchmark of the GB300 angular-correlation path.

One step = the whole hot path on the pages' workload shape: DD, DR and RR histograms of two
100,000-galaxy catalogs (D clustered, R uniform; 720 bins of 0.25 degrees) plus omega, with the
catalogs already resident in HBM. Reported value: logical pairs per second, (n_d^2 + n_d n_r +
n_r^2) / step time, in G pairs/s ("CUDA Deep Dive: 10B Galaxy Pairs on an RTX 5080", section "The
problem": N^2 pairs per family, three families).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config 1]

--impl reference times the fp64 CPU oracle (the reference arm) on a bounded row sample of the same
workload. With N > 1 (launched by torch.distributed.run) every rank runs an independent replica
of the job on its own GPU (weak scaling); the reference arm runs on rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402

METRIC = "G pairs/s (DD+DR+RR, N=100k each) and % of FP32 issue roofline"
UNIT = "Gpairs/s"
# Thread instructions per pair of each pair-kernel path: the general chord + polynomial loop is 25
# (dot product, sign, chord, polynomial, sqrt, sign-dependent constant, rounding fma, address,
# shared atomic); where the caps fix the sign of the dot product the dot, the sign operation and the
# constant choice drop out (18); where every theta' stays below 72 degrees the polynomial is of
# degree 5 instead of 7 (16); the dot form for groups between 55 and 125 degrees is 11 (dot, square,
# degree-4 polynomial, rounding fma, address, atomic). Exact-mode flagging adds 3: the fine code
# (a second rounding fma, or a shift of the one code), the masked zero test of its fraction, a
# 3-input predicate OR shared by 2 pairs, and one warp vote with its branch per j (4 pairs per lane).
INST_PER_PATH = {"pairs_fixed": 18, "pairs_general": 25, "pairs_fixed_exact": 21, "pairs_general_exact": 28,
                 "pairs_mid": 11, "pairs_mid_exact": 14, "pairs_small": 16, "pairs_small_exact": 19}
INST_MASKED = 25  # diagonal / ragged units run the general loop on every computed pair
INST_MASKED_EXACT = 4  # and with flags: fine-code shift, fraction mask, test, branch per pair
SMS, LANES_PER_SM, SM_MAX_MHZ = 152, 128, 2070.0
# The pages' kernel time for three 100k histograms on an RTX 5080 (another machine: context only)
PAGE_KERNEL_MS = 22.747


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(values: list[float], world: int) -> list[float]:
    """Element-wise max over ranks (host-side gloo all-reduce; no data-path collective)."""
    if world <= 1:
        return values
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def logical_pairs(n_d: int, n_r: int) -> int:
    return n_d * n_d + n_d * n_r + n_r * n_r


def evaluated_pairs(n_d: int, n_r: int) -> int:
    """Pairs the kernels must evaluate: every DR pair, each unordered DD and RR pair once."""
    return n_d * n_r + n_d * (n_d - 1) // 2 + n_r * (n_r - 1) // 2


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int, path: str | None):
        self.device, self.path, self.proc = device, path, None

    def __enter__(self):
        try:
            self.fh = open(self.path, "w") if self.path else subprocess.DEVNULL
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.device), "-lms", "200"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
            if self.path:
                self.fh.write(out)
                self.fh.close()

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def code_only(text: str) -> str:
    """C++/CUDA source without comments, trailing blanks and empty lines (what the compiler sees)."""
    out, i, n, quote = [], 0, len(text), None
    while i < n:
        ch = text[i]
        if quote:
            out.append(ch)
            if ch == "\\" and i + 1 < n:
                out.append(text[i + 1])
                i += 1
            elif ch == quote:
                quote = None
        elif ch in "\"'":
            quote = ch
            out.append(ch)
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
            continue
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            continue
        else:
            out.append(ch)
        i += 1
    return "\n".join(line.rstrip() for line in "".join(out).splitlines() if line.strip())


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code (comments excluded), to tie recorded ncu counters to them."""
    h = hashlib.sha256()
    for rel in ("all_pairs_angular_gb300/csrc/acf_kernels.cuh", "all_pairs_angular_gb300/csrc/acf.cu"):
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


# How each arm treats the L2 cache between timed steps: one statement, the same in both arms'
# `config`, so that the two lines describe the same workload
L2_NOTE = "GPU arm: L2 flushed between timed steps (256 MiB device write); CPU reference arm: n/a"


def bench_config(cat, workload: str, options: dict) -> dict:
    """The workload as both arms report it (launch facts go to a separate `launch` object)."""
    cfg = {"workload": workload, "n_d": cat.n_d, "n_r": cat.n_r, "bin_width_deg": cat.bin_width_deg,
           "nbins": cat.nbins, "l2": L2_NOTE}
    if options:
        cfg["options"] = options
    return cfg


def recorded_counters(workload: str) -> dict | None:
    """The committed ncu record of the pair kernel on this workload (per-launch DRAM bytes and
    executed instructions), if it was captured from the current kernel source."""
    path = os.path.join(ROOT, "profiles", "pair_kernel_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash() or rec.get("workload") != workload:
        return None
    return rec


def executed_roofline(rec: dict | None, pair_ms_per_step: float, alg_inst_per_step: float, peak: float) -> dict | None:
    """The pair kernel's fraction of the issue roofline on the basis of the instructions it really
    executed (ncu smsp__thread_inst_executed.sum of the DD, DR and RR launches of one step, from
    the committed record) over the event-timed pair-kernel time of a step."""
    if not rec or pair_ms_per_step <= 0:
        return None
    per = rec.get("per_launch", {})
    try:
        inst = sum(float(per[f]["thread_inst_executed"]) for f in ("DD", "DR", "RR"))
    except (KeyError, TypeError, ValueError):
        return None
    achieved = inst / (pair_ms_per_step / 1e3) / 1e12
    out = {"basis": "executed thread-instructions per step (ncu smsp__thread_inst_executed.sum, committed record)",
           "thread_inst_per_step": inst, "achieved": achieved, "frac": achieved / peak,
           "inst_overhead": inst / alg_inst_per_step if alg_inst_per_step else None}
    if "issue_active_pct" in rec:
        out["ncu_issue_active_pct"] = rec["issue_active_pct"]
    return out


def cpu_baseline(cat, rows: int, seed: int, threads: int = 0) -> dict:
    """Time the fp64 oracle on a row sample: `rows` rows of D against D, of D against R and of R
    against R. Returns the oracle rate in logical G pairs/s."""
    import oracle
    idx_d = synth.sample_rows(cat.n_d, rows, seed)
    idx_r = synth.sample_rows(cat.n_r, rows, seed + 1)
    w, nb = cat.bin_width_deg, cat.nbins
    t0 = time.perf_counter()
    oracle.histogram(cat.ra_d[idx_d], cat.dec_d[idx_d], cat.ra_d, cat.dec_d, w, nb, threads=threads)
    oracle.histogram(cat.ra_d[idx_d], cat.dec_d[idx_d], cat.ra_r, cat.dec_r, w, nb, threads=threads)
    oracle.histogram(cat.ra_r[idx_r], cat.dec_r[idx_r], cat.ra_r, cat.dec_r, w, nb, threads=threads)
    dt = time.perf_counter() - t0
    pairs = rows * (2 * cat.n_d + cat.n_r)
    cores = threads if threads > 0 else (os.cpu_count() or 1)
    return {"value": pairs / dt / 1e9, "unit": UNIT, "cores": cores, "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{rows} random rows each of DD, DR and RR against the full catalogs ({pairs:.3g} pairs)"}


def run_reference(args, cat, workload, rank, world):
    if rank != 0:
        return 0
    rows = args.ref_rows
    times = []
    for s in range(args.warmup + args.steps):
        r = cpu_baseline(cat, rows, seed=1000 + s)
        if s >= args.warmup:
            times.append(r["seconds"])
    per_step_pairs = rows * (2 * cat.n_d + cat.n_r)
    total = sum(times)
    value = per_step_pairs * len(times) / total / 1e9
    cb = {"value": value, "unit": UNIT, "cores": os.cpu_count() or 1, "kind": "oracle",
          "sample": f"each step: {rows} random rows each of DD, DR and RR against the full catalogs"}
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(cat, workload, {}),
            "cpu_baseline": cb, "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args, cat, workload, rank, world, local):
    import torch

    import all_pairs_angular_gb300 as acf

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(dev)
    ctx = acf.Context(local, stream)
    ctx.set_option("kernel_timing", 1)
    for k, v in parse_options(args.option).items():
        ctx.set_option(k, v)
    w, nb = cat.bin_width_deg, cat.nbins
    with torch.cuda.stream(stream):
        ra_d = torch.from_numpy(cat.ra_d).to(dev)
        dec_d = torch.from_numpy(cat.dec_d).to(dev)
        ra_r = torch.from_numpy(cat.ra_r).to(dev)
        dec_r = torch.from_numpy(cat.dec_r).to(dev)
        dd = torch.empty(nb, dtype=torch.int64, device=dev)
        dr = torch.empty_like(dd)
        rr = torch.empty_like(dd)
        om = torch.empty(nb, dtype=torch.float64, device=dev)
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)  # > 129 MB L2

    def step():
        # the whole hot path: both catalogs sorted and converted, DD, DR, RR and omega
        acf.acf_correlate(ctx.handle, ra_d, dec_d, cat.n_d, ra_r, dec_r, cat.n_r, w, nb, dd, dr, rr, om)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        ctx.kernel_times()  # discard warm-up launches
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        barrier(world)
        torch.cuda.synchronize(dev)
        # the raw nvidia-smi samples go to a file only when ACF_CLOCK_LOG_DIR names a folder
        log_dir = os.environ.get("ACF_CLOCK_LOG_DIR", "")
        clock_log = os.path.join(log_dir, f"clocks_rank{rank}.csv") if log_dir and os.path.isdir(log_dir) else None
        launched_before = ctx.info("kernel_launches")
        replays_before = ctx.info("graph_replays")
        with ClockSampler(local, clock_log) as clk:
            for s in range(args.steps):
                flush.zero_()                     # evict L2 outside the timed region
                ev[s][0].record(stream)
                step()
                ev[s][1].record(stream)
            stream.synchronize()
        torch.cuda.synchronize(dev)
        barrier(world)
    gpu_launches = ctx.info("kernel_launches") - launched_before  # this library's kernels, timed steps only
    # timed steps the library served from its CUDA graph of the call (option "graphs", default on:
    # the first warm-up step runs as usual, the second is captured, later ones replay it)
    graph_steps = ctx.info("graph_replays") - replays_before
    step_ms = [a.elapsed_time(b) for a, b in ev]
    kt = ctx.kernel_times()
    # instructions the algorithm needs per step: one untimed step, reading each call's path counts
    ctx.set_option("kernel_timing", 0)
    alg_inst, alg_pairs = 0, 0
    path_pairs = {}
    with torch.cuda.stream(stream):
        for call in (lambda: acf.acf_histogram(ctx.handle, ra_d, dec_d, cat.n_d, None, None, 0, w, nb, dd),
                     lambda: acf.acf_histogram(ctx.handle, ra_d, dec_d, cat.n_d, ra_r, dec_r, cat.n_r, w, nb, dr),
                     lambda: acf.acf_histogram(ctx.handle, ra_r, dec_r, cat.n_r, None, None, 0, w, nb, rr)):
            call()
            for key, ipp in INST_PER_PATH.items():
                n_pairs = ctx.info(key)
                alg_inst += ipp * n_pairs
                alg_pairs += n_pairs
                path_pairs[key] = path_pairs.get(key, 0) + n_pairs
            masked = ctx.info("pairs_masked")
            path_pairs["pairs_masked"] = path_pairs.get("pairs_masked", 0) + masked
            exact_on = sum(ctx.info(k) for k in ("pairs_fixed_exact", "pairs_general_exact", "pairs_small_exact",
                                                 "pairs_mid_exact")) > 0
            alg_inst += (INST_MASKED + (INST_MASKED_EXACT if exact_on else 0)) * masked
            alg_pairs += masked
    # the exact mode's fix-ups, timed by themselves (kernel_timing 2) over a few more untimed steps
    fixup = None
    if exact_on:
        ctx.set_option("kernel_timing", 2)
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
        ft = ctx.kernel_times()
        ctx.set_option("kernel_timing", 0)
        fixup = {"ms_per_step": sum(ft) / 3, "launches_per_step": len(ft) // 3,
                 "basis": "CUDA events around each fix-up launch, 3 untimed steps"}
    total_ms = sum(step_ms)
    total_ms_max, = reduce_max([total_ms], world)
    pairs = logical_pairs(cat.n_d, cat.n_r)
    value = world * pairs * args.steps / (total_ms_max / 1e3) / 1e9
    # dominant kernel: the pair kernel (three launches per step: DD, DR, RR)
    evals = evaluated_pairs(cat.n_d, cat.n_r)
    pair_ms = sum(kt)
    clocks = clk.summary()
    peak = SMS * LANES_PER_SM * SM_MAX_MHZ * 1e6 / 1e12  # T thread-instructions / s at the maximum clock
    achieved = alg_inst * args.steps / (pair_ms / 1e3) / 1e12 if pair_ms > 0 else None
    rec = recorded_counters(workload)
    roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Tinst/s",
            "frac": (achieved / peak) if achieved else None,
            "frac_basis": "algorithmic instructions: a per-path instruction model (bench.py INST_PER_PATH) "
                          "times the kernel's own per-path pair counters, over event-timed pair-kernel time",
            "traffic": rec.get("dram_bytes_per_launch") if rec else None,
            "inst_per_pair": alg_inst / max(alg_pairs, 1), "pairs_computed_per_step": alg_pairs,
            "path_share": {k[len("pairs_"):]: round(v / max(alg_pairs, 1), 4) for k, v in path_pairs.items() if v},
            "pair_kernel_ms_per_launch": pair_ms / max(len(kt), 1),
            "pair_kernel_launches": len(kt),
            "peak_basis": f"{SMS} SMs x {LANES_PER_SM} FP32 lanes x {SM_MAX_MHZ:.0f} MHz (maximum SM clock)"}
    roof["executed"] = executed_roofline(rec, pair_ms / args.steps, alg_inst, peak)
    if clocks.get("sm_mhz"):
        roof["frac_at_observed_clock"] = achieved / (SMS * LANES_PER_SM * clocks["sm_mhz"] * 1e6 / 1e12)
    # the FP32 issue ceiling measured on this GPU in this run (independent FMA chains)
    fma_rate, _ = acf.acf_fp32_peak(ctx.handle, 1 << 16)
    roof["fma_chain_ceiling"] = fma_rate / 1e12
    roof["frac_of_fma_chain_ceiling"] = achieved / (fma_rate / 1e12) if achieved else None

    # end to end through the C ABI with pinned host buffers: copies inside the timed region
    h = {k: torch.from_numpy(getattr(cat, k)).pin_memory() for k in ("ra_d", "dec_d", "ra_r", "dec_r")}
    hout = [torch.empty(nb, dtype=torch.int64).pin_memory() for _ in range(3)] + [
        torch.empty(nb, dtype=torch.float64).pin_memory()]

    def e2e_step():
        acf.acf_correlate_host(ctx.handle, h["ra_d"], h["dec_d"], cat.n_d, h["ra_r"], h["dec_r"], cat.n_r, w, nb,
                               *hout)

    for _ in range(args.warmup):
        e2e_step()
    barrier(world)
    e2e_times = []
    for _ in range(args.steps):
        flush.zero_()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_step()  # synchronises before returning
        e2e_times.append(time.perf_counter() - t0)
    e2e_total, = reduce_max([sum(e2e_times)], world)
    e2e_value = world * pairs * args.steps / e2e_total / 1e9
    h2d = 4 * (2 * cat.n_d + 2 * cat.n_r)
    d2h = 8 * 4 * nb
    assert np.array_equal(acf.as_uint64(hout[0]), acf.as_uint64(dd)), "e2e and device paths disagree"

    if rank == 0:
        cb = cpu_baseline(cat, args.cpu_rows, seed=77) if args.cpu_rows > 0 else None
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak",
            # the pages' number is for two 100k catalogs in 0.25-degree bins only
            # (and with the default options only)
            "vs_baseline": (value / (pairs / (PAGE_KERNEL_MS / 1e3) / 1e9)
                            if args.config == 1 and not args.option else None),
            "dtype": "f32", "data": "synthetic",
            "config": bench_config(cat, workload, parse_options(args.option)),
            "launch": {"parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "grid": ctx.info("grid"), "threads": ctx.info("threads"), "layout": ctx.info("layout")},
            "evaluated_gpairs_per_s": world * evals * args.steps / (total_ms_max / 1e3) / 1e9,
            # per-step spread on rank 0 (the pages' protocol reports the median and the minimum)
            "step_ms_stats": {"first": step_ms[0], "median": statistics.median(step_ms), "min": min(step_ms),
                              "max": max(step_ms)},
            "roofline": roof, "cpu_baseline": cb,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": 1e3 * e2e_total / args.steps,
                    # host-timed, so a host hiccup shows here: the spread of the steps on rank 0
                    "step_ms_stats": {"first": 1e3 * e2e_times[0], "median": 1e3 * statistics.median(e2e_times),
                                      "min": 1e3 * min(e2e_times), "max": 1e3 * max(e2e_times)}},
            "gpu_launches": gpu_launches, "clocks": clocks, "fixup": fixup, "graph_replayed_steps": graph_steps,
        }
        print(json.dumps(line), flush=True)
    ctx.close()
    return 0


def run_profile(args, cat):
    """One warm-up step and one step of DD, DR, RR and omega, nothing else: a short, fixed launch
    list for Nsight Compute (pair kernel launches: 3 warm-up, then DD, DR, RR)."""
    import torch

    import all_pairs_angular_gb300 as acf

    dev = torch.device("cuda", 0)
    ctx = acf.Context(0)
    for k, v in parse_options(args.option).items():
        ctx.set_option(k, v)
    w, nb = cat.bin_width_deg, cat.nbins
    t = {k: torch.from_numpy(getattr(cat, k)).to(dev) for k in ("ra_d", "dec_d", "ra_r", "dec_r")}
    out = [torch.empty(nb, dtype=torch.int64, device=dev) for _ in range(3)]
    om = torch.empty(nb, dtype=torch.float64, device=dev)
    for _ in range(2):
        ctx.correlate(t["ra_d"], t["dec_d"], t["ra_r"], t["dec_r"], w, nb, out=(*out, om))
    torch.cuda.synchronize()
    sums = [int(acf.as_uint64(o).sum()) for o in out]
    print(json.dumps({"profile": cat.name, "sums": sums, "grid": ctx.info("grid"), "threads": ctx.info("threads"),
                      "kernel_source_hash": kernel_source_hash()}), flush=True)
    ctx.close()
    return 0 if sums == [cat.n_d ** 2, cat.n_d * cat.n_r, cat.n_r ** 2] else 1


# The page's kernel times per ladder level on its RTX 5080 (section "The ladder"): context only.
PAGE_LADDER_MS = {0: 188.653, 1: 169.209, 2: 163.435, 3: 34.027, 4: 24.528, 5: 22.747}
ABLATION_VARIANTS = [
    ("default (exact 2, range forms)", {}),
    ("exact mode 1 (re-decide within 20 deg of 0 and 180)", {"exact": 1}),
    ("exact mode 0 (fp32 bins only)", {"exact": 0}),
    ("range forms off (full-range chord for every pair), exact 2", {"range_forms": 0}),
    ("range forms off, exact 0", {"range_forms": 0, "exact": 0}),
    ("dot product + acosf (the page's form)", {"bin_method": 1}),
    ("dot product + A&S 4.4.45 arccos (approximate mode)", {"bin_method": 2}),
    ("one block-shared histogram instead of 32 lane copies", {"layout": 2}),
    ("512 threads per block", {"threads": 512}),
]


def run_ablation(args, cat) -> int:
    """The page's optimisation ladder rebuilt on this GPU, then one change at a time from this
    library's default, all on one workload: pair-kernel time and what each does to the counts
    against the oracle's (tests/golden, for the workloads that have a golden file)."""
    import statistics

    import torch

    import all_pairs_angular_gb300 as acf

    dev = torch.device("cuda", 0)
    w, nb = cat.bin_width_deg, cat.nbins
    t = {k: torch.from_numpy(getattr(cat, k)).to(dev) for k in ("ra_d", "dec_d", "ra_r", "dec_r")}
    gold = None
    gpath = os.path.join(ROOT, "tests", "golden", f"config{args.config}_oracle.json")
    if os.path.exists(gpath):
        with open(gpath) as f:
            g = json.load(f)
        if g.get("digest") == cat.digest():
            gold = g

    def compare(hs):
        if gold is None:
            return {}
        moved = {}
        for fam, h in zip(("DD", "DR", "RR"), hs):
            ref = np.array(gold[fam]["hist"], np.int64)
            moved[fam] = int(np.abs(np.cumsum(h.astype(np.int64) - ref)).sum())
        rr = np.array(gold["RR"]["hist"], np.float64)
        nd2, ndr, nr2 = float(cat.n_d) ** 2, float(cat.n_d) * cat.n_r, float(cat.n_r) ** 2
        with np.errstate(invalid="ignore", divide="ignore"):
            om = (hs[0] / nd2 - 2.0 * hs[1] / ndr + hs[2] / nr2) / (hs[2] / nr2)
        ref_om = np.array([np.nan if x is None else x for x in gold["omega"]])
        big = rr >= 1000
        return {"moved_pairs": moved, "max_abs_domega_rr_ge_1000": float(np.nanmax(np.abs(om[big] - ref_om[big])))}

    rows = []
    evaluated = cat.n_d * cat.n_r + cat.n_d * (cat.n_d + 1) // 2 + cat.n_r * (cat.n_r + 1) // 2
    if cat.n_d == cat.n_r:
        for level in range(6):
            hs = [torch.empty(nb, dtype=torch.int64, device=dev) for _ in range(3)]
            times = [acf.acf_ladder(level, t["ra_d"], t["dec_d"], t["ra_r"], t["dec_r"], w, nb, *hs)
                     for _ in range(3 if level < 3 else 5)]
            ms = statistics.median(times[1:])
            pairs = 3 * cat.n_d * cat.n_d if level == 0 else evaluated
            rows.append({"row": f"page ladder L{level}", "kernel_ms": ms, "evaluated_gpairs_per_s": pairs / ms / 1e6,
                         "page_rtx5080_ms": PAGE_LADDER_MS[level], **compare([acf.as_uint64(h) for h in hs])})
            print(json.dumps(rows[-1]), flush=True)
    for name, opts in ABLATION_VARIANTS:
        ctx = acf.Context(0)
        for k, v in opts.items():
            ctx.set_option(k, v)
        ctx.set_option("kernel_timing", 1)
        out = None
        step_ms = []
        for rep in range(4):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            out = ctx.correlate(t["ra_d"], t["dec_d"], t["ra_r"], t["dec_r"], w, nb)
            e1.record()
            torch.cuda.synchronize()
            if rep:
                step_ms.append(e0.elapsed_time(e1))
        kt = ctx.kernel_times()
        pair_ms = sum(kt[len(kt) // 4:]) / 3.0  # the last three of four steps
        hs = [acf.as_uint64(h) for h in out[:3]]
        rows.append({"row": name, "options": opts, "step_ms": statistics.median(step_ms), "pair_kernels_ms": pair_ms,
                     "logical_gpairs_per_s": logical_pairs(cat.n_d, cat.n_r) / statistics.median(step_ms) / 1e6,
                     **compare(hs)})
        print(json.dumps(rows[-1]), flush=True)
        ctx.close()
    return 0


def parse_options(items) -> dict:
    """["exact=0", "layout=3"] -> {"exact": 0, "layout": 3}"""
    out = {}
    for it in items:
        k, sep, v = it.partition("=")
        if not sep or not k:
            raise SystemExit(f"--option wants KEY=VALUE, got {it!r}")
        out[k] = int(v)
    return out


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=1, help="workload index (default 1: two 100k catalogs)")
    ap.add_argument("--cpu-rows", type=int, default=2000, help="rows per family for the CPU baseline (0: skip)")
    ap.add_argument("--ref-rows", type=int, default=200, help="rows per family per reference-arm step")
    ap.add_argument("--profile", action="store_true", help="one warm-up step + one step only (for ncu)")
    ap.add_argument("--option", action="append", default=[], metavar="KEY=VALUE",
                    help="a library option (acf_set_option) for the timed run, e.g. exact=0; repeatable")
    ap.add_argument("--ablation", action="store_true",
                    help="the page's ladder and one-change variants of the library, timed and checked")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local = dist_env()
    if world != args.gpus:
        world = max(world, 1)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    cat = synth.config(args.config)
    workload = (f"{cat.name}: D {cat.n_d} (half uniform, half in {synth.CONFIGS[args.config]['n_clumps']} clumps), "
                f"R {cat.n_r} uniform, {cat.nbins} bins of {cat.bin_width_deg} deg, seed {cat.seed}")
    if args.profile:
        return run_profile(args, cat)
    if args.ablation:
        return run_ablation(args, cat)
    try:
        if args.impl == "reference":
            return run_reference(args, cat, workload, rank, world)
        return run_ours(args, cat, workload, rank, world, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
