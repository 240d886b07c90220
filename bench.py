"""Benchmark: seconds per GPTQ group (fold + q4tp sweep) at n = 17408.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--codec q4tp|q2tp]

One step = one full pass of the hot path on one synthetic Hessian group
already resident in HBM: fold (builder, Cholesky, inverse, U), dead-column
zeroing, ladder, q4tp sweep, through the C ABI (gptq_quantize_group).  With
N > 1 (torchrun) every rank folds and quantizes its own group (independent
problems, no collective on the data path): weak scaling.  ``--codec q2tp``
times the same step with the q2tp "placed" rule instead (placed ladder,
31-rung search, 2-bit codes: gptq_quantize_group_q2tp), under its own metric.

The default line also carries the 11-group batch (config "batch": seeds
0..10, four streams, total wall time and groups/s) measured after the
headline (``--no-batch`` leaves it out), the whole fold's and the sweep
GEMMs' fractions of the 3xTF32 peak, and that peak measured in-process
(cuBLAS TF32).

``--impl reference`` times the CPU oracle (the plain f64/f32 restatement of
the pages) on the host cores, on a bounded sample of the same workload
scaled to seconds per group.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "s per GPTQ group (fold+q4tp) at n=17408"
METRIC_Q2 = "s per GPTQ group (fold+q2tp placed) at n=17408"
UNIT = "s/group"

# Peaks for the roofline denominators when the driver's measured file is absent.
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Nominal dense tensor ratios (TF32 : BF16 = 1.1 : 2.25 PFLOP/s).
TF32_PER_BF16 = 1.1 / 2.25
# DRAM bytes (read + write) per launch of the update kinds at the bench
# workload, from a one-pass ncu launch list of the current kernels (the
# fold's 33 K = 512 trailing updates: 30.52 GB); drop an entry whenever its
# kernels change.
TRAFFIC = {"fold_gemm": 924.73e6}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK), "fallback"


def workload_desc(cfg, codec="q4tp"):
    return (f"{cfg.name}: one Hessian group, n={cfg.n} channels, W [{cfg.rows}, {cfg.n}] f32 "
            f"N(0, {cfg.w_std}^2); H = X X^T / T, X [{cfg.n}, {cfg.T}] N(0,1) with lognormal(0, {cfg.sigma}) "
            f"channel scales, {cfg.n_outlier} outlier channels x100, {cfg.n_dead} dead; "
            f"lambda={cfg.lam}, group 32, " + ("q4tp" if codec == "q4tp" else "q2tp placed rule"))


def fold_gemm_flops(n, NB=128, part="all", G=4):
    """Algorithmic flops of the fold's update GEMM launches over one fold, on
    the padded size, following the library's schedule: steps in groups of G
    blocks (fewer at the end).  After step i of a group, a K = NB strip
    update of the group's remaining block columns; after the group, one
    K = G NB trailing update.
    part: "trailing" (the group updates, kind fold_gemm), "strip" (the K = NB
    strips, kind fold_strip) or "all"."""
    N = (n + NB - 1) // NB * NB
    strip = trail = 0
    k = 0
    while k < N:
        g = min(G, (N - k) // NB)
        sg = k + g * NB
        for i in range(g - 1):
            kn = k + (i + 1) * NB
            w = sg - kn
            # SYRK strip: the rows below the group, and the lower triangle of
            # the group's remaining square; the inverse's rows above kn.
            strip += 2 * NB * ((N - sg) * w + w * (w + 1) // 2)
            strip += 2 * NB * kn * w
        m = N - sg
        if m > 0:
            # SYRK of the group, then the inverse rectangle: step i's panel
            # meets the rows c < k_i + NB only (its rows of later blocks of the
            # group are zero: X is lower triangular, so the launch multiplies
            # them but they are no work of the method).
            trail += 2 * (g * NB) * (m * (m + 1) // 2)
            trail += sum(2 * NB * (k + (i + 1) * NB) * m for i in range(g))
        k = sg
    return {"trailing": trail, "strip": strip, "all": trail + strip}[part]


def sweep_gemm_flops(rows, n, SB=128):
    tot = 0
    for b0 in range(0, n, SB):
        b1 = min(b0 + SB, n)
        if b1 < n:
            tot += 2 * (b1 - b0) * rows * (n - b1)
    return tot


def hbm_report(per_kind, n, rows, codec="q4tp", peak_gbs=None, NB=128, SB=128):
    """Achieved HBM rate of the sequential, memory-facing kernels: their
    algorithmic bytes per group over their measured time per group (kinds
    absent from ``per_kind`` are left out)."""
    N = (n + NB - 1) // NB * NB
    gpr = n // 32
    codes = rows * n // (4 if codec == "q2tp" else 2)
    tabs = rows * 34 * 4
    parts = {
        "build": ("a2 builder: read the packed H, write the N x N working matrix", n * (n + 1) // 2 * 4 + N * N * 4),
        "trsm": ("a6 U = P X P D^-1 fused into the panel products' store: U's upper triangle written "
                 "(the tensor-core panel product itself is bound by launch and load latency)", n * (n + 1) // 2 * 4),
        "ladder": ("a7 dead-column zeroing fused with the ladder: read W and diag H, write the zeroed W, "
                   "tab and lost", 2 * rows * n * 4 + n * 4 + tabs),
        "place": ("q2tp placement: read W, write tab and lost", rows * n * 4 + tabs),
        "copy": ("dead-column zeroing: read and write W", 2 * rows * n * 4),
        "sweep_block": ("a8, a9, a11: read W and U's diagonal blocks, write codes, rungs and scales "
                        "(latency-bound rounding chain)", rows * n * 4 + n * SB * 4 + codes + rows * gpr * 5),
    }
    out = {}
    for kind, (what, nbytes) in parts.items():
        ms = per_kind.get(kind, {}).get("ms_per_step")
        if not ms:
            continue
        gbs = nbytes / (ms / 1e3) / 1e9
        out[kind] = {"what": what, "bytes_per_group": nbytes, "ms_per_group": ms, "gbs": gbs,
                     "frac": gbs / peak_gbs if peak_gbs else None}
    return out


def measure_tf32_tflops(torch, dev, size=8192, reps=10):
    """Dense TF32 peak of this GPU, measured here: cuBLAS f32 matmul with TF32
    allowed at size^3 (2 size^3 flops), best of `reps` after warm-up, timed
    with CUDA events on the current stream.  A burst figure: the roofline
    denominators of kernels timed in a seconds-long run at full clocks."""
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device=dev)
        g.manual_seed(7)
        a = torch.randn(size, size, device=dev, generator=g)
        b = torch.randn(size, size, device=dev, generator=g)
        c = torch.empty(size, size, device=dev)
        for _ in range(3):
            torch.matmul(a, b, out=c)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            torch.matmul(a, b, out=c)
            e1.record()
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        del a, b, c
        return 2.0 * size ** 3 / (best / 1e3) / 1e12
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev


class ClockSampler:
    """nvidia-smi clocks, power and throttle reasons sampled every 20 ms;
    only the samples inside [t0, t1] (host clock) count."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def stop(self, t0=None, t1=None):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, pw, mx, reasons = [], [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            try:
                pw.append(float(f[3]))
            except ValueError:
                pass
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "sm_min_mhz": min(sm),
                "power_w": statistics.median(pw) if pw else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def cpu_baseline_sample(cfg, n_fold=None, rows_sweep=8, codec="q4tp"):
    """Oracle on a bounded sample, scaled to seconds per full group:
    the fold on the leading n_fold x n_fold block of the group's H (cost
    scaled by (n / n_fold)^3) and the sweep (ladder included) of `rows_sweep`
    rows at full n against that block's operator padded with the identity
    (cost scaled by rows / rows_sweep)."""
    import numpy as np
    import torch

    import oracle
    import synth

    n_fold = n_fold or max(256, (cfg.n // 4) // 32 * 32)
    sub = synth.Config(cfg.name + "_sample", n_fold, rows_sweep, max(1, cfg.T * n_fold // cfg.n), cfg.w_std,
                       cfg.sigma, max(1, cfg.n_outlier * n_fold // cfg.n), max(1, cfg.n_dead * n_fold // cfg.n),
                       cfg.lam, cfg.seed)
    hp = synth.make_h_packed(sub, "cpu").numpy()
    w = synth.make_w(synth.Config(cfg.name, cfg.n, rows_sweep, cfg.T, cfg.w_std, cfg.sigma, cfg.n_outlier,
                                  cfg.n_dead, cfg.lam, cfg.seed), "cpu").numpy()
    t0 = time.perf_counter()
    u, d, dead, lam = oracle.fold(hp, n_fold, cfg.lam)
    t_fold = time.perf_counter() - t0
    # Sweep at full width: the sample operator on the leading block, identity
    # elsewhere (the sweep's cost does not depend on U's values).
    big = np.eye(cfg.n, dtype=np.float32)
    big[:n_fold, :n_fold] = u.astype(np.float32)
    hw = np.ones(cfg.n, dtype=np.float32)
    t0 = time.perf_counter()
    if codec == "q4tp":
        tab, lost = oracle.ladder(w)
        oracle.sweep_q4tp(w, big, hw, tab, lost)
    else:
        tab, lost, _ = oracle.ladder_q2tp(w, hw)
        oracle.sweep_q2tp(w, big, hw, tab)
    t_sweep = time.perf_counter() - t0
    est = t_fold * (cfg.n / n_fold) ** 3 + t_sweep * (cfg.rows / rows_sweep)
    sample = (f"oracle fold at n={n_fold} ({t_fold:.2f} s, x(n/{n_fold})^3) + oracle {codec} ladder and "
              f"sweep of {rows_sweep} rows at n={cfg.n} ({t_sweep:.2f} s, x{cfg.rows}/{rows_sweep}); "
              f"the fold's matrix products in numpy's BLAS/LAPACK on all cores, the sweep's loops on one")
    return est, sample, t_fold + t_sweep


def run_reference(args, cfg, rank):
    if rank != 0:
        return
    cores = os.cpu_count()
    vals = []
    sample = ""
    for i in range(args.warmup + args.steps):
        est, sample, spent = cpu_baseline_sample(cfg, n_fold=args.ref_n, rows_sweep=args.ref_rows,
                                                 codec=args.codec)
        if i >= args.warmup:
            vals.append(est)
    v = statistics.median(vals)
    line = {"metric": METRIC if args.codec == "q4tp" else METRIC_Q2, "value": v, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": v * 1e3, "higher_is_better": False, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_desc(cfg, args.codec)},
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def aggregate(t_local: float, steps: int, world: int, pg=None):
    """Whole-job seconds per group: the slowest rank's time for `steps` steps
    (max over ranks), divided by the groups all ranks processed (one group
    per rank per step).  Returns (t_max, value)."""
    t = float(t_local)
    if pg is not None and world > 1:
        import torch

        tt = torch.tensor([t], dtype=torch.float64)
        if pg.get_backend() == "nccl":
            tt = tt.cuda()
        pg.all_reduce(tt, op=pg.ReduceOp.MAX)
        t = float(tt.item())
    return t, t / (steps * world)


def batch_measure(args, dev, lib, _lib, torch, synth, steps, warmup):
    """11 independent n = 17408 groups (seeds 0..10) back to back on one GPU:
    `--streams` host threads, each with its own CUDA stream and workspace,
    take groups in turn.  Device-timed from one event that every stream
    waits on to one event that waits on every stream.  Returns a dict."""
    import concurrent.futures as cf

    ngroups = 11
    cfgs = [synth.config("n17408", seed=i) for i in range(ngroups)]
    probs = [synth.make_problem(c, dev) for c in cfgs]
    n, rows = cfgs[0].n, cfgs[0].rows
    gpr = n // 32
    S = max(1, args.streams)
    streams = [torch.cuda.Stream(dev) for _ in range(S)]
    wss = [_lib.workspace(lib.gptq_group_workspace_bytes(rows, n), dev) for _ in range(S)]
    outs = [(torch.empty(rows * n // 2, dtype=torch.uint8, device=dev),
             torch.empty(rows * gpr, dtype=torch.uint8, device=dev),
             torch.empty(rows * gpr, dtype=torch.float32, device=dev)) for _ in range(S)]

    def lane(i):
        with torch.cuda.stream(streams[i]):
            for g in range(i, ngroups, S):
                hp, w = probs[g]
                _lib.quantize_group(hp, n, w, cfgs[g].lam, ws=wss[i], want_u=False, want_aux=False, stream=streams[i],
                                    out=outs[i])

    def one_pass(pool):
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream(dev)
        start.record(cur)
        for st in streams:
            st.wait_event(start)
        list(pool.map(lane, range(S)))
        for st in streams:
            ev = torch.cuda.Event()
            ev.record(st)
            cur.wait_event(ev)
        end.record(cur)
        return start, end

    with cf.ThreadPoolExecutor(S) as pool:
        for _ in range(max(warmup, 0)):
            one_pass(pool)
        torch.cuda.synchronize()
        sampler = ClockSampler(dev.index or 0)
        sampler.start()
        time.sleep(0.3)
        l0 = _lib.launch_count()
        t_h0 = time.perf_counter()
        marks = [one_pass(pool) for _ in range(steps)]
        torch.cuda.synchronize()
        t_h1 = time.perf_counter()
        launches = _lib.launch_count() - l0
        clocks = sampler.stop(t_h0, t_h1)
    t = sum(s.elapsed_time(e) for s, e in marks) / 1e3
    out = {"workload": f"batch: {ngroups} independent groups, each " + workload_desc(cfgs[0]).split(": ", 1)[1]
                       + f"; seeds 0..{ngroups - 1}; {S} streams",
           "groups": ngroups, "streams": S, "passes": steps, "warmup": warmup,
           "total_s_per_pass": t / steps, "s_per_group": t / steps / ngroups,
           "groups_per_s": ngroups * steps / t, "gpu_launches": launches, "clocks": clocks,
           "timing": "CUDA events: one event every stream waits on, one that waits on every stream"}
    del probs, wss, outs
    torch.cuda.empty_cache()
    return out


def run_batch(args, rank, world, dev, lib, _lib, torch, synth):
    b = batch_measure(args, dev, lib, _lib, torch, synth, args.steps, args.warmup)
    t_max, value = aggregate(b["s_per_group"] * args.steps, args.steps, world, None)
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": b["total_s_per_pass"] * 1e3, "higher_is_better": False,
                "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": b["workload"], "groups_per_step": b["groups"],
                           "groups_per_s": b["groups_per_s"], "l2": "inputs larger than L2; no flush"},
                "gpu_launches": b["gpu_launches"], "clocks": b["clocks"]}
        print(json.dumps(line), flush=True)


def run_gram(args, rank, world, dev, lib, _lib, torch, synth):
    """The calibration step in front of the fold: H += X^T X for one window
    of T = 32768 tokens at n = 17408 (X = the group's activations as
    [tokens, channels]), into a packed H resident in HBM."""
    cfg = synth.config("n17408", seed=rank)
    n, T = cfg.n, cfg.T
    x = synth.make_x(cfg, dev).T.contiguous()  # [T, n]
    hp = torch.zeros(n * (n + 1) // 2, dtype=torch.float32, device=dev)
    ws = _lib.workspace(lib.gptq_gram_workspace_bytes(n), dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(args.warmup, 0)):
        _lib.gram_add(hp, x, ws=ws, stream=stream)
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    time.sleep(0.3)
    l0 = _lib.launch_count()
    _lib.profile_start(100000)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        _lib.gram_add(hp, x, ws=ws, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    prof = _lib.profile_stop()
    launches = _lib.launch_count() - l0
    clocks = sampler.stop()
    t, value = aggregate(e0.elapsed_time(e1) / 1e3, args.steps, world, None)
    flops = n * (n + 1) // 2 * 2 * T
    pk, src = peaks()
    peak = pk.get("bf16_tflops_sustained", pk.get("bf16_tflops")) * TF32_PER_BF16 / 3.0
    ms_g, cnt_g = prof.get("gram_gemm", (0.0, 0))
    ach = flops * args.steps / (ms_g / 1e3) / 1e12 if ms_g > 0 else None
    if rank == 0:
        line = {"metric": "s per calibration window: H += X^T X at n=17408, T=32768 tokens", "value": value,
                "unit": "s/window", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": t / args.steps * 1e3, "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "f32", "data": "synthetic",
                "config": {"workload": f"Gram accumulation, X [{T}, {n}] f32 (the n17408 group's activations), "
                                       "H packed upper f32", "l2": "inputs larger than L2; no flush"},
                "roofline": {"bound": "tensor", "kernel": "gram_gemm", "achieved": ach, "peak": peak,
                             "unit": "TFLOP/s", "frac": (ach / peak) if ach else None, "traffic": None,
                             "flop_per_launch": flops * args.steps / max(cnt_g, 1)},
                "tflops_whole_call": flops / (t / args.steps) / 1e12,
                "per_kernel": {k: {"ms_per_step": v[0] / args.steps, "launches_per_step": v[1] / args.steps}
                               for k, v in prof.items() if not k.startswith("_") and v[1] > 0},
                "gpu_launches": launches, "clocks": clocks}
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="n17408")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--ref-n", type=int, default=None)
    ap.add_argument("--ref-rows", type=int, default=8)
    ap.add_argument("--n", type=int, default=None, help="override n (T = 2n) for small profiling cases")
    ap.add_argument("--rows", type=int, default=None)
    ap.add_argument("--streams", type=int, default=4, help="host threads / streams for --config batch")
    ap.add_argument("--codec", choices=["q4tp", "q2tp"], default="q4tp")
    ap.add_argument("--no-batch", action="store_true",
                    help="leave out the 11-group batch measured after the headline (n17408 q4tp only)")
    ap.add_argument("--batch-passes", type=int, default=3)
    ap.add_argument("--debias", action="store_true",
                    help="add the output debias (W H on the tensor cores, per-row lo shift) to the step")
    args = ap.parse_args()

    import synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = synth.config("n17408" if args.config in ("batch", "gram") else args.config, seed=rank)
    if args.n is not None:
        cfg = dataclasses.replace(cfg, n=args.n, T=2 * args.n, name=f"{args.config}_n{args.n}")
    if args.rows is not None:
        cfg = dataclasses.replace(cfg, rows=args.rows)
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import numpy as np  # noqa: F401
    import torch

    from gptq_post_weight_gb300 import _lib

    if not os.path.exists(_lib.LIB_PATH):
        raise SystemExit("libgptqfold.so is not built (python -m gptq_post_weight_gb300.build)")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=dev)
        pg = dist
    lib = _lib.load()
    if args.config == "batch":
        run_batch(args, rank, world, dev, lib, _lib, torch, synth)
        return
    if args.config == "gram":
        run_gram(args, rank, world, dev, lib, _lib, torch, synth)
        return

    hp, w = synth.make_problem(cfg, dev)
    n, rows = cfg.n, cfg.rows
    gpr = n // 32
    ws = _lib.workspace(lib.gptq_group_workspace_bytes(rows, n), dev)
    q2 = args.codec == "q2tp"
    # Without the debias, the ladder and D are not needed back: they stay in
    # the workspace, and every step passes the library the same arguments
    # (its graph replay keys on them).
    group_call = _lib.quantize_group_q2tp if q2 else _lib.quantize_group

    def quantize(*a, **kw):
        return group_call(*a, want_aux=args.debias, **kw)
    outs = (torch.empty(rows * n // (4 if q2 else 2), dtype=torch.uint8, device=dev),
            torch.empty(rows * gpr, dtype=torch.uint8, device=dev),
            torch.empty(rows * gpr, dtype=torch.float32, device=dev))
    stream = torch.cuda.current_stream(dev)

    ws_db = _lib.workspace(lib.gptq_debias_workspace_bytes(rows, n), dev) if args.debias else None

    def step():
        res = quantize(hp, n, w, cfg.lam, ws=ws, want_u=False, stream=stream, out=outs)
        if args.debias:
            _lib.debias(2 if q2 else 4, w, hp, outs[0], outs[1], res["tab"], res["lost"], outs[2],
                        ws=ws_db, stream=stream)
        return res

    res = None
    for _ in range(max(args.warmup, 0)):
        res = step()
    torch.cuda.synchronize()
    lam_used = res["lam"] if res is not None else None
    tf32_meas = measure_tf32_tflops(torch, dev)

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(local)
    barrier()
    sampler.start()
    time.sleep(0.3)
    launches0 = _lib.launch_count()
    # The headline steps carry no per-launch events (bracketing the 270
    # update launches of a step costs about a millisecond); the roofline's
    # live kernel timing comes from a second timed region below.
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    t_host0 = time.perf_counter()
    e0.record(stream)
    for _ in range(args.steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.perf_counter()
    launches = _lib.launch_count() - launches0
    clocks = sampler.stop(t_host0, t_host1)
    t_dev, value = aggregate(e0.elapsed_time(e1) / 1e3, args.steps, world, pg)

    # Second timed region: the same number of steps with CUDA events around
    # every launch of the two tensor-core update kinds (on the launching
    # stream), for the roofline's achieved rate.
    barrier()
    _lib.profile_start(200000, kinds=("fold_gemm", "fold_strip", "sweep_gemm"))
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = _lib.profile_stop()

    # Per-kernel breakdown: one more (untimed) step with every launch bracketed.
    _lib.profile_start(200000)
    step()
    torch.cuda.synchronize()
    breakdown = _lib.profile_stop()

    # The fold alone through its own entry (the stream path, its pivot-flag
    # readback included), CUDA events on the stream: the fold's wall time per
    # group, side-stream work that overlaps the main stream counted once.
    fold_wall_ms = None
    if not args.debias:
        _lib.fold(hp, n, cfg.lam, ws=ws, stream=stream, want_d=False)
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for _ in range(args.steps):
            _lib.fold(hp, n, cfg.lam, ws=ws, stream=stream, want_d=False)
        f1.record(stream)
        torch.cuda.synchronize()
        fold_wall_ms = f0.elapsed_time(f1) / args.steps

    # End to end through the public call with host buffers: every step
    # copies its group's inputs from pinned host memory, runs the call and
    # reads its outputs back.  Two device buffer sets and a copy stream let
    # the next group's upload run under the current group's compute (the
    # call returns once its stream is idle, so a set is free again by then).
    e2e = None
    if not args.no_e2e:
        hp_h = hp.cpu().pin_memory()
        w_h = w.cpu().pin_memory()
        outs_h = [tuple(torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs) for _ in range(2)]
        sets = [(torch.empty_like(hp), torch.empty_like(w), outs),
                (torch.empty_like(hp), torch.empty_like(w), tuple(torch.empty_like(o) for o in outs))]
        copy = torch.cuda.Stream(dev)
        ready = [torch.cuda.Event(), torch.cuda.Event()]

        def upload(j):
            hp_d, w_d, _ = sets[j % 2]
            with torch.cuda.stream(copy):
                hp_d.copy_(hp_h, non_blocking=True)
                w_d.copy_(w_h, non_blocking=True)
                ready[j % 2].record(copy)

        def e2e_run(k):
            upload(0)
            for j in range(k):
                if j + 1 < k:
                    upload(j + 1)
                hp_d, w_d, o_d = sets[j % 2]
                stream.wait_event(ready[j % 2])
                res_d = quantize(hp_d, n, w_d, cfg.lam, ws=ws, want_u=False, stream=stream, out=o_d)
                if args.debias:
                    _lib.debias(2 if q2 else 4, w_d, hp_d, o_d[0], o_d[1], res_d["tab"], res_d["lost"], o_d[2],
                                ws=ws_db, stream=stream)
                copy.wait_stream(stream)
                with torch.cuda.stream(copy):
                    for o_h, o in zip(outs_h[j % 2], o_d):
                        o_h.copy_(o, non_blocking=True)
            torch.cuda.synchronize()

        # A run of groups as the pages quantize them (rounds of 11): the first
        # group's upload and the last group's readback have nothing to hide
        # under, and a run of 11 spreads them as a run of that length does.
        e2e_steps = max(args.steps, 11)
        e2e_run(max(args.warmup, 4))  # both buffer sets seen twice: replayed from then on
        barrier()
        t0 = time.perf_counter()
        e2e_run(e2e_steps)
        t_e2e, v_e2e = aggregate(time.perf_counter() - t0, e2e_steps, world, pg)
        e2e = {"value": v_e2e, "unit": UNIT,
               "h2d_bytes_per_step": hp.numel() * 4 + w.numel() * 4,
               "d2h_bytes_per_step": sum(o.numel() * o.element_size() for o in outs),
               "steps": e2e_steps,
               "overlap": "next group's upload on a copy stream under the current group's compute; "
                          "the first upload and the last readback are inside the timed run"}

    # The 11-group batch (seeds 0..10 on several streams), after the headline.
    batch = None
    if (not args.no_batch and world == 1 and not q2 and not args.debias and args.config == "n17408"
            and args.n is None and args.rows is None):
        batch = batch_measure(args, dev, lib, _lib, torch, synth, max(1, args.batch_passes), 2)

    # Roofline of the dominant kernel kind, from the live event timings.
    # 3xTF32: three TF32 MMAs per f32 product, so the algorithmic rate is held
    # against one third of the TF32 dense peak.  That peak is measured here
    # (cuBLAS TF32, a burst figure); it is used as is when the SM clocks
    # stayed at their maximum through the timed region (no power or thermal
    # reason), else scaled by the driver's sustained / burst bf16 ratio.
    pk, src = peaks()
    at_max = bool(clocks and clocks.get("sm_max_mhz") and clocks["sm_mhz"] >= 0.98 * clocks["sm_max_mhz"]
                  and not clocks.get("reasons"))
    if tf32_meas:
        tf32 = tf32_meas if at_max else tf32_meas * pk.get("bf16_tflops_sustained", 1.0) / pk.get("bf16_tflops", 1.0)
        peak_src = (f"measured here: cuBLAS TF32 8192^3 best of 10 = {tf32_meas:.1f} TFLOP/s"
                    + ("" if at_max else " x the driver's bf16 sustained/burst ratio (clocks left their maximum)")
                    + " / 3 (3xTF32 split)")
    else:
        tf32 = pk.get("bf16_tflops_sustained", pk.get("bf16_tflops")) * TF32_PER_BF16
        peak_src = f"{src} bf16 sustained x 1.1/2.25 (nominal TF32 ratio) / 3 (3xTF32 split)"
    peak = tf32 / 3.0
    kinds = {k: v for k, v in prof.items() if k in ("fold_gemm", "sweep_gemm")}
    top = max(kinds, key=lambda k: kinds[k][0])
    ms_top, cnt_top = kinds[top]
    flops = {"fold_gemm": fold_gemm_flops(n, part="trailing") * args.steps,
             "sweep_gemm": sweep_gemm_flops(rows, n) * args.steps}
    roof = None
    if top in flops and cnt_top > 0:
        per_launch = flops[top] / cnt_top
        achieved = per_launch / (ms_top / cnt_top / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": top, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": TRAFFIC.get(top),
                "timing": f"CUDA events around each launch of this kind over a second timed region of "
                          f"{args.steps} steps (the headline steps carry no events)",
                "peak_source": peak_src, "flop_per_launch": per_launch}
    fold_flops = 2 * n ** 3 / 3
    per_kind = {k: {"ms_per_step": v[0], "launches_per_step": v[1]}
                for k, v in breakdown.items() if not k.startswith("_") and v[1] > 0}
    fold_kinds = ("fold_gemm", "build", "potrf", "trsm", "diag", "fold_strip")
    fold_ms_kinds = sum(per_kind.get(k, {}).get("ms_per_step", 0.0) for k in fold_kinds)
    fold_ms = fold_wall_ms if fold_wall_ms else fold_ms_kinds
    fold_tflops = fold_flops / (fold_ms / 1e3) / 1e12 if "fold_gemm" in per_kind and fold_ms > 0 else None
    sweep_ms = per_kind.get("sweep_gemm", {}).get("ms_per_step")
    sweep_tflops = sweep_gemm_flops(rows, n) / (sweep_ms / 1e3) / 1e12 if sweep_ms else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        est, sample, spent = cpu_baseline_sample(cfg, n_fold=args.ref_n, rows_sweep=args.ref_rows,
                                                 codec=args.codec)
        cpu = {"value": est, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": (METRIC_Q2 if q2 else METRIC).replace(") at", "+debias) at") if args.debias
                      else (METRIC_Q2 if q2 else METRIC), "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_dev / args.steps * 1e3, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": workload_desc(cfg, args.codec), "n": n, "rows": rows, "lambda_used": lam_used,
                       "l2": "inputs larger than L2 (H_packed %.0f MB, W %.0f MB, U %.0f MB); no flush"
                             % (hp.numel() * 4 / 1e6, w.numel() * 4 / 1e6, n * n * 4 / 1e6),
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": roof,
            "fold_tflops_algorithmic": fold_tflops,
            "fold_frac": fold_tflops / peak if fold_tflops else None,
            "fold_frac_what": ("whole fold, 2 n^3 / 3 algorithmic flops over "
                               + ("its wall time per group (the fold entry alone, CUDA events on its stream, "
                                  "stream path: no graph replay)" if fold_wall_ms else
                                  "the sum of its kernels' times per group")
                               + ", against the 3xTF32 peak of roofline.peak"),
            "fold_ms": fold_ms,
            "fold_ms_sum_of_kernels": fold_ms_kinds,
            "sweep_gemm_tflops_algorithmic": sweep_tflops,
            "sweep_gemm_frac": sweep_tflops / peak if sweep_tflops else None,
            "sweep_gemm_frac_what": "every trailing update of the sweep (thin and K = 512), rows n^2 algorithmic "
                                    "flops over their time per group, against the same peak",
            "batch": batch,
            "per_kernel": per_kind,
            "per_kernel_source": "one extra untimed step with every launch bracketed by events",
            "hbm": {"unit": "GB/s", "peak": pk.get("hbm_gbs"), "peak_source": src,
                    "kernels": hbm_report(per_kind, n, rows, args.codec, pk.get("hbm_gbs"))},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
            "peaks": {"source": src, "hbm_gbs": pk.get("hbm_gbs"), "bf16_tflops": pk.get("bf16_tflops"),
                      "bf16_tflops_sustained": pk.get("bf16_tflops_sustained"),
                      "tf32_tflops_measured": tf32_meas,
                      "tf32_tflops_nominal_ratio": pk.get("bf16_tflops", 0) * TF32_PER_BF16,
                      "tf32_used": tf32, "clocks_at_max": at_max},
        }
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
