"""Benchmark of the swizzled GEMM hot path on GB300.

One step = one C = A*B on the 8192^3 BF16 workload (A, B ~ N(0,1), FP32
accumulate and output), 2-CTA clusters with 256 x 256 cluster tiles and the
cluster-persistent scheduler (num_clusters = co-resident CTA pairs), in the
headline tile order.  Inputs are resident in HBM; L2 is flushed (a write of
twice its size) before every timed step and the step is timed alone with CUDA
events on the launching stream.

Also reported on the same JSON line:
  sweep        every order of the headline configuration: TFLOP/s, fraction
               of the measured peak, the offline L2 model's hit rate and DRAM
               bytes (the first page's model, and the two-die reading run on
               the kernel's own K order: odd waves descending in persistent
               launches), and the ncu figures recorded for this kernel source
  configs      the same sweep for the specification's other configurations:
               1024x1024x512 fp16, 4096^3 fp16 (1-CTA 128 x 256 tiles,
               persistent and one CTA per tile), 6144x10240x4096 fp16
               (128 x 128 CTA tiles)
  roofline     the GEMM kernel against the measured bf16 tensor peak
  e2e          the same GEMM through the public API from pinned host buffers,
               host->device and device->host copies inside the timed region
  transpose    swz_transpose 16384 x 32768 (naive / padded / xor) in GB/s
  cpu_baseline the CPU oracle (FP64, all host cores) on a bounded row sample
  clocks       nvidia-smi samples taken over the timed headline steps and one
               second more of the same steps (clocks_whole_run: the whole run)

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl swz|reference]
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GEMM TFLOP/s & % FP16 tensor peak per swizzle order; L2 hit rate vs model"
# The configurations of the specification.  The default (timed headline) is
# the 8192^3 bf16 CTA-pair one; the others are selectable with --workload.
_ALL = [("row", 1), ("col", 1), ("panel", 2), ("panel", 4), ("panel", 8), ("panel", 16),
        ("serpentine", 4), ("serpentine", 8), ("serpentine", 16), ("morton", 1), ("xor", 1)]
WORKLOADS = {
    # sweep: the orders each configuration of the specification names
    "gemm8192_bf16_pair": dict(M=8192, N=8192, K=8192, dtype="bf16", dist="normal",
                               cfg=dict(cta_pair=True), tile=(128, 256), cluster_m=2,
                               sweep=[o for o in _ALL if o != ("panel", 2)]),
    "gemm4096_fp16": dict(M=4096, N=4096, K=4096, dtype="fp16", dist="uniform",
                          cfg=dict(tile_n=256), tile=(128, 256), cluster_m=1,
                          sweep=_ALL + [("serpentine", 2)]),
    "gemm4096_fp16_pair": dict(M=4096, N=4096, K=4096, dtype="fp16", dist="uniform",
                               cfg=dict(cta_pair=True), tile=(128, 256), cluster_m=2,
                               sweep=_ALL + [("serpentine", 2)]),
    "gemm6144x10240x4096_fp16": dict(M=6144, N=10240, K=4096, dtype="fp16", dist="uniform",
                                     cfg=dict(tile_n=128), tile=(128, 128), cluster_m=1,
                                     sweep=[("row", 1), ("col", 1), ("panel", 4), ("panel", 8),
                                            ("panel", 16), ("serpentine", 4),
                                            ("serpentine", 8), ("serpentine", 16)]),
    "gemm6144x10240x4096_fp16_pair": dict(M=6144, N=10240, K=4096, dtype="fp16",
                                          dist="uniform", cfg=dict(cta_pair=True, tile_n=128),
                                          tile=(128, 128), cluster_m=2,
                                          sweep=[("row", 1), ("col", 1), ("panel", 4),
                                                 ("panel", 8), ("panel", 16),
                                                 ("serpentine", 4), ("serpentine", 8),
                                                 ("serpentine", 16)]),
    "gemm1024x1024x512_fp16": dict(M=1024, N=1024, K=512, dtype="fp16", dist="uniform",
                                   cfg=dict(tile_n=128), tile=(128, 128), cluster_m=1,
                                   sweep=[("row", 1), ("col", 1), ("panel", 4), ("morton", 1),
                                          ("xor", 1), ("serpentine", 2)]),
}
HEADLINE = dict(order="serpentine", group=8, persistent=True)
SWEEP = WORKLOADS["gemm8192_bf16_pair"]["sweep"]

# The other configurations of the specification, timed in the default run
# beside the headline, each in a sub-object of the line: (key, workload,
# launch modes) and the orders each names.
_G = (2, 4, 8, 16)
CONFIG_SWEEPS = [
    ("cfg1_1024x1024x512_fp16", "gemm1024x1024x512_fp16", (True,)),
    ("cfg2_4096_fp16_tile128x256", "gemm4096_fp16", (True, False)),
    ("cfg2_4096_fp16_tile128x256_pair", "gemm4096_fp16_pair", (True, False)),
    ("cfg4_6144x10240x4096_fp16_tile128x128", "gemm6144x10240x4096_fp16_pair", (True,)),
]
CONFIG_ORDERS = {
    "cfg1_1024x1024x512_fp16": [("row", 1), ("col", 1), ("panel", 4), ("morton", 1),
                                ("xor", 1), ("serpentine", 2)],
    "cfg2_4096_fp16_tile128x256": ([("row", 1), ("col", 1)] + [("panel", g) for g in _G]
                                   + [("serpentine", g) for g in _G]
                                   + [("morton", 1), ("xor", 1)]),
    "cfg2_4096_fp16_tile128x256_pair": ([("row", 1), ("col", 1)] + [("panel", g) for g in _G]
                                        + [("serpentine", g) for g in _G]
                                        + [("morton", 1), ("xor", 1)]),
    "cfg4_6144x10240x4096_fp16_tile128x128": ([("row", 1), ("col", 1)]
                                              + [("panel", g) for g in (4, 8, 16)]
                                              + [("serpentine", g) for g in (4, 8, 16)]),
}

# ncu figures of the GEMM kernel, per workload: one cold launch per order
# (`--only sweep`: the L2 hit rate lts__t_sector_hit_rate.pct and
# dram__bytes_read.sum) and the DRAM traffic (read + write) of the headline
# launch.  They are counters of a capture, not of this run, and hold only
# for the gemm.cu code they were taken on (code_hash: the SHA-256 prefix of
# the source without comments and whitespace); for any other code they are
# left out of the line.
NCU = {
    "gemm8192_bf16_pair": {
        "source": {"gemm_cu_code_hash": "61c4fd4006e5d62d", "captured": "2026-12-02",
                   "kernel": "gemm_kernel<256, 1, 0, 128, 0>", "stream_k": True,
                   "command": "ncu --metrics lts__t_sector_hit_rate.pct,dram__bytes_read.sum --clock-control none "
                              "-k regex:gemm_kernel -s 10 -c 10 python bench.py --workload gemm8192_bf16_pair "
                              "--only sweep --no-cpu; traffic: ncu --set full -k regex:gemm_kernel -s 3 -c 1 "
                              "python bench.py --only gemm --steps 1 --warmup 3 --no-cpu"},
        "traffic_bytes": 873719296 + 276592640, "traffic_order": ("serpentine", 8),
        "orders": {("row", 1): (66.9, 1498279936), ("col", 1): (66.22, 1487829504),
                   ("panel", 4): (70.69, 1263904000), ("panel", 8): (75.16, 952798720),
                   ("panel", 16): (73.42, 925908224), ("serpentine", 4): (73.44, 1078299904),
                   ("serpentine", 8): (76.76, 874268416), ("serpentine", 16): (75.54, 917067776),
                   ("morton", 1): (70.1, 1084324096), ("xor", 1): (70.37, 1453511424)}},
    "gemm4096_fp16": {
        "source": {"gemm_cu_code_hash": "61c4fd4006e5d62d", "captured": "2026-12-02",
                   "kernel": "gemm_kernel<256, 0, 0, 128, 0>", "stream_k": True,
                   "command": "ncu --metrics lts__t_sector_hit_rate.pct,dram__bytes_read.sum --clock-control none "
                              "-k regex:gemm_kernel -s 12 -c 12 python bench.py --workload gemm4096_fp16 "
                              "--only sweep --no-cpu"},
        "orders": {("row", 1): (80.78, 84835328), ("col", 1): (75.93, 87338496),
                   ("panel", 2): (79.43, 87023616), ("panel", 4): (80.59, 92467200),
                   ("panel", 8): (78.62, 96026880), ("panel", 16): (74.01, 111985664),
                   ("serpentine", 4): (79.83, 97025280), ("serpentine", 8): (78.52, 100045568),
                   ("serpentine", 16): (81.52, 84868352), ("morton", 1): (75.17, 109900544),
                   ("xor", 1): (73.91, 111733504), ("serpentine", 2): (76.14, 93911040)}},
    "gemm6144x10240x4096_fp16_pair": {
        "source": {"gemm_cu_code_hash": "61c4fd4006e5d62d", "captured": "2026-12-02",
                   "kernel": "gemm_kernel<128, 1, 0, 128, 0>", "stream_k": True,
                   "command": "ncu --metrics lts__t_sector_hit_rate.pct,dram__bytes_read.sum --clock-control none "
                              "-k regex:gemm_kernel -s 8 -c 8 python bench.py --workload gemm6144x10240x4096_fp16_pair "
                              "--only sweep --no-cpu"},
        "orders": {("row", 1): (70.57, 864301824), ("col", 1): (82.7, 264039680),
                   ("panel", 4): (77.38, 561634048), ("panel", 8): (83.48, 322198784),
                   ("panel", 16): (84.62, 247439360), ("serpentine", 4): (82.12, 380236032),
                   ("serpentine", 8): (83.33, 323559168), ("serpentine", 16): (83.25, 294002432)}},
}


def code_hash(text):
    """SHA-256 prefix of C++ source text with its comments and whitespace
    removed: two sources that differ only in comments or layout share it."""
    parts, code, i, n = [], [], 0, len(text)

    def flush():
        parts.append(re.sub(r"\s+", " ", "".join(code)))
        code.clear()
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            flush()
            parts.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            i = text.find("\n", i)
            i = n if i < 0 else i
            code.append(" ")
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            code.append(" ")
        else:
            code.append(c)
            i += 1
    flush()
    joined = "".join(parts).strip()
    # spaces next to punctuation carry no meaning either
    joined = re.sub(r" ?([{}()\[\];,]) ?", r"\1", joined)
    return hashlib.sha256(joined.encode()).hexdigest()[:16]


def _gemm_src_hash():
    """The code hash of csrc/gemm.cu (ncu figures hold for one kernel code)."""
    with open(os.path.join(ROOT, "thread_block_smem_gb300", "csrc", "gemm.cu")) as f:
        return code_hash(f.read())


def ncu_record(workload):
    """The recorded ncu figures of `workload` if they were taken on the
    current gemm.cu source, else None."""
    rec = NCU.get(workload)
    if rec is None or rec["source"]["gemm_cu_code_hash"] != _gemm_src_hash():
        return None
    return rec


def resolve_workload(args):
    """The workload of the run: a named configuration, or a custom shape
    (--m/--n/--k with --dtype, --tile-n, --pair; the first page's benchmark
    flags), with the sweep's grouped orders at --group-sizes."""
    if args.m or args.n or args.k:
        if not (args.m and args.n and args.k):
            raise SystemExit("--m, --n and --k go together")
        tn = args.tile_n or 256
        wl = dict(M=args.m, N=args.n, K=args.k, dtype=args.dtype,
                  dist="normal" if args.dtype == "bf16" else "uniform",
                  cfg=dict(cta_pair=True, tile_n=tn) if args.pair else dict(tile_n=tn),
                  tile=(128, tn), cluster_m=2 if args.pair else 1, sweep=list(_ALL))
        args.workload = (f"custom{args.m}x{args.n}x{args.k}_{args.dtype}"
                         + (f"_pair{tn}" if args.pair else f"_tile{tn}"))
    else:
        wl = dict(WORKLOADS[args.workload])
    if args.group_sizes:
        gs = [int(x) for x in args.group_sizes.split(",") if x]
        if any(g < 1 for g in gs):
            raise SystemExit("--group-sizes: positive integers")
        wl["sweep"] = ([o for o in wl["sweep"] if o[0] not in ("panel", "serpentine")]
                       + [("panel", g) for g in gs] + [("serpentine", g) for g in gs])
    return wl


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clock, utilisation and throttle reasons while
    running; mark(tag) labels the samples taken from then on (None: no
    label), so that a summary can cover one phase of the run."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,utilization.gpu,"
         "clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.marks = []  # (time, tag)
        self.rows = []

    def mark(self, tag):
        self.marks.append((time.time(), tag))

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.rows = []
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [[x.strip() for x in line.split(",")] for line in out.strip().splitlines()]
        for r in rows:
            if len(r) < 10:
                continue
            try:  # the sample's local wall time
                t = datetime.datetime.strptime(r[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            r = r[1:]
            tag = None
            for tm, tg in self.marks:
                if tm <= t:
                    tag = tg
            self.rows.append((tag, r))

    def summary(self, *tags):
        """Median SM clock over the samples of the phases `tags` (all samples
        when none is given) taken while the GPU was busy (utilisation >= 50
        %), the maximum clock and every throttle reason seen active."""
        rows = [r for tg, r in self.rows if not tags or tg in tags]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        busy = [r for r in rows if (num(r[3]) or 0) >= 50]
        sm = [num(r[0]) for r in (busy or rows) if num(r[0])]
        pw = [num(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(num(r[1]) or 0 for r in rows),
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(rows), "samples_busy": len(busy)}


def spearman(xs, ys):
    """Rank correlation as the first page's benchmark reports it: ranks are
    positions after a stable ascending sort (no tie averaging), then the
    Pearson correlation of the ranks; 0 when a rank vector is constant."""
    def pos(v):
        r = [0] * len(v)
        for p, i in enumerate(sorted(range(len(v)), key=lambda i: v[i])):
            r[i] = p
        return r
    if len(xs) < 2:
        return 0.0
    rx, ry = pos(xs), pos(ys)
    mx, my = statistics.mean(rx), statistics.mean(ry)
    sxy = sum((a - mx) * (b - my) for a, b in zip(rx, ry))
    sxx = sum((a - mx) ** 2 for a in rx)
    syy = sum((b - my) ** 2 for b in ry)
    return sxy / (sxx * syy) ** 0.5 if sxx and syy else 0.0


def max_over_ranks(value, device=None):
    """Max of a float over all ranks of the initialised process group (the
    identity without one).  Used for the per-step time: the slowest replica
    sets the job's time."""
    import torch
    import torch.distributed as tdist
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def _dist():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def cpu_baseline(M, N, K, dtype, dist, target_s=12.0):
    """Times the CPU oracle (FP64 GEMM, all host cores) on a bounded sample:
    whole rows of C, as many 8-row slabs as fit in about ``target_s``."""
    import torch
    import synth_inputs as si
    from oracle import ref
    A, B = si.gemm_inputs(M, N, K, dtype, dist, seed=0)
    a64, b64 = A.double(), B.double()
    del A, B
    ref.gemm_f64_widened(a64, b64, 0, 1)  # warm (page in B)
    rows, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < target_s and rows < M:
        ref.gemm_f64_widened(a64, b64, rows, min(rows + 8, M))
        rows = min(rows + 8, M)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": ref.num_threads(),
            "kind": "oracle", "sample": f"rows 0..{rows} of the {M}x{N}x{K} {dtype} product "
            f"({flops / 1e9:.1f} GFLOP in {dt:.1f} s, FP64)"}


def run_reference(args):
    rank, world, _ = _dist()
    if rank != 0:
        return
    wl = resolve_workload(args)
    M, N, K = wl["M"], wl["N"], wl["K"]
    import synth_inputs as si
    from oracle import ref
    A, B = si.gemm_inputs(M, N, K, wl["dtype"], wl["dist"], seed=0)
    a64, b64 = A.double(), B.double()
    rows = 8  # one step = an 8-row slab of C (about a second of host work)
    for _ in range(args.warmup):
        ref.gemm_f64_widened(a64, b64, 0, rows)
    t0 = time.perf_counter()
    for s in range(args.steps):
        r0 = (s * rows) % M
        ref.gemm_f64_widened(a64, b64, r0, r0 + rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * N * K * args.steps
    v = flops / dt / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}: gemm {M}x{N}x{K} {wl['dtype']} -> fp32",
                       "note": "CPU oracle, FP64; each step computes 8 rows of C"},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": ref.num_threads(),
                             "kind": "oracle", "sample": f"{rows} rows of C per step"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_swz(args):
    import torch
    import torch.distributed as tdist

    import synth_inputs as si
    import thread_block_smem_gb300 as swz
    from thread_block_smem_gb300 import build

    rank, world, local = _dist()
    if world > 1:
        tdist.init_process_group("nccl")
    torch.cuda.set_device(local)
    build.build()
    dev = torch.device("cuda", local)
    rc, (sms, l2_bytes, ccmaj, ccmin) = swz.swz_device_info()
    peaks, peak_src = _peaks()
    stream = torch.cuda.current_stream()
    flush = torch.empty(2 * max(l2_bytes, 64 << 20) // 4, dtype=torch.float32, device=dev)
    do_gemm = args.only in ("all", "gemm", "sweep", "swizzle", "launch")
    do_transpose = args.only in ("all", "transpose") and not args.no_transpose
    do_mma_sync = args.only in ("all", "mma_sync") and not args.no_mma_sync

    wl = resolve_workload(args)
    M, N, K = wl["M"], wl["N"], wl["K"]
    cfg = dict(wl["cfg"])
    persistent = not args.non_persistent
    if args.num_programs:  # the headline GEMM on fewer programs (per-SM rate)
        cfg["num_programs"] = args.num_programs
    flops = 2.0 * M * N * K
    line = {"metric": METRIC, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl["dtype"], "data": "synthetic"}
    if args.die_split:
        dies = swz.calibrate()
        line["die_calibration"] = {"sms_per_die": [dies.count(0), dies.count(1)]}
    head_order = args.order or HEADLINE["order"]
    head_group = args.group or HEADLINE["group"]

    if do_gemm and args.stream_k is None:
        # by default Stream-K where the launch has a full wave of tiles (see sweep())
        _, (_, _, sm_, sn_, cap) = swz.swz_gemm_plan(M, N, K, 1,
                                                    swz.make_opts(stream_k=True, **cfg))
        args.stream_k = persistent and sm_ * sn_ >= cap // (2 if cfg.get("cta_pair") else 1)
    args.stream_k = bool(args.stream_k) and persistent
    if do_gemm:
        A, B = si.gemm_inputs(M, N, K, wl["dtype"], wl["dist"], seed=0)
        Ad, Bd = A.to(dev), B.to(dev)
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
        _, (_, _, _, _, programs) = swz.swz_gemm_plan(
            M, N, K, int(persistent), swz.make_opts(stream_k=args.stream_k, **cfg))
        ws = None
        if args.stream_k:
            nws = swz.workspace_size(M, N, K, persistent, **cfg)
            ws = torch.zeros(max(nws, 256), dtype=torch.uint8, device=dev)

    def gemm_once(order, group, span=0):
        swz.gemm(Ad, Bd, order, group, persistent, out=C, stream_k=args.stream_k,
                 workspace=ws, smem_swizzle=span, die_split=args.die_split, **cfg)

    def timed(fn, steps, warmup):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        ev = []
        for _ in range(steps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            ev.append((e0, e1))
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev]

    def model(order, g, w, conc, parts, k_alternate=False):
        """The offline L2 model at the kernel's tiling: hit % and DRAM bytes."""
        tk = 128 if w["tile"][1] == 128 else 64  # K per stage: two atoms for 128-wide tiles
        return swz.l2_model_predict(order, g, w["M"], w["N"], w["K"], w["tile"][0], w["tile"][1],
                                    tk, 2, model_l2, conc, w["cluster_m"], l2_partitions=parts,
                                    k_alternate=k_alternate)

    model_l2 = int(args.l2_cache_mb * 2**20) if args.l2_cache_mb else l2_bytes

    def sweep(name, w, persist, steps, warmup):
        """Every order of workload `w`: median TFLOP/s of L2-flushed launches,
        fraction of the measured peak, the L2 model (the first page's, and the
        two-die reading) and, where recorded for this kernel source, ncu."""
        wM, wN, wK = w["M"], w["N"], w["K"]
        wf = 2.0 * wM * wN * wK
        wA, wB = si.gemm_inputs(wM, wN, wK, w["dtype"], w["dist"], seed=0)
        wA, wB = wA.to(dev), wB.to(dev)
        wC = torch.empty((wM, wN), dtype=torch.float32, device=dev)
        wcfg = dict(w["cfg"])
        _, (_, _, _, _, progs) = swz.swz_gemm_plan(wM, wN, wK, int(persist), swz.make_opts(**wcfg))
        _, (_, _, sm_, sn_, cap) = swz.swz_gemm_plan(wM, wN, wK, 1,
                                                    swz.make_opts(stream_k=True, **wcfg))
        cl = 2 if wcfg.get("cta_pair") else 1
        # the headline's scheduler, Stream-K, where the launch has a full wave
        # of tiles to overlap its exchange with (with fewer tiles than
        # programs every tile would be split and the exchange is exposed)
        if persist and args.stream_k is not False and sm_ * sn_ >= cap // cl:
            nws = swz.workspace_size(wM, wN, wK, True, **wcfg)
            wcfg.update(stream_k=True,
                        workspace=torch.zeros(max(nws, 256), dtype=torch.uint8, device=dev))
        # the model's wave: resident CTAs (the first page's min(tiles, capacity)),
        # unless overridden (its --num-sms)
        conc = args.num_sms if args.num_sms else progs
        rec = ncu_record(name) if persist else None
        out = []
        for order, g in w["sweep"]:
            fn = lambda: swz.gemm(wA, wB, order, g, persist, out=wC, **wcfg)
            try:
                t = timed(fn, steps, warmup)
            except swz.SwzError as e:  # Morton / XOR on a grid they do not permute
                out.append({"order": order, "group": g, "error": swz.strerror(e.code)})
                continue
            med = statistics.median(t)
            hit, dram = model(order, g, w, conc, 1)
            # the two-die reading on the K order the kernel runs: in a
            # persistent launch every other wave takes K descending
            hit2, dram2 = model(order, g, w, conc, 2, k_alternate=persist)
            o = {"order": order, "group": g, "ms": med, "tflops": wf / med / 1e9,
                 "frac_of_peak": wf / med / 1e9 / peaks["bf16_tflops"],
                 "l2_model_hit_pct": hit, "l2_model_dram_read_bytes": dram,
                 "l2_model_2die_hit_pct": hit2, "l2_model_2die_dram_read_bytes": dram2}
            if rec and (order, g) in rec["orders"]:
                nh, nd = rec["orders"][(order, g)]
                o.update({"ncu_l2_hit_pct": nh, "ncu_dram_read_bytes": nd,
                          "l2_model_2die_dram_err": (dram2 - nd) / nd})
            out.append(o)
        del wA, wB, wC
        res = {"shape": [wM, wN, wK], "dtype": w["dtype"],
               "cfg": {k: v for k, v in wcfg.items() if k != "workspace"},
               "persistent": persist, "programs": progs, "orders": out,
               "model": {"l2_bytes": model_l2, "concurrency_ctas": conc}}
        good = [o for o in out if "tflops" in o]
        if len(good) > 1:
            res["spearman_l2_model_vs_tflops"] = spearman(
                [o["l2_model_hit_pct"] for o in good], [o["tflops"] for o in good])
        meas = [o for o in good if "ncu_dram_read_bytes" in o]
        if len(meas) > 1:
            res["ncu_source"] = rec["source"]
            res["spearman_model_dram_vs_ncu_dram"] = {
                "full_l2": spearman([o["l2_model_dram_read_bytes"] for o in meas],
                                    [o["ncu_dram_read_bytes"] for o in meas]),
                "two_die": spearman([o["l2_model_2die_dram_read_bytes"] for o in meas],
                                    [o["ncu_dram_read_bytes"] for o in meas])}
            res["l2_model_2die_dram_abs_err_max"] = max(abs(o["l2_model_2die_dram_err"])
                                                        for o in meas)
        return res

    def back_to_back(w, order, g, calls=50, reps=7):
        """Device time per call of `calls` GEMMs of workload `w` recorded in one
        CUDA graph and replayed back to back (each kernel starts its prologue
        while the previous one finishes: programmatic dependent launch).  L2
        is flushed before each replay; the operands stay in L2 after the
        first call."""
        bM, bN, bK = w["M"], w["N"], w["K"]
        bA, bB = si.gemm_inputs(bM, bN, bK, w["dtype"], w["dist"], seed=0)
        bA, bB = bA.to(dev), bB.to(dev)
        bC = torch.empty((bM, bN), dtype=torch.float32, device=dev)

        def run():
            for _ in range(calls):
                swz.gemm(bA, bB, order, g, True, out=bC, **w["cfg"])

        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            run()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            run()
        graph.replay()
        torch.cuda.synchronize()
        per = []
        for _ in range(reps):
            flush.fill_(1.0)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) / 1e3 / calls)
        del graph, bA, bB, bC
        t = statistics.median(per)
        return {"order": order, "group": g, "calls": calls, "persistent": True,
                "device_us_per_call": t * 1e6, "tflops": 2.0 * bM * bN * bK / t / 1e12,
                "how": "one CUDA graph of back-to-back calls, CUDA events around each "
                       "replay; L2 flushed before each replay"}

    sampler = ClockSampler(local)
    ms = None
    with sampler:
        if args.only in ("all", "gemm"):
            # ---- headline: K timed steps ------------------------------
            if world > 1:
                tdist.barrier()
            torch.cuda.synchronize()
            sampler.mark("timed")
            ms = timed(lambda: gemm_once(head_order, head_group), args.steps, args.warmup)
            torch.cuda.synchronize()
            # the same steps again, untimed, for about a second: nvidia-smi
            # samples every 50 ms, too coarse for the timed steps alone
            sampler.mark("window")
            t_end = time.time() + 1.0
            while time.time() < t_end:
                timed(lambda: gemm_once(head_order, head_group), 20, 0)
            sampler.mark(None)
            if world > 1:
                tdist.barrier()
        if args.only == "sweep":
            # one cold (L2-flushed) launch per order, for counter capture
            for order, g in wl["sweep"]:
                gemm_once(order, g)
            torch.cuda.synchronize()
            for order, g in wl["sweep"]:
                timed(lambda: gemm_once(order, g), 1, 0)
        elif args.only == "all" and not args.no_sweep:
            line["sweep"] = sweep(args.workload, wl, persistent, max(5, args.steps // 4), 3)
            # the other configurations of the specification, each in its own
            # sub-object (order sweeps; the 4096^3 one also non-persistent)
            if not args.no_configs:
                cf = {}
                for key, wname, modes in CONFIG_SWEEPS:
                    if wname == args.workload:
                        continue
                    w = resolve_workload(argparse.Namespace(**{**vars(args), "workload": wname,
                                                               "m": 0, "n": 0, "k": 0}))
                    cf[key] = {("persistent" if p else "non_persistent"): sweep(wname, w, p, 5, 3)
                               for p in modes}
                    if key.startswith("cfg1"):
                        cf[key]["back_to_back"] = back_to_back(w, "row", 1)
                line["configs"] = cf
        # ---- operand-stage swizzle span (TMA + tensor-core layout) ---------
        spans = []
        if args.only == "swizzle":  # one cold launch per span, for counter capture
            for sp in (128, 64, 32):
                gemm_once(head_order, head_group, sp)
            torch.cuda.synchronize()
        elif args.only == "all" and not args.no_swizzle:
            for sp in (128, 64, 32):
                t = timed(lambda: gemm_once(head_order, head_group, sp), max(5, args.steps // 4),
                          3)
                med = statistics.median(t)
                spans.append({"span_bytes": sp, "ms": med, "tflops": flops / med / 1e9})
        # ---- static (work_idx striding) vs dynamic (atomic counter) -------
        sched = {}
        if args.only == "all" and not args.no_dynamic and persistent:
            dws = torch.zeros(256, dtype=torch.uint8, device=dev)
            nws = swz.workspace_size(M, N, K, True, **cfg)
            sws = torch.zeros(max(nws, 256), dtype=torch.uint8, device=dev)
            for name, kw in (("static", {}), ("stream_k", dict(stream_k=True, workspace=sws)),
                             ("dynamic", dict(dynamic=True, workspace=dws))):
                fn = lambda: swz.gemm(Ad, Bd, head_order, head_group, True, out=C, **kw, **cfg)
                t = timed(fn, max(5, args.steps // 4), 3)
                sched[name] = {"ms": statistics.median(t),
                               "tflops": flops / statistics.median(t) / 1e9}
    # the clock of the headline: samples of the timed steps and of the
    # second of the same steps after them; under sustained dense load the
    # power cap (sw_power_cap) takes the clock down from its maximum within
    # that second, so the median is a lower bound of the timed steps' clock
    clocks = sampler.summary("timed", "window")
    clocks["timed_steps"] = sampler.summary("timed")
    clocks_all = sampler.summary()
    if spans:
        line["smem_swizzle_spans"] = spans
    if sched:
        line["scheduler"] = sched

    if ms is not None:
        ms_step = max_over_ranks(statistics.mean(ms), dev)
        achieved = flops / statistics.mean(ms) / 1e9
        # the captured launch is the default workload's headline launch only
        rec = ncu_record(args.workload)
        traffic = (rec["traffic_bytes"] if rec and "traffic_bytes" in rec and persistent
                   and not args.num_programs
                   and bool(args.stream_k) == rec["source"].get("stream_k", False)
                   and (head_order, head_group) == rec["traffic_order"] else None)
        line.update({
            "value": world * flops / ms_step / 1e9, "ms_per_step": ms_step,
            "config": {"workload": f"{args.workload}: gemm {M}x{N}x{K} {wl['dtype']} "
                                   f"{'N(0,1)' if wl['dist'] == 'normal' else 'U[-1,1)'} -> fp32, "
                                   + (f"2-CTA clusters 256x{cfg.get('tile_n') or 256}"
                                      if cfg.get("cta_pair") else
                                      f"1-CTA tiles 128x{cfg.get('tile_n')}")
                                   + (", persistent" if persistent else ", one CTA per tile")
                                   + (", Stream-K tail" if args.stream_k else ""),
                       "order": head_order, "group": head_group,
                       "programs": programs,
                       "l2": "flushed before every timed step (write of 2x L2)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "device": {"sms": sms, "l2_bytes": l2_bytes, "cc": f"{ccmaj}.{ccmin}"}},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                         "traffic": traffic,
                         "traffic_source": rec["source"] if traffic is not None else None,
                         "peak_source": f"bf16 burst, of {peak_src}"},
            "gpu_launches": args.steps,
        })
    line["clocks"] = clocks
    line["clocks_whole_run"] = clocks_all

    # ---- end to end through the public API from pinned host buffers --------
    # swz_gemm_host: B in, then A in / GEMM / C out overlapped in row slabs;
    # the timed region holds every byte of host<->device traffic of the step.
    if args.only == "all":
        hA, hB = A.pin_memory(), B.pin_memory()
        hC = torch.empty((M, N), dtype=torch.float32).pin_memory()

        def e2e_time(**kw):
            t = []
            for i in range(3 + 5):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                swz.gemm_host(hA, hB, hC, Ad, Bd, C, head_order, head_group,
                              stream_k=args.stream_k, workspace=ws, **kw, **cfg)
                e1.record(stream)
                torch.cuda.synchronize()
                if i >= 3:
                    t.append(e0.elapsed_time(e1))
            # median: a single host-side stall (page-ins of pinned memory,
            # another process on the host) must not decide the figure
            return statistics.median(t)

        # a job of several GEMMs from host memory: consecutive calls alternate
        # between two streams, each with its own device buffers and pinned C,
        # so one call's C leaves while the next call's A and B arrive (the
        # link carries 340 GB/s both ways at once against 210 one way).  Every
        # call still copies its own inputs and result inside the timed region.
        def e2e_streamed(n_calls, **kw):
            sts = [stream, torch.cuda.Stream(device=dev)]
            bufs = [(Ad, Bd, C, hC, ws),
                    (torch.empty_like(Ad), torch.empty_like(Bd), torch.empty_like(C),
                     torch.empty_like(hC).pin_memory(), None if ws is None else torch.zeros_like(ws))]
            t = []
            for rep in range(2 + 5):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                sts[1].wait_stream(stream)
                for i in range(n_calls):
                    a, b, c, h, w = bufs[i % 2]
                    swz.gemm_host(hA, hB, h, a, b, c, head_order, head_group,
                                  stream_k=args.stream_k, workspace=w, stream=sts[i % 2],
                                  **kw, **cfg)
                stream.wait_stream(sts[1])
                e1.record(stream)
                torch.cuda.synchronize()
                if rep >= 2:
                    t.append(e0.elapsed_time(e1) / n_calls)
            return statistics.median(t)  # host memory is shared: one slow rep must not decide

        ms_slabs = e2e_time(slabs=args.e2e_slabs)
        n_calls = max(args.steps, 4)
        ms_job = e2e_streamed(n_calls, slabs=args.e2e_slabs)
        line["e2e"] = {"value": world * flops / ms_job / 1e9, "unit": "TFLOP/s",
                       "h2d_bytes_per_step": hA.numel() * 2 + hB.numel() * 2,
                       "d2h_bytes_per_step": hC.numel() * 4,
                       "api": f"swz_gemm_host, {args.e2e_slabs} row slabs, pinned host "
                              f"buffers; a job of {n_calls} GEMMs on two alternating "
                              "streams, each call with its own copies in and out",
                       "single_call": {"value": world * flops / ms_slabs / 1e9,
                                     "api": f"swz_gemm_host, {args.e2e_slabs} row slabs, "
                                            "one call timed alone"}}
        del hA, hB, hC
    # ---- launch cost: R GEMMs back to back, called one by one and recorded
    # in one CUDA graph (--only launch; for small shapes, where the host work
    # of a call is comparable with its kernel).  Wall clock from the first
    # enqueue to the end of the last kernel, per call; the graph's device
    # time from events around a replay.  L2 stays warm (operands reused).
    if args.only == "launch":
        R, reps = 50, 7

        def calls():
            for _ in range(R):
                gemm_once(head_order, head_group)

        for _ in range(3):
            calls()
        torch.cuda.synchronize()
        eager, enqueue = [], []
        for _ in range(reps):
            t0 = time.perf_counter()
            calls()
            t1 = time.perf_counter()
            torch.cuda.synchronize()
            eager.append((time.perf_counter() - t0) / R)
            enqueue.append((t1 - t0) / R)
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            calls()
        stream.wait_stream(side)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            calls()
        graph.replay()
        torch.cuda.synchronize()
        replay, replay_dev = [], []
        for _ in range(reps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            t0 = time.perf_counter()
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            replay.append((time.perf_counter() - t0) / R)
            replay_dev.append(e0.elapsed_time(e1) / 1e3 / R)
        cold = statistics.median(timed(lambda: gemm_once(head_order, head_group), 10, 3)) / 1e3
        med = statistics.median
        line["launch"] = {
            "calls": R, "reps": reps, "order": head_order, "group": head_group,
            "eager_us_per_call": med(eager) * 1e6,
            "eager_enqueue_us_per_call": med(enqueue) * 1e6,
            "eager_tflops": flops / med(eager) / 1e12,
            "graph_us_per_call": med(replay) * 1e6,
            "graph_device_us_per_call": med(replay_dev) * 1e6,
            "graph_tflops": flops / med(replay) / 1e12,
            "single_launch_cold_l2_us": cold * 1e6}
        del graph

    if do_gemm:
        del A, B, Ad, Bd, C

    # ---- transpose (HBM-bound) ---------------------------------------------
    if do_transpose:
        tr = {}
        sizes = [(16384, 32768)] if args.only == "all" else [(1024, 2048), (16384, 32768)]
        for tm, tn in sizes:
            x = torch.empty((tm, tn), dtype=torch.int32, device=dev).random_()
            y = torch.empty((tn, tm), dtype=torch.int32, device=dev)
            for lay in ("naive", "padded", "xor"):
                t = timed(lambda: swz.transpose(x, lay, out=y), 10 if args.only == "all" else 1,
                          3 if args.only == "all" else 1)
                med = statistics.median(t)
                gbs = 2.0 * tm * tn * 4 / med / 1e6
                tr[f"{lay} {tm}x{tn}"] = {"ms": med, "GB/s": gbs,
                                          "frac_hbm": gbs / peaks["hbm_gbs"]}
            del x, y
        line["transpose"] = tr

    # ---- cuBLAS on the same shape, for counter comparison only -------------
    # (--only cublas: torch.matmul's bf16 kernel with bf16 and with fp32
    # output, three warm-up launches and one cold launch each; never timed
    # into the line's numbers)
    if args.only == "cublas":
        g = torch.Generator().manual_seed(0)
        Ab = torch.randn((M, K), generator=g).to(torch.bfloat16).to(dev)
        Bb = torch.randn((K, N), generator=g).to(torch.bfloat16).to(dev)
        cub = {}
        for name, fn in (("bf16_out", lambda: torch.matmul(Ab, Bb)),
                         ("fp32_out", lambda: torch.mm(Ab, Bb, out_dtype=torch.float32))):
            try:
                t = timed(fn, 1, 3)
                cub[name] = {"ms": t[0], "tflops": flops / t[0] / 1e9}
            except (RuntimeError, TypeError) as e:  # out_dtype not in this torch
                cub[name] = {"error": type(e).__name__}
        line["cublas_reference"] = cub
        del Ab, Bb

    # ---- TF32 path (fp32 inputs, B stored N x K), 8192^3 ---------------------
    # (--only tf32: three warm-up launches and one cold launch, for capture)
    if (args.only == "all" and not args.no_tf32) or args.only == "tf32":
        g = torch.Generator().manual_seed(0)
        A32 = (torch.rand((M, K), generator=g) * 2 - 1).to(dev)
        Bt32 = (torch.rand((N, K), generator=g) * 2 - 1).to(dev)
        C32 = torch.empty((M, N), dtype=torch.float32, device=dev)
        # the headline's scheduler (Stream-K tail when the headline uses it)
        sk32 = {}
        if args.stream_k:
            n32 = swz.workspace_size(M, N, K, True, cta_pair=True)
            sk32 = dict(stream_k=True,
                        workspace=torch.zeros(max(n32, 256), dtype=torch.uint8, device=dev))
        t = timed(lambda: swz.gemm(A32, Bt32, head_order, head_group, True, out=C32,
                                   b_transposed=True, cta_pair=True, **sk32),
                  10 if args.only == "all" else 1, 3)
        med = statistics.median(t)
        # the measured bf16 peak scaled by the TF32 / bf16 rate ratio of the
        # library's own tcgen05 MMAs: 1/2 (4,095 vs 8,190 FLOP per clock per
        # SM); replaced below by this run's ratio when tc_rate runs
        peak_tf32 = peaks["bf16_tflops"] * 0.5
        line["tf32_8192"] = {"ms": med, "tflops": flops / med / 1e9, "stream_k": bool(sk32),
                             "peak": peak_tf32, "frac": flops / med / 1e9 / peak_tf32,
                             "peak_source": "measured bf16 burst x the tcgen05 tf32/bf16 rate "
                                            "ratio 1/2"}
        del A32, Bt32, C32, sk32

    # ---- tensor-core rate of the library's own tcgen05 code (swz_tc_rate) ----
    # FLOP per clock per SM from back-to-back MMAs on shared-memory operands;
    # peaks = SMs x that x SM clock at the maximum clock, at the clock of a
    # short run, and at the clock after about 2 s of full load.
    if args.only in ("all", "tc_rate") and not args.no_tc_rate:
        tc = {}
        max_mhz = clocks.get("sm_max_mhz") or None
        for name, dt, k_row in (("bf16", torch.bfloat16, 64), ("fp16", torch.float16, 64),
                                ("tf32", torch.float32, 32)):
            g = torch.Generator().manual_seed(0)
            At = (torch.rand((128, k_row), generator=g) * 2 - 1).to(dt).to(dev)
            Bt = (torch.rand((256, k_row), generator=g) * 2 - 1).to(dt).to(dev)
            swz.tc_rate(At, Bt, 1024)  # warm-up
            n_short = 16384
            times, flop, _ = swz.tc_rate(At, Bt, n_short)
            cyc, ns = times[:, 0].double(), times[:, 1].double()
            fpc = float((n_short * flop / cyc).median())
            burst_mhz = float((cyc / ns * 1e3).median())
            rec = {"mma": f"128x256x{flop // (2 * 128 * 256)} {name}, one CTA per SM",
                   "flop_per_clk_per_sm": fpc, "short_run_sm_mhz": burst_mhz,
                   "peak_short_run_tflops": sms * fpc * burst_mhz / 1e6}
            if max_mhz:
                rec["sm_max_mhz"] = max_mhz
                rec["peak_max_clock_tflops"] = sms * fpc * max_mhz / 1e6
            if name != "fp16":
                t_end = time.time() + 2.0
                while True:
                    times, _, _ = swz.tc_rate(At, Bt, 1 << 20)
                    if time.time() >= t_end:
                        break
                cyc, ns = times[:, 0].double(), times[:, 1].double()
                load_mhz = float((cyc / ns * 1e3).median())
                rec["loaded_sm_mhz"] = load_mhz
                rec["peak_loaded_tflops"] = sms * fpc * load_mhz / 1e6
            tc[name] = rec
            del At, Bt
        # the issuing thread's stage loop: per stage a barrier test, the
        # tensor fence, S MMAs and a commit (swz_tc_rate_ex), 2-CTA MMAs of
        # 256 x 128 and 256 x 256; fraction of the back-to-back rate above
        g = torch.Generator().manual_seed(1)
        At = (torch.rand((128, 64), generator=g) * 2 - 1).to(torch.bfloat16).to(dev)
        Bt = (torch.rand((256, 64), generator=g) * 2 - 1).to(torch.bfloat16).to(dev)
        issue = []
        for n, stage in ((128, 0), (128, 4), (128, 8), (128, 16), (256, 4), (256, 8)):
            times, flop, _ = swz.tc_rate(At, Bt[:n].contiguous(), 16384, cta_pair=True,
                                         mmas_per_stage=stage)
            cyc = times[:, 0].double()
            f = float((16384 * flop / cyc).median())
            issue.append({"mma": f"256x{n}x16 bf16, CTA pair", "mmas_per_stage": stage,
                          "cycles_per_mma": float((cyc / 16384).median()),
                          "frac_of_rate": f / tc["bf16"]["flop_per_clk_per_sm"]})
        tc["issue_loop"] = issue
        del At, Bt
        if "roofline" in line and "peak_max_clock_tflops" in tc["bf16"]:
            a = line["roofline"]["achieved"]
            tc["headline_frac_of_bf16_max_clock_peak"] = a / tc["bf16"]["peak_max_clock_tflops"]
            tc["headline_frac_of_bf16_loaded_peak"] = a / tc["bf16"]["peak_loaded_tflops"]
        if "tf32_8192" in line:
            t32 = line["tf32_8192"]
            ratio = tc["tf32"]["flop_per_clk_per_sm"] / tc["bf16"]["flop_per_clk_per_sm"]
            t32["peak"] = peaks["bf16_tflops"] * ratio
            t32["frac"] = t32["tflops"] / t32["peak"]
            t32["peak_source"] = (f"measured bf16 burst x this run's tcgen05 tf32/bf16 rate "
                                  f"ratio {ratio:.4f}")
            t32["frac_of_tf32_loaded_peak"] = t32["tflops"] / tc["tf32"]["peak_loaded_tflops"]
        line["tc_rate"] = tc

    # ---- ldmatrix / mma.sync path: operand layout vs bank conflicts ---------
    if do_mma_sync:
        mm = 4096
        Am, Bm = si.gemm_inputs(mm, mm, mm, "fp16", "uniform", seed=0)
        Am, Bm = Am.to(dev), Bm.to(dev)
        Cm = torch.empty((mm, mm), dtype=torch.float32, device=dev)
        res = {}
        for name in ("naive", "padded", "swizzle64", "swizzle128"):
            fn = lambda: swz.gemm_mma_sync(Am, Bm, name, "panel", 8, out=Cm)
            t = timed(fn, 10 if args.only == "all" else 1, 3 if args.only == "all" else 1)
            med = statistics.median(t)
            res[name] = {"ms": med, "tflops": 2.0 * mm ** 3 / med / 1e9,
                         "layout": list(swz.SMEM_LAYOUTS[name])}
        line["mma_sync_4096_fp16"] = res
        del Am, Bm, Cm

    if rank != 0:
        if world > 1:
            tdist.destroy_process_group()
        return
    if world > 1:
        tdist.destroy_process_group()
    if world == 1 and not args.no_cpu and args.only == "all":
        line["cpu_baseline"] = cpu_baseline(M, N, K, wl["dtype"], wl["dist"])
    print(json.dumps(line), flush=True)


def make_parser():
    """The command line of bench.py."""
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["swz", "reference"], default="swz")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-transpose", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="gemm8192_bf16_pair")
    ap.add_argument("--m", type=int, default=0, help="custom shape (with --n, --k)")
    ap.add_argument("--n", type=int, default=0)
    ap.add_argument("--k", type=int, default=0)
    ap.add_argument("--dtype", choices=["fp16", "bf16"], default="fp16",
                    help="custom shape: operand type (bf16 draws N(0,1), fp16 U[-1,1))")
    ap.add_argument("--tile-n", type=int, default=0, choices=[0, 128, 256],
                    help="custom shape: tile width (default 256)")
    ap.add_argument("--pair", action="store_true", help="custom shape: 2-CTA clusters")
    ap.add_argument("--group-sizes", default="",
                    help="comma-separated G / S values of the sweep's grouped orders")
    ap.add_argument("--order", choices=["row", "col", "panel", "morton", "xor", "serpentine"],
                    default=None, help="headline tile order (default panel)")
    ap.add_argument("--group", type=int, default=None, help="G or S of the headline order")
    ap.add_argument("--stream-k", action=argparse.BooleanOptionalAction, default=None,
                    help="Stream-K tail of persistent launches (default: on when the launch "
                         "has a full wave of tiles; --no-stream-k: whole tiles only, the plain "
                         "work-index stride; --stream-k: always)")
    ap.add_argument("--die-split", action="store_true",
                    help="each die's clusters take their own share of the tiles (calibrates "
                         "the device first; persistent only)")
    ap.add_argument("--non-persistent", action="store_true", help="one CTA (pair) per tile")
    ap.add_argument("--e2e-slabs", type=int, default=8, help="row slabs of the host pipeline")
    ap.add_argument("--no-mma-sync", action="store_true")
    ap.add_argument("--no-tf32", action="store_true")
    ap.add_argument("--no-tc-rate", action="store_true")
    ap.add_argument("--no-swizzle", action="store_true")
    ap.add_argument("--l2-cache-mb", type=float, default=0.0,
                    help="L2 size the offline model assumes (default: the device's)")
    ap.add_argument("--num-sms", type=int, default=0,
                    help="concurrent CTAs the offline model assumes, as SMs (default: the "
                         "launch's resident programs)")
    ap.add_argument("--num-programs", type=int, default=0,
                    help="persistent launches of the headline GEMM on this many CTAs "
                         "(with --only gemm; default: the resident capacity)")
    ap.add_argument("--no-dynamic", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other configurations' order sweeps")
    ap.add_argument("--only", choices=["all", "gemm", "sweep", "transpose", "mma_sync",
                                       "tc_rate", "swizzle", "tf32", "cublas", "launch"],
                    default="all",
                    help="gemm: headline steps only; sweep / swizzle: one cold launch per "
                         "order / operand swizzle span; "
                         "transpose: the transposes only; tf32: the TF32 8192^3 GEMM, "
                         "3 warm-up launches and one cold one; cublas: torch.matmul on the "
                         "workload's shape for counter comparison (profiling modes); "
                         "launch: 50 calls back to back, eager and replayed from a CUDA "
                         "graph, per-call wall time")
    return ap


def main():
    args = make_parser().parse_args()
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    if args.non_persistent:
        args.stream_k = False  # Stream-K shares the tail of a persistent launch
    if args.impl == "reference":
        run_reference(args)
    else:
        run_swz(args)


if __name__ == "__main__":
    main()
