"""Host-side checks of bench.py: the multi-rank aggregation on two gloo ranks,
the reference arm's JSON line under a 2-rank launch, and the rank statistic."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, out):
    import torch.distributed as tdist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        got = bench.max_over_ranks(1.5 + rank * 2.25)
        tdist.barrier()
        out.put((rank, got))
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(2))
    assert res == {0: 3.75, 1: 3.75}


def test_max_over_ranks_without_group():
    assert bench.max_over_ranks(2.5) == 2.5


def test_spearman_matches_page_convention():
    assert bench.spearman([1, 2, 3, 4], [4, 3, 2, 1]) == pytest.approx(-1.0)
    assert bench.spearman([5, 5, 5], [1, 2, 3]) == pytest.approx(1.0)
    assert bench.spearman([1.0], [2.0]) == 0.0


@pytest.mark.slow
def test_reference_arm_two_ranks_prints_one_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    port = 29600 + os.getpid() % 1000
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["steps"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_resolve_workload_custom_and_group_sizes():
    import argparse
    base = dict(workload="gemm8192_bf16_pair", m=0, n=0, k=0, dtype="fp16", tile_n=0,
                pair=False, group_sizes="")
    wl = bench.resolve_workload(argparse.Namespace(**base))
    assert (wl["M"], wl["N"], wl["K"], wl["dtype"]) == (8192, 8192, 8192, "bf16")
    a = argparse.Namespace(**dict(base, m=2048, n=1024, k=512, tile_n=128, pair=True,
                                  group_sizes="3,5"))
    wl = bench.resolve_workload(a)
    assert (wl["M"], wl["N"], wl["K"]) == (2048, 1024, 512)
    assert wl["cfg"] == dict(cta_pair=True, tile_n=128) and wl["cluster_m"] == 2
    assert a.workload == "custom2048x1024x512_fp16_pair128"
    grouped = [o for o in wl["sweep"] if o[0] in ("panel", "serpentine")]
    assert grouped == [("panel", 3), ("panel", 5), ("serpentine", 3), ("serpentine", 5)]
    assert ("row", 1) in wl["sweep"] and ("morton", 1) in wl["sweep"]
    with pytest.raises(SystemExit):
        bench.resolve_workload(argparse.Namespace(**dict(base, m=64)))


def test_workloads_and_capture_modes():
    import argparse
    base = dict(m=0, n=0, k=0, dtype="fp16", tile_n=0, pair=False, group_sizes="")
    wl = bench.resolve_workload(argparse.Namespace(
        **dict(base, workload="gemm6144x10240x4096_fp16_pair")))
    assert ("morton", 1) not in wl["sweep"] and ("xor", 1) not in wl["sweep"]
    # every named workload resolves, with a non-empty order sweep
    for name in bench.WORKLOADS:
        w = bench.resolve_workload(argparse.Namespace(**dict(base, workload=name)))
        assert w["M"] > 0 and w["sweep"]
    # the capture modes the profiles' commands use are accepted
    src = open(bench.__file__).read()
    for mode in ("gemm", "sweep", "swizzle", "transpose", "mma_sync", "tc_rate", "tf32",
                 "cublas", "launch"):
        assert f'"{mode}"' in src


def test_clock_sampler_summarises_one_phase():
    # nvidia-smi rows are placed by their own timestamps; only the samples of
    # the marked phase taken while the GPU was busy set the median clock
    import datetime

    def stamp(t):
        return datetime.datetime.fromtimestamp(t).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]

    t0 = 1_800_000_000.0
    rows = [(t0 + 0.1, 2070, 0, "Not Active"), (t0 + 1.1, 1950, 100, "Active"),
            (t0 + 1.2, 1930, 100, "Active"), (t0 + 1.3, 2070, 10, "Not Active"),
            (t0 + 2.5, 1800, 100, "Not Active")]
    text = "\n".join(f"{stamp(t)}, {mhz}, 2070, 900.0, {util}, 0x0, Not Active, Not Active, "
                     f"Not Active, {cap}" for t, mhz, util, cap in rows)

    class FakeProc:
        def terminate(self):
            pass

        def communicate(self, timeout=None):
            return text, ""

    s = bench.ClockSampler(0)
    s.proc = FakeProc()
    s.marks = [(t0 + 1.0, "headline"), (t0 + 2.0, None)]
    s.__exit__(None, None, None)
    h = s.summary("headline")
    assert s.summary("headline", None)["samples"] == 5
    assert h["samples"] == 3 and h["samples_busy"] == 2
    assert h["sm_mhz"] == 1940 and h["reasons"] == ["sw_power_cap"]
    assert s.summary()["samples"] == 5


def test_config_sweeps_cover_the_specification():
    # every configuration of the specification other than the headline is in
    # the default line, with the orders it names
    keys = {k for k, _, _ in bench.CONFIG_SWEEPS}
    assert keys == set(bench.CONFIG_ORDERS)
    for key, wname, modes in bench.CONFIG_SWEEPS:
        assert wname in bench.WORKLOADS
    o2 = bench.CONFIG_ORDERS["cfg2_4096_fp16_tile128x256"]
    assert {g for o, g in o2 if o == "panel"} == {2, 4, 8, 16}
    assert {g for o, g in o2 if o == "serpentine"} == {2, 4, 8, 16}
    assert ("morton", 1) in o2 and ("xor", 1) in o2
    o4 = bench.CONFIG_ORDERS["cfg4_6144x10240x4096_fp16_tile128x128"]
    assert not {o for o, _ in o4} & {"morton", "xor"}  # not bijective on 48 x 80
    assert len(bench.CONFIG_ORDERS["cfg1_1024x1024x512_fp16"]) == 6
    # configuration 2's tile grid runs as single CTAs and as CTA pairs
    assert set(bench.CONFIG_ORDERS["cfg2_4096_fp16_tile128x256_pair"]) == set(o2)
    assert dict((k, m) for k, _, m in bench.CONFIG_SWEEPS)["cfg2_4096_fp16_tile128x256"] == (
        True, False)
    # the capture mode (--only sweep) of each workload covers the same orders
    for key, wname, _ in bench.CONFIG_SWEEPS:
        assert set(bench.WORKLOADS[wname]["sweep"]) == set(bench.CONFIG_ORDERS[key]), key


def test_code_hash_ignores_comments_and_layout_only():
    # the ncu records are keyed on the kernel's code, not on its comments
    a = 'int f(int x) {  // doubles\n  return 2 * x; /* twice */ }\nconst char* s = "// kept";'
    b = 'int f(int x) {\n    return 2 * x;\n}\nconst char* s = "// kept";'
    assert bench.code_hash(a) == bench.code_hash(b)
    assert bench.code_hash(a) != bench.code_hash(a.replace("2 * x", "3 * x"))
    assert bench.code_hash(a) != bench.code_hash(a.replace('"// kept"', '"/ kept"'))
    # the records in the bench are keyed this way
    for rec in bench.NCU.values():
        assert len(rec["source"]["gemm_cu_code_hash"]) == 16


def test_profile_commands_parse():
    # every `python bench.py ...` command the profile summaries give is a
    # valid command line of this bench.py (placeholders of a command family
    # replaced by one of their values)
    import glob
    import os
    import re
    import shlex
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    fill = {"W": ["gemm4096_fp16"], "O": ["row"], "G": ["1"], "P": ["76"],
            "[F]": ["--stream-k", "--die-split"]}
    ap = bench.make_parser()
    seen = 0
    for path in glob.glob(os.path.join(root, "profiles", "*.md")):
        text = re.sub(r"\\\n\s*", " ", open(path).read())  # join continued lines
        for m in re.finditer(r"python bench\.py([^\n#`]*)", text):
            argv = [a for t in shlex.split(m.group(1)) for a in fill.get(t, [t])]
            argv = [a for a in argv if a not in (">", "2>&1")]
            ap.parse_args(argv)
            seen += 1
    assert seen >= 10
