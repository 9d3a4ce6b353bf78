"""Host-side pieces of bench.py: the replica aggregation over ranks (gloo,
world size 2), the algorithmic byte count, the reference arm's JSON line (also
under torchrun with two ranks) and the code hash that keys recorded DRAM
traffic."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    el, units = bench.aggregate(10.0 + 5.0 * rank, 100.0 * (rank + 1), world, dist)
    q.put((rank, el, units))
    dist.destroy_process_group()


def test_aggregate_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + (os.getpid() % 1000)
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get() for _ in range(2))
    for _, el, units in res:
        assert el == 15.0 and units == 300.0


def test_single_rank_aggregate_is_identity():
    assert bench.aggregate(3.0, 7.0, 1) == (3.0, 7.0)


def test_head_bytes_verify():
    cfg = bench.synth.CONFIGS["verify"]
    # 262144 rows x (2560*4/8 packed bytes + 2 arrays x 40 groups x 2 bytes)
    assert bench.head_bytes(cfg) == 262144 * (1280 + 160) == 377_487_360


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    # the contract's keys, with the arm's own metric, unit and direction
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert k in line, k
    assert line["steps"] == 2 and line["warmup"] == 1 and line["n_gpus"] == 1
    assert line["higher_is_better"] is True and line["vs_baseline"] is None
    assert line["config"]["workload"].startswith("tiny")
    cb = line["cpu_baseline"]
    assert cb["value"] == line["value"] and cb["unit"] == line["unit"] and cb["cores"] >= 1
    assert cb["sample"]
    assert line["e2e"]["value"] == line["value"] and line["e2e"]["unit"] == line["unit"]
    assert line["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_under_torchrun_prints_once():
    # Launched the way the driver launches N > 1: rank 0 alone runs the
    # oracle and prints; the other rank exits 0 without work.
    port = 29700 + (os.getpid() % 200)
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
                        "--nproc-per-node", "2", "--master-addr", "127.0.0.1",
                        "--master-port", str(port), os.path.join(ROOT, "bench.py"),
                        "--impl", "reference", "--config", "tiny", "--gpus", "2",
                        "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["value"] > 0


def test_recorded_traffic_is_keyed_by_code_not_comments():
    a = "int f(int x) {  // doubles\n  return 2 * x; /* no\n overflow check */ }\n"
    b = "/* header */\nint f(int x) {\n    return 2 * x;\n}\n// end\n"
    c = "int f(int x) { return 3 * x; }\n"
    assert bench.code_of(a) == bench.code_of(b) == "int f(int x) { return 2 * x; }"
    assert bench.code_of(c) != bench.code_of(a)
    # every recorded figure names sources that exist (a figure whose code has
    # changed since is reported as null by the bench, not failed here)
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        d = json.load(f)
    for kernel, per in d.items():
        for workload, e in per.items():
            assert bench.source_hash(e["sources"]) is not None, (kernel, workload)
