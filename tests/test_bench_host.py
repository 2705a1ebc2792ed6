"""Host logic of bench.py without a GPU: the N-replica timing reduction over two gloo
ranks, the whole-job aggregation, and the reference arm (the CPU oracle) end to end."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    w, r, _ = bench.dist_info()
    bench.init_dist(w, "gloo")
    ms = 10.0 + 5.0 * r                    # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, w)
    bench.barrier(w)
    q.put((r, worst, bench.aggregate_value(1e12, w, worst)))
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r, worst, value in out:
        assert worst == 15.0                           # max over ranks, seen by every rank
        assert value == pytest.approx(2 * 1e12 / 15e-3 / 1e12)


def test_reference_arm_prints_one_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "2", "--warmup", "1",
                        "--ref-sample-tokens", "16"], capture_output=True, text=True, env=env,
                       timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == "TFLOP/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--config", "tiny", "--steps", "1", "--warmup", "0"],
                       capture_output=True, text=True, env=env, timeout=120, cwd=ROOT)
    assert r.returncode == 0 and r.stdout.strip() == ""


def test_peak_regime_follows_the_clock_record():
    sys.path.insert(0, ROOT)
    import bench
    peaks = {"sm_max_mhz": 2070.0}
    # the region held the maximum clock with no cap: the burst GEMM peak applies
    assert bench.peak_regime({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []},
                             peaks)[0] == "burst"
    # the power cap pulled the clock down: the sustained (power-capped) peak applies
    assert bench.peak_regime({"sm_mhz": 1781.0, "sm_max_mhz": 2070.0,
                              "reasons": ["sw_power_cap"]}, peaks)[0] == "sustained"
    assert bench.peak_regime({"sm_mhz": 1700.0, "sm_max_mhz": 2070.0, "reasons": []},
                             peaks)[0] == "sustained"
    assert bench.peak_regime({"sm_mhz": None, "reasons": ["no samples"]}, peaks)[0] == "sustained"
