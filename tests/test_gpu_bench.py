"""bench.py's own arm on the GPU: one short run of the 4k-token workload must print one
JSON line with every key of the benchmark contract, self-consistent (value from the
step time and the algorithmic FLOPs, the roofline fraction from its own achieved and
peak, the launch count from the kernels a BF16 step enqueues)."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_bench_line_contract():
    steps = 3
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--config", "qwen3_30b_4k",
                        "--steps", str(steps), "--warmup", "3", "--graph",
                        "--cpu-sample-tokens", "64"],
                       capture_output=True, text=True, env=env, timeout=900, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    j = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks", "graph"):
        assert key in j, key
    assert j["n_gpus"] == 1 and j["steps"] == steps and j["higher_is_better"] is True
    assert j["scaling"] == "weak" and j["data"] == "synthetic" and j["unit"] == "TFLOP/s"
    assert j["config"]["workload"] == "qwen3_30b_4k"
    # value = algorithmic FLOPs of a step (18 R H I) over the step time
    R, H, I = 4096 * 8, 2048, 768
    assert j["value"] == pytest.approx(18 * R * H * I / (j["ms_per_step"] * 1e-3) / 1e12, rel=1e-6)
    roof = j["roofline"]
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["achieved"] > 0 and roof["peak"] > 0
    assert roof["frac"] == pytest.approx(roof["achieved"] / roof["peak"], rel=1e-9)
    assert roof["traffic"] is None or roof["traffic"] > 0
    cpu = j["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] > 0 and cpu["sample"]
    e2e = j["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert e2e["unit"] == "TFLOP/s"
    assert j["gpu_launches"] == 12 * steps        # 7 forward + 5 backward launches per step
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(j["clocks"])
    assert j["graph"]["ms_per_step"] > 0
