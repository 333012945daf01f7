"""bench.py on the host, without a GPU: the reference arm (the CPU oracle)
prints one well-formed JSON line with the benchmark's keys, and the launch
count follows the kernel dispatch."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--workload", "tiny_T4_H256_I64_E16_k2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC
    assert d["unit"] == "tokens/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["steps"] >= 1 and d["config"]["workload"] == "tiny_T4_H256_I64_E16_k2"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_launch_count_follows_the_dispatch():
    assert bench.layer_launches(1, 10) == 1        # one cooperative kernel
    assert bench.layer_launches(8, 10) == 1
    assert bench.layer_launches(4096, 10) == 6     # route, align, gather, gate/up, down, combine
    assert bench.layer_launches(32, 10) == 5       # route+align in one launch
    assert bench.layer_launches(9, 10) == 3        # decode step kernels
