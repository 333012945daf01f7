"""bench.py on the host, without a GPU:
- the reference arm (the CPU oracle) prints one well-formed JSON line with
  the benchmark's keys, and ranks other than 0 print nothing;
- the launch count follows the kernel dispatch;
- the replicas path (world size 2, gloo) times the job by its slowest rank
  and counts every rank's tokens."""
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


class _FakeLib:
    """moe_step_kernel_path by a fixed rule (no device here)."""
    MOE_PATH_DECODE, MOE_PATH_TENSOR_CORE, MOE_PATH_STREAM = 1, 2, 3

    def __init__(self, path):
        self.path = path

    def moe_step_kernel_path(self, T, E, k, H, I):
        return self.path


def test_launch_count_follows_the_dispatch():
    dec, tc, st = _FakeLib(1), _FakeLib(2), _FakeLib(3)
    q = (512, 10, 2560, 640)
    assert bench.layer_launches(dec, 1, *q) == 1        # one cooperative kernel
    assert bench.layer_launches(tc, 8, *q) == 1
    assert bench.layer_launches(tc, 4096, *q) == 6      # route, align, gather, gate/up, down, combine
    assert bench.layer_launches(tc, 32, *q) == 6
    assert bench.layer_launches(dec, 9, *q) == 4        # route, align, decode step kernels (combine fused)
    assert bench.layer_launches(st, 12, *q) == 5        # route, align, stream kernels, combine


def _rank_main(rank, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=2)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slower one
        slowest = bench.max_over_ranks(ms)
        q.put((rank, slowest, bench.whole_job_rate(dist.get_world_size(), 4, 10, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank():
    """The N > 1 bench path on CPU (gloo, world size 2): every rank gets the
    slowest rank's time, and the whole-job rate counts both replicas' tokens."""
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, slowest, rate in got:
        assert slowest == 15.0
        assert abs(rate - 2 * 4 * 10 / 0.015) < 1e-6


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1", "--workload", "tiny_T4_H256_I64_E16_k2"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_large_batches_run_the_oracle_on_every_core():
    import concurrent.futures as cf

    from w4a16_group_quantized_moe_gb300 import inputs
    small = inputs.Workload("t_T4_H256_I64_E16_k2", inputs.MoEShape(4, 256, 64, 16, 2))
    assert bench.oracle_plan(small) == (4, 1)  # whole layers on one thread
    wl = inputs.Workload("t_T64_H256_I64_E16_k2", inputs.MoEShape(64, 256, 64, 16, 2))
    n_tok, threads = bench.oracle_plan(wl)
    assert threads == bench.oracle_threads() and n_tok == 4 * threads
    w13, w2 = inputs.make_weights(16, 256, 64, 0)
    with cf.ThreadPoolExecutor(threads) as pool:
        n, dt = bench.oracle_step(wl, 0, 4, w13, w2, n_tok, pool)
    assert n == n_tok and dt > 0
