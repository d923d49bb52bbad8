"""CPU tests of the benchmark's host logic: the multi-rank path (world size 2 over gloo, the
max-over-ranks timing and barriers), the byte accounting, and the reference arm's JSON."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, w, l = bench.dist_env()
    bench.dist_init(w, "gloo")
    bench.dist_barrier(w)
    m = bench.dist_max(10.0 * (rank + 1), w)
    q.put((r, w, l, m))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in ps)
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == [(0, 2, 0, 20.0), (1, 2, 1, 20.0)]


def test_algorithmic_bytes_headline():
    wl = bench.workload()
    f, b = bench.algorithmic_bytes(wl)
    N = 4 * 2048 * 2048
    assert 10 * N < f + b < 10 * N + 5e6          # 10N + parameters (~4.3 MB)
    assert abs((f + b) / 8e12 * 1e6 - 21.4) < 0.5  # ~21.4 us at 8 TB/s


def test_reference_arm_json_line():
    env = dict(os.environ, OMP_NUM_THREADS="2")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "2", "--warmup", "3", "--ref-sample-T", "16"],
                         capture_output=True, text=True, env=env, timeout=300, check=True).stdout
    line = json.loads(out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["cores"] == 2
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["metric"] == bench.METRIC
