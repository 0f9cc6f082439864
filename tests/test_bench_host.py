"""Host-side logic of bench.py on CPU: the per-step work figures, the
multi-rank aggregation (gloo, world size 2: max over ranks, whole-job
throughput), and the reference arm's rank handling."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_step_work_figures():
    flops, b = bench.step_work(4096, 7168, 2048)
    assert flops["fprop"] == 2.0 * 4096 * 7168 * 2048
    assert set(b) == {"quant_128x128(W)", "quant_dual_stash(X)", "fprop", "quant_dual(dY)", "dgrad", "wgrad"}
    # dual cast: one 2-byte read, two 1-byte payloads, both scale arrays
    assert b["quant_dual(dY)"] == 4096 * 2048 * 4 + 4 * 16 * 4096 + 4 * 32 * 2048
    # forward cast of X with the stash requant: the same traffic as a dual cast
    assert b["quant_dual_stash(X)"] == 4096 * 7168 * 4 + 4 * 56 * 4096 + 4 * 32 * 7168


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist = bench.init_dist(world, "gloo")
    m = bench.max_over_ranks(dist, 1.5 + rank)
    bench.barrier(dist)
    out.put((rank, m, bench.whole_job_throughput(100.0, world, m)))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]            # max over ranks
    assert all(abs(r[2] - 200.0 / 2.5) < 1e-12 for r in res)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""


@pytest.mark.slow
def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0", "--cpu-sample", "0.03125"], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["cpu_baseline"]["kind"] == "oracle"


def test_cpulist_parsing_and_unbound_placement():
    """sysfs cpulist syntax, and the pinned-buffer placement helper falls back
    to an unbound allocation (affinity unchanged) where no GPU is visible."""
    assert bench._cpulist("0-3,8,10-11\n") == {0, 1, 2, 3, 8, 10, 11}
    assert bench._cpulist("") == set()
    before = os.sched_getaffinity(0)
    out, note = bench.alloc_pinned_near_gpu(torch, 0, lambda: 42)
    assert out == 42 and os.sched_getaffinity(0) == before
    assert set(note) == {"gpu_numa_node", "bound_cpus"}
