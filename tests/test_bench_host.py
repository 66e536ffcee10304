"""Host-side logic of bench.py, on CPU: the multi-rank timing reduction over gloo
(world size 2), the whole-job throughput, and the oracle reference arm (rank 0 only)."""

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    m = bench.max_over_ranks(1.5 + rank, world)
    out[rank] = m
    bench.barrier(world)
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    # 2 ranks x 1e12 FLOPs each in 2 ms (slowest rank) = 1000 TFLOP/s
    assert abs(bench.job_throughput(2, 1e12, 2.0) - 1000.0) < 1e-9


def _run_ref(rank, world):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                           "--steps", "1", "--warmup", "0", "--workload", "tiny_full"],
                          capture_output=True, text=True, env=env, timeout=300)


def test_reference_arm_rank0_prints_one_line():
    r = _run_ref(0, 2)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run_ref(1, 2)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
