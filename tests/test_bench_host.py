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


def test_kernel_family_follows_the_forward_dispatch():
    """bench.py keys measured traffic to the kernel family that runs a workload; its
    rule restates the library's (fa_api.cu use_onetile): the one-tile kernel for
    d = 256, and for d = 64 / 128 when a row space holds at most 128 rows, a row space
    being one head's queries or, with at most 64 queries and grouped heads, those of
    all query heads of one K/V head, or when the problem's 256-row units fill at most
    half of the SMs (152 on GB300)."""
    sys.path.insert(0, ROOT)
    import dataclasses
    import bench
    from tiled_attention_03_gb300.workloads import BY_NAME
    fam = lambda name: bench.kernel_family(BY_NAME[name], sms=152)
    assert fam("full_b4h32n4096d128") == "fwd"
    assert fam("full_b4h32n4096d32") == "fwd"
    assert fam("full_b4h32n4096d64") == "fwd"
    assert fam("chunk_b1h32kv8_nq512_nk16384_d128") == "fwd"
    assert fam("varlen_causal_b16h32n4096d128") == "fwd"
    assert fam("varlen_causal_b16h16n4096d256") == "fwd1t"
    for name in ("decode_b8h32kv8_nq1_nk32768_d128", "decode_b8h32kv8_nq1_nk32768_d64",
                 "decode_b8h16kv4_nq1_nk32768_d256", "chunk_b1h16kv4_nq512_nk16384_d256",
                 "full_b4h16n4096d256", "causal_b4h16n4096d256"):
        assert fam(name) == "fwd1t", name
    assert fam("bwd_b4h32n4096d128") == "bwd"
    assert fam("bwd_b4h16n4096d256") == "bwd256"
    base = BY_NAME["full_b4h32n4096d128"]
    cut = lambda **kw: bench.kernel_family(dataclasses.replace(base, **kw), sms=152)
    assert cut(B=40, H=4, N=128) == "fwd1t" and cut(B=40, H=4, N=129) == "fwd"
    # small problems: 256-row units on at most half of the 152 SMs
    for name in ("tiny_full", "causal_short"):
        assert fam(name) == "fwd1t", name
    assert fam("mqa_causal_b2h16kv1n2048d64") == "fwd"  # 256 units
    assert cut(B=19, H=4, N=129) == "fwd1t" and cut(B=20, H=4, N=129) == "fwd"  # 76 / 80 units
    assert cut(B=40, H=16, H_kv=2, Nq=16) == "fwd1t"    # 8 heads x 16 queries = 128 rows
    assert cut(B=40, H=16, H_kv=2, Nq=17) == "fwd"      # 136 rows
    assert cut(B=40, H=4, H_kv=2, Nq=100) == "fwd1t"    # not packed (Nq > 64): 100 rows
    assert cut(H=4, N=100, d=32) == "fwd"               # d = 32 has no one-tile form


def test_kernel_source_hash_covers_every_included_header():
    """A family's traffic figure is reported only while the hash of its sources is
    unchanged, so those sources must include every local header its kernel file pulls
    in, directly or through another header."""
    sys.path.insert(0, ROOT)
    import re
    import bench
    csrc = os.path.join(ROOT, "tiled_attention_03_gb300", "csrc")

    def includes(name, seen):
        if name in seen:
            return seen
        seen.add(name)
        with open(os.path.join(csrc, name), encoding="utf-8") as f:
            for inc in re.findall(r'#include "([^"]+)"', f.read()):
                if os.path.exists(os.path.join(csrc, inc)):
                    includes(inc, seen)
        return seen

    kernels = {"fwd": "fa_fwd_kernel.cuh", "fwd1t": "fa_fwd1t_kernel.cuh",
               "bwd": "fa_bwd_kernel.cuh", "bwd256": "fa_bwd256_kernel.cuh"}
    for family, top in kernels.items():
        hashed = {os.path.basename(p) for p in bench.KERNEL_SOURCES[family]}
        missing = includes(top, set()) - hashed
        assert not missing, (family, missing)
