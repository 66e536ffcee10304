"""Benchmark of the attention forward pass on GB300.

One step = one forward pass (fa_forward, one kernel launch) over the
B4 H32 N4096 d128 bf16 non-causal workload, inputs resident in HBM. Prints one
JSON line (rank 0). Under torchrun every rank runs its own replica of the
workload (independent problems, no collective on the data path) and the
max-over-ranks time is reported with the whole-job throughput.

--impl reference times the fp64 CPU oracle on this host's cores, on a bounded
sample of the same workload, in the same metric.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "attn fwd TFLOP/s (% of GB300 BF16 tensor peak); tokens/s @B4 H32 N4096 d128"
METRIC_BWD = "attn bwd TFLOP/s (10 N^2 d FLOPs per head: dQ, dK, dV with S recomputed)"
WORKLOAD = "full_b4h32n4096d128"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
# The sources each kernel family compiles from: a traffic figure stays valid while
# the sources of the kernels it was measured on are unchanged.
CSRC = "tiled_attention_03_gb300/csrc/"
KERNEL_SOURCES = {
    "fwd": (CSRC + "fa_fwd_kernel.cuh", CSRC + "fa_combine.cuh", CSRC + "fa_mask.cuh",
            CSRC + "fa_tmem_max.cuh", CSRC + "ptx.cuh"),
    "fwd1t": (CSRC + "fa_fwd1t_kernel.cuh", CSRC + "fa_combine.cuh", CSRC + "fa_mask.cuh",
              CSRC + "fa_tmem_max.cuh", CSRC + "ptx.cuh"),
    "bwd": (CSRC + "fa_bwd_kernel.cuh", CSRC + "fa_mask.cuh", CSRC + "ptx.cuh"),
    "bwd256": (CSRC + "fa_bwd256_kernel.cuh", CSRC + "fa_bwd_kernel.cuh", CSRC + "fa_mask.cuh",
               CSRC + "ptx.cuh"),
}
TRAFFIC_DIR = os.path.join(ROOT, "profiles")


def sm_count() -> int:
    import torch
    if torch.cuda.is_available():
        return torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return 152  # GB300


def one_tile(w, sms: int | None = None) -> bool:
    """Whether the library runs this forward on its one-tile kernel: always at d = 256,
    and at d = 64 / 128 when a row space (one head's queries, or the queries of all
    query heads of one K/V head when each has at most 64) holds at most 128 rows, or
    when the call has one key split and the two-tile kernel's 256-row units would
    fill at most half of the SMs."""
    if w.backward:
        return False
    if w.d == 256:
        return True
    if w.varlen:
        return False
    if w.d not in (64, 128):
        return False
    packed = w.kv_heads < w.H and w.q_rows <= 64
    rows = (w.H // w.kv_heads if packed else 1) * w.q_rows
    if rows <= 128:
        return True
    sms = sms if sms is not None else sm_count()
    spaces = w.B * (w.kv_heads if packed else w.H)
    units = spaces * ((rows + 255) // 256)
    tiles = (w.N + 127) // 128
    # the split count the call runs: the workload's, or the library's default (one wave)
    splits = 1 if w.splits < 0 else w.splits if w.splits > 0 else (
        1 if units >= sms else max(1, min(sms // units, max(1, tiles // 4), 256)))
    return min(splits, tiles) == 1 and 2 * units <= sms


def kernel_family(w, sms: int | None = None) -> str:
    if w.backward:
        return "bwd256" if w.d == 256 else "bwd"
    return "fwd1t" if one_tile(w, sms) else "fwd"


def kernel_source_hash(family: str) -> str:
    """Hash of the family's sources with comments and whitespace removed, so that
    an edit of comments alone keeps the measured counters."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_traffic(w):
    """DRAM bytes per step from the committed ncu summary (profiles/*_traffic.txt)
    of this workload, if it was taken on the current kernel source; else None."""
    try:
        names = sorted(os.listdir(TRAFFIC_DIR))
    except OSError:
        return None
    for name in names:
        if not name.endswith("_traffic.txt"):
            continue
        try:
            vals = {}
            with open(os.path.join(TRAFFIC_DIR, name)) as f:
                for line in f:
                    if ":" in line and not line.startswith("#"):
                        key, val = line.split(":", 1)
                        vals[key.strip()] = val.strip()
            if (vals.get("workload") == w.name
                    and vals.get("kernel_source_hash") == kernel_source_hash(kernel_family(w))):
                return float(vals["dram_bytes_per_launch"])
        except (OSError, KeyError, ValueError):
            continue
    return None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["bf16_tflops"]), float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    def __init__(self, gpu_index: int, interval_ms: int = 100):
        self.proc = None
        self.out = None
        try:
            self.out = open(_tmp_path("clocks"), "w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={CLOCK_FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={interval_ms}"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.count(",") >= 8]
        self.out.close()
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if "Active" in r[5 + i]
                          and "Not" not in r[5 + i]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def _tmp_path(tag):
    return os.path.join(tempfile.gettempdir(), f".bench_{tag}_{os.getpid()}.csv")


def dist_setup(n_gpus: int):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Max of a per-rank scalar (the timing reduction; nothing of the data path)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_rank: float, ms_per_step_max: float) -> float:
    """Whole-job TFLOP/s: every rank runs its own replica; the slowest rank sets the time."""
    return world * flops_per_rank / (ms_per_step_max * 1e-3) / 1e12


def oracle_slab(w):
    """One (b, h) slab of the workload's shape, drawn with its recipe."""
    from tiled_attention_03_gb300.workloads import make_qkv
    return make_qkv(1, 1, w.N, w.d, w.dtype, seed=w.seed, q_std=w.q_std, Nq=w.Nq)


def cpu_oracle_rate(w, min_seconds: float, max_units: int | None = None, slab=None):
    """Time the fp64 oracle on a sample of (1 head, 128-row block) units of the
    workload, using every core of this host. Returns (TFLOP/s, cores, sample, seconds)."""
    import oracle
    from tiled_attention_03_gb300.workloads import visible_in_rows
    cores = len(os.sched_getaffinity(0))
    q, k, v = oracle_slab(w) if slab is None else slab
    rows = w.q_rows
    nblk = (rows + 127) // 128
    n = cores if max_units is None else min(cores, max_units)
    while True:
        units = [(0, (u % nblk) * 128, min(rows, (u % nblk + 1) * 128)) for u in range(n)]
        t0 = time.perf_counter()
        oracle.attention(q, k, v, w.scale, {0: "none", 1: "causal", 2: "window"}[w.mask],
                         (w.window_left, w.window_right), units=units, nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= min_seconds or (max_units is not None and n >= max_units) or n >= 64 * cores:
            break
        n *= 2
    # algorithmic flops of the sampled rows: 4 d per visible (query, key) pair
    pairs = sum(visible_in_rows(w.N, w.mask, w.window_left, w.window_right, r0, r1, w.Nq)
                for _, r0, r1 in units)
    flops = 4.0 * w.d * pairs
    return flops / dt / 1e12, cores, f"{len(units)} x (1 head, {min(128, rows)}-row block, all {w.N} keys)", dt


def cpu_oracle_full(w, min_seconds: float, threads: int):
    """Time the fp64 oracle on the WHOLE workload (every head, every row), repeated
    until min_seconds have passed, on `threads` host threads. Only for the small
    workloads that the oracle finishes in milliseconds. Returns (TFLOP/s, seconds per
    pass)."""
    import oracle
    from tiled_attention_03_gb300.workloads import algorithmic_flops, workload_inputs
    q, k, v = workload_inputs(w)[:3]
    mask = {0: "none", 1: "causal", 2: "window"}[w.mask]
    reps, dt = 0, 0.0
    t0 = time.perf_counter()
    while dt < min_seconds or reps == 0:
        oracle.attention(q, k, v, w.scale, mask, (w.window_left, w.window_right), nthreads=threads)
        reps += 1
        dt = time.perf_counter() - t0
    return algorithmic_flops(w) * reps / dt / 1e12, dt / reps


# The two small parity workloads: the oracle runs them whole, on all cores and on one.
SMALL_WORKLOADS = ("tiny_full", "causal_short")


def cpu_oracle_rate_bwd(w, min_seconds: float, max_heads: int | None = None):
    """Time the fp64 gradient oracle on a sample of whole K/V heads (each with the
    query heads reading it) of the workload's shape, on every core. Returns
    (TFLOP/s, cores, sample, seconds)."""
    import oracle
    from tiled_attention_03_gb300.workloads import make_qkv, visible_pairs
    cores = len(os.sched_getaffinity(0))
    group = w.H // w.kv_heads
    n = max(1, cores // group) if max_heads is None else max(1, min(max_heads, cores // group))
    while True:
        q, k, v = make_qkv(1, n * group, w.N, w.d, w.dtype, seed=w.seed, q_std=w.q_std, H_kv=n)
        do = make_qkv(1, n * group, w.N, w.d, w.dtype, seed=w.seed + 10000)[0]
        t0 = time.perf_counter()
        oracle.attention_bwd(q, k, v, do, w.scale, {0: "none", 1: "causal", 2: "window"}[w.mask],
                             (w.window_left, w.window_right), nthreads=cores)
        dt = time.perf_counter() - t0
        if dt >= min_seconds or max_heads is not None or n >= 8 * cores:
            break
        n *= 2
    flops = 10.0 * w.d * n * group * visible_pairs(w.N, w.mask, w.window_left, w.window_right)
    return flops / dt / 1e12, cores, f"{n} K/V head(s) x {group} query head(s), all {w.N} rows", dt


def run_reference(args, w):
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return
    n = len(os.sched_getaffinity(0))
    if w.backward:
        def sample_once():
            return cpu_oracle_rate_bwd(w, 0.0, max_heads=n)
    else:
        slab = oracle_slab(w)

        def sample_once():
            return cpu_oracle_rate(w, 0.0, max_units=n, slab=slab)
    for _ in range(args.warmup):
        sample_once()
    flops_total, secs_total = 0.0, 0.0
    for _ in range(args.steps):
        r, cores, sample, dt = sample_once()
        flops_total += r * 1e12 * dt
        secs_total += dt
    value = flops_total / secs_total / 1e12
    wall = secs_total
    line = {
        "impl": "reference", "metric": METRIC_BWD if w.backward else METRIC, "value": value,
        "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * wall / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                   "mask": {0: "none", 1: "causal", 2: "window"}[w.mask], "input_dtype": w.dtype_name,
                   "step": "oracle over one bounded sample of the workload"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_e2e(args, w, q_h, k_h, v_h, mask, stream, dev, world, flops):
    """Same metric through the public API (tiled_attention_03_gb300.forward) with
    pinned host inputs and pinned result buffers: every step copies Q, K, V to the
    device, runs the kernel and copies O and LSE back (overlapped in chunks of
    about 64 MB by the library's fa_forward_host)."""
    import tiled_attention_03_gb300 as fa
    qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
    splits = None if w.splits < 0 else w.splits
    # the caller's reusable pinned result buffers
    out = torch.empty(q_h.shape, dtype=q_h.dtype, pin_memory=True)
    lse_out = torch.empty(q_h.shape[:-1], dtype=torch.float32, pin_memory=True)

    def run():
        fa.forward(qp, kp, vp, w.scale, mask, (w.window_left, w.window_right),
                   num_splits=splits, out=out, lse_out=lse_out)

    for _ in range(2):
        run()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    # an event after every step (the stream waits for each step's last copy out)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.e2e_steps + 1)]
    ev[0].record(stream)
    for i in range(args.e2e_steps):
        run()
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    wall_ms = (time.perf_counter() - t0) * 1e3 / args.e2e_steps
    e2e_ms = max_over_ranks(max(ev[0].elapsed_time(ev[-1]) / args.e2e_steps, wall_ms), world)
    per = sorted(ev[i].elapsed_time(ev[i + 1]) for i in range(args.e2e_steps))
    pct = lambda f: per[min(len(per) - 1, int(f * len(per)))]
    elems = q_h.numel()  # O has Q's shape
    h2d = (q_h.numel() + k_h.numel() + v_h.numel()) * q_h.element_size()
    d2h = elems * q_h.element_size() + (elems // w.d) * 4
    return {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
            "step_ms": {"p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9)},
            "copy_floor": copy_floor(qp, kp, vp, out, lse_out, dev)}


def copy_floor(qp, kp, vp, out, lse_out, dev, reps: int = 5):
    """The step's copies alone, in the same run: Q, K, V host -> device, then O and LSE
    device -> host, each direction by itself and both at once on two streams (the
    least time the end-to-end step could take). Median of `reps`, in ms and GB/s."""
    ins = [torch.empty_like(t, device=dev) for t in (qp, kp, vp)]
    outs = [torch.empty_like(t, device=dev) for t in (out, lse_out)]
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(do_in, do_out):
        ts = []
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            if do_in:
                with torch.cuda.stream(s_in):
                    for d, h in zip(ins, (qp, kp, vp)):
                        d.copy_(h, non_blocking=True)
            if do_out:
                with torch.cuda.stream(s_out):
                    for h, d in zip((out, lse_out), outs):
                        h.copy_(d, non_blocking=True)
            torch.cuda.synchronize(dev)
            ts.append((time.perf_counter() - t0) * 1e3)
        return sorted(ts)[len(ts) // 2]

    b_in = sum(t.numel() * t.element_size() for t in (qp, kp, vp))
    b_out = sum(t.numel() * t.element_size() for t in (out, lse_out))
    t_in, t_out, t_both = timed(True, False), timed(False, True), timed(True, True)
    return {"h2d_ms": t_in, "h2d_gbs": b_in / t_in / 1e6, "d2h_ms": t_out,
            "d2h_gbs": b_out / t_out / 1e6, "both_ms": t_both}


def run_e2e_varlen(args, w, host, max_q, mask, stream, dev, world, flops):
    """Variable-length forward through the public binding with pinned host tensors:
    every step copies Q, K, V and cu_seqlens to the device, runs
    fa_forward_varlen and copies O and LSE back."""
    import tiled_attention_03_gb300 as fa
    pinned = [t.pin_memory() for t in host]

    def run():
        q, k, v, cu = (t.to(dev, non_blocking=True) for t in pinned)
        o = torch.empty_like(q)
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=dev)
        fa.fa_forward_varlen(q, k, v, o, lse, cu, cu, max_q, w.scale, mask, w.window_left,
                             w.window_right)
        oh = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        lh = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        oh.copy_(o, non_blocking=True)
        lh.copy_(lse, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    for _ in range(2):
        run()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        run()
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, world)
    q = host[0]
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = q.numel() * q.element_size() + (q.numel() // w.d) * 4
    return {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def run_e2e_varlen_bwd(args, w, host, max_q, mask, dev, world, flops):
    """Variable-length backward through the public binding with pinned host
    tensors: every step copies Q, K, V, O, LSE, dO and cu_seqlens to the device,
    runs fa_backward_varlen and copies dQ, dK, dV back."""
    import tiled_attention_03_gb300 as fa
    pinned = [t.pin_memory() for t in host]
    outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in host[:3]]

    def run():
        q, k, v, o, lse, do, cu = (t.to(dev, non_blocking=True) for t in pinned)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        fa.fa_backward_varlen(q, k, v, o, do, lse, cu, cu, dq, dk, dv, max_q, max_q, w.scale, mask,
                              w.window_left, w.window_right)
        for dst, g in zip(outs, (dq, dk, dv)):
            dst.copy_(g, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    for _ in range(2):
        run()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        run()
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    return {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def run_e2e_bwd(args, w, host, mask, stream, dev, world, flops):
    """Backward through the public API (tiled_attention_03_gb300.backward) with
    pinned host tensors: every step copies Q, K, V, O, LSE and dO to the device,
    runs the backward and copies dQ, dK and dV back."""
    import tiled_attention_03_gb300 as fa
    pinned = [t.pin_memory() for t in host]

    def run():
        q, k, v, o, lse, do = (t.to(dev, non_blocking=True) for t in pinned)
        grads = fa.backward(q, k, v, o, lse, do, w.scale, mask, (w.window_left, w.window_right))
        outs = [torch.empty(g.shape, dtype=g.dtype, pin_memory=True) for g in grads]
        for dst, g in zip(outs, grads):
            dst.copy_(g, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()
        return outs

    for _ in range(2):
        run()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        run()
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3 / args.e2e_steps, world)
    h2d = sum(t.numel() * t.element_size() for t in host)
    q, k = host[0], host[1]
    d2h = (q.numel() + 2 * k.numel()) * q.element_size()
    return {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--l2-flush", action="store_true",
                    help="write a 256 MB buffer before every step (not timed), for workloads "
                         "whose inputs fit in L2")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from tiled_attention_03_gb300.workloads import BY_NAME, algorithmic_bytes, algorithmic_flops
    w = BY_NAME[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
        return

    import tiled_attention_03_gb300 as fa
    from tiled_attention_03_gb300.workloads import workload_inputs

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fa.load_library()

    q_h, k_h, v_h = workload_inputs(w)
    q, k, v = q_h.to(dev), k_h.to(dev), v_h.to(dev)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    mask = {0: "none", 1: "causal", 2: "window"}[w.mask]
    stream = torch.cuda.current_stream(dev)

    if w.varlen:
        from tiled_attention_03_gb300.workloads import (varlen_inputs, varlen_lengths,
                                                        workload_grad_output)
        splits = 1
        vq_h, vk_h, vv_h, cu_h = varlen_inputs(w)
        vq, vk, vv, cu = vq_h.to(dev), vk_h.to(dev), vv_h.to(dev), cu_h.to(dev)
        vo = torch.empty_like(vq)
        vlse = torch.empty(vq.shape[:2], dtype=torch.float32, device=dev)
        max_q = max(varlen_lengths(w))
        if w.backward:
            # O and LSE from one forward outside the timed region; a step is the backward
            fa.fa_forward_varlen(vq, vk, vv, vo, vlse, cu, cu, max_q, w.scale, mask,
                                 w.window_left, w.window_right, stream)
            lens = varlen_lengths(w)
            dfull = workload_grad_output(w)
            do_h = torch.cat([dfull[b, :, :lens[b]].transpose(0, 1) for b in range(w.B)], 0).contiguous()
            vdo = do_h.to(dev)
            vdq, vdk, vdv = torch.empty_like(vq), torch.empty_like(vk), torch.empty_like(vv)
            vws = torch.empty(fa.fa_backward_varlen_workspace_bytes(w.B, w.H, vq.shape[0]),
                              dtype=torch.uint8, device=dev)

            def step():
                fa.fa_backward_varlen(vq, vk, vv, vo, vdo, vlse, cu, cu, vdq, vdk, vdv, max_q, max_q,
                                      w.scale, mask, w.window_left, w.window_right, vws, stream)
        else:
            def step():
                fa.fa_forward_varlen(vq, vk, vv, vo, vlse, cu, cu, max_q, w.scale, mask,
                                     w.window_left, w.window_right, stream)
    elif w.backward:
        # O and LSE from one forward, outside the timed region; a step is the backward.
        from tiled_attention_03_gb300.workloads import workload_grad_output
        splits = 1
        fa.fa_forward_gqa(q, k, v, o, lse, w.scale, mask, w.window_left, w.window_right, stream)
        do_h = workload_grad_output(w)
        do = do_h.to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.fa_backward_workspace_bytes(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                         device=dev)

        def step():
            fa.fa_backward(q, k, v, o, do, lse, dq, dk, dv, w.scale, mask, w.window_left,
                           w.window_right, ws, stream)
    elif w.splits >= 0:
        splits = w.splits or fa.fa_splitkv_default_splits(w.B, w.H, w.kv_heads, w.q_rows, w.N)
        ws = torch.empty(max(16, fa.fa_splitkv_workspace_bytes(w.B, w.H, w.q_rows, w.d, splits)),
                         dtype=torch.uint8, device=dev)

        def step():
            fa.fa_forward_splitkv(q, k, v, o, lse, w.scale, mask, w.window_left, w.window_right,
                                  splits, ws, stream)
    else:
        splits = 1
        call = fa.fa_forward if w.kv_heads == w.H else fa.fa_forward_gqa

        def step():
            call(q, k, v, o, lse, w.scale, mask, w.window_left, w.window_right, stream)

    for _ in range(args.warmup):
        step()
    st = fa.fa_sync_status(stream)
    if st != fa.FA_OK:
        raise SystemExit(f"device status after warm-up: {fa.fa_status_string(st)}")

    flops = algorithmic_flops(w)
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = fa.fa_launch_count()
    # one event between consecutive steps: the total and each step's own duration.
    # With --l2-flush, a 256 MB write (larger than L2) precedes every step, outside
    # that step's events, and the time is the sum of the steps alone.
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if args.l2_flush else None
    if flush is None:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        ev[0].record(stream)
        for i in range(args.steps):
            step()
            ev[i + 1].record(stream)
        pairs = [(ev[i], ev[i + 1]) for i in range(args.steps)]
    else:
        pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                 for _ in range(args.steps)]
        for a, b in pairs:
            flush.fill_(1)
            a.record(stream)
            step()
            b.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    launches = fa.fa_launch_count() - launches0
    clocks = sampler.stop() if sampler else None
    st = fa.fa_sync_status(stream)
    if st != fa.FA_OK:
        raise SystemExit(f"device status after the timed region: {fa.fa_status_string(st)}")
    per_step = [a.elapsed_time(b) for a, b in pairs]
    ms_local = pairs[0][0].elapsed_time(pairs[-1][1]) if flush is None else sum(per_step)
    per_step.sort()
    pct = lambda f: per_step[min(len(per_step) - 1, int(f * len(per_step)))]
    ms_total = max_over_ranks(ms_local, world)
    ms_step = ms_total / args.steps
    value = job_throughput(world, flops, ms_step)
    kernel_ms = ms_local / args.steps  # the step's launches, all on this stream

    # ---- end to end through the public API with pinned host buffers
    e2e = None
    if args.e2e_steps > 0 and w.varlen and w.backward:
        host = [vq_h, vk_h, vv_h, vo.cpu(), vlse.cpu(), do_h, cu_h]
        e2e = run_e2e_varlen_bwd(args, w, host, max_q, mask, dev, world, flops)
    elif args.e2e_steps > 0 and w.varlen:
        e2e = run_e2e_varlen(args, w, [vq_h, vk_h, vv_h, cu_h], max_q, mask, stream, dev, world,
                             flops)
    elif args.e2e_steps > 0 and w.backward:
        host = [q_h, k_h, v_h, o.cpu(), lse.cpu(), do_h]
        e2e = run_e2e_bwd(args, w, host, mask, stream, dev, world, flops)
    elif args.e2e_steps > 0:
        e2e = run_e2e(args, w, q_h, k_h, v_h, mask, stream, dev, world, flops)

    if rank == 0:
        peak_tf, peak_gbs, peak_src = peaks()
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        nbytes = algorithmic_bytes(w)
        # tensor-bound above the ridge (peak FLOP/s / peak B/s), HBM-bound below it
        tensor_bound = flops / nbytes > peak_tf * 1e12 / (peak_gbs * 1e9)
        traffic = measured_traffic(w)
        cpu = None
        if args.cpu_seconds > 0 and w.backward:
            cpu_v, cores, sample, _ = cpu_oracle_rate_bwd(w, args.cpu_seconds)
            cpu = {"value": cpu_v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                   "sample": sample}
        elif args.cpu_seconds > 0 and w.name in SMALL_WORKLOADS:
            cores = len(os.sched_getaffinity(0))
            cpu_v, per_pass = cpu_oracle_full(w, min(args.cpu_seconds, 5.0), cores)
            one_v, one_pass = cpu_oracle_full(w, min(args.cpu_seconds, 5.0), 1)
            cpu = {"value": cpu_v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                   "sample": f"the whole workload ({per_pass * 1e3:.2f} ms per pass)",
                   "one_core": {"value": one_v, "unit": "TFLOP/s", "cores": 1,
                                "sample": f"the whole workload ({one_pass * 1e3:.2f} ms per pass)"}}
        elif args.cpu_seconds > 0:
            cpu_v, cores, sample, _ = cpu_oracle_rate(w, args.cpu_seconds)
            cpu = {"value": cpu_v, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                   "sample": sample}
        in_t = ((vq, vk, vv, vdo) if w.varlen and w.backward else (vq, vk, vv) if w.varlen
                else (q, k, v, do) if w.backward else (q, k, v))
        in_bytes = sum(t.numel() * t.element_size() for t in in_t)
        line = {
            "metric": METRIC_BWD if w.backward else METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "step_ms": {"p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9), "rank": 0},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype_name, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "N": w.N, "d": w.d,
                       "mask": mask, "seed": w.seed,
                       "parallelism": f"{world} independent replica(s), no collective",
                       "kv_heads": w.kv_heads,
                       "l2": ("256 MB written before every step (not timed)" if args.l2_flush
                              else f"inputs ({in_bytes / 1e6:.0f} MB) larger than L2, no flush"
                              if in_bytes > 129e6 else "inputs smaller than L2, no flush")},
            "tokens_per_s": world * (vq.shape[0] if w.varlen else w.B * w.q_rows) / (ms_step * 1e-3),
            "pct_of_peak": 100.0 * value / (world * peak_tf),
            "roofline": ({"bound": "tensor", "achieved": achieved, "peak": peak_tf,
                          "unit": "TFLOP/s", "frac": achieved / peak_tf,
                          "peak_source": f"{peak_src} bf16 burst"}
                         if tensor_bound else
                         {"bound": "hbm", "achieved": nbytes / (kernel_ms * 1e-3) / 1e9,
                          "peak": peak_gbs, "unit": "GB/s",
                          "frac": nbytes / (kernel_ms * 1e-3) / 1e9 / peak_gbs,
                          "peak_source": f"{peak_src} copy bandwidth"}) | {
                "traffic": traffic, "algorithmic_bytes": nbytes,
                "kernel": ((f"fa_bwd prep + dV, dK, dQ passes <256, {w.dtype_name}>" if w.d == 256
                            else f"fa_bwd prep + dK/dV + dQ kernels <{w.d}, {w.dtype_name}"
                            + (", varlen>" if w.varlen else ">")) if w.backward
                           else (f"fa_fwd1t_kernel<{w.d}, {w.dtype_name}, varlen>" if w.d == 256
                                 else f"fa_fwd_kernel<{w.d}, {w.dtype_name}, varlen>") if w.varlen
                           else (f"fa_fwd1t_kernel<{w.d}, {w.dtype_name}>" if one_tile(w)
                                 else f"fa_fwd_kernel<{w.d}, {w.dtype_name}>")
                           + (f" + merge ({splits} key splits)" if splits > 1 else ""))},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
