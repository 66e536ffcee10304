"""Seeded synthetic inputs for the attention forward pass.

This module only draws random numbers and describes workload shapes. It holds
none of the attention arithmetic, so both the CUDA path and the CPU oracle can
be fed from it without sharing any of the method.

The five workloads are the shapes the pages use: a tiny full-attention case, a
short causal case, the benchmark shape of "ai6s.net/6a0ed07b662f9a54cb761aa2"
(performance table: batch 4, 32 heads, head_dim 128, seq 4096), a
sliding-window case with a sequence length that is not a tile multiple and
peaky logits (the NaN-at-window-edges pitfall on the same page), and a long
causal case with LLaMA-13B-like heads ("aicoding.csdn.net/6a69d3ff10ee7a33f2941f44",
memory table, B=8 H=40).

Recipe (the pages name no generator): a CPU ``torch.Generator`` seeded with
the workload's seed draws Q, K, V in that order, each as float32
``randn(B, H, N, d)``; Q is multiplied by ``q_std``; each is then rounded to the
workload's 16-bit dtype. Both sides read the rounded 16-bit values.
"""

from __future__ import annotations

import dataclasses
import math

import numpy as np

import torch

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_WINDOW = 2

MASK_NAMES = {MASK_NONE: "none", MASK_CAUSAL: "causal", MASK_WINDOW: "window"}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: torch.dtype
    mask: int
    window_left: int
    window_right: int
    seed: int
    q_std: float = 1.0
    H_kv: int = 0  # K/V heads (grouped-query attention); 0 means H
    Nq: int = 0    # query rows per head when fewer than the N keys (the last Nq positions); 0 means N
    splits: int = -1  # key splits for the split-KV entry point (0: its default); -1: not split
    backward: bool = False  # time the backward pass (dQ, dK, dV) instead of the forward
    varlen: bool = False    # B sequences of seeded lengths in [N/8, N], packed token-major

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), rounded to float32 as the C ABI takes it."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    @property
    def dtype_name(self) -> str:
        return {torch.float16: "fp16", torch.bfloat16: "bf16"}[self.dtype]

    @property
    def kv_heads(self) -> int:
        return self.H_kv or self.H

    @property
    def q_rows(self) -> int:
        return self.Nq or self.N

    def describe(self) -> str:
        m = MASK_NAMES[self.mask]
        if self.mask == MASK_WINDOW:
            m += f"({self.window_left},{self.window_right})"
        kv = f" Hkv{self.kv_heads}" if self.kv_heads != self.H else ""
        nq = f" Nq{self.q_rows}" if self.q_rows != self.N else ""
        return f"B{self.B} H{self.H}{kv}{nq} N{self.N} d{self.d} {self.dtype_name} {m}"


WORKLOADS = [
    Workload("tiny_full", 1, 1, 256, 64, torch.float16, MASK_NONE, 0, 0, seed=0),
    Workload("causal_short", 1, 8, 1024, 64, torch.float16, MASK_CAUSAL, 0, 0, seed=1),
    Workload("full_b4h32n4096d128", 4, 32, 4096, 128, torch.bfloat16, MASK_NONE, 0, 0, seed=2),
    Workload("window_ragged_peaky", 2, 32, 4000, 128, torch.float16, MASK_WINDOW, 1024, 0,
             seed=3, q_std=3.0),
    Workload("causal_long_b8h40n8192", 8, 40, 8192, 128, torch.bfloat16, MASK_CAUSAL, 0, 0, seed=4),
]

# Shapes for the widened rows (grouped-query attention): the bench shape with 8 K/V
# heads shared by 32 query heads, and a multi-query causal case.
EXTRA_WORKLOADS = [
    Workload("gqa_b4h32kv8n4096d128", 4, 32, 4096, 128, torch.bfloat16, MASK_NONE, 0, 0,
             seed=5, H_kv=8),
    Workload("mqa_causal_b2h16kv1n2048d64", 2, 16, 2048, 64, torch.float16, MASK_CAUSAL, 0, 0,
             seed=6, H_kv=1),
    # split-KV: one decode step over a long cache (memory-bound), and a 512-query chunk
    # appended to a 16k-token cache
    Workload("decode_b8h32kv8_nq1_nk32768_d128", 8, 32, 32768, 128, torch.bfloat16, MASK_CAUSAL,
             0, 0, seed=7, H_kv=8, Nq=1, splits=0),
    Workload("chunk_b1h32kv8_nq512_nk16384_d128", 1, 32, 16384, 128, torch.bfloat16, MASK_CAUSAL,
             0, 0, seed=8, H_kv=8, Nq=512, splits=0),
    # the d = 64 decode step (one-tile kernel with 128-key tiles at d = 64)
    Workload("decode_b8h32kv8_nq1_nk32768_d64", 8, 32, 32768, 64, torch.bfloat16, MASK_CAUSAL,
             0, 0, seed=22, H_kv=8, Nq=1, splits=0),
    # head dimension 32 (64-byte swizzled tiles) and 64 on the bench shape
    # the long causal workload with 4 of its 8 batch entries: the same per-head shape
    # and scheduling, small enough for a many-pass ncu capture (its traffic doubles to
    # the full one's)
    Workload("causal_b4h40n8192", 4, 40, 8192, 128, torch.bfloat16, MASK_CAUSAL, 0, 0, seed=4),
    Workload("full_b4h32n4096d32", 4, 32, 4096, 32, torch.bfloat16, MASK_NONE, 0, 0, seed=13),
    Workload("full_b4h32n4096d64", 4, 32, 4096, 64, torch.bfloat16, MASK_NONE, 0, 0, seed=18),
    # head dimension 256 (its own kernel), same FLOPs as the bench shape
    Workload("full_b4h16n4096d256", 4, 16, 4096, 256, torch.bfloat16, MASK_NONE, 0, 0, seed=14),
    Workload("causal_b4h16n4096d256", 4, 16, 4096, 256, torch.bfloat16, MASK_CAUSAL, 0, 0, seed=15),
    # split-KV at head dimension 256: a decode step and a 512-query chunk on a long cache
    Workload("decode_b8h16kv4_nq1_nk32768_d256", 8, 16, 32768, 256, torch.bfloat16, MASK_CAUSAL,
             0, 0, seed=20, H_kv=4, Nq=1, splits=0),
    Workload("chunk_b1h16kv4_nq512_nk16384_d256", 1, 16, 16384, 256, torch.bfloat16, MASK_CAUSAL,
             0, 0, seed=21, H_kv=4, Nq=512, splits=0),
]

# Backward pass on the bench shape (dO drawn after Q, K, V from the same generator).
BWD_WORKLOADS = [
    Workload("bwd_b4h32n4096d128", 4, 32, 4096, 128, torch.bfloat16, MASK_NONE, 0, 0, seed=9,
             backward=True),
    Workload("bwd_causal_b4h32n4096d128", 4, 32, 4096, 128, torch.bfloat16, MASK_CAUSAL, 0, 0,
             seed=10, backward=True),
    Workload("bwd_gqa_causal_b2h32kv8n4096d64", 2, 32, 4096, 64, torch.float16, MASK_CAUSAL, 0, 0,
             seed=11, H_kv=8, backward=True),
    Workload("bwd_b4h32n4096d32", 4, 32, 4096, 32, torch.bfloat16, MASK_NONE, 0, 0, seed=19,
             backward=True),
    # head dimension 256 (its own three-pass kernels)
    Workload("bwd_b4h16n4096d256", 4, 16, 4096, 256, torch.bfloat16, MASK_NONE, 0, 0, seed=24,
             backward=True),
    Workload("bwd_causal_b4h16n4096d256", 4, 16, 4096, 256, torch.bfloat16, MASK_CAUSAL, 0, 0,
             seed=25, backward=True),
]

# A packed batch of 16 causal sequences of mixed lengths (N/8 .. N), token-major.
VARLEN_WORKLOADS = [
    Workload("varlen_causal_b16h32n4096d128", 16, 32, 4096, 128, torch.bfloat16, MASK_CAUSAL, 0, 0,
             seed=12, varlen=True),
    # the same length mix at head dimension 256 (16 heads)
    Workload("varlen_causal_b16h16n4096d256", 16, 16, 4096, 256, torch.bfloat16, MASK_CAUSAL, 0, 0,
             seed=23, varlen=True),
    # its backward (dO drawn like the dense backward workloads, then packed)
    Workload("bwd_varlen_causal_b16h32n4096d128", 16, 32, 4096, 128, torch.bfloat16, MASK_CAUSAL,
             0, 0, seed=12, varlen=True, backward=True),
    # and at head dimension 256
    Workload("bwd_varlen_causal_b16h16n4096d256", 16, 16, 4096, 256, torch.bfloat16, MASK_CAUSAL,
             0, 0, seed=23, varlen=True, backward=True),
]

BY_NAME = {w.name: w for w in WORKLOADS + EXTRA_WORKLOADS + BWD_WORKLOADS + VARLEN_WORKLOADS}


def varlen_lengths(w: Workload) -> list[int]:
    """Seeded sequence lengths of a variable-length workload, uniform in [N/8, N]."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 20000)
    return [int(x) for x in torch.randint(w.N // 8, w.N + 1, (w.B,), generator=g)]


def varlen_inputs(w: Workload):
    """Token-major Q, K, V (total, heads, d) and cu_seqlens (B + 1,) int32: sequence b
    is the first L_b positions of batch entry b of workload_inputs(w)."""
    q, k, v = workload_inputs(w)
    lens = varlen_lengths(w)
    pack = lambda t: torch.cat([t[b, :, :lens[b]].transpose(0, 1) for b in range(w.B)], 0).contiguous()
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32)
    return pack(q), pack(k), pack(v), cu


def make_qkv(B: int, H: int, N: int, d: int, dtype: torch.dtype, seed: int,
             q_std: float = 1.0, H_kv: int = 0, Nq: int = 0):
    """Return CPU tensors Q (B, H, Nq or N, d) and K, V (B, H_kv or H, N, d) in ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    Hk = H_kv or H
    q = torch.randn(B, H, Nq or N, d, generator=g, dtype=torch.float32)
    if q_std != 1.0:
        q.mul_(q_std)
    q = q.to(dtype)
    k = torch.randn(B, Hk, N, d, generator=g, dtype=torch.float32).to(dtype)
    v = torch.randn(B, Hk, N, d, generator=g, dtype=torch.float32).to(dtype)
    return q, k, v


def workload_inputs(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.d, w.dtype, w.seed, w.q_std, w.H_kv, w.Nq)


def workload_grad_output(w: Workload):
    """dO for a backward workload: N(0, 1) of Q's shape, from seed + 10000."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 10000)
    return torch.randn(w.B, w.H, w.q_rows, w.d, generator=g, dtype=torch.float32).to(w.dtype)


def sample_units(w: Workload, n: int = 16, block: int = 128, seed: int | None = None):
    """Seeded sample of (bh, row0, row1) slices: always the first block, the
    last (possibly ragged) block and one middle block, plus random ones."""
    nblk = (w.q_rows + block - 1) // block
    BH = w.B * w.H
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 + w.seed if seed is None else seed)
    picks = [(0, 0), (BH - 1, nblk - 1), (BH // 2, nblk // 2)]
    while len(picks) < n:
        bh = int(torch.randint(0, BH, (1,), generator=g))
        blk = int(torch.randint(0, nblk, (1,), generator=g))
        if (bh, blk) not in picks:
            picks.append((bh, blk))
    return [(bh, blk * block, min(w.q_rows, (blk + 1) * block)) for bh, blk in picks[:n]]


def visible_in_rows(N: int, mask: int, wl: int, wr: int, r0: int, r1: int, Nq: int = 0) -> int:
    """Number of (query, key) pairs a mask leaves visible for query rows
    [r0, r1) of one (b, h) with N keys (query i at key position i + N - Nq):
    the count the algorithmic FLOP figure is built on (4*d per pair)."""
    off = N - (Nq or N)
    if mask == MASK_NONE:
        return (r1 - r0) * N
    if mask == MASK_CAUSAL:
        wl, wr = N, 0
    total = 0
    for i in range(r0, r1):
        lo = max(0, i + off - wl)
        hi = min(N - 1, i + off + wr)
        total += max(0, hi - lo + 1)
    return total


def visible_pairs(N: int, mask: int, wl: int, wr: int, Nq: int = 0) -> int:
    """Visible (query, key) pairs of one (b, h)."""
    return visible_in_rows(N, mask, wl, wr, 0, Nq or N, Nq)


def algorithmic_flops(w: Workload) -> float:
    """Forward: 2 products of 2 d FLOPs per visible pair. Backward: 5 (dV, dP, dQ,
    dK and the recomputed S), i.e. 2.5x the forward."""
    per_pair = 10.0 if w.backward else 4.0
    if w.varlen:
        pairs = sum(visible_pairs(n, w.mask, w.window_left, w.window_right) for n in varlen_lengths(w))
        return per_pair * w.d * w.H * pairs
    return per_pair * w.d * w.B * w.H * visible_pairs(w.N, w.mask, w.window_left, w.window_right, w.Nq)


def algorithmic_bytes(w: Workload) -> int:
    """Forward: Q, K, V read once and O (16-bit) plus LSE (fp32) written once.
    Backward: Q, K, V, O, dO and LSE read once, dQ, dK, dV written once."""
    tokens = sum(varlen_lengths(w)) if w.varlen else w.B * w.q_rows
    q_elems = tokens * w.H * w.d
    kv_elems = (tokens if w.varlen else w.B * w.N) * w.kv_heads * w.d
    rows = tokens * w.H
    if w.backward:
        return (4 * q_elems + 4 * kv_elems) * 2 + rows * 4
    return (2 * q_elems + 2 * kv_elems) * 2 + rows * 4
