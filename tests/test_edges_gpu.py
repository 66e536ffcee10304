"""Edge cases at the limits of the index arithmetic and of the masks."""

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

from parity_util import TOL_LSE, TOL_O, compare, run_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_long_sequence_sampled(mask):
    """N = 65536 keys per head (row/key indices far past 16 bits, 512 key tiles per
    row block): first, last and a middle row block against the oracle."""
    N = 65536
    q, k, v = make_qkv(1, 2, N, 64, torch.bfloat16, seed=21)
    o, lse = run_cuda(q, k, v, 0.125, mask)
    units = [(0, 0, 128), (1, N - 128, N), (1, 30000, 30128)]
    compare(o, lse, q, k, v, 0.125, mask, units=units)


def test_zero_width_window_returns_own_value():
    """Window (0, 0): every query sees only its own key, so P = 1, O = V_i exactly
    (rounded) and LSE = its own logit."""
    q, k, v = make_qkv(2, 3, 777, 128, torch.float16, seed=22)
    o, lse = run_cuda(q, k, v, 0.1, "window", (0, 0))
    assert torch.equal(o.cpu(), v)
    compare(o, lse, q, k, v, 0.1, "window", (0, 0))


def test_many_heads_short_rows():
    """B*H = 4096 heads of 3 rows: a large unit count with one ragged tile each."""
    q, k, v = make_qkv(64, 64, 3, 64, torch.bfloat16, seed=23)
    o, lse = run_cuda(q, k, v, 0.125, "causal")
    compare(o, lse, q, k, v, 0.125, "causal", units=[(0, 0, 3), (4095, 0, 3), (1234, 0, 3)])


def test_backward_bench_size_head():
    """Backward at the bench's sequence length and head dim, one K/V head checked
    against the oracle (32 query blocks per key block, 32 key blocks per query block)."""
    from test_bwd_gpu import compare as bwd_compare, run_bwd
    q, k, v = make_qkv(1, 2, 4096, 128, torch.bfloat16, seed=24)
    do = make_qkv(1, 2, 4096, 128, torch.bfloat16, seed=25)[0]
    dq, dk, dv = run_bwd(q, k, v, do, 128 ** -0.5, "none")
    bwd_compare(q, k, v, do, 128 ** -0.5, "none", (0, 0), dq, dk, dv, kv_heads=[1])
