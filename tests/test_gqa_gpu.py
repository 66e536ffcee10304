"""Grouped-query / multi-query attention (fa_forward_gqa) against the oracle."""

import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import EXTRA_WORKLOADS, make_qkv, sample_units, workload_inputs

from parity_util import compare, run_cuda

pytestmark = pytest.mark.gpu

MASK_ARG = {0: "none", 1: "causal", 2: "window"}


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("H,Hk", [(8, 2), (8, 1), (6, 3)])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (70, 3))])
@pytest.mark.parametrize("N", [1, 200, 513])
def test_gqa_parity(N, mask, window, H, Hk, d, dtype):
    q, k, v = make_qkv(2, H, N, d, dtype, seed=N + H * 3 + Hk, H_kv=Hk)
    o, lse = run_cuda(q, k, v, d ** -0.5, mask, window)
    compare(o, lse, q, k, v, d ** -0.5, mask, window)


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_gqa_bit_exact_vs_repeated_kv(mask):
    # Sharing a K/V head must give exactly what multi-head attention gives on
    # copies of that head: the same arithmetic runs for every query row.
    H, Hk, N, d = 8, 2, 700, 128
    q, k, v = make_qkv(1, H, N, d, torch.bfloat16, seed=3, H_kv=Hk)
    o1, l1 = run_cuda(q, k, v, d ** -0.5, mask)
    kr = k.repeat_interleave(H // Hk, dim=1).contiguous()
    vr = v.repeat_interleave(H // Hk, dim=1).contiguous()
    o2, l2 = run_cuda(q, kr, vr, d ** -0.5, mask)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("w", [w for w in EXTRA_WORKLOADS if not w.Nq], ids=lambda w: w.name)
def test_gqa_workloads_sampled(w):
    q, k, v = workload_inputs(w)
    o, lse = run_cuda(q, k, v, w.scale, MASK_ARG[w.mask], (w.window_left, w.window_right))
    compare(o, lse, q, k, v, w.scale, MASK_ARG[w.mask], (w.window_left, w.window_right),
            units=sample_units(w))


def test_gqa_rejects_non_dividing_heads():
    q, k, v = make_qkv(1, 6, 64, 64, torch.float16, seed=0, H_kv=4)
    with pytest.raises(fa.FaError):
        run_cuda(q, k, v, 0.125, "none")
