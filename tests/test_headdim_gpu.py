"""Head dimension 32 (64-byte swizzled tiles) on every forward entry point, and head
dimension 256 (its own kernel) on fa_forward / fa_forward_gqa, against the oracle."""

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

from parity_util import TOL_LSE, TOL_O, compare, run_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("N", [1, 63, 128, 129, 300, 1000])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (77, 9))])
def test_d32_parity(mask, window, N, dtype):
    q, k, v = make_qkv(2, 3, N, 32, dtype, seed=N + 32)
    o, lse = run_cuda(q, k, v, 32 ** -0.5, mask, window)
    compare(o, lse, q, k, v, 32 ** -0.5, mask, window)


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_d32_gqa(mask):
    q, _, _ = make_qkv(2, 8, 500, 32, torch.bfloat16, seed=4)
    _, k, v = make_qkv(2, 2, 500, 32, torch.bfloat16, seed=5, H_kv=2)
    o, lse = run_cuda(q, k, v, 0.2, mask)
    compare(o, lse, q, k, v, 0.2, mask)


@pytest.mark.parametrize("splits", [1, 4])
def test_d32_splitkv_decode(splits):
    dev = torch.device("cuda", 0)
    q, _, _ = make_qkv(2, 8, 3, 32, torch.float16, seed=6)
    _, k, v = make_qkv(2, 2, 2000, 32, torch.float16, seed=7, H_kv=2)
    o = torch.empty(q.shape, dtype=q.dtype, device=dev)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    fa.fa_forward_splitkv(q.to(dev), k.to(dev), v.to(dev), o, lse, 0.17, "causal", 0, 0, splits)
    assert fa.fa_sync_status() == fa.FA_OK
    compare(o, lse, q, k, v, 0.17, "causal")


def test_d32_varlen():
    dev = torch.device("cuda", 0)
    lens = [5, 130, 1, 257]
    H, d = 4, 32
    qs = [make_qkv(1, H, L, d, torch.bfloat16, seed=40 + i) for i, L in enumerate(lens)]
    pack = lambda ts: torch.cat([t[0].transpose(0, 1) for t in ts], 0).contiguous()
    Q, K, V = pack([x[0] for x in qs]), pack([x[1] for x in qs]), pack([x[2] for x in qs])
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lens)]), dtype=torch.int32, device=dev)
    o = torch.empty(Q.shape, dtype=Q.dtype, device=dev)
    lse = torch.empty(Q.shape[:2], dtype=torch.float32, device=dev)
    fa.fa_forward_varlen(Q.to(dev), K.to(dev), V.to(dev), o, lse, cu, cu, max(lens), 0.3, "causal")
    assert fa.fa_sync_status() == fa.FA_OK
    t0 = 0
    for (q, k, v), L in zip(qs, lens):
        O, LSE = oracle.attention(q, k, v, 0.3, "causal")
        got = o[t0:t0 + L].cpu().transpose(0, 1).reshape(-1, d).double().numpy()
        gl = lse[t0:t0 + L].cpu().transpose(0, 1).reshape(-1).double().numpy()
        assert np.abs(got - O).max() <= TOL_O[torch.bfloat16]
        assert np.abs(gl - LSE).max() <= TOL_LSE
        t0 += L


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("N", [1, 63, 64, 65, 129, 300, 1000])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (100, 7))])
def test_d256_parity(mask, window, N, dtype):
    q, k, v = make_qkv(1, 3, N, 256, dtype, seed=N + 256)
    o, lse = run_cuda(q, k, v, 256 ** -0.5, mask, window)
    compare(o, lse, q, k, v, 256 ** -0.5, mask, window)


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_d256_gqa_long(mask):
    """Many 64-key blocks per unit, GQA, a late dominant key per row (forces the
    lazy O rescale) on some rows."""
    q, _, _ = make_qkv(2, 4, 2000, 256, torch.bfloat16, seed=8, q_std=2.0)
    _, k, v = make_qkv(2, 2, 2000, 256, torch.bfloat16, seed=9, H_kv=2)
    k[:, :, 1900:] *= 3.0
    o, lse = run_cuda(q, k, v, 256 ** -0.5, mask)
    compare(o, lse, q, k, v, 256 ** -0.5, mask)


def test_d256_varlen_uneven_lengths():
    """d = 256 in a packed batch of uneven sequences (the one-tile kernel's
    variable-length form): every sequence against the oracle, GQA, causal."""
    from test_varlen_gpu import check, packed_inputs, run_varlen
    seqs, Q, K, V, cu_q, cu_k = packed_inputs([30, 0, 300, 129], [30, 0, 700, 129], 4, 2, 256,
                                              torch.bfloat16, seed=31)
    o, lse = run_varlen(Q, K, V, cu_q, cu_k, 300, 0.0625, "causal", (0, 0))
    check(seqs, o, lse, cu_q, 0.0625, "causal", (0, 0), torch.bfloat16)