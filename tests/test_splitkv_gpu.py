"""Split-KV attention (fa_forward_splitkv): keys cut into chunks processed in parallel
and merged through their log-sum-exps; fewer queries than keys allowed (queries at the
last positions). Checked against the oracle and against the unsplit kernel."""

import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

from parity_util import TOL_LSE, TOL_O, compare, run_cuda

pytestmark = pytest.mark.gpu


def run_split(q, k, v, scale, mask="none", window=(0, 0), splits=0):
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev).contiguous() for t in (q, k, v))
    o = torch.full_like(q, -777.0)
    lse = torch.full(q.shape[:-1], -12345.0, dtype=torch.float32, device=dev)
    fa.fa_forward_splitkv(q, k, v, o, lse, scale, mask, window[0], window[1], splits)
    st = fa.fa_sync_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    return o, lse


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 129), (1, 5000), (4, 1000), (100, 3000), (300, 300)])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (500, 0))])
@pytest.mark.parametrize("splits", [1, 3, 40])
def test_splitkv_parity(splits, mask, window, Nq, Nk, d, dtype):
    q, _, _ = make_qkv(1, 4, Nq, d, dtype, seed=Nq + splits)
    _, k, v = make_qkv(1, 2, Nk, d, dtype, seed=Nk + 3 * splits, H_kv=2)
    o, lse = run_split(q, k, v, d ** -0.5, mask, window, splits)
    compare(o, lse, q, k, v, d ** -0.5, mask, window)


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_splitkv_matches_unsplit_kernel(mask):
    q, k, v = make_qkv(2, 8, 2000, 128, torch.bfloat16, seed=5)
    o1, l1 = run_cuda(q, k, v, 0.088, mask)
    for splits in (2, 5, 16):
        o2, l2 = run_split(q, k, v, 0.088, mask, splits=splits)
        assert float((o1.float() - o2.float()).abs().max()) <= TOL_O[torch.bfloat16]
        assert float((l1 - l2).abs().max()) <= TOL_LSE


def test_splitkv_default_splits_and_decode_shape():
    # a decode step: one query per head, a long key sequence, GQA
    B, H, Hk, Nk, d = 4, 32, 8, 16384, 128
    q, _, _ = make_qkv(B, H, 1, d, torch.bfloat16, seed=1)
    _, k, v = make_qkv(B, Hk, Nk, d, torch.bfloat16, seed=2, H_kv=Hk)
    s = fa.fa_splitkv_default_splits(B, H, 1, Nk)
    assert s > 1
    o, lse = run_split(q, k, v, d ** -0.5, "causal", splits=0)
    compare(o, lse, q, k, v, d ** -0.5, "causal", units=[(0, 0, 1), (B * H - 1, 0, 1), (77, 0, 1)])


def test_splitkv_workspace_checks():
    q, k, v = (t.cuda() for t in make_qkv(1, 2, 4, 64, torch.float16, seed=0))
    _, kk, vv = (t.cuda() for t in make_qkv(1, 2, 1024, 64, torch.float16, seed=1))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], device="cuda")
    need = fa.fa_splitkv_workspace_bytes(1, 2, 4, 64, 4)
    assert need > 0
    small = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FaError):
        fa.fa_forward_splitkv(q, kk, vv, o, lse, 0.125, "none", 0, 0, 4, small)
    with pytest.raises(fa.FaError):   # masks need Nq <= Nk
        fa.fa_forward_splitkv(kk, q, v, torch.empty_like(kk), torch.empty(kk.shape[:-1], device="cuda"),
                              0.125, "causal", 0, 0, 2)
    assert fa.fa_sync_status() == fa.FA_OK
