"""Split-KV attention (fa_forward_splitkv): keys cut into chunks processed in parallel
and merged through their log-sum-exps; fewer queries than keys allowed (queries at the
last positions). Checked against the oracle and against the unsplit kernel."""

import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import (EXTRA_WORKLOADS, make_qkv, sample_units,
                                                workload_inputs)

from parity_util import GUARD, SENT_L, TOL_LSE, TOL_O, compare, run_cuda

pytestmark = pytest.mark.gpu


def run_split(q, k, v, scale, mask="none", window=(0, 0), splits=0):
    """Split-KV call with sentinel guard bands around O and LSE."""
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev).contiguous() for t in (q, k, v))
    n, rows = q.numel(), q.numel() // q.shape[-1]
    obuf = torch.full((n + 2 * GUARD,), -777.0, dtype=q.dtype, device=dev)
    lbuf = torch.full((rows + 2 * GUARD,), SENT_L, dtype=torch.float32, device=dev)
    o = obuf[GUARD:GUARD + n].view(q.shape)
    lse = lbuf[GUARD:GUARD + rows].view(q.shape[:-1])
    fa.fa_forward_splitkv(q, k, v, o, lse, scale, mask, window[0], window[1], splits)
    st = fa.fa_sync_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    for buf, sent in ((obuf, -777.0), (lbuf, SENT_L)):
        assert bool((buf[:GUARD] == sent).all()), "write before the output"
        assert bool((buf[-GUARD:] == sent).all()), "write past the output"
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


# d = 256 runs its own kernel (64-key K/V tiles, so a split of s 128-key tiles is 2s of
# its tiles); queries may also outnumber the keys when there is no mask.
@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 5000), (4, 1000), (100, 3000), (300, 300), (200, 70)])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (500, 0))])
@pytest.mark.parametrize("splits", [1, 3, 40])
def test_splitkv_parity_d256(splits, mask, window, Nq, Nk, dtype):
    if Nq > Nk and mask != "none":
        pytest.skip("masks place the queries at the last key positions: Nq <= Nk")
    q, _, _ = make_qkv(1, 4, Nq, 256, dtype, seed=Nq + splits + 1)
    _, k, v = make_qkv(1, 2, Nk, 256, dtype, seed=Nk + 3 * splits + 1, H_kv=2)
    o, lse = run_split(q, k, v, 0.0625, mask, window, splits)
    compare(o, lse, q, k, v, 0.0625, mask, window)


# Row spaces of at most 128 rows run on the one-tile kernel at d = 64 and 128 too
# (128-key K/V tiles there): queries fewer or more than the keys, a single key, a
# full 128-row tile, every split count.
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk,mask", [(100, 50, "none"), (128, 1, "none"), (1, 1, "causal"),
                                        (64, 200, "causal"), (128, 129, "causal"),
                                        (77, 1000, "window"), (120, 4000, "none")])
@pytest.mark.parametrize("splits", [1, 2, 7])
def test_one_tile_rows(splits, mask, Nq, Nk, d):
    q, _, _ = make_qkv(2, 3, Nq, d, torch.float16, seed=Nq + 5 * splits)
    _, k, v = make_qkv(2, 3, Nk, d, torch.float16, seed=Nk + 11 * splits)
    window = (300, 40) if mask == "window" else (0, 0)
    o, lse = run_split(q, k, v, d ** -0.5, mask, window, splits)
    compare(o, lse, q, k, v, d ** -0.5, mask, window)


# Few queries per head with grouped K/V heads: the query heads of a K/V head share
# one row space, so 128-row tiles hold several heads and cut through heads (row
# spaces of at most 128 rows on the one-tile kernel, longer ones on the two-tile
# kernel at d = 64 and 128).
@pytest.mark.parametrize("B,H,Hk,Nq,Nk", [
    (2, 16, 2, 1, 3000), (1, 16, 2, 33, 1500), (1, 8, 1, 64, 700), (3, 12, 4, 7, 129),
    (1, 32, 8, 5, 40), (2, 6, 3, 64, 64), (1, 4, 2, 65, 900)])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)),
                                         ("window", (200, 0)), ("window", (30, 20))])
@pytest.mark.parametrize("splits", [1, 4])
@pytest.mark.parametrize("d", [64, 128, 256])
def test_packed_query_heads(d, splits, mask, window, B, H, Hk, Nq, Nk):
    dtype = torch.bfloat16
    q, _, _ = make_qkv(B, H, Nq, d, dtype, seed=Nq * 7 + splits)
    _, k, v = make_qkv(B, Hk, Nk, d, dtype, seed=Nk + H, H_kv=Hk)
    o, lse = run_split(q, k, v, 0.09, mask, window, splits)
    compare(o, lse, q, k, v, 0.09, mask, window)


@pytest.mark.parametrize("d", [128, 256])
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_splitkv_matches_unsplit_kernel(mask, d):
    q, k, v = make_qkv(2, 8, 2000, d, torch.bfloat16, seed=5)
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
    s = fa.fa_splitkv_default_splits(B, H, Hk, 1, Nk)
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


@pytest.mark.parametrize("w", [w for w in EXTRA_WORKLOADS if w.Nq], ids=lambda w: w.name)
def test_splitkv_workloads_sampled(w):
    """The decode and chunked-prefill workloads at full size, in the split count
    the benchmark uses, on sampled rows."""
    q, k, v = workload_inputs(w)
    window = (w.window_left, w.window_right)
    mask = {0: "none", 1: "causal", 2: "window"}[w.mask]
    o, lse = run_split(q, k, v, w.scale, mask, window, max(w.splits, 0))
    compare(o, lse, q, k, v, w.scale, mask, window, units=sample_units(w))
