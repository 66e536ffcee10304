"""Backward pass (fa_backward) against the fp64 gradient oracle: the CUDA forward
gives O and LSE, the CUDA backward dQ, dK, dV; the oracle differentiates the
definition directly. Guard bands around every output catch stray writes."""

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu

# Error bound, relative to the largest magnitude of the exact gradient tensor.
# The kernel rounds P and dS to the 16-bit input type before their products
# (relative error 2^-9 for bf16, 2^-12 for fp16) and uses the forward's rounded
# O for the row term D; every sum runs in fp32. The bound leaves a margin of
# about 5x over the worst errors measured on these cases.
TOL_REL = {torch.float16: 5e-3, torch.bfloat16: 3e-2}
GUARD = 4096


def guarded(shape, dtype, dev, sentinel=-555.0):
    n = int(np.prod(shape))
    buf = torch.full((n + 2 * GUARD,), sentinel, dtype=dtype, device=dev)
    return buf, buf[GUARD:GUARD + n].view(shape)


def run_bwd(q, k, v, do, scale, mask="none", window=(0, 0)):
    dev = torch.device("cuda", 0)
    q, k, v, do = (t.to(dev).contiguous() for t in (q, k, v, do))
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32, device=dev)
    fa.fa_forward_gqa(q, k, v, o, lse, scale, mask, window[0], window[1])
    bufs = [guarded(q.shape, q.dtype, dev), guarded(k.shape, k.dtype, dev), guarded(v.shape, v.dtype, dev)]
    dq, dk, dv = (b[1] for b in bufs)
    ws_n = fa.fa_backward_workspace_bytes(*q.shape)
    wsb = torch.full((ws_n + 2 * GUARD,), 77, dtype=torch.uint8, device=dev)
    ws = wsb[GUARD:GUARD + ws_n]
    fa.fa_backward(q, k, v, o, do, lse, dq, dk, dv, scale, mask, window[0], window[1], ws)
    st = fa.fa_sync_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    for buf, _ in bufs:
        assert bool((buf[:GUARD] == -555.0).all()) and bool((buf[-GUARD:] == -555.0).all()), "stray write"
    assert bool((wsb[:GUARD] == 77).all()) and bool((wsb[-GUARD:] == 77).all()), "workspace overrun"
    return dq, dk, dv


def check(got, ref, dtype, what):
    g = got.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(g).all(), f"{what}: NaN/Inf"
    err = np.abs(g - ref).max()
    # relative to the tensor's largest entry, with a floor for gradients that
    # vanish exactly (one visible key: dQ = 0) while rounding leaves ~1e-7
    scale = max(np.abs(ref).max(), 0.1)
    assert err <= TOL_REL[dtype] * scale, f"{what}: max err {err:.3g} vs max |ref| {scale:.3g}"
    return err / scale


def compare(q, k, v, do, scale, mask, window, dq, dk, dv, kv_heads=None):
    B, H, N, d = q.shape
    Hk = k.shape[1]
    g = H // Hk
    rQ, rK, rV = oracle.attention_bwd(q, k, v, do, scale, mask, window, kv_heads=kv_heads)
    if kv_heads is None:
        kv_heads = list(range(B * Hk))
    dqc = dq.cpu().reshape(B * Hk, g, N, d)
    dkc = dk.cpu().reshape(B * Hk, N, d)
    dvc = dv.cpu().reshape(B * Hk, N, d)
    idx = torch.tensor(kv_heads)
    return (check(dqc[idx], rQ, q.dtype, "dQ"), check(dkc[idx], rK, q.dtype, "dK"),
            check(dvc[idx], rV, q.dtype, "dV"))


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
@pytest.mark.parametrize("N", [1, 63, 128, 129, 300])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (70, 5))])
def test_bwd_parity(mask, window, N, d, dtype):
    B, H = 1, 2
    q, k, v = make_qkv(B, H, N, d, dtype, seed=N + d)
    do = make_qkv(B, H, N, d, dtype, seed=N + 1000)[0]
    scale = d ** -0.5
    dq, dk, dv = run_bwd(q, k, v, do, scale, mask, window)
    compare(q, k, v, do, scale, mask, window, dq, dk, dv)


@pytest.mark.parametrize("Hk", [1, 2])
@pytest.mark.parametrize("mask", ["none", "causal"])
def test_bwd_gqa(mask, Hk):
    B, H, N, d = 2, 4, 200, 64
    q, _, _ = make_qkv(B, H, N, d, torch.bfloat16, seed=3)
    _, k, v = make_qkv(B, Hk, N, d, torch.bfloat16, seed=4, H_kv=Hk)
    do = make_qkv(B, H, N, d, torch.bfloat16, seed=5)[0]
    dq, dk, dv = run_bwd(q, k, v, do, 0.125, mask)
    compare(q, k, v, do, 0.125, mask, (0, 0), dq, dk, dv)


def test_bwd_long_sampled():
    """Many query blocks per key block (accumulation over 8 Q tiles and 2 heads of a group)."""
    B, H, Hk, N, d = 1, 4, 2, 1024, 128
    q, _, _ = make_qkv(B, H, N, d, torch.bfloat16, seed=8)
    _, k, v = make_qkv(B, Hk, N, d, torch.bfloat16, seed=9, H_kv=Hk)
    do = make_qkv(B, H, N, d, torch.bfloat16, seed=10)[0]
    dq, dk, dv = run_bwd(q, k, v, do, d ** -0.5, "causal")
    compare(q, k, v, do, d ** -0.5, "causal", (0, 0), dq, dk, dv, kv_heads=[1])


@pytest.mark.parametrize("Hk", [1, 2])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (200, 30))])
def test_bwd_d256_gqa(mask, window, Hk):
    """Head dimension 256 (its own three-pass kernels): grouped K/V heads, 64-row
    streamed tiles crossing 128-row blocks, a ragged last block."""
    B, H, N, d = 2, 4, 333, 256
    q, _, _ = make_qkv(B, H, N, d, torch.bfloat16, seed=31)
    _, k, v = make_qkv(B, Hk, N, d, torch.bfloat16, seed=32, H_kv=Hk)
    do = make_qkv(B, H, N, d, torch.bfloat16, seed=33)[0]
    dq, dk, dv = run_bwd(q, k, v, do, d ** -0.5, mask, window)
    compare(q, k, v, do, d ** -0.5, mask, window, dq, dk, dv)


def test_bwd_d256_long_sampled():
    """d = 256 with many streamed tiles per unit (1024 positions, causal, 2 query heads
    per K/V head), checked on one K/V head."""
    B, H, Hk, N, d = 1, 4, 2, 1024, 256
    q, _, _ = make_qkv(B, H, N, d, torch.float16, seed=34)
    _, k, v = make_qkv(B, Hk, N, d, torch.float16, seed=35, H_kv=Hk)
    do = make_qkv(B, H, N, d, torch.float16, seed=36)[0]
    dq, dk, dv = run_bwd(q, k, v, do, d ** -0.5, "causal")
    compare(q, k, v, do, d ** -0.5, "causal", (0, 0), dq, dk, dv, kv_heads=[0])


@pytest.mark.parametrize("d", [128, 256])
def test_bwd_many_units_per_cta(d):
    """256 units per pass on 152 SMs: the CTAs that take a second unit (from the
    launch-wide counter) load its resident tile and restart their accumulators
    between units. Checked on the first K/V head (first units) and the last one
    (second units)."""
    B, H, N = 1, 16, 2048
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=37)
    do = make_qkv(B, H, N, d, torch.bfloat16, seed=38)[0]
    dq, dk, dv = run_bwd(q, k, v, do, d ** -0.5, "causal")
    compare(q, k, v, do, d ** -0.5, "causal", (0, 0), dq, dk, dv, kv_heads=[0, H - 1])


@pytest.mark.parametrize("d", [64, 256])
def test_bwd_deterministic(d):
    """dQ, dK and dV are accumulated in tensor memory in a fixed order, without
    atomics: reruns are bit-identical."""
    q, k, v = make_qkv(1, 4, 500, d, torch.float16, seed=12)
    do = make_qkv(1, 4, 500, d, torch.float16, seed=13)[0]
    a = run_bwd(q, k, v, do, 0.125, "causal")
    b = run_bwd(q, k, v, do, 0.125, "causal")
    assert all(torch.equal(x, y) for x, y in zip(a, b))


def test_bwd_rejects_bad_workspace():
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in make_qkv(1, 2, 64, 64, torch.float16, seed=0))
    o, lse = torch.empty_like(q), torch.empty(1, 2, 64, device=dev)
    small = torch.empty(fa.fa_backward_workspace_bytes(1, 2, 64, 64) - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FaError):
        fa.fa_backward(q, k, v, o, q, lse, torch.empty_like(q), torch.empty_like(k),
                       torch.empty_like(v), 0.125, "none", 0, 0, small)
    with pytest.raises(fa.FaError):  # dQ aliasing Q
        fa.fa_backward(q, k, v, o, q.clone(), lse, q, torch.empty_like(k), torch.empty_like(v), 0.125)
    assert fa.fa_sync_status() == fa.FA_OK
