"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Tolerances (max abs error): O <= 4e-3 for fp16 and <= 2e-2 for bf16, LSE <=
1e-3, no NaN/Inf, and nothing written outside O and LSE (sentinel guards).
"""

import math

import numpy as np
import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import WORKLOADS, make_qkv, sample_units, workload_inputs

from parity_util import compare, run_cuda

pytestmark = pytest.mark.gpu

MASK_ARG = {0: "none", 1: "causal", 2: "window"}


def _window(w):
    return (w.window_left, w.window_right)


@pytest.mark.parametrize("idx", [0, 1])
def test_workload_full(idx):
    w = WORKLOADS[idx]
    q, k, v = workload_inputs(w)
    o, lse = run_cuda(q, k, v, w.scale, MASK_ARG[w.mask], _window(w))
    compare(o, lse, q, k, v, w.scale, MASK_ARG[w.mask], _window(w))


@pytest.mark.parametrize("idx", [2, 3, 4])
def test_workload_sampled(idx):
    w = WORKLOADS[idx]
    q, k, v = workload_inputs(w)
    o, lse = run_cuda(q, k, v, w.scale, MASK_ARG[w.mask], _window(w))
    units = sample_units(w)
    compare(o, lse, q, k, v, w.scale, MASK_ARG[w.mask], _window(w), units=units)
    # every row of the outputs is finite
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


SWEEP_N = [1, 2, 63, 64, 65, 127, 128, 129, 255, 1000]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (37, 5))])
@pytest.mark.parametrize("N", SWEEP_N)
def test_sweep(N, mask, window, d, dtype):
    q, k, v = make_qkv(1, 2, N, d, dtype, seed=N * 7 + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = run_cuda(q, k, v, scale, mask, window)
    compare(o, lse, q, k, v, scale, mask, window)


@pytest.mark.parametrize("window", [(0, 0), (100, 0), (128, 128), (1, 300), (5000, 0), (0, 5000),
                                    (127, 1), (129, 0), (256, 255)])
def test_window_edges(window):
    N, d = 700, 128
    q, k, v = make_qkv(1, 2, N, d, torch.float16, seed=sum(window), q_std=3.0)
    o, lse = run_cuda(q, k, v, d ** -0.5, "window", window)
    compare(o, lse, q, k, v, d ** -0.5, "window", window)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_many_heads_short_rows(dtype):
    q, k, v = make_qkv(4, 96, 72, 64, dtype, seed=3)
    o, lse = run_cuda(q, k, v, 0.125, "causal")
    compare(o, lse, q, k, v, 0.125, "causal")


def test_scale_values():
    q, k, v = make_qkv(1, 1, 300, 64, torch.bfloat16, seed=4)
    for scale in (1.0, 0.125, 0.01):
        o, lse = run_cuda(q, k, v, scale, "none")
        compare(o, lse, q, k, v, scale, "none")


def test_v_all_ones_gives_ones():
    N, d = 500, 128
    q, k, _ = make_qkv(1, 2, N, d, torch.bfloat16, seed=5, q_std=2.0)
    v = torch.ones_like(q)
    o, lse = run_cuda(q, k, v, d ** -0.5, "causal")
    assert float((o.float() - 1).abs().max()) <= 2e-2


def test_uniform_scores_mean_of_visible_v():
    N, d = 300, 64
    _, k, v = make_qkv(1, 1, N, d, torch.float16, seed=6)
    q = torch.zeros_like(k)
    o, lse = run_cuda(q, k, v, 0.125, "causal")
    V = v.double()[0, 0]
    mean = torch.cumsum(V, 0) / torch.arange(1, N + 1, dtype=torch.float64)[:, None]
    assert float((o.double().cpu()[0, 0] - mean).abs().max()) <= 4e-3
    ln = torch.log(torch.arange(1, N + 1, dtype=torch.float64))
    assert float((lse.double().cpu()[0, 0] - ln).abs().max()) <= 1e-3


def test_dominant_key_in_last_tile():
    N, d = 520, 64
    _, _, v = make_qkv(1, 1, N, d, torch.bfloat16, seed=21)
    q = torch.zeros(1, 1, N, d, dtype=torch.bfloat16)
    q[..., 0] = 4.0
    k = torch.zeros(1, 1, N, d, dtype=torch.bfloat16)
    k[..., 1] = torch.linspace(-1, 1, N).to(torch.bfloat16)
    k[0, 0, N - 1, 0] = 8.0  # logit 32 against 0 for all other keys: the max jumps late
    o, lse = run_cuda(q, k, v, 1.0, "none")
    assert float((o.float().cpu()[0, 0] - v.float()[0, 0, N - 1]).abs().max()) <= 2e-2
    assert float((lse.cpu() - 32.0).abs().max()) <= 1e-3


@pytest.mark.parametrize("mask,window", [("causal", (0, 0)), ("window", (60, 2))])
def test_mask_invariance_bit_exact(mask, window):
    N, d, i0 = 400, 128, 250
    q, k, v = make_qkv(1, 1, N, d, torch.float16, seed=7)
    k2, v2 = k.clone(), v.clone()
    g = torch.Generator().manual_seed(8)
    if mask == "causal":
        sl, rows = slice(i0 + 1, N), slice(0, i0 + 1)
    else:
        sl, rows = slice(0, i0 - window[0]), slice(i0, N)
    k2[..., sl, :] = (torch.randn(k2[..., sl, :].shape, generator=g) * 4).to(k.dtype)
    v2[..., sl, :] = (torch.randn(v2[..., sl, :].shape, generator=g) * 4).to(v.dtype)
    o1, l1 = run_cuda(q, k, v, d ** -0.5, mask, window)
    o2, l2 = run_cuda(q, k2, v2, d ** -0.5, mask, window)
    assert torch.equal(o1[..., rows, :], o2[..., rows, :])
    assert torch.equal(l1[..., rows], l2[..., rows])


def test_deterministic_and_stream():
    q, k, v = make_qkv(2, 4, 777, 128, torch.bfloat16, seed=9)
    o1, l1 = run_cuda(q, k, v, 0.088, "causal")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o2, l2 = run_cuda(q, k, v, 0.088, "causal")
    s.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_forward_host_tensors():
    q, k, v = make_qkv(1, 2, 300, 64, torch.float16, seed=10)
    o, lse = fa.forward(q.pin_memory(), k.pin_memory(), v.pin_memory(), 0.125, "causal")
    assert o.device.type == "cpu" and lse.device.type == "cpu"
    compare(o, lse, q, k, v, 0.125, "causal")


def test_forward_host_tensors_pipelined_into_caller_buffers():
    """Several batch entries (copies and kernels overlapped per chunk), GQA, the
    caller's pinned result buffers; and a rectangular (Nq < Nk) host call."""
    q, _, _ = make_qkv(3, 8, 257, 128, torch.bfloat16, seed=11)
    _, k, v = make_qkv(3, 2, 257, 128, torch.bfloat16, seed=12, H_kv=2)
    out = torch.full(q.shape, -7.0, dtype=q.dtype).pin_memory()
    lse_out = torch.full(q.shape[:-1], -7.0).pin_memory()
    o, lse = fa.forward(q.pin_memory(), k.pin_memory(), v.pin_memory(), 0.09, "causal",
                        out=out, lse_out=lse_out)
    assert o.data_ptr() == out.data_ptr() and lse.data_ptr() == lse_out.data_ptr()
    compare(o, lse, q, k, v, 0.09, "causal")
    q2 = q[:, :, -5:].contiguous()
    o2, l2 = fa.forward(q2, k, v, 0.09, "causal")
    compare(o2, l2, q2, k, v, 0.09, "causal")


@pytest.mark.parametrize("d", [32, 64, 256])
@pytest.mark.parametrize("chunk_bytes", [1, 300_000])
def test_forward_host_tensors_chunked_by_heads(monkeypatch, chunk_bytes, d):
    """The host pipeline cut into chunks of K/V heads (one K/V head with its query
    heads per chunk, or more), grouped heads, and a split-KV (Nq < Nk) call."""
    from tiled_attention_03_gb300 import binding
    monkeypatch.setattr(binding, "HOST_CHUNK_BYTES", chunk_bytes)
    q, _, _ = make_qkv(2, 6, 200, d, torch.float16, seed=13)
    _, k, v = make_qkv(2, 3, 200, d, torch.float16, seed=14, H_kv=3)
    o, lse = fa.forward(q.pin_memory(), k.pin_memory(), v.pin_memory(), 0.125, "causal")
    compare(o, lse, q, k, v, 0.125, "causal")
    q2 = q[:, :, -3:].contiguous()
    o2, l2 = fa.forward(q2, k, v, 0.125, "causal")
    compare(o2, l2, q2, k, v, 0.125, "causal")


def test_forward_host_pipeline_splits_pageable_and_checks():
    """fa_forward_host with key splits on Nq == Nk, with pageable (not pinned)
    host tensors, and its own rejections: a device pointer among the host
    buffers, a workspace that is too small."""
    q, k, v = make_qkv(2, 4, 300, 64, torch.bfloat16, seed=15)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], dtype=torch.float32)
    fa.fa_forward_host(q, k, v, o, lse, 0.125, "causal", num_splits=3, chunk_bytes=1)
    torch.cuda.synchronize()
    compare(o, lse, q, k, v, 0.125, "causal")
    lib = fa.load_library()
    need = fa.fa_forward_host_workspace_bytes(2, 4, 4, 300, 300, 64)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    args = (2, 4, 4, 300, 300, 64, 0.125, 0, 0, 0, 1, 0, 0)
    qd = q.cuda()
    assert lib.fa_forward_host(qd.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               *args, ws.data_ptr(), need, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               *args, ws.data_ptr(), need - 256, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_forward_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               *args, ws.data_ptr(), need, None) == fa.FA_OK
    torch.cuda.synchronize()
    compare(o, lse, q, k, v, 0.125, "none")
    assert fa.fa_sync_status() == fa.FA_OK


@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (200, 17))])
def test_forward_host_bit_identical_to_device_call(monkeypatch, mask, window):
    """Each row's arithmetic does not depend on how heads are grouped into launches,
    so the host pipeline (chunks of one K/V head) gives exactly the device call's
    O and LSE."""
    from tiled_attention_03_gb300 import binding
    monkeypatch.setattr(binding, "HOST_CHUNK_BYTES", 1)
    q, _, _ = make_qkv(2, 8, 700, 128, torch.bfloat16, seed=16)
    _, k, v = make_qkv(2, 4, 700, 128, torch.bfloat16, seed=17, H_kv=4)
    o_h, l_h = fa.forward(q.pin_memory(), k.pin_memory(), v.pin_memory(), 0.088, mask, window)
    o_d, l_d = fa.forward(q.cuda(), k.cuda(), v.cuda(), 0.088, mask, window)
    torch.cuda.synchronize()
    assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


def test_rejects_host_pointer_in_abi():
    q, k, v = make_qkv(1, 1, 64, 64, torch.float16, seed=0)
    lib = fa.load_library()
    dq = q.cuda()
    o = torch.empty_like(dq)
    lse = torch.empty(1, 1, 64, device="cuda")
    rc = lib.fa_forward(q.data_ptr(), dq.data_ptr(), dq.data_ptr(), o.data_ptr(), lse.data_ptr(),
                        1, 1, 64, 64, 0.125, 0, 0, 0, 0, None)
    assert rc == fa.FA_ERR_INVALID_ARG
    assert fa.fa_sync_status() == fa.FA_OK
