"""Failure path on the GPU without a GPU fault: a bounded in-kernel wait is made to run
out (a K tile that is never loaded), the kernel gives up cleanly, fa_sync_status reports
FA_ERR_TIMEOUT, and the context keeps working."""

import time

import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

from parity_util import compare, run_cuda

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("d,mask", [(128, "none"), (64, "causal")])
def test_wait_timeout_is_reported_and_gpu_recovers(d, mask):
    q, k, v = make_qkv(1, 4, 1024, d, torch.bfloat16, seed=1)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(dq)
    lse = torch.empty(dq.shape[:-1], device="cuda")
    assert fa.fa_sync_status() == fa.FA_OK
    fa.fa_set_wait_budget_ns(50_000_000)  # 50 ms
    try:
        fa.fa_test_arm_fault(0)
        t0 = time.time()
        fa.fa_forward(dq, dk, dv, o, lse, d ** -0.5, mask)
        st = fa.fa_sync_status()
        elapsed = time.time() - t0
    finally:
        fa.fa_set_wait_budget_ns(0)
    assert st == fa.FA_ERR_TIMEOUT, fa.fa_status_string(st)
    assert elapsed < 5.0
    # the status word was cleared and the next launches are correct
    assert fa.fa_sync_status() == fa.FA_OK
    o2, lse2 = run_cuda(q, k, v, d ** -0.5, mask)
    compare(o2, lse2, q, k, v, d ** -0.5, mask)


def test_hook_is_one_shot():
    q, k, v = make_qkv(1, 2, 600, 64, torch.float16, seed=2)
    fa.fa_set_wait_budget_ns(50_000_000)
    try:
        fa.fa_test_arm_fault(0)
        fa.fa_test_arm_fault(-1)  # disarmed again
        o, lse = run_cuda(q, k, v, 0.125, "none")
    finally:
        fa.fa_set_wait_budget_ns(0)
    compare(o, lse, q, k, v, 0.125, "none")


@pytest.mark.parametrize("varlen", [False, True])
def test_backward_wait_timeout_is_reported_and_gpu_recovers(varlen):
    """The same for the backward: the dK/dV kernel's first unit in every CTA never
    gets its K/V tile; its waits run out, every role gives up, the status reads
    FA_ERR_TIMEOUT, and the next backward is correct."""
    from test_bwd_gpu import compare as bwd_compare, run_bwd
    q, k, v = make_qkv(1, 4, 700, 64, torch.bfloat16, seed=3)
    do = make_qkv(1, 4, 700, 64, torch.bfloat16, seed=4)[0]
    dev = torch.device("cuda", 0)
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qd)
    lse = torch.empty(qd.shape[:-1], device=dev)
    fa.fa_forward(qd, kd, vd, o, lse, 0.125, "causal")
    assert fa.fa_sync_status() == fa.FA_OK
    grads = [torch.empty_like(t) for t in (qd, kd, vd)]
    fa.fa_set_wait_budget_ns(50_000_000)
    try:
        fa.fa_test_arm_fault(0)
        t0 = time.time()
        if varlen:
            tok = lambda t: t[0].transpose(0, 1).contiguous()
            cu = torch.tensor([0, 700], dtype=torch.int32, device=dev)
            fa.fa_backward_varlen(tok(qd), tok(kd), tok(vd), tok(o), tok(dod),
                                  lse[0].transpose(0, 1).contiguous(), cu, cu,
                                  *(tok(g) for g in grads), 700, 700, 0.125, "causal")
        else:
            fa.fa_backward(qd, kd, vd, o, dod, lse, *grads, 0.125, "causal")
        st = fa.fa_sync_status()
        elapsed = time.time() - t0
    finally:
        fa.fa_set_wait_budget_ns(0)
    assert st == fa.FA_ERR_TIMEOUT, fa.fa_status_string(st)
    assert elapsed < 5.0
    assert fa.fa_sync_status() == fa.FA_OK
    dq, dk, dv = run_bwd(q, k, v, do, 0.125, "causal")
    bwd_compare(q, k, v, do, 0.125, "causal", (0, 0), dq, dk, dv)


@pytest.mark.parametrize("d,n", [(256, 600), (128, 100)])
def test_onetile_timeout_consumes_the_hook(d, n):
    """The one-tile kernel (every d = 256 forward; a d = 128 head of at most 128
    queries) takes the hook too: its launch times out and reports it, and the hook
    is spent, so the next launch of the two-tile kernel is correct."""
    q, k, v = make_qkv(1, 2, n, d, torch.bfloat16, seed=5)
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(dq)
    lse = torch.empty(dq.shape[:-1], device="cuda")
    assert fa.fa_sync_status() == fa.FA_OK
    fa.fa_set_wait_budget_ns(50_000_000)
    try:
        fa.fa_test_arm_fault(0)
        t0 = time.time()
        fa.fa_forward(dq, dk, dv, o, lse, d ** -0.5, "none")
        st = fa.fa_sync_status()
        elapsed = time.time() - t0
        # the hook was consumed by that launch: this one (two-tile kernel) runs clean
        q2, k2, v2 = make_qkv(1, 2, 600, 64, torch.float16, seed=6)
        o2, lse2 = run_cuda(q2, k2, v2, 0.125, "causal")
        st2 = fa.fa_sync_status()
    finally:
        fa.fa_set_wait_budget_ns(0)
    assert st == fa.FA_ERR_TIMEOUT, fa.fa_status_string(st)
    assert elapsed < 5.0
    assert st2 == fa.FA_OK, fa.fa_status_string(st2)
    compare(o2, lse2, q2, k2, v2, 0.125, "causal")
    o3, lse3 = run_cuda(q, k, v, d ** -0.5, "none")
    compare(o3, lse3, q, k, v, d ** -0.5, "none")
