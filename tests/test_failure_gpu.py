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
