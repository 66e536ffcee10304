"""fa_forward_splitkv_static: split-KV attention for callers that cannot allocate
device memory (runtimes that reserve all their memory up front, hosts that give the
library no allocator). Its scratch is a fixed array inside the library.

Called through the C ABI on two calls in a row (the second call, on other inputs and
a smaller shape, runs on the scratch the first one left behind). Both calls run the
same kernels with the same split count as fa_forward_splitkv with a caller workspace,
so their results must be bit-identical to it; they are also compared element by
element with the oracle. This file is collected last."""

import ctypes

import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.binding import FA_DTYPE_BF16, FA_DTYPE_FP16, load_library
from tiled_attention_03_gb300.workloads import make_qkv

from parity_util import compare

pytestmark = pytest.mark.gpu

MASKS = {"none": 0, "causal": 1, "window": 2}


def _lib():
    lib = load_library()
    lib.fa_forward_splitkv_static.restype = ctypes.c_int
    lib.fa_forward_splitkv_static.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
        ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
        ctypes.c_int64, ctypes.c_void_p]
    return lib


def _static(lib, q, k, v, o, lse, scale, mask, window, splits):
    B, H, Nq, d = q.shape
    dt = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    return lib.fa_forward_splitkv_static(
        q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, k.shape[1],
        Nq, k.shape[2], d, scale, MASKS[mask], window[0], window[1], dt, splits,
        torch.cuda.current_stream().cuda_stream)


CASES = [
    # (B, H, H_kv, Nq, Nk, d, dtype, mask, window, splits, seed)
    (2, 8, 2, 64, 6000, 128, torch.bfloat16, "causal", (0, 0), 12, 1),
    (1, 4, 4, 3, 2500, 64, torch.float16, "window", (700, 0), 5, 2),
]


def test_static_scratch_matches_workspace_entry_on_two_calls():
    lib = _lib()
    for (B, H, Hk, Nq, Nk, d, dtype, mask, window, splits, seed) in CASES:
        q, _, _ = make_qkv(B, H, Nq, d, dtype, seed=seed)
        _, k, v = make_qkv(B, Hk, Nk, d, dtype, seed=seed + 100, H_kv=Hk)
        q, k, v = q.cuda(), k.cuda(), v.cuda()
        scale = d ** -0.5
        assert fa.fa_splitkv_workspace_bytes(B, H, Nq, d, splits) <= fa.FA_SPLITKV_STATIC_SCRATCH_BYTES
        o_ref = torch.empty_like(q)
        l_ref = torch.empty(q.shape[:-1], device="cuda")
        fa.fa_forward_splitkv(q, k, v, o_ref, l_ref, scale, mask, window[0], window[1], splits)
        o = torch.full_like(q, -777.0)
        lse = torch.full(q.shape[:-1], -12345.0, device="cuda")
        rc = _static(lib, q, k, v, o, lse, scale, mask, window, splits)
        assert rc == fa.FA_OK, fa.fa_status_string(rc)
        assert fa.fa_sync_status() == fa.FA_OK
        # same kernels, same splits: bit for bit the workspace entry's result
        assert torch.equal(o, o_ref)
        assert torch.equal(lse, l_ref)
        compare(o, lse, q.cpu(), k.cpu(), v.cpu(), scale, mask, window)


def test_static_scratch_checks_the_split_count_it_runs():
    """The size rule counts the splits the call runs: a split count far above the
    number of 128-key tiles is clamped to it, and is accepted when the clamped
    count fits the scratch."""
    lib = _lib()
    B, H, Nq, Nk, d, splits = 1, 8, 256, 256, 128, 1000
    assert fa.fa_splitkv_workspace_bytes(B, H, Nq, d, splits) > fa.FA_SPLITKV_STATIC_SCRATCH_BYTES
    assert fa.fa_splitkv_workspace_bytes(B, H, Nq, d, 2) <= fa.FA_SPLITKV_STATIC_SCRATCH_BYTES
    q, k, v = make_qkv(B, H, Nq, d, torch.bfloat16, seed=7)
    q, k, v = q.cuda(), k.cuda(), v.cuda()
    o_ref = torch.empty_like(q)
    l_ref = torch.empty(q.shape[:-1], device="cuda")
    fa.fa_forward_splitkv(q, k, v, o_ref, l_ref, d ** -0.5, "causal", 0, 0, 2)
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], device="cuda")
    rc = _static(lib, q, k, v, o, lse, d ** -0.5, "causal", (0, 0), splits)
    assert rc == fa.FA_OK, fa.fa_status_string(rc)
    assert fa.fa_sync_status() == fa.FA_OK
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_static_scratch_rejects_requests_beyond_its_size():
    lib = _lib()
    B, H, Nq, d, splits = 4, 32, 512, 128, 64
    assert fa.fa_splitkv_workspace_bytes(B, H, Nq, d, splits) > fa.FA_SPLITKV_STATIC_SCRATCH_BYTES
    q = torch.zeros(B, H, Nq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(B, H, 8192, d, dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:-1], device="cuda")
    rc = _static(lib, q, k, k, o, lse, 0.1, "none", (0, 0), splits)
    assert rc == fa.FA_ERR_UNSUPPORTED
    assert fa.fa_sync_status() == fa.FA_OK
