"""C-ABI checks that need no GPU: the library loads, exports every function
include/*.h declares, and rejects invalid arguments before touching CUDA."""

import ctypes

import pytest

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.binding import declared_functions, load_library
from tiled_attention_03_gb300.build import build_library


@pytest.fixture(scope="module")
def lib():
    build_library()
    return load_library()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"fa_forward", "fa_status_string", "fa_sync_status"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for code in range(5):
        s = fa.fa_status_string(code)
        assert s.startswith("FA_")
    assert "unknown" in fa.fa_status_string(99)


A = 0x10000  # aligned fake addresses: never dereferenced, every call below fails its checks first
B_ = 0x20000000
C = 0x40000000
O_ = 0x60000000
L_ = 0x70000000


def call(lib, q=A, k=B_, v=C, o=O_, lse=L_, B=1, H=1, N=16, d=64, scale=0.125, mask=0,
         wl=0, wr=0, dtype=0):
    return lib.fa_forward(q, k, v, o, lse, B, H, N, d, scale, mask, wl, wr, dtype, None)


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(k=0), dict(v=0), dict(o=0), dict(lse=0),
    dict(B=0), dict(H=0), dict(N=0), dict(d=0), dict(N=-5),
    dict(dtype=2), dict(dtype=-1), dict(mask=3), dict(mask=-1),
    dict(mask=2, wl=-1), dict(mask=2, wr=-1),
    dict(scale=0.0), dict(scale=-0.5), dict(scale=float("inf")), dict(scale=float("nan")),
    dict(q=A + 8), dict(o=O_ + 2), dict(lse=L_ + 2),
    dict(o=O_ + 16),        # O takes 32-byte stores: 16-byte alignment is not enough
    dict(o=A),              # O aliases Q
    dict(lse=O_ + 64),      # LSE inside O
])
def test_invalid_arguments(lib, kw):
    assert call(lib, **kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [16, 96, 80, 512])
def test_unsupported_head_dim(lib, d):
    assert call(lib, d=d) == fa.FA_ERR_UNSUPPORTED


@pytest.mark.parametrize("hk", [0, -1, 3, 5])
def test_gqa_invalid_kv_heads(lib, hk):
    rc = lib.fa_forward_gqa(A, B_, C, O_, L_, 1, 4, hk, 16, 64, 0.125, 0, 0, 0, 0, None)
    assert rc == fa.FA_ERR_INVALID_ARG


def test_window_args_ignored_unless_window(lib):
    # Negative window values are only an error in window mode: in the other modes
    # the call gets past argument checks (and then fails on this GPU-less host).
    rc = call(lib, mask=1, wl=-3, wr=-3)
    assert rc != fa.FA_ERR_INVALID_ARG


def test_wait_budget_and_counter(lib):
    fa.fa_set_wait_budget_ns(0)
    assert fa.fa_launch_count() >= 0


def test_python_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float16)
    with pytest.raises(fa.FaError):
        fa.fa_forward(q, q, q, q.clone(), torch.zeros(1, 1, 8), 0.125)


# fa_backward: Q K V O dO LSE dQ dK dV at distinct aligned fake addresses (never dereferenced)
BW = dict(q=0x100000, k=0x200000, v=0x300000, o=0x400000, do=0x500000, lse=0x600000,
          dq=0x700000, dk=0x800000, dv=0x900000, ws=0xA00000)


def bwd_call(lib, B=1, H=2, Hk=2, N=16, d=64, scale=0.125, mask=0, wl=0, wr=0, dtype=0,
             ws_bytes=None, **ptrs):
    a = dict(BW, **ptrs)
    if ws_bytes is None:
        ws_bytes = lib.fa_backward_workspace_bytes(B, H, N, d)
    return lib.fa_backward(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                           a["dv"], B, H, Hk, N, d, scale, mask, wl, wr, dtype, a["ws"], ws_bytes, None)


def test_backward_workspace_size(lib):
    assert lib.fa_backward_workspace_bytes(0, 1, 1, 64) == 0
    small = lib.fa_backward_workspace_bytes(1, 1, 1, 64)
    big = lib.fa_backward_workspace_bytes(2, 4, 1000, 128)
    assert 0 < small < big


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(do=0), dict(lse=0), dict(dq=0), dict(dv=0), dict(ws=0),
    dict(B=0), dict(N=0), dict(Hk=0), dict(Hk=3), dict(dtype=5), dict(mask=7),
    dict(mask=2, wl=-1), dict(scale=0.0), dict(scale=float("nan")),
    dict(q=0x100008), dict(dk=0x800004), dict(ws=0xA00002),
    dict(dq=0x700010), dict(dk=0x800010), dict(dv=0x900010), dict(ws=0xA00010),  # 32-byte stores
    dict(dq=0x100000),            # dQ aliases Q
    dict(dk=0x700000),            # dK overlaps dQ
    dict(ws=0x500000),            # workspace overlaps dO
    dict(ws_bytes=16),            # workspace too small
])
def test_backward_invalid_arguments(lib, kw):
    assert bwd_call(lib, **kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("d", [16, 96, 512])
def test_backward_unsupported_head_dim(lib, d):
    assert bwd_call(lib, d=d) == fa.FA_ERR_UNSUPPORTED


def varlen_call(lib, B=2, H=2, Hk=2, tq=100, tk=100, maxq=60, d=64, scale=0.125, mask=0, wl=0,
                wr=0, dtype=0, **ptrs):
    a = dict(q=0x100000, k=0x200000, v=0x300000, o=0x400000, lse=0x600000, cq=0x700000,
             ck=0x800000)
    a.update(ptrs)
    return lib.fa_forward_varlen(a["q"], a["k"], a["v"], a["o"], a["lse"], a["cq"], a["ck"], B, H, Hk,
                                 tq, tk, maxq, d, scale, mask, wl, wr, dtype, None)


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(cq=0), dict(ck=0), dict(B=0), dict(Hk=3), dict(tk=0), dict(tq=-1),
    dict(dtype=4), dict(mask=2, wr=-1), dict(scale=-1.0), dict(q=0x100004), dict(cq=0x700002),
    dict(o=0x400010),            # O 16- but not 32-byte aligned
    dict(o=0x100000),            # O aliases Q
    dict(lse=0x400010),          # LSE inside O
])
def test_varlen_invalid_arguments(lib, kw):
    assert varlen_call(lib, **kw) == fa.FA_ERR_INVALID_ARG


def test_varlen_empty_is_ok_without_pointers(lib):
    assert varlen_call(lib, tq=0, maxq=0, q=0, k=0, v=0, o=0, lse=0, cq=0, ck=0) == fa.FA_OK


@pytest.mark.parametrize("kw", [dict(d=96), dict(maxq=101)])
def test_varlen_unsupported(lib, kw):
    assert varlen_call(lib, **kw) == fa.FA_ERR_UNSUPPORTED


def bwd_varlen_call(lib, d=64, **kw):
    # host checks only: every pointer is fake and every check before the device
    # lookup is on the arguments alone
    B, H, tq = 2, 2, 100
    return lib.fa_backward_varlen(0x100000, 0x200000, 0x300000, 0x400000, 0x500000, 0x600000,
                                  0x700000, 0x700100, 0x800000, 0x900000, 0xA00000, B, H, H, tq, tq,
                                  60, 60, d, 0.125, 0, 0, 0, 0, 0xB00000,
                                  lib.fa_backward_varlen_workspace_bytes(B, H, tq), None)


@pytest.mark.parametrize("d", [16, 96, 512])
def test_backward_varlen_unsupported_head_dim(lib, d):
    assert bwd_varlen_call(lib, d=d) == fa.FA_ERR_UNSUPPORTED


def host_call(lib, B=1, H=2, Hk=2, Nq=128, Nk=128, d=64, scale=0.125, mask=0, wl=0, wr=0,
              dtype=0, splits=0, chunk=0, ws_bytes=1 << 30, **ptrs):
    a = dict(q=0x100000, k=0x200000, v=0x300000, o=0x400000, lse=0x600000, ws=0x700000)
    a.update(ptrs)
    return lib.fa_forward_host(a["q"], a["k"], a["v"], a["o"], a["lse"], B, H, Hk, Nq, Nk, d, scale,
                               mask, wl, wr, dtype, splits, chunk, a["ws"], ws_bytes, None)


def test_host_pipeline_workspace_size(lib):
    # Q, K, V, O copies (32 KiB each) and the LSE copy (1 KiB); no key-split scratch
    assert lib.fa_forward_host_workspace_bytes(1, 2, 2, 128, 128, 64, 0, 0) == 4 * 32768 + 1024
    # Nq < Nk adds the split scratch of the largest chunk
    assert (lib.fa_forward_host_workspace_bytes(1, 2, 2, 4, 4096, 64, 0, 0) >
            lib.fa_forward_host_workspace_bytes(1, 2, 2, 4, 4, 64, 0, 0))
    # d = 256 takes the split form too (Nq < Nk, or splits requested)
    assert (lib.fa_forward_host_workspace_bytes(1, 2, 2, 64, 128, 256, 0, 0) >
            lib.fa_forward_host_workspace_bytes(1, 2, 2, 64, 64, 256, 0, 0) > 0)
    assert (lib.fa_forward_host_workspace_bytes(1, 2, 2, 1024, 1024, 256, 2, 0) >
            lib.fa_forward_host_workspace_bytes(1, 2, 2, 1024, 1024, 256, 0, 0) > 0)
    for bad in [(0, 2, 2, 128, 128, 64, 0, 0), (1, 3, 2, 128, 128, 64, 0, 0),
                (1, 2, 2, 128, 128, 96, 0, 0), (1, 2, 2, 128, 128, 64, -1, 0)]:
        assert lib.fa_forward_host_workspace_bytes(*bad) == 0


@pytest.mark.parametrize("kw", [
    dict(q=0), dict(o=0), dict(lse=0), dict(ws=0), dict(B=0), dict(Hk=3), dict(Nq=0),
    dict(dtype=2), dict(mask=3), dict(mask=2, wl=-1), dict(scale=0.0), dict(splits=-1),
    dict(mask=1, Nq=200), dict(lse=0x600002),
    dict(ws=0x700010),           # workspace 16- but not 32-byte aligned
])
def test_host_pipeline_invalid_arguments(lib, kw):
    assert host_call(lib, **kw) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("kw", [dict(d=96), dict(d=16), dict(d=512)])
def test_host_pipeline_unsupported(lib, kw):
    assert host_call(lib, **kw) == fa.FA_ERR_UNSUPPORTED


def test_splitkv_workspace_must_be_32_byte_aligned(lib):
    # the split scratch takes 32-byte stores: a workspace only 16-byte aligned is refused
    # before anything else is looked at
    args = [0x100000, 0x200000, 0x300000, 0x400000, 0x600000, 1, 2, 2, 4, 4096, 64, 0.125, 0, 0,
            0, 0, 4]
    assert lib.fa_forward_splitkv(*args, 0x700010, 1 << 24, None) == fa.FA_ERR_INVALID_ARG
    assert lib.fa_forward_splitkv(*args, 0x700008, 1 << 24, None) == fa.FA_ERR_INVALID_ARG


def test_release_build_has_no_debug_checks(lib):
    assert lib.fa_debug_flags() == 0
    lib.fa_test_arm_row_shift(0)  # accepted (and ignored) by release builds
