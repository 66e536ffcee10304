"""The library's debug builds (include/fa.h, "Debug builds"), built here from the same
sources with one extra flag each and loaded next to the release build:

  * FA_DEBUG_SERIALIZE: the two-tile forward with the least overlap its protocol allows;
  * FA_DEBUG_BOUNDS: every store of the two-tile forward checked against the output.

Each runs a small parity sweep against the oracle. The bounds build also shows that a
launch whose stored rows are shifted past the output (its test hook) stores nothing,
reports FA_ERR_BOUNDS through fa_sync_status instead of faulting, and that the next
launch is correct."""

import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.binding import FA_DTYPE_BF16, FA_DTYPE_FP16, load_library_at
from tiled_attention_03_gb300.build import build_library
from tiled_attention_03_gb300.workloads import make_qkv

from parity_util import GUARD, SENT_L, SENT_O, compare

pytestmark = pytest.mark.gpu

MASKS = {"none": 0, "causal": 1, "window": 2}


@pytest.fixture(scope="module", params=["serialize", "bounds"])
def debug_lib(request):
    lib = load_library_at(build_library(debug=request.param))
    flag = {"serialize": fa.FA_DEBUG_SERIALIZE_FLAG, "bounds": fa.FA_DEBUG_BOUNDS_FLAG}[request.param]
    assert lib.fa_debug_flags() == flag
    return request.param, lib


def run(lib, q, k, v, scale, mask, window, splits=0, shift=0):
    """One forward through `lib` with sentinel guard bands around O and LSE; returns
    (O, LSE, guard bands intact, device status)."""
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev).contiguous() for t in (q, k, v))
    B, H, N, d = q.shape
    n = q.numel()
    obuf = torch.full((n + 2 * GUARD,), SENT_O[q.dtype], dtype=q.dtype, device=dev)
    lbuf = torch.full((B * H * N + 2 * GUARD,), SENT_L, dtype=torch.float32, device=dev)
    o = obuf[GUARD:GUARD + n].view(q.shape)
    lse = lbuf[GUARD:GUARD + B * H * N].view(B, H, N)
    dt = FA_DTYPE_BF16 if q.dtype == torch.bfloat16 else FA_DTYPE_FP16
    stream = torch.cuda.current_stream().cuda_stream
    if shift:
        lib.fa_test_arm_row_shift(shift)
    if splits:
        ws = torch.empty(lib.fa_splitkv_workspace_bytes(B, H, N, d, splits), dtype=torch.uint8,
                         device=dev)
        rc = lib.fa_forward_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                    lse.data_ptr(), B, H, H, N, N, d, scale, MASKS[mask],
                                    window[0], window[1], dt, splits, ws.data_ptr(), ws.numel(),
                                    stream)
    else:
        rc = lib.fa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                            B, H, N, d, scale, MASKS[mask], window[0], window[1], dt, stream)
    assert rc == fa.FA_OK, fa.fa_status_string(rc)
    st = lib.fa_sync_status(stream)
    guards = all(bool((b[:GUARD] == s).all()) and bool((b[-GUARD:] == s).all())
                 for b, s in ((obuf, SENT_O[q.dtype]), (lbuf, SENT_L)))
    return o, lse, guards, st, (obuf, lbuf)


# 80 heads of 300 rows: 160 two-tile units, more than half of the SMs, so the
# two-tile kernel (the one the debug flags change) runs every case.
CASES = [(d, mask, window, dtype) for d in (32, 64, 128)
         for mask, window in (("none", (0, 0)), ("causal", (0, 0)), ("window", (100, 20)))
         for dtype in ((torch.float16,) if d == 64 else (torch.bfloat16,))]


@pytest.mark.parametrize("d,mask,window,dtype", CASES)
def test_debug_build_parity(debug_lib, d, mask, window, dtype):
    _, lib = debug_lib
    q, k, v = make_qkv(1, 80, 300, d, dtype, seed=d + len(mask))
    o, lse, guards, st, _ = run(lib, q, k, v, d ** -0.5, mask, window)
    assert st == fa.FA_OK, fa.fa_status_string(st)
    assert guards, "write outside O or LSE"
    compare(o, lse, q, k, v, d ** -0.5, mask, window)


def test_debug_build_split_parity(debug_lib):
    """Key splits: the fp32 partial buffers and the merge."""
    _, lib = debug_lib
    q, k, v = make_qkv(1, 80, 300, 128, torch.bfloat16, seed=5)
    o, lse, guards, st, _ = run(lib, q, k, v, 128 ** -0.5, "causal", (0, 0), splits=2)
    assert st == fa.FA_OK and guards
    compare(o, lse, q, k, v, 128 ** -0.5, "causal")


def test_bounds_check_refuses_and_reports(debug_lib):
    name, lib = debug_lib
    if name != "bounds":
        pytest.skip("the bounds build's hook")
    q, k, v = make_qkv(1, 80, 300, 64, torch.float16, seed=9)
    rows = 80 * 300
    # every stored row shifted by the output's size: each store is refused
    o, lse, guards, st, (obuf, lbuf) = run(lib, q, k, v, 0.125, "causal", (0, 0), shift=rows)
    assert st == fa.FA_ERR_BOUNDS, fa.fa_status_string(st)
    assert bool((obuf == SENT_O[q.dtype]).all()) and bool((lbuf == SENT_L).all()), "a refused row was stored"
    assert lib.fa_sync_status(torch.cuda.current_stream().cuda_stream) == fa.FA_OK  # cleared
    o, lse, guards, st, _ = run(lib, q, k, v, 0.125, "causal", (0, 0))
    assert st == fa.FA_OK and guards
    compare(o, lse, q, k, v, 0.125, "causal")
