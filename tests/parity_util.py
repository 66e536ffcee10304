"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
with sentinel guard bands around O and LSE, and compare with the oracle."""

import numpy as np
import torch

import oracle
import tiled_attention_03_gb300 as fa

TOL_O = {torch.float16: 4e-3, torch.bfloat16: 2e-2}
TOL_LSE = 1e-3
GUARD = 4096  # elements of sentinel before and after each output
SENT_O = {torch.float16: -777.0, torch.bfloat16: -777.0}
SENT_L = -12345.0


def run_cuda(q, k, v, scale, mask="none", window=(0, 0), check_guards=True):
    """q, k, v: CPU or CUDA (B, H, N, d) tensors. Returns CUDA (O, LSE)."""
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev).contiguous() for t in (q, k, v))
    B, H, N, d = q.shape
    n = B * H * N * d
    obuf = torch.full((n + 2 * GUARD,), SENT_O[q.dtype], dtype=q.dtype, device=dev)
    lbuf = torch.full((B * H * N + 2 * GUARD,), SENT_L, dtype=torch.float32, device=dev)
    o = obuf[GUARD:GUARD + n].view(B, H, N, d)
    lse = lbuf[GUARD:GUARD + B * H * N].view(B, H, N)
    if k.shape[1] == q.shape[1]:
        fa.fa_forward(q, k, v, o, lse, scale, mask, window[0], window[1])
    else:
        fa.fa_forward_gqa(q, k, v, o, lse, scale, mask, window[0], window[1])
    st = fa.fa_sync_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    if check_guards:
        for buf, s in ((obuf, SENT_O[q.dtype]), (lbuf, SENT_L)):
            assert bool((buf[:GUARD] == s).all()), "write before the output"
            assert bool((buf[-GUARD:] == s).all()), "write past the output"
    return o, lse


def compare(o, lse, q, k, v, scale, mask="none", window=(0, 0), units=None, tol_o=None):
    """Element-wise comparison against the oracle on `units` (default: all rows)."""
    B, H, N, d = q.shape
    O, LSE = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale, mask, window, units=units)
    oc = o.float().cpu().reshape(B * H, N, d)
    lc = lse.cpu().reshape(B * H, N)
    if units is None:
        units = [(bh, 0, N) for bh in range(B * H)]
    got_o = np.concatenate([oc[bh, r0:r1].numpy() for bh, r0, r1 in units]).astype(np.float64)
    got_l = np.concatenate([lc[bh, r0:r1].numpy() for bh, r0, r1 in units]).astype(np.float64)
    assert np.isfinite(got_o).all() and np.isfinite(got_l).all(), "NaN/Inf in the output"
    err_o = np.abs(got_o - O).max()
    err_l = np.abs(got_l - LSE).max()
    tol = TOL_O[q.dtype] if tol_o is None else tol_o
    assert err_o <= tol, f"max|O - oracle| = {err_o:.3g} > {tol}"
    assert err_l <= TOL_LSE, f"max|LSE - oracle| = {err_l:.3g} > {TOL_LSE}"
    return err_o, err_l
