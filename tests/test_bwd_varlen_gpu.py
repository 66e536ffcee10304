"""Variable-length backward (fa_backward_varlen): packed sequences, each compared with
the fp64 gradient oracle run on that sequence alone."""

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

from test_bwd_gpu import TOL_REL

pytestmark = pytest.mark.gpu


def check(got, ref, dtype, what):
    g = got.float().numpy().astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: NaN/Inf"
    err = np.abs(g - ref).max() if ref.size else 0.0
    scale = max(np.abs(ref).max() if ref.size else 0.0, 0.1)
    assert err <= TOL_REL[dtype] * scale, f"{what}: max err {err:.3g} vs {scale:.3g}"


def run_case(lens_q, lens_k, H, Hk, d, dtype, mask, window, seed):
    dev = torch.device("cuda", 0)
    seqs = []
    for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        q = make_qkv(1, H, max(lq, 1), d, dtype, seed=seed + 4 * b)[0][:, :, :lq]
        _, k, v = make_qkv(1, Hk, max(lk, 1), d, dtype, seed=seed + 4 * b + 1, H_kv=Hk)
        do = make_qkv(1, H, max(lq, 1), d, dtype, seed=seed + 4 * b + 2)[0][:, :, :lq]
        seqs.append((q, k[:, :, :lk], v[:, :, :lk], do))
    pack = lambda ts: torch.cat([t[0].transpose(0, 1) for t in ts], 0).contiguous().to(dev)
    Q, K, V, DO = (pack([s[i] for s in seqs]) for i in range(4))
    cu = lambda ls: torch.tensor(np.concatenate([[0], np.cumsum(ls)]), dtype=torch.int32, device=dev)
    cq, ck = cu(lens_q), cu(lens_k)
    scale = d ** -0.5
    O = torch.empty_like(Q)
    LSE = torch.empty(Q.shape[:2], dtype=torch.float32, device=dev)
    fa.fa_forward_varlen(Q, K, V, O, LSE, cq, ck, max(lens_q), scale, mask, window[0], window[1])
    # outputs inside sentinel-filled buffers: a store outside them shows as a changed guard
    G = 4096
    bufs = [torch.full((t.numel() + 2 * G,), -555.0, dtype=t.dtype, device=dev) for t in (Q, K, V)]
    dQ, dK, dV = (b[G:G + t.numel()].view(t.shape) for b, t in zip(bufs, (Q, K, V)))
    for t in (dQ, dK, dV):
        t.fill_(9.0)
    fa.fa_backward_varlen(Q, K, V, O, DO, LSE, cq, ck, dQ, dK, dV, max(lens_q), max(lens_k), scale,
                          mask, window[0], window[1])
    st = fa.fa_sync_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    for b in bufs:
        assert bool((b[:G] == -555.0).all()) and bool((b[-G:] == -555.0).all()), "stray write"
    dQ, dK, dV = dQ.cpu(), dK.cpu(), dV.cpu()
    for b, (q, k, v, do) in enumerate(seqs):
        lq, lk = q.shape[2], k.shape[2]
        t0, s0 = int(cq[b]), int(ck[b])
        gk = dK[s0:s0 + lk].transpose(0, 1)
        gv = dV[s0:s0 + lk].transpose(0, 1)
        if lq == 0:
            assert bool((gk == 0).all()) and bool((gv == 0).all()), f"sequence {b}: keys without queries"
            continue
        rQ, rK, rV = oracle.attention_bwd(q, k, v, do, float(torch.tensor(scale, dtype=torch.float32)),
                                          mask, window)
        gq = dQ[t0:t0 + lq].transpose(0, 1).reshape(Hk, H // Hk, lq, d)
        check(gq, rQ, dtype, f"seq {b} dQ")
        check(gk, rK, dtype, f"seq {b} dK")
        check(gv, rV, dtype, f"seq {b} dV")


CASES = [
    ([1, 127, 128, 129, 300], None, 2, 2),
    ([200, 0, 64, 257], None, 4, 2),          # an empty sequence: its keys get zero gradients
    ([5, 40, 130], [700, 40, 1000], 4, 1),    # fewer queries than keys
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [32, 64, 128, 256])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (90, 3))])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_bwd_varlen_parity(case, mask, window, d, dtype):
    lens_q, lens_k, H, Hk = CASES[case]
    run_case(lens_q, lens_k or lens_q, H, Hk, d, dtype, mask, window, seed=31 * case + d)


@pytest.mark.parametrize("d", [128, 256])
def test_bwd_varlen_many_units_per_cta(d):
    """16 sequences of up to 512 tokens, 4 heads: 256 units per pass on 152 SMs, so
    CTAs run a second unit of another sequence."""
    lens = [512, 300, 129, 512, 64, 511, 200, 512, 384, 1, 450, 512, 257, 128, 500, 33]
    run_case(lens, lens, 4, 4, d, torch.bfloat16, "causal", (0, 0), seed=71)


@pytest.mark.parametrize("d", [64, 256])
def test_bwd_varlen_matches_dense(d):
    """Equal lengths: bit-identical to fa_backward on the (B, H, N, d) layout."""
    from test_bwd_gpu import run_bwd
    dev = torch.device("cuda", 0)
    B, H, N = 3, 4, 333
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=5)
    do = make_qkv(B, H, N, d, torch.bfloat16, seed=6)[0]
    dq_d, dk_d, dv_d = run_bwd(q, k, v, do, 0.125, "causal")
    tok = lambda t: t.transpose(1, 2).reshape(B * N, H, d).contiguous().to(dev)
    Q, K, V, DO = tok(q), tok(k), tok(v), tok(do)
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32, device=dev)
    O = torch.empty_like(Q)
    LSE = torch.empty(B * N, H, dtype=torch.float32, device=dev)
    fa.fa_forward_varlen(Q, K, V, O, LSE, cu, cu, N, 0.125, "causal")
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    fa.fa_backward_varlen(Q, K, V, O, DO, LSE, cu, cu, dQ, dK, dV, N, N, 0.125, "causal")
    assert fa.fa_sync_status() == fa.FA_OK
    assert torch.equal(dQ.cpu(), tok(dq_d.cpu()).cpu())
    assert torch.equal(dK.cpu(), tok(dk_d.cpu()).cpu())
    assert torch.equal(dV.cpu(), tok(dv_d.cpu()).cpu())
