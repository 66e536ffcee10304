"""Variable-length batches (fa_forward_varlen): sequences of different lengths packed
token-major; each sequence is compared with the oracle run on that sequence alone."""

import numpy as np
import pytest
import torch

import oracle
import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

from parity_util import GUARD, SENT_L, TOL_LSE, TOL_O

pytestmark = pytest.mark.gpu


def packed_inputs(lens_q, lens_k, H, Hk, d, dtype, seed):
    """Per-sequence (1, H, L, d) tensors drawn with the workload recipe, and their
    token-major packing (total, H, d)."""
    seqs = []
    for b, (lq, lk) in enumerate(zip(lens_q, lens_k)):
        q, _, _ = make_qkv(1, H, max(lq, 1), d, dtype, seed=seed + 3 * b)
        _, k, v = make_qkv(1, Hk, max(lk, 1), d, dtype, seed=seed + 3 * b + 1, H_kv=Hk)
        seqs.append((q[:, :, :lq], k[:, :, :lk], v[:, :, :lk]))
    pack = lambda ts: torch.cat([t[0].transpose(0, 1) for t in ts], 0).contiguous()
    Q = pack([s[0] for s in seqs])
    K = pack([s[1] for s in seqs])
    V = pack([s[2] for s in seqs])
    cu = lambda ls: torch.tensor(np.concatenate([[0], np.cumsum(ls)]), dtype=torch.int32)
    return seqs, Q, K, V, cu(lens_q), cu(lens_k)


def run_varlen(Q, K, V, cu_q, cu_k, max_q, scale, mask, window):
    dev = torch.device("cuda", 0)
    Q, K, V, cu_q, cu_k = (t.to(dev) for t in (Q, K, V, cu_q, cu_k))
    n, rows = Q.numel(), Q.shape[0] * Q.shape[1]
    obuf = torch.full((n + 2 * GUARD,), -777.0, dtype=Q.dtype, device=dev)
    lbuf = torch.full((rows + 2 * GUARD,), SENT_L, dtype=torch.float32, device=dev)
    o = obuf[GUARD:GUARD + n].view(Q.shape)
    lse = lbuf[GUARD:GUARD + rows].view(Q.shape[0], Q.shape[1])
    fa.fa_forward_varlen(Q, K, V, o, lse, cu_q, cu_k, max_q, scale, mask, window[0], window[1])
    st = fa.fa_sync_status()
    assert st == fa.FA_OK, fa.fa_status_string(st)
    for buf, sent in ((obuf, -777.0), (lbuf, SENT_L)):
        assert bool((buf[:GUARD] == sent).all()) and bool((buf[-GUARD:] == sent).all()), "stray write"
    return o.cpu(), lse.cpu()


def check(seqs, o, lse, cu_q, scale, mask, window, dtype):
    for b, (q, k, v) in enumerate(seqs):
        lq = q.shape[2]
        if lq == 0:
            continue
        O, LSE = oracle.attention(q, k, v, scale, mask, window)   # rows (h, i) in that order
        t0 = int(cu_q[b])
        got_o = o[t0:t0 + lq].transpose(0, 1).reshape(-1, q.shape[3]).double().numpy()
        got_l = lse[t0:t0 + lq].transpose(0, 1).reshape(-1).double().numpy()
        assert np.isfinite(got_o).all() and np.isfinite(got_l).all()
        assert np.abs(got_o - O).max() <= TOL_O[dtype], f"sequence {b}: O"
        assert np.abs(got_l - LSE).max() <= TOL_LSE, f"sequence {b}: LSE"


CASES = [
    # lens_q, lens_k, H, Hk
    ([1, 127, 128, 129, 300], None, 2, 2),
    ([513, 0, 64, 200], None, 4, 2),          # an empty sequence in the middle
    ([5, 40, 128], [700, 40, 1000], 4, 1),    # fewer queries than keys (chunked prefill)
    ([1, 1, 1, 1], [3000, 17, 129, 256], 8, 2),  # one decode step per sequence
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (90, 3))])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_varlen_parity(case, mask, window, d, dtype):
    lens_q, lens_k, H, Hk = CASES[case]
    lens_k = lens_k or lens_q
    seqs, Q, K, V, cu_q, cu_k = packed_inputs(lens_q, lens_k, H, Hk, d, dtype, seed=17 * case + d)
    scale = d ** -0.5
    o, lse = run_varlen(Q, K, V, cu_q, cu_k, max(lens_q), scale, mask, window)
    check(seqs, o, lse, cu_q, scale, mask, window, dtype)


@pytest.mark.parametrize("d", [128, 256])
def test_varlen_matches_dense_batch(d):
    """Equal lengths: the same numbers as fa_forward on the (B, H, N, d) layout."""
    B, H, N = 3, 4, 333
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=3)
    dev = torch.device("cuda", 0)
    o_d, l_d = fa.forward(q.to(dev), k.to(dev), v.to(dev), d ** -0.5, "causal")
    tok = lambda t: t.transpose(1, 2).reshape(B * N, H, d).contiguous()
    cu = torch.arange(0, (B + 1) * N, N, dtype=torch.int32)
    o_v, l_v = run_varlen(tok(q), tok(k), tok(v), cu, cu, N, d ** -0.5, "causal", (0, 0))
    assert torch.equal(o_v, tok(o_d.cpu()))
    assert torch.equal(l_v, l_d.cpu().transpose(1, 2).reshape(B * N, H))


def test_varlen_no_queries_is_a_no_op():
    dev = torch.device("cuda", 0)
    q = torch.zeros(0, 2, 64, dtype=torch.float16, device=dev)
    k = torch.randn(10, 2, 64, dtype=torch.float16, device=dev)
    cu_q = torch.zeros(3, dtype=torch.int32, device=dev)
    cu_k = torch.tensor([0, 5, 10], dtype=torch.int32, device=dev)
    fa.fa_forward_varlen(q, k, k, torch.empty_like(q), torch.empty(0, 2, device=dev), cu_q, cu_k,
                         0, 0.125)
    assert fa.fa_sync_status() == fa.FA_OK


@pytest.mark.parametrize("name", ["varlen_causal_b16h32n4096d128", "varlen_causal_b16h16n4096d256"])
def test_varlen_workload_sampled(name):
    """The benchmark's packed batches at full size, in their launch configuration;
    sampled (sequence, head, 128-row block) slices against the oracle."""
    from tiled_attention_03_gb300.workloads import BY_NAME, varlen_inputs, varlen_lengths
    w = BY_NAME[name]
    Q, K, V, cu = varlen_inputs(w)
    lens = varlen_lengths(w)
    o, lse = run_varlen(Q, K, V, cu, cu, max(lens), w.scale, "causal", (0, 0))
    g = torch.Generator().manual_seed(1012)
    for b in (0, w.B - 1, int(torch.randint(0, w.B, (1,), generator=g))):
        t0, L = int(cu[b]), lens[b]
        q = Q[t0:t0 + L].transpose(0, 1).unsqueeze(0)
        k = K[t0:t0 + L].transpose(0, 1).unsqueeze(0)
        v = V[t0:t0 + L].transpose(0, 1).unsqueeze(0)
        nblk = (L + 127) // 128
        units = [(0, 0, min(128, L)), (w.H - 1, (nblk - 1) * 128, L)]
        h = int(torch.randint(0, w.H, (1,), generator=g))
        blk = int(torch.randint(0, nblk, (1,), generator=g))
        units.append((h, blk * 128, min(L, blk * 128 + 128)))
        O, LSE = oracle.attention(q, k, v, w.scale, "causal", units=units)
        got_o = np.concatenate([o[t0 + r0:t0 + r1, hh].double().numpy() for hh, r0, r1 in units])
        got_l = np.concatenate([lse[t0 + r0:t0 + r1, hh].double().numpy() for hh, r0, r1 in units])
        assert np.abs(got_o - O).max() <= TOL_O[w.dtype]
        assert np.abs(got_l - LSE).max() <= TOL_LSE
