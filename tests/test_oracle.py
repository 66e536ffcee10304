"""Pins for the fp64 CPU oracle (no GPU needed).

Each check ties the oracle to something other than itself: a library routine,
a closed form, an invariant of softmax attention, a hand-worked fixture, or an
independent brute-force evaluation. Together they are chosen so that a dropped
term, a wrong sign or index, a transposed operand, a missing scale or a wrong
mask boundary fails at least one of them.
"""

import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from tiled_attention_03_gb300.workloads import make_qkv

HERE = os.path.dirname(os.path.abspath(__file__))
DTYPES = [torch.float16, torch.bfloat16]


def _f64(t):
    return t.to(torch.float64).numpy()


def brute_force(q, k, v, scale, mask, wl=0, wr=0):
    """Independent evaluation with numpy matmuls and scipy's softmax/logsumexp.
    Query i of Nq stands at key position i + Nk - Nq."""
    B, H, Nq, d = q.shape
    N = k.shape[2]
    Q, K, V = _f64(q), _f64(k), _f64(v)
    S = scale * np.einsum("bhid,bhjd->bhij", Q, K)
    i = np.arange(Nq)[:, None] + (N - Nq)
    j = np.arange(N)[None, :]
    if mask == "causal":
        vis = j <= i
    elif mask == "window":
        vis = (j >= i - wl) & (j <= i + wr)
    else:
        vis = np.ones((Nq, N), dtype=bool)
    S = np.where(vis, S, -np.inf)
    P = scipy.special.softmax(S, axis=-1)
    O = np.einsum("bhij,bhjd->bhid", P, V)
    LSE = scipy.special.logsumexp(S, axis=-1)
    return O.reshape(-1, d), LSE.reshape(-1), P.reshape(-1, N)


# --- 16-bit decoding against library conversions --------------------------------

def test_decode_fp16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode16(int(b), torch.float16) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


def test_decode_bf16_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.decode16(int(b), torch.bfloat16) for b in bits])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


# --- brute force on tiny inputs ---------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("N,d", [(1, 4), (5, 4), (17, 64), (64, 64), (33, 8)])
@pytest.mark.parametrize("mask,wl,wr", [("none", 0, 0), ("causal", 0, 0),
                                        ("window", 3, 2), ("window", 0, 0), ("window", 7, 0)])
def test_brute_force(dtype, N, d, mask, wl, wr):
    q, k, v = make_qkv(2, 2, N, d, dtype, seed=N * 31 + d, q_std=2.0)
    scale = 1.0 / math.sqrt(d)
    O, LSE, P = oracle.attention(q, k, v, scale, mask, (wl, wr), return_p=True, nthreads=2)
    Ob, LSEb, Pb = brute_force(q, k, v, scale, mask, wl, wr)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, LSEb, rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(P, Pb, rtol=0, atol=1e-14)


def test_unit_subsets_match_full():
    q, k, v = make_qkv(2, 3, 300, 64, torch.float16, seed=5)
    O, LSE = oracle.attention(q, k, v, 0.125, "causal")
    units = [(4, 128, 256), (0, 0, 128), (5, 256, 300)]
    Os, LSEs = oracle.attention(q, k, v, 0.125, "causal", units=units)
    rows = np.concatenate([bh * 300 + np.arange(r0, r1) for bh, r0, r1 in units])
    np.testing.assert_array_equal(Os, O[rows])
    np.testing.assert_array_equal(LSEs, LSE[rows])


# --- the online recurrence equals the direct definition ---------------------------

@pytest.mark.parametrize("bc", [1, 7, 64, 128])
@pytest.mark.parametrize("mask,wl,wr", [("none", 0, 0), ("causal", 0, 0), ("window", 50, 3)])
def test_online_recurrence_equals_direct(bc, mask, wl, wr):
    q, k, v = make_qkv(1, 2, 203, 64, torch.bfloat16, seed=bc, q_std=3.0)
    O, LSE = oracle.attention(q, k, v, 0.125, mask, (wl, wr))
    Oo, LSEo = oracle.attention(q, k, v, 0.125, mask, (wl, wr), online_bc=bc)
    np.testing.assert_allclose(Oo, O, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(LSEo, LSE, rtol=1e-12, atol=1e-12)


# --- closed forms -----------------------------------------------------------------

def _read_golden(name):
    rows = []
    with open(os.path.join(HERE, "golden", name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                m, wl, wr, i, o0, o1, n = line.split()
                rows.append((m, int(wl), int(wr), int(i), float(o0), float(o1), int(n)))
    return rows


@pytest.mark.parametrize("dtype", DTYPES)
def test_golden_uniform_scores(dtype):
    q = torch.zeros(1, 1, 4, 2, dtype=dtype)
    k = torch.zeros(1, 1, 4, 2, dtype=dtype)
    v = torch.tensor([[1, 2], [3, 4], [5, 6], [7, 8]], dtype=dtype).view(1, 1, 4, 2)
    for m, wl, wr, i, o0, o1, n in _read_golden("uniform_scores_n4_d2.txt"):
        O, LSE = oracle.attention(q, k, v, 1.0, m, (wl, wr))
        assert O[i, 0] == pytest.approx(o0, abs=1e-14)
        assert O[i, 1] == pytest.approx(o1, abs=1e-14)
        assert LSE[i] == pytest.approx(math.log(n), abs=1e-14)


@pytest.mark.parametrize("mask,wl,wr", [("none", 0, 0), ("causal", 0, 0), ("window", 37, 5)])
def test_uniform_scores_mean_of_visible_v(mask, wl, wr):
    N, d = 150, 16
    _, k, v = make_qkv(1, 1, N, d, torch.float16, seed=11)
    q = torch.zeros_like(k)
    O, LSE = oracle.attention(q, k, v, 0.3, mask, (wl, wr))
    V = _f64(v)[0, 0]
    for i in range(N):
        if mask == "none":
            lo, hi = 0, N - 1
        elif mask == "causal":
            lo, hi = 0, i
        else:
            lo, hi = max(0, i - wl), min(N - 1, i + wr)
        cnt = hi - lo + 1
        mean = [sum(V[j, c] for j in range(lo, hi + 1)) / cnt for c in range(d)]
        np.testing.assert_allclose(O[i], mean, rtol=0, atol=1e-13)
        assert LSE[i] == pytest.approx(math.log(cnt), abs=1e-13)


def test_single_row_is_that_value():
    # N = 1: the only key gets weight 1; LSE is its logit.
    q, k, v = make_qkv(1, 1, 1, 8, torch.bfloat16, seed=3)
    O, LSE = oracle.attention(q, k, v, 0.5, "none")
    np.testing.assert_array_equal(O[0], _f64(v)[0, 0, 0])
    logit = 0.5 * float(np.dot(_f64(q)[0, 0, 0], _f64(k)[0, 0, 0]))
    assert LSE[0] == pytest.approx(logit, abs=1e-14)


def test_exact_weights_three_keys():
    # q = (1, 0), keys (0,0), (1,0), (2,0), scale 1 -> logits 0, 1, 2; weights e^x / sum.
    q = torch.tensor([[1.0, 0.0]] * 3, dtype=torch.float16).view(1, 1, 3, 2)
    k = torch.tensor([[0.0, 0.0], [1.0, 0.0], [2.0, 0.0]], dtype=torch.float16).view(1, 1, 3, 2)
    v = torch.tensor([[1.0, -1.0], [2.0, 4.0], [-3.0, 0.5]], dtype=torch.float16).view(1, 1, 3, 2)
    O, LSE = oracle.attention(q, k, v, 1.0, "causal")
    e = math.e
    # row 2 sees all three keys
    z = 1 + e + e * e
    w = [1 / z, e / z, e * e / z]
    assert O[2, 0] == pytest.approx(w[0] * 1 + w[1] * 2 + w[2] * -3, abs=1e-14)
    assert O[2, 1] == pytest.approx(w[0] * -1 + w[1] * 4 + w[2] * 0.5, abs=1e-14)
    assert LSE[2] == pytest.approx(math.log(z), abs=1e-14)
    # row 1 sees keys 0, 1
    z1 = 1 + e
    assert O[1, 0] == pytest.approx((1 + 2 * e) / z1, abs=1e-14)
    assert LSE[1] == pytest.approx(math.log(z1), abs=1e-14)
    # row 0 sees key 0 only: logit 0
    assert O[0, 0] == 1.0 and O[0, 1] == -1.0 and LSE[0] == 0.0


@pytest.mark.parametrize("online_bc", [0, 64])
def test_dominant_key_late(online_bc):
    # One key aligned with the query and far above the rest, placed last, so the
    # running max jumps in the final block: O_i must equal that key's V row.
    N, d = 200, 64
    _, _, v = make_qkv(1, 1, N, d, torch.bfloat16, seed=21)
    q = torch.zeros(1, 1, N, d, dtype=torch.bfloat16)
    q[..., 0] = 4.0
    k = torch.zeros(1, 1, N, d, dtype=torch.bfloat16)
    k[..., 1] = torch.linspace(-1, 1, N).to(torch.bfloat16)  # orthogonal to q: logit 0
    k[0, 0, N - 1, 0] = 8.0  # logit 32 for every query
    O, LSE = oracle.attention(q, k, v, 1.0, "none", online_bc=online_bc)
    V = _f64(v)[0, 0]
    gap = math.exp(-32.0) * N * np.abs(V).max()
    np.testing.assert_allclose(O, np.broadcast_to(V[N - 1], O.shape), rtol=0, atol=2 * gap)
    expect_lse = 32.0 + math.log1p((N - 1) * math.exp(-32.0))
    np.testing.assert_allclose(LSE, expect_lse, rtol=0, atol=1e-12)


# --- invariants -------------------------------------------------------------------

@pytest.mark.parametrize("mask,wl,wr", [("none", 0, 0), ("causal", 0, 0), ("window", 9, 4)])
def test_rows_of_p_sum_to_one_and_respect_mask(mask, wl, wr):
    N = 70
    q, k, v = make_qkv(1, 2, N, 32, torch.float16, seed=2, q_std=3.0)
    _, _, P = oracle.attention(q, k, v, 0.2, mask, (wl, wr), return_p=True)
    np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert (P >= 0).all()
    rows = np.arange(P.shape[0]) % N
    j = np.arange(N)[None, :]
    i = rows[:, None]
    if mask == "causal":
        hidden = j > i
    elif mask == "window":
        hidden = (j < i - wl) | (j > i + wr)
    else:
        hidden = np.zeros_like(j > i)
    assert (P[hidden] == 0).all()
    assert (P[~hidden] > 0).all()


@pytest.mark.parametrize("dtype", DTYPES)
def test_affine_v(dtype):
    # O(2V + 0.5) = 2 O(V) + 0.5; V on a coarse grid so 2V + 0.5 is exact in 16 bits.
    N, d = 90, 32
    q, k, _ = make_qkv(1, 1, N, d, dtype, seed=8)
    g = torch.Generator().manual_seed(9)
    v = (torch.randint(-32, 33, (1, 1, N, d), generator=g).to(torch.float32) / 8).to(dtype)
    v2 = (2 * v.to(torch.float32) + 0.5).to(dtype)
    assert torch.equal(v2.to(torch.float32), 2 * v.to(torch.float32) + 0.5)
    O1, L1 = oracle.attention(q, k, v, 0.25, "causal")
    O2, L2 = oracle.attention(q, k, v2, 0.25, "causal")
    np.testing.assert_allclose(O2, 2 * O1 + 0.5, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(L1, L2)


@pytest.mark.parametrize("mask,wl,wr", [("causal", 0, 0), ("window", 20, 3)])
def test_mask_invariance_bit_exact(mask, wl, wr):
    N, d, i0 = 160, 64, 100
    q, k, v = make_qkv(1, 1, N, d, torch.float16, seed=4)
    k2, v2 = k.clone(), v.clone()
    g = torch.Generator().manual_seed(5)
    if mask == "causal":
        # keys after i0 are hidden from rows <= i0
        sl, rows = slice(i0 + 1, N), slice(0, i0 + 1)
    else:
        # keys before i0 - wl are hidden from rows >= i0 ... as long as i + wr stays below
        # the perturbed region's start, which it does since only earlier keys are changed
        sl, rows = slice(0, i0 - wl), slice(i0, N)
    k2[..., sl, :] = torch.randn(k2[..., sl, :].shape, generator=g).to(k.dtype) * 5
    v2[..., sl, :] = torch.randn(v2[..., sl, :].shape, generator=g).to(v.dtype) * 5
    O1, L1 = oracle.attention(q, k, v, 0.125, mask, (wl, wr))
    O2, L2 = oracle.attention(q, k2, v2, 0.125, mask, (wl, wr))
    np.testing.assert_array_equal(O1[rows], O2[rows])
    np.testing.assert_array_equal(L1[rows], L2[rows])
    # and the perturbation is seen by rows that can see those keys
    other = slice(i0 + 1, N) if mask == "causal" else slice(0, i0 - wl)
    assert not np.array_equal(O1[other], O2[other])


def test_key_permutation_invariance():
    N, d = 130, 64
    q, k, v = make_qkv(1, 2, N, d, torch.bfloat16, seed=6)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(7))
    O1, L1 = oracle.attention(q, k, v, 0.1, "none")
    O2, L2 = oracle.attention(q, k[:, :, perm], v[:, :, perm], 0.1, "none")
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L2, L1, rtol=1e-14, atol=1e-13)


def test_query_permutation_equivariance():
    # Non-causal rows are independent of each other: permuting queries permutes outputs.
    N, d = 77, 32
    q, k, v = make_qkv(1, 1, N, d, torch.float16, seed=12)
    perm = torch.randperm(N, generator=torch.Generator().manual_seed(13))
    O1, L1 = oracle.attention(q, k, v, 0.2, "none")
    O2, L2 = oracle.attention(q[:, :, perm], k, v, 0.2, "none")
    np.testing.assert_array_equal(O2, O1[perm.numpy()])
    np.testing.assert_array_equal(L2, L1[perm.numpy()])


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_logit_shift(mask):
    # K[..., d-1] = 1 and Q[..., d-1] = c/scale: every visible logit of a row moves by c.
    N, d, scale, c = 96, 64, 0.125, 2.0
    q, k, v = make_qkv(1, 1, N, d, torch.float16, seed=14)
    k[..., d - 1] = 1.0
    q0 = q.clone()
    q0[..., d - 1] = 0.0
    q1 = q.clone()
    q1[..., d - 1] = c / scale
    O0, L0 = oracle.attention(q0, k, v, scale, mask)
    O1, L1 = oracle.attention(q1, k, v, scale, mask)
    np.testing.assert_allclose(O1, O0, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L1 - L0, c, rtol=0, atol=1e-12)


def test_scale_enters_logits():
    # Doubling the scale equals doubling Q (exact in 16 bits).
    q, k, v = make_qkv(1, 1, 64, 16, torch.bfloat16, seed=15)
    O1, L1 = oracle.attention(q, k, v, 0.5, "none")
    O2, L2 = oracle.attention((q.float() * 2).to(q.dtype), k, v, 0.25, "none")
    np.testing.assert_allclose(O2, O1, rtol=0, atol=1e-13)
    np.testing.assert_allclose(L2, L1, rtol=0, atol=1e-13)


def test_rejects_bad_arguments():
    q, k, v = make_qkv(1, 1, 8, 4, torch.float16, seed=0)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 1.0, "window", (-1, 0))
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 1.0, "none", units=[(0, 0, 9)])


# --- grouped-query attention ------------------------------------------------------

@pytest.mark.parametrize("H,Hk", [(4, 2), (6, 1), (8, 4)])
@pytest.mark.parametrize("mask,wl,wr", [("none", 0, 0), ("causal", 0, 0), ("window", 9, 2)])
def test_gqa_equals_mha_on_repeated_kv(H, Hk, mask, wl, wr):
    # Grouped K/V heads are shared by H / Hk consecutive query heads: the result equals
    # multi-head attention with each K/V head repeated H / Hk times (same arithmetic).
    B, N, d = 2, 70, 16
    q, _, _ = make_qkv(B, H, N, d, torch.bfloat16, seed=H * 10 + Hk)
    _, k, v = make_qkv(B, Hk, N, d, torch.bfloat16, seed=H * 10 + Hk + 1)
    O1, L1 = oracle.attention(q, k, v, 0.25, mask, (wl, wr))
    rep = H // Hk
    O2, L2 = oracle.attention(q, k.repeat_interleave(rep, dim=1).contiguous(),
                              v.repeat_interleave(rep, dim=1).contiguous(), 0.25, mask, (wl, wr))
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
    # and brute force on the repeated form
    Ob, Lb, _ = brute_force(q, k.repeat_interleave(rep, dim=1), v.repeat_interleave(rep, dim=1),
                            0.25, mask, wl, wr)
    np.testing.assert_allclose(O1, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L1, Lb, rtol=1e-13, atol=1e-12)


def test_gqa_rejects_non_dividing_heads():
    q, _, _ = make_qkv(1, 3, 8, 4, torch.float16, seed=0)
    _, k, v = make_qkv(1, 2, 8, 4, torch.float16, seed=1)
    with pytest.raises(ValueError):
        oracle.attention(q, k, v, 1.0, "none")


# --- fewer queries than keys (queries at the last positions) ---------------------

@pytest.mark.parametrize("Nq,Nk", [(1, 1), (1, 50), (7, 50), (50, 50), (33, 200)])
@pytest.mark.parametrize("mask,wl,wr", [("none", 0, 0), ("causal", 0, 0), ("window", 11, 3)])
def test_rectangular_brute_force(Nq, Nk, mask, wl, wr):
    q, _, _ = make_qkv(2, 2, Nq, 16, torch.float16, seed=Nq + Nk, q_std=2.0)
    _, k, v = make_qkv(2, 2, Nk, 16, torch.float16, seed=Nq * 7 + Nk)
    O, LSE = oracle.attention(q, k, v, 0.25, mask, (wl, wr))
    Ob, Lb, _ = brute_force(q, k, v, 0.25, mask, wl, wr)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, Lb, rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("mask,wl,wr", [("none", 0, 0), ("causal", 0, 0), ("window", 20, 0)])
def test_rectangular_equals_last_rows_of_square(mask, wl, wr):
    # Queries placed at the last Nq positions compute exactly the last Nq rows of the
    # square problem whose last rows are those queries.
    Nk, Nq, d = 120, 9, 32
    qs, k, v = make_qkv(1, 2, Nk, d, torch.bfloat16, seed=77)
    q = qs[:, :, Nk - Nq:].contiguous()
    Os, Ls = oracle.attention(qs, k, v, 0.2, mask, (wl, wr))
    O, L = oracle.attention(q, k, v, 0.2, mask, (wl, wr))
    rows = np.concatenate([bh * Nk + np.arange(Nk - Nq, Nk) for bh in range(2)])
    np.testing.assert_array_equal(O, Os[rows])
    np.testing.assert_array_equal(L, Ls[rows])


def test_single_query_uniform_scores_is_mean_of_all_values():
    _, k, v = make_qkv(1, 1, 300, 16, torch.float16, seed=8)
    q = torch.zeros(1, 1, 1, 16, dtype=torch.float16)
    O, L = oracle.attention(q, k, v, 0.5, "causal")  # the one query stands at the last key
    np.testing.assert_allclose(O[0], _f64(v)[0, 0].mean(axis=0), rtol=0, atol=1e-13)
    assert L[0] == pytest.approx(math.log(300), abs=1e-13)
