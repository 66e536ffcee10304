"""Pins of the fp64 gradient oracle (oracle.attention_bwd) against things other than
itself: torch.autograd on the naive three-matmul form, central finite differences of
an independent numpy forward, a two-key case worked by hand, and invariants that hold
for the gradient of any softmax attention."""

import math

import numpy as np
import pytest
import torch

import oracle
from tiled_attention_03_gb300.workloads import make_qkv


def visible(Nq, N, mask, window):
    """Boolean (Nq, N) visibility: query i stands at key position i + N - Nq."""
    pos = np.arange(Nq)[:, None] + (N - Nq)
    j = np.arange(N)[None, :]
    if mask == "causal":
        return j <= pos
    if mask == "window":
        return (j >= pos - window[0]) & (j <= pos + window[1])
    return np.ones((Nq, N), dtype=bool)


def autograd_grads(q, k, v, do, scale, mask, window):
    """torch float64 autograd of sum(O * dO) with O = softmax(scale QK^T + M) V."""
    B, H, Nq, d = q.shape
    Hk, N = k.shape[1], k.shape[2]
    Q = q.double().requires_grad_(True)
    K = k.double().requires_grad_(True)
    V = v.double().requires_grad_(True)
    Ke = K.repeat_interleave(H // Hk, dim=1)
    Ve = V.repeat_interleave(H // Hk, dim=1)
    s = scale * Q @ Ke.transpose(-1, -2)
    m = torch.from_numpy(visible(Nq, N, mask, window))
    s = s.masked_fill(~m, float("-inf"))
    o = torch.softmax(s, dim=-1) @ Ve
    (o * do.double()).sum().backward()
    return Q.grad.numpy(), K.grad.numpy(), V.grad.numpy()


def as_full(dQ, dK, dV, B, H, Hk):
    """Oracle outputs (all K/V heads, in order) reshaped to (B, H, ...), (B, Hk, ...)."""
    g = H // Hk
    return (dQ.reshape(B, Hk * g, *dQ.shape[2:]), dK.reshape(B, Hk, *dK.shape[1:]),
            dV.reshape(B, Hk, *dV.shape[1:]))


CASES = [
    # B, H, Hk, Nq, N, d, mask, window
    (1, 1, 1, 5, 5, 4, "none", (0, 0)),
    (1, 2, 2, 17, 17, 8, "causal", (0, 0)),
    (2, 2, 1, 9, 9, 4, "window", (3, 1)),
    (1, 4, 2, 3, 12, 8, "causal", (0, 0)),
    (1, 4, 2, 6, 20, 4, "window", (5, 0)),
    (1, 3, 3, 33, 33, 16, "none", (0, 0)),
]


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_matches_autograd(case, dtype):
    B, H, Hk, Nq, N, d, mask, window = case
    q, _, _ = make_qkv(B, H, Nq, d, dtype, seed=N + d)
    _, k, v = make_qkv(B, Hk, N, d, dtype, seed=3 * N + 1, H_kv=Hk)
    do = make_qkv(B, H, Nq, d, dtype, seed=7 * N + 2)[0]
    scale = 0.37
    dQ, dK, dV = as_full(*oracle.attention_bwd(q, k, v, do, scale, mask, window), B, H, Hk)
    gQ, gK, gV = autograd_grads(q, k, v, do, scale, mask, window)
    for got, ref in ((dQ, gQ), (dK, gK), (dV, gV)):
        assert np.abs(got - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max())


def numpy_loss(q, k, v, do, scale, vis):
    """sum(O * dO) of one head, by numpy in float64 (no torch, no oracle)."""
    s = scale * (q @ k.T)
    s = np.where(vis, s, -np.inf)
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s)
    p = e / e.sum(axis=1, keepdims=True)
    return float(((p @ v) * do).sum())


@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (2, 1))])
def test_matches_finite_differences(mask, window):
    Nq, N, d, scale = 7, 11, 6, 0.45
    q, _, _ = make_qkv(1, 1, Nq, d, torch.float16, seed=11)
    _, k, v = make_qkv(1, 1, N, d, torch.float16, seed=12)
    do = make_qkv(1, 1, Nq, d, torch.float16, seed=13)[0]
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, scale, mask, window)
    Q, K, V, DO = (t[0, 0].double().numpy() for t in (q, k, v, do))
    vis = visible(Nq, N, mask, window)
    h = 1e-6
    rng = np.random.default_rng(5)
    for name, X, G in (("Q", Q, dQ[0, 0]), ("K", K, dK[0]), ("V", V, dV[0])):
        for _ in range(12):
            r, c = int(rng.integers(X.shape[0])), int(rng.integers(d))
            Xp, Xm = X.copy(), X.copy()
            Xp[r, c] += h
            Xm[r, c] -= h
            args_p = {"Q": (Xp, K, V), "K": (Q, Xp, V), "V": (Q, K, Xp)}[name]
            args_m = {"Q": (Xm, K, V), "K": (Q, Xm, V), "V": (Q, K, Xm)}[name]
            fd = (numpy_loss(*args_p, DO, scale, vis) - numpy_loss(*args_m, DO, scale, vis)) / (2 * h)
            assert abs(fd - G[r, c]) <= 1e-6 * max(1.0, abs(fd)), (name, r, c, fd, G[r, c])


def test_two_keys_by_hand():
    """q = 1 (d = 1), keys 0 and 1, values 0 and 1, scale 1, dO = 1. With
    P = (1, e)/(1 + e): dV = P, dP = (0, 1), sum_j P_j dP_j = P_1, dS = (-P0 P1, P0 P1),
    dq = dS_1 * 1 = P0 P1, dk = dS * q. Causal with two queries at positions 0 and 1:
    row 0 sees key 0 only (P = (1, 0): no gradient to q_0 or k), row 1 as above."""
    f16 = torch.float16
    p0, p1 = 1 / (1 + math.e), math.e / (1 + math.e)
    k = torch.tensor([0.0, 1.0], dtype=f16).view(1, 1, 2, 1)
    v = torch.tensor([0.0, 1.0], dtype=f16).view(1, 1, 2, 1)
    q1 = torch.tensor([1.0], dtype=f16).view(1, 1, 1, 1)
    dQ, dK, dV = oracle.attention_bwd(q1, k, v, torch.ones_like(q1), 1.0)
    assert dQ[0, 0, 0, 0] == pytest.approx(p0 * p1, abs=1e-15)
    assert dK[0, :, 0] == pytest.approx([-p0 * p1, p0 * p1], abs=1e-15)
    assert dV[0, :, 0] == pytest.approx([p0, p1], abs=1e-15)
    q2 = torch.ones(1, 1, 2, 1, dtype=f16)
    dQ, dK, dV = oracle.attention_bwd(q2, k, v, torch.ones_like(q2), 1.0, "causal")
    assert dQ[0, 0, :, 0] == pytest.approx([0.0, p0 * p1], abs=1e-15)
    assert dK[0, :, 0] == pytest.approx([-p0 * p1, p0 * p1], abs=1e-15)
    assert dV[0, :, 0] == pytest.approx([1 + p0, p1], abs=1e-15)


@pytest.mark.parametrize("mask,window", [("none", (0, 0)), ("causal", (0, 0)), ("window", (40, 3))])
def test_invariants(mask, window):
    """Shifting every key by the same vector leaves each softmax row unchanged, so
    the keys' gradients sum to zero; P rows sum to one, so the values' gradients
    sum to the summed dO; the gradient is linear in dO (doubling is exact)."""
    B, H, Hk, N, d = 1, 4, 2, 150, 32
    q, k, v = make_qkv(B, H, N, d, torch.float16, seed=21, H_kv=Hk)
    do = make_qkv(B, H, N, d, torch.float16, seed=22)[0]
    dQ, dK, dV = oracle.attention_bwd(q, k, v, do, 0.2, mask, window)
    assert np.abs(dK.sum(axis=1)).max() <= 1e-11
    dsum = do.double().numpy().reshape(B * Hk, H // Hk * N, d).sum(axis=1)
    assert np.abs(dV.sum(axis=1) - dsum).max() <= 1e-11
    dQ2, dK2, dV2 = oracle.attention_bwd(q, k, v, do * 2, 0.2, mask, window)
    assert np.array_equal(dQ2, 2 * dQ) and np.array_equal(dK2, 2 * dK) and np.array_equal(dV2, 2 * dV)


def test_uniform_scores():
    """Q = 0: every visible key gets weight 1/n_i, so dK = 0 exactly and
    dV_j = sum over the queries i that see key j of dO_i / n_i."""
    Nq, N, d = 40, 64, 16
    _, k, v = make_qkv(1, 1, N, d, torch.bfloat16, seed=31)
    q = torch.zeros(1, 1, Nq, d, dtype=torch.bfloat16)
    do = make_qkv(1, 1, Nq, d, torch.bfloat16, seed=32)[0]
    for mask, window in (("none", (0, 0)), ("causal", (0, 0)), ("window", (9, 2))):
        _, dK, dV = oracle.attention_bwd(q, k, v, do, 0.25, mask, window)
        assert np.all(dK == 0.0)
        vis = visible(Nq, N, mask, window).astype(np.float64)
        w = vis / vis.sum(axis=1, keepdims=True)
        ref = w.T @ do[0, 0].double().numpy()
        assert np.abs(dV[0] - ref).max() <= 1e-12


def test_hidden_keys_get_no_gradient():
    """Keys no query can see (before every window) have dK = dV = 0 exactly."""
    Nq, N, d = 8, 60, 8
    q, _, _ = make_qkv(1, 2, Nq, d, torch.float16, seed=41)
    _, k, v = make_qkv(1, 1, N, d, torch.float16, seed=42, H_kv=1)
    do = make_qkv(1, 2, Nq, d, torch.float16, seed=43)[0]
    _, dK, dV = oracle.attention_bwd(q, k, v, do, 0.3, "window", (5, 0))
    first = N - Nq - 5  # the earliest key any query sees
    assert np.all(dK[0, :first] == 0) and np.all(dV[0, :first] == 0)
    assert np.abs(dV[0, first:]).min(axis=1).max() > 0


def test_rejects_bad_arguments():
    q, k, v = make_qkv(1, 3, 4, 4, torch.float16, seed=0, H_kv=2)
    with pytest.raises((ValueError, AssertionError)):
        oracle.attention_bwd(q, k, v, q, 0.5)
