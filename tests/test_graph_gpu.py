"""The entry points under CUDA-graph capture: a forward, a split-KV forward and a
backward captured once and replayed on new inputs (copied into the captured
buffers) give bit-identical results to direct calls. Each launch keeps the
scheduler-counter slot it took at capture; its last CTA resets the slot, so
sequential replays reuse it safely."""

import pytest
import torch

import tiled_attention_03_gb300 as fa
from tiled_attention_03_gb300.workloads import make_qkv

pytestmark = pytest.mark.gpu


def test_capture_and_replay_matches_direct_calls():
    dev = torch.device("cuda", 0)
    B, H, Hk, N, d, Nq = 2, 8, 2, 600, 128, 3
    q = torch.empty(B, H, N, d, dtype=torch.bfloat16, device=dev)
    k = torch.empty(B, Hk, N, d, dtype=torch.bfloat16, device=dev)
    v = torch.empty_like(k)
    do = torch.empty_like(q)
    qs = torch.empty(B, H, Nq, d, dtype=torch.bfloat16, device=dev)
    o, lse = torch.empty_like(q), torch.empty(B, H, N, device=dev)
    os_, lses = torch.empty_like(qs), torch.empty(B, H, Nq, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    splits = 3
    ws_split = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, splits), dtype=torch.uint8,
                           device=dev)
    ws_bwd = torch.empty(fa.fa_backward_workspace_bytes(B, H, N, d), dtype=torch.uint8, device=dev)

    def fill(seed):
        a, _, _ = make_qkv(B, H, N, d, torch.bfloat16, seed=seed)
        _, b, c = make_qkv(B, Hk, N, d, torch.bfloat16, seed=seed + 1, H_kv=Hk)
        g = make_qkv(B, H, N, d, torch.bfloat16, seed=seed + 2)[0]
        q.copy_(a); k.copy_(b); v.copy_(c); do.copy_(g); qs.copy_(a[:, :, -Nq:])

    def step(stream):
        fa.fa_forward_gqa(q, k, v, o, lse, 0.088, "causal", 0, 0, stream)
        fa.fa_forward_splitkv(qs, k, v, os_, lses, 0.088, "causal", 0, 0, splits, ws_split, stream)
        fa.fa_backward(q, k, v, o, do, lse, dq, dk, dv, 0.088, "causal", 0, 0, ws_bwd, stream)

    s = torch.cuda.Stream(dev)
    fill(40)
    with torch.cuda.stream(s):
        step(s)  # warm-up: kernel attributes and device state set outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        step(s)
    torch.cuda.synchronize()
    for seed in (50, 60, 70):
        fill(seed)
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_sync_status() == fa.FA_OK
        got = [t.clone() for t in (o, lse, os_, lses, dq, dk, dv)]
        with torch.cuda.stream(s):
            step(s)
        torch.cuda.synchronize()
        assert fa.fa_sync_status() == fa.FA_OK
        for g, r in zip(got, (o, lse, os_, lses, dq, dk, dv)):
            assert torch.equal(g, r)
