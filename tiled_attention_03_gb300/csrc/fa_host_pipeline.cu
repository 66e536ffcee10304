// fa_host_pipeline.cu -- fa_forward_host: the forward pass over host buffers,
// with the copies and the kernels overlapped chunk by chunk.
//
// A chunk is one batch entry and a range of K/V heads together with their query
// heads. In the B x H x N x d layout its slices of Q, K, V, O and LSE are
// contiguous, so each moves with a single copy. Chunk c's copy in (stream s_in),
// kernel (the caller's stream) and copy out (stream s_out) are ordered by
// events, so the copy in of chunk c+1, the kernel on chunk c and the copy out
// of chunk c-1 run at the same time. The host link, not the kernel, bounds this
// path: the copies in and out share it.
#include <cmath>
#include <mutex>

#include "fa.h"
#include "fa_host.h"

namespace {

constexpr int kMaxDevices = 64;
// Measured on B4 H32 N4096 d128 (GB300, 2 x ~200 GB/s host link): 16 MiB chunks
// 2.53 ms per step, 32 MiB 2.44, 64 MiB 2.34, 96 MiB 2.53. Smaller chunks leave
// the kernel of each too few work units for the SMs; larger ones lengthen the
// exposed first copy in and last copy out.
constexpr int64_t kDefaultChunkBytes = int64_t{64} << 20;
constexpr int64_t kElem = 2;  // bytes of one fp16 / bf16 element

// The library's own copy streams and events of one device, created on first use.
// One event per role suffices: a stream wait takes the event's latest record at
// the time of the wait, so re-recording it for the next chunk is safe. The lock
// keeps two callers from interleaving their records and waits.
struct Pipe {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_in = nullptr, ev_k = nullptr, ev_done = nullptr;
    std::mutex mu;
};
Pipe g_pipe[kMaxDevices];

Pipe *pipe_for(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    Pipe &p = g_pipe[dev];
    std::call_once(p.once, [&p] {
        cudaError_t e = cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking);
        if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking);
        cudaEvent_t *evs[] = {&p.ev_start, &p.ev_in, &p.ev_k, &p.ev_done};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) cudaGetLastError();
        p.err = e;
    });
    return &p;
}

// Sizes of the device copies and of one chunk's key-split scratch, and the
// number of K/V heads per chunk.
struct Plan {
    bool split = false;
    int64_t group = 1, step = 1;
    size_t q_bytes = 0, kv_bytes = 0, lse_bytes = 0;
    size_t off_k = 0, off_v = 0, off_o = 0, off_lse = 0, off_split = 0, split_bytes = 0;
    size_t total = 0;
};

// Shape checks of fa_forward_splitkv; false when invalid, with the status to return.
bool plan(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d,
          int64_t num_splits, int64_t chunk_bytes, Plan &pl, fa_status &why) {
    why = FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || H_kv < 1 || Nq < 1 || Nk < 1 || d < 1 || num_splits < 0) return false;
    if (H % H_kv != 0) return false;
    why = FA_ERR_UNSUPPORTED;
    if (d != 32 && d != 64 && d != 128 && d != 256) return false;
    if (Nq > (int64_t{1} << 29) || Nk > (int64_t{1} << 29) || B * H > (int64_t{1} << 31))
        return false;
    pl.split = num_splits > 0 || Nq != Nk;
    pl.group = H / H_kv;
    const int64_t per_kv_head = (pl.group * Nq + 2 * Nk) * d * kElem;
    const int64_t chunk = chunk_bytes > 0 ? chunk_bytes : kDefaultChunkBytes;
    pl.step = chunk / per_kv_head;
    if (pl.step < 1) pl.step = 1;
    if (pl.step > H_kv) pl.step = H_kv;
    using fa_host::align256;
    pl.q_bytes = static_cast<size_t>(B * H * Nq * d * kElem);
    pl.kv_bytes = static_cast<size_t>(B * H_kv * Nk * d * kElem);
    pl.lse_bytes = static_cast<size_t>(B * H * Nq) * sizeof(float);
    pl.off_k = align256(pl.q_bytes);
    pl.off_v = pl.off_k + align256(pl.kv_bytes);
    pl.off_o = pl.off_v + align256(pl.kv_bytes);
    pl.off_lse = pl.off_o + align256(pl.q_bytes);
    pl.off_split = pl.off_lse + align256(pl.lse_bytes);
    if (pl.split) {
        // fa_splitkv_default_splits never exceeds max(1, min(256, key tiles / 4))
        const int64_t tiles = (Nk + 127) / 128;
        int64_t s = num_splits;
        if (s == 0) {
            s = tiles / 4;
            if (s > 256) s = 256;
            if (s < 1) s = 1;
        }
        pl.split_bytes = fa_splitkv_workspace_bytes(1, pl.step * pl.group, Nq, d, s);
    }
    pl.total = pl.off_split + align256(pl.split_bytes);
    return true;
}

// Host memory: page-locked or pageable, not device or managed memory.
bool host_memory(const void *p) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return a.type == cudaMemoryTypeHost || a.type == cudaMemoryTypeUnregistered;
}

bool ok(cudaError_t e) {
    if (e == cudaSuccess) return true;
    cudaGetLastError();
    return false;
}

}  // namespace

extern "C" {

size_t fa_forward_host_workspace_bytes(int64_t B, int64_t H, int64_t H_kv, int64_t Nq,
                                       int64_t Nk, int64_t d, int64_t num_splits,
                                       int64_t chunk_bytes) {
    Plan pl;
    fa_status why;
    return plan(B, H, H_kv, Nq, Nk, d, num_splits, chunk_bytes, pl, why) ? pl.total : 0;
}

fa_status fa_forward_host(const void *Q, const void *K, const void *V, void *O, float *LSE,
                          int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d,
                          float scale, fa_mask_mode mask_mode, int64_t window_left,
                          int64_t window_right, fa_dtype dtype, int64_t num_splits,
                          int64_t chunk_bytes, void *workspace, size_t workspace_bytes,
                          void *stream) {
    // ---- every check before anything is enqueued
    if (!Q || !K || !V || !O || !LSE || !workspace) return FA_ERR_INVALID_ARG;
    Plan pl;
    fa_status why;
    if (!plan(B, H, H_kv, Nq, Nk, d, num_splits, chunk_bytes, pl, why)) return why;
    if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
    if (mask_mode != FA_MASK_NONE && mask_mode != FA_MASK_CAUSAL && mask_mode != FA_MASK_WINDOW)
        return FA_ERR_INVALID_ARG;
    if (mask_mode == FA_MASK_WINDOW && (window_left < 0 || window_right < 0))
        return FA_ERR_INVALID_ARG;
    if (mask_mode != FA_MASK_NONE && Nq > Nk) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (!fa_host::aligned4(LSE)) return FA_ERR_INVALID_ARG;
    const void *host[] = {Q, K, V, O, LSE};
    for (const void *p : host)
        if (!host_memory(p)) return FA_ERR_INVALID_ARG;
    const void *ins[] = {Q, K, V};
    const size_t in_len[] = {pl.q_bytes, pl.kv_bytes, pl.kv_bytes};
    for (int i = 0; i < 3; ++i)
        if (fa_host::overlaps(O, pl.q_bytes, ins[i], in_len[i]) ||
            fa_host::overlaps(LSE, pl.lse_bytes, ins[i], in_len[i]))
            return FA_ERR_INVALID_ARG;
    if (fa_host::overlaps(O, pl.q_bytes, LSE, pl.lse_bytes)) return FA_ERR_INVALID_ARG;
    int dev = 0;
    if (!ok(cudaGetDevice(&dev))) return FA_ERR_CUDA;
    if (!fa_host::aligned32(workspace) || !fa_host::on_device(workspace, dev) ||
        workspace_bytes < pl.total)
        return FA_ERR_INVALID_ARG;
    Pipe *pp = pipe_for(dev);
    if (pp == nullptr) return FA_ERR_UNSUPPORTED;
    if (pp->err != cudaSuccess) return FA_ERR_CUDA;
    Pipe &P = *pp;

    uint8_t *w = static_cast<uint8_t *>(workspace);
    uint8_t *dQ = w, *dK = w + pl.off_k, *dV = w + pl.off_v, *dO = w + pl.off_o;
    float *dL = reinterpret_cast<float *>(w + pl.off_lse);
    void *dS = pl.split_bytes > 0 ? w + pl.off_split : nullptr;
    const uint8_t *hQ = static_cast<const uint8_t *>(Q), *hK = static_cast<const uint8_t *>(K),
                  *hV = static_cast<const uint8_t *>(V);
    uint8_t *hO = static_cast<uint8_t *>(O);
    const cudaStream_t st = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(P.mu);
    // The staging buffers are free once the caller's earlier work on `stream`
    // (including an earlier call's kernels and, through its final wait, copies) is done.
    if (!ok(cudaEventRecord(P.ev_start, st)) || !ok(cudaStreamWaitEvent(P.s_in, P.ev_start, 0)))
        return FA_ERR_CUDA;
    fa_status status = FA_OK;
    for (int64_t b = 0; b < B && status == FA_OK; ++b) {
        for (int64_t hk0 = 0; hk0 < H_kv && status == FA_OK; hk0 += pl.step) {
            const int64_t nh = hk0 + pl.step <= H_kv ? pl.step : H_kv - hk0;
            const int64_t qh = nh * pl.group;
            const size_t q_off = static_cast<size_t>((b * H + hk0 * pl.group) * Nq * d * kElem);
            const size_t q_len = static_cast<size_t>(qh * Nq * d * kElem);
            const size_t k_off = static_cast<size_t>((b * H_kv + hk0) * Nk * d * kElem);
            const size_t k_len = static_cast<size_t>(nh * Nk * d * kElem);
            const size_t l_off = static_cast<size_t>((b * H + hk0 * pl.group) * Nq);
            const size_t l_len = static_cast<size_t>(qh * Nq) * sizeof(float);
            if (!ok(cudaMemcpyAsync(dQ + q_off, hQ + q_off, q_len, cudaMemcpyHostToDevice, P.s_in)) ||
                !ok(cudaMemcpyAsync(dK + k_off, hK + k_off, k_len, cudaMemcpyHostToDevice, P.s_in)) ||
                !ok(cudaMemcpyAsync(dV + k_off, hV + k_off, k_len, cudaMemcpyHostToDevice, P.s_in)) ||
                !ok(cudaEventRecord(P.ev_in, P.s_in)) || !ok(cudaStreamWaitEvent(st, P.ev_in, 0))) {
                status = FA_ERR_CUDA;
                break;
            }
            if (pl.split) {
                const int64_t s = num_splits > 0 ? num_splits
                                                 : fa_splitkv_default_splits(1, qh, nh, Nq, Nk);
                status = fa_forward_splitkv(dQ + q_off, dK + k_off, dV + k_off, dO + q_off,
                                            dL + l_off, 1, qh, nh, Nq, Nk, d, scale, mask_mode,
                                            window_left, window_right, dtype, s, dS,
                                            pl.split_bytes, stream);
            } else {
                status = fa_forward_gqa(dQ + q_off, dK + k_off, dV + k_off, dO + q_off, dL + l_off,
                                        1, qh, nh, Nq, d, scale, mask_mode, window_left,
                                        window_right, dtype, stream);
            }
            if (status != FA_OK) break;
            if (!ok(cudaEventRecord(P.ev_k, st)) || !ok(cudaStreamWaitEvent(P.s_out, P.ev_k, 0)) ||
                !ok(cudaMemcpyAsync(hO + q_off, dO + q_off, q_len, cudaMemcpyDeviceToHost, P.s_out)) ||
                !ok(cudaMemcpyAsync(LSE + l_off, dL + l_off, l_len, cudaMemcpyDeviceToHost, P.s_out)))
                status = FA_ERR_CUDA;
        }
    }
    // `stream` waits for every copy out (also after a failure, so that the
    // caller's next use of the workspace stays ordered after them).
    if (!ok(cudaEventRecord(P.ev_done, P.s_out)) || !ok(cudaStreamWaitEvent(st, P.ev_done, 0)))
        return FA_ERR_CUDA;
    return status;
}

}  // extern "C"
