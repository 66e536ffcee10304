// fa_bwd_api.cu -- the backward entry points of include/fa.h: argument checks,
// workspace layout, TMA maps and the three launches (prep, dK/dV, dQ).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"
#include "fa_bwd256_kernel.cuh"
#include "fa_bwd_kernel.cuh"
#include "fa_host.h"

namespace {

using fa_host::align256;

constexpr int kMaxDevices = 64;

struct BwdDeviceState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
};
BwdDeviceState g_bwd_dev[kMaxDevices];

// Opt in to the kernel's shared memory and check that the launch's registers
// cover the setmaxnreg split (a split above them would make setmaxnreg.inc wait
// forever).
template <typename Kernel>
cudaError_t configure_one(Kernel k, int smem) {
    cudaFuncAttributes attr{};
    cudaError_t e = cudaFuncGetAttributes(&attr, k);
    if (e != cudaSuccess) return e;
    if (attr.numRegs * fa::bwd::kThreads < fa::bwd::kRegsNeeded) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

template <int D, bool BF16>
cudaError_t configure_bwd() {
    using namespace fa::bwd;
    cudaError_t e = configure_one(fa_bwd_dkdv_kernel<D, BF16, false>, KvSmem<D>::kAlloc);
    if (e == cudaSuccess) e = configure_one(fa_bwd_dq_kernel<D, BF16, false>, QSmem<D>::kAlloc);
    if (e == cudaSuccess) e = configure_one(fa_bwd_dkdv_kernel<D, BF16, true>, KvSmem<D>::kAlloc);
    if (e == cudaSuccess) e = configure_one(fa_bwd_dq_kernel<D, BF16, true>, QSmem<D>::kAlloc);
    return e;
}

// d = 256: the three passes of fa_bwd256_kernel.cuh (192 threads, no setmaxnreg).
template <bool BF16, bool VARLEN>
cudaError_t configure_bwd256() {
    using namespace fa::bwd256;
    cudaError_t e = cudaFuncSetAttribute(fa_bwd256_kernel<kPassDQ, BF16, VARLEN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Layout<kPassDQ>::kAlloc);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fa_bwd256_kernel<kPassDK, BF16, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<kPassDK>::kAlloc);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(fa_bwd256_kernel<kPassDV, BF16, VARLEN>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<kPassDV>::kAlloc);
    return e;
}

cudaError_t bwd_device_init(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    BwdDeviceState &s = g_bwd_dev[dev];
    std::call_once(s.once, [&s] {
        cudaError_t e = configure_bwd<32, false>();
        if (e == cudaSuccess) e = configure_bwd<32, true>();
        if (e == cudaSuccess) e = configure_bwd<64, false>();
        if (e == cudaSuccess) e = configure_bwd<64, true>();
        if (e == cudaSuccess) e = configure_bwd<128, false>();
        if (e == cudaSuccess) e = configure_bwd<128, true>();
        if (e == cudaSuccess) e = configure_bwd256<false, false>();
        if (e == cudaSuccess) e = configure_bwd256<true, false>();
        if (e == cudaSuccess) e = configure_bwd256<false, true>();
        if (e == cudaSuccess) e = configure_bwd256<true, true>();
        s.err = e;
    });
    return s.err;
}

int64_t padded_rows(int64_t N) { return (N + fa::bwd::kTile - 1) / fa::bwd::kTile * fa::bwd::kTile; }

// Workspace: the row terms L = LSE log2(e) and D = rowsum(dO O), fp32, rows padded
// to 128 per head.
struct BwdWorkspace {
    size_t l, d, total;
};
BwdWorkspace bwd_layout(int64_t B, int64_t H, int64_t N) {
    const size_t rows = static_cast<size_t>(B) * H * padded_rows(N);
    BwdWorkspace w;
    w.l = 0;
    w.d = align256(rows * sizeof(float));
    w.total = w.d + align256(rows * sizeof(float));
    return w;
}

template <int D, bool BF16, bool VARLEN>
cudaError_t launch_main(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                        const CUtensorMap &mdo, const fa::bwd::BwdParams &pkv,
                        const fa::bwd::BwdParams &pq, int sms, cudaStream_t st);

template <int D, bool BF16>
cudaError_t launch_bwd(const fa::bwd::PrepParams &pp, const CUtensorMap &mq, const CUtensorMap &mk,
                       const CUtensorMap &mv, const CUtensorMap &mdo, const fa::bwd::BwdParams &pkv,
                       const fa::bwd::BwdParams &pq, int sms, cudaStream_t st) {
    using namespace fa::bwd;
    const int64_t prep_rows = static_cast<int64_t>(pp.BH) * pp.Npad;
    fa_bwd_prep_kernel<D, BF16><<<static_cast<unsigned>((prep_rows + kPrepWarps - 1) / kPrepWarps),
                                  kPrepWarps * 32, 0, st>>>(pp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_main<D, BF16, false>(mq, mk, mv, mdo, pkv, pq, sms, st);
}

template <int D, bool BF16, bool VARLEN>
cudaError_t launch_main(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                        const CUtensorMap &mdo, const fa::bwd::BwdParams &pkv,
                        const fa::bwd::BwdParams &pq, int sms, cudaStream_t st) {
    using namespace fa::bwd;
    // Persistent grids: one CTA per SM (each holds all of its SM's tensor memory).
    fa_bwd_dkdv_kernel<D, BF16, VARLEN><<<static_cast<unsigned>(pkv.n_units < sms ? pkv.n_units : sms),
                                          kThreads, KvSmem<D>::kAlloc, st>>>(mq, mk, mv, mdo, pkv);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    fa_bwd_dq_kernel<D, BF16, VARLEN><<<static_cast<unsigned>(pq.n_units < sms ? pq.n_units : sms),
                                        kThreads, QSmem<D>::kAlloc, st>>>(mq, mk, mv, mdo, pq);
    return cudaGetLastError();
}

// d = 256: the dV, dK and dQ passes (fa_bwd256_kernel.cuh) after the row-term
// prep. Maps: q128 / do128 and k128 / v128 are the 128-row views of the resident
// tiles, q64 / do64 and k64 / v64 the 64-row views of the streamed ones.
template <bool BF16, bool VARLEN>
cudaError_t launch_bwd256_passes(const CUtensorMap &q128, const CUtensorMap &do128,
                                 const CUtensorMap &k128, const CUtensorMap &v128,
                                 const CUtensorMap &q64, const CUtensorMap &do64,
                                 const CUtensorMap &k64, const CUtensorMap &v64,
                                 const fa::bwd256::Params &pdq, const fa::bwd256::Params &pdk,
                                 const fa::bwd256::Params &pdv, int sms, cudaStream_t st) {
    using namespace fa::bwd256;
    cudaError_t e;
    auto grid = [sms](const Params &q) { return static_cast<unsigned>(q.n_units < sms ? q.n_units : sms); };
    fa_bwd256_kernel<kPassDV, BF16, VARLEN>
        <<<grid(pdv), kThreads, Layout<kPassDV>::kAlloc, st>>>(k128, k128, q64, do64, pdv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fa_bwd256_kernel<kPassDK, BF16, VARLEN>
        <<<grid(pdk), kThreads, Layout<kPassDK>::kAlloc, st>>>(k128, v128, q64, do64, pdk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fa_bwd256_kernel<kPassDQ, BF16, VARLEN>
        <<<grid(pdq), kThreads, Layout<kPassDQ>::kAlloc, st>>>(q128, do128, k64, v64, pdq);
    return cudaGetLastError();
}

template <bool BF16>
cudaError_t launch_bwd256(const fa::bwd::PrepParams &pp, const CUtensorMap &q128,
                          const CUtensorMap &do128, const CUtensorMap &k128, const CUtensorMap &v128,
                          const CUtensorMap &q64, const CUtensorMap &do64, const CUtensorMap &k64,
                          const CUtensorMap &v64, const fa::bwd256::Params &pdq,
                          const fa::bwd256::Params &pdk, const fa::bwd256::Params &pdv, int sms,
                          cudaStream_t st) {
    const int64_t prep_rows = static_cast<int64_t>(pp.BH) * pp.Npad;
    fa::bwd::fa_bwd_prep_kernel<256, BF16>
        <<<static_cast<unsigned>((prep_rows + fa::bwd::kPrepWarps - 1) / fa::bwd::kPrepWarps),
           fa::bwd::kPrepWarps * 32, 0, st>>>(pp);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_bwd256_passes<BF16, false>(q128, do128, k128, v128, q64, do64, k64, v64, pdq, pdk,
                                             pdv, sms, st);
}

// Variable-length batches at d = 256: padded row offsets, the row terms, then the
// three passes over token-major maps.
template <bool BF16>
cudaError_t launch_bwd256_varlen(const fa::bwd::PrepVarlenParams &pp, const CUtensorMap &q128,
                                 const CUtensorMap &do128, const CUtensorMap &k128,
                                 const CUtensorMap &v128, const CUtensorMap &q64,
                                 const CUtensorMap &do64, const CUtensorMap &k64,
                                 const CUtensorMap &v64, const fa::bwd256::Params &pdq,
                                 const fa::bwd256::Params &pdk, const fa::bwd256::Params &pdv,
                                 int sms, cudaStream_t st) {
    using namespace fa::bwd;
    fa_bwd_cu_pad_kernel<<<1, 32, 0, st>>>(pp.cu_q, pp.B, pp.total_q, const_cast<int *>(pp.cu_pad));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(pp.H) * pp.vstride;
    fa_bwd_prep_varlen_kernel<256, BF16><<<static_cast<unsigned>((rows + kPrepWarps - 1) / kPrepWarps),
                                           kPrepWarps * 32, 0, st>>>(pp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_bwd256_passes<BF16, true>(q128, do128, k128, v128, q64, do64, k64, v64, pdq, pdk,
                                            pdv, sms, st);
}

template <int D, bool BF16>
cudaError_t launch_bwd_varlen(const fa::bwd::PrepVarlenParams &pp, const CUtensorMap &mq,
                              const CUtensorMap &mk, const CUtensorMap &mv, const CUtensorMap &mdo,
                              const fa::bwd::BwdParams &pkv, const fa::bwd::BwdParams &pq, int sms,
                              cudaStream_t st) {
    using namespace fa::bwd;
    fa_bwd_cu_pad_kernel<<<1, 32, 0, st>>>(pp.cu_q, pp.B, pp.total_q, const_cast<int *>(pp.cu_pad));
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t rows = static_cast<int64_t>(pp.H) * pp.vstride;
    fa_bwd_prep_varlen_kernel<D, BF16><<<static_cast<unsigned>((rows + kPrepWarps - 1) / kPrepWarps),
                                         kPrepWarps * 32, 0, st>>>(pp);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_main<D, BF16, true>(mq, mk, mv, mdo, pkv, pq, sms, st);
}

}  // namespace

extern "C" {

size_t fa_backward_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d) {
    if (B < 1 || H < 1 || N < 1 || d < 1) return 0;
    return bwd_layout(B, H, N).total;
}

fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                      const float *LSE, void *dQ, void *dK, void *dV, int64_t B, int64_t H,
                      int64_t H_kv, int64_t N, int64_t d, float scale, fa_mask_mode mask_mode,
                      int64_t window_left, int64_t window_right, fa_dtype dtype, void *workspace,
                      size_t workspace_bytes, void *stream) {
    using fa_host::aligned16;
    using fa_host::on_device;
    using fa_host::overlaps;
    // ---- host-side checks: nothing is enqueued on failure
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace)
        return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
    if (mask_mode != FA_MASK_NONE && mask_mode != FA_MASK_CAUSAL && mask_mode != FA_MASK_WINDOW)
        return FA_ERR_INVALID_ARG;
    if (mask_mode == FA_MASK_WINDOW && (window_left < 0 || window_right < 0))
        return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    const void *ptrs[] = {Q, K, V, O, dO};
    for (const void *q : ptrs)
        if (!aligned16(q)) return FA_ERR_INVALID_ARG;
    // the gradients and the workspace take 32-byte vector stores
    const void *stored[] = {dQ, dK, dV, workspace};
    for (const void *q : stored)
        if (!fa_host::aligned32(q)) return FA_ERR_INVALID_ARG;
    if (!fa_host::aligned4(LSE)) return FA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (N > (int64_t{1} << 29) || B * H > (int64_t{1} << 31)) return FA_ERR_UNSUPPORTED;
    const int64_t BH = B * H, BHkv = B * H_kv;
    const int64_t Npad = padded_rows(N);
    const int64_t n_blk = Npad / fa::bwd::kTile;
    if (BH * Npad > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    const BwdWorkspace wl = bwd_layout(B, H, N);
    if (workspace_bytes < wl.total) return FA_ERR_INVALID_ARG;
    const size_t qb = static_cast<size_t>(BH) * N * d * 2;     // Q, O, dO, dQ
    const size_t kb = static_cast<size_t>(BHkv) * N * d * 2;   // K, V, dK, dV
    const size_t lb = static_cast<size_t>(BH) * N * sizeof(float);
    // Outputs and workspace overlap no input and no other output.
    const void *outs[] = {dQ, dK, dV, workspace};
    const size_t out_n[] = {qb, kb, kb, wl.total};
    const void *ins[] = {Q, K, V, O, dO, LSE};
    const size_t in_n[] = {qb, kb, kb, qb, qb, lb};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_n[a], ins[b], in_n[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_n[a], outs[b], out_n[b])) return FA_ERR_INVALID_ARG;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    const fa_host::DeviceInfo info = fa_host::device_info(dev);
    if (info.err != cudaSuccess) return FA_ERR_CUDA;
    if (!(info.cc_major == 10 && info.cc_minor == 3)) return FA_ERR_UNSUPPORTED;
    if (bwd_device_init(dev) != cudaSuccess) return FA_ERR_CUDA;
    for (const void *q : ptrs)
        if (!on_device(q, dev)) return FA_ERR_INVALID_ARG;

    const bool bf16 = dtype == FA_DTYPE_BF16;
    CUtensorMap mq, mk, mv, mdo;
    if (!fa_host::make_map(&mq, Q, bf16, BH, N, d) || !fa_host::make_map(&mk, K, bf16, BHkv, N, d) ||
        !fa_host::make_map(&mv, V, bf16, BHkv, N, d) || !fa_host::make_map(&mdo, dO, bf16, BH, N, d))
        return FA_ERR_CUDA;
    CUtensorMap mq64, mk64, mv64, mdo64;  // d = 256: 64-row views of the streamed tiles
    if (d == 256 &&
        (!fa_host::make_map(&mq64, Q, bf16, BH, N, d, 64) ||
         !fa_host::make_map(&mk64, K, bf16, BHkv, N, d, 64) ||
         !fa_host::make_map(&mv64, V, bf16, BHkv, N, d, 64) ||
         !fa_host::make_map(&mdo64, dO, bf16, BH, N, d, 64)))
        return FA_ERR_CUDA;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    fa::bwd::PrepParams pp{};
    pp.O = O;
    pp.dO = dO;
    pp.LSE = LSE;
    pp.Lw = reinterpret_cast<float *>(ws + wl.l);
    pp.Dw = reinterpret_cast<float *>(ws + wl.d);
    pp.BH = static_cast<int>(BH);
    pp.N = static_cast<int>(N);
    pp.Npad = static_cast<int>(Npad);

    fa::bwd::BwdParams p{};
    p.dQ = dQ;
    p.dK = dK;
    p.dV = dV;
    p.Lw = pp.Lw;
    p.Dw = pp.Dw;
    p.N = static_cast<int>(N);
    p.Npad = static_cast<int>(Npad);
    p.H = static_cast<int>(H);
    p.Hkv = static_cast<int>(H_kv);
    p.group = static_cast<int>(H / H_kv);
    p.BH = static_cast<int>(BH);
    p.BHkv = static_cast<int>(BHkv);
    p.n_blk = static_cast<int>(n_blk);
    // visibility i - wl <= j <= i + wr, with N standing in for "unbounded"
    int64_t wlv = N, wrv = N;
    if (mask_mode == FA_MASK_CAUSAL) wrv = 0;
    if (mask_mode == FA_MASK_WINDOW) {
        wlv = window_left < N ? window_left : N;
        wrv = window_right < N ? window_right : N;
    }
    p.wl = static_cast<int>(wlv);
    p.wr = static_cast<int>(wrv);
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.wait_budget_ns = fa_host::wait_budget();
    p.status = info.status;
    p.fault_unit = -1;
    fa::bwd::BwdParams pkv = p, pq = p;
    pkv.fault_unit = fa_host::take_fault_position();
    pkv.n_units = static_cast<int>(BHkv * n_blk);  // (K/V head, key block)
    pq.n_units = static_cast<int>(BH * n_blk);     // (query head, query block)
    pkv.sched = fa_host::next_sched_slot(info.sched);
    pq.sched = fa_host::next_sched_slot(info.sched);
    pq.heavy_first = wrv < N ? 1 : 0;              // later blocks see more keys

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (d == 256) {
        fa::bwd256::Params b{};
        b.Lw = pp.Lw;
        b.Dw = pp.Dw;
        b.N = p.N;
        b.Npad = p.Npad;
        b.H = p.H;
        b.Hkv = p.Hkv;
        b.group = p.group;
        b.n_blk = p.n_blk;
        b.wl = p.wl;
        b.wr = p.wr;
        b.scale_log2 = p.scale_log2;
        b.wait_budget_ns = p.wait_budget_ns;
        b.status = p.status;
        b.fault_unit = -1;
        fa::bwd256::Params pdq = b, pdk = b, pdv = b;
        pdq.out = dQ;
        pdq.res0 = Q;
        pdk.res0 = K;
        pdv.res0 = K;
        pdq.out_scale = scale;
        pdq.n_units = static_cast<int>(BH * n_blk);      // (query head, 128-query block)
        pdk.out = dK;
        pdk.out_scale = scale;
        pdk.n_units = static_cast<int>(BHkv * n_blk);    // (K/V head, 128-key block)
        pdv.out = dV;
        pdv.out_scale = 1.f;
        pdv.n_units = pdk.n_units;
        pdv.fault_unit = pkv.fault_unit;                 // the hook applies to the first pass
        pdq.sched = pq.sched;
        pdk.sched = pkv.sched;
        pdv.sched = fa_host::next_sched_slot(info.sched);
        const cudaError_t e =
            bf16 ? launch_bwd256<true>(pp, mq, mdo, mk, mv, mq64, mdo64, mk64, mv64, pdq, pdk, pdv,
                                       info.sm_count, st)
                 : launch_bwd256<false>(pp, mq, mdo, mk, mv, mq64, mdo64, mk64, mv64, pdq, pdk, pdv,
                                        info.sm_count, st);
        if (e != cudaSuccess) return FA_ERR_CUDA;
        fa_host::count_launches(4);
        return FA_OK;
    }
    cudaError_t e;
    if (d == 32)
        e = bf16 ? launch_bwd<32, true>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st)
                 : launch_bwd<32, false>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st);
    else if (d == 64)
        e = bf16 ? launch_bwd<64, true>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st)
                 : launch_bwd<64, false>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st);
    else
        e = bf16 ? launch_bwd<128, true>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st)
                 : launch_bwd<128, false>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    fa_host::count_launches(3);
    return FA_OK;
}

// Workspace of the variable-length backward: padded sequence starts (B + 1), then
// L and D as H rows of vstride floats each.
struct VarlenBwdWorkspace {
    size_t pad, l, d, total;
    int64_t vstride;
};
VarlenBwdWorkspace varlen_bwd_layout(int64_t B, int64_t H, int64_t total_q) {
    VarlenBwdWorkspace w;
    w.vstride = (total_q + fa::bwd::kTile * B + fa::bwd::kTile - 1) / fa::bwd::kTile * fa::bwd::kTile;
    const size_t vec = static_cast<size_t>(H) * w.vstride * sizeof(float);
    w.pad = 0;
    w.l = align256(static_cast<size_t>(B + 1) * sizeof(int32_t));
    w.d = w.l + align256(vec);
    w.total = w.d + align256(vec);
    return w;
}

size_t fa_backward_varlen_workspace_bytes(int64_t B, int64_t H, int64_t total_q) {
    if (B < 1 || H < 1 || total_q < 0) return 0;
    return varlen_bwd_layout(B, H, total_q).total;
}

fa_status fa_backward_varlen(const void *Q, const void *K, const void *V, const void *O,
                             const void *dO, const float *LSE, const int32_t *cu_seqlens_q,
                             const int32_t *cu_seqlens_k, void *dQ, void *dK, void *dV, int64_t B,
                             int64_t H, int64_t H_kv, int64_t total_q, int64_t total_k,
                             int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d, float scale,
                             fa_mask_mode mask_mode, int64_t window_left, int64_t window_right,
                             fa_dtype dtype, void *workspace, size_t workspace_bytes,
                             void *stream) {
    using fa_host::aligned16;
    using fa_host::on_device;
    using fa_host::overlaps;
    // ---- host-side checks: nothing is enqueued on failure
    if (B < 1 || H < 1 || d < 1 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 ||
        max_seqlen_k < 0)
        return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (dtype != FA_DTYPE_FP16 && dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
    if (mask_mode != FA_MASK_NONE && mask_mode != FA_MASK_CAUSAL && mask_mode != FA_MASK_WINDOW)
        return FA_ERR_INVALID_ARG;
    if (mask_mode == FA_MASK_WINDOW && (window_left < 0 || window_right < 0))
        return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (total_q > (int64_t{1} << 29) || total_k > (int64_t{1} << 29) || max_seqlen_q > total_q ||
        max_seqlen_k > total_k || B > (int64_t{1} << 20))
        return FA_ERR_UNSUPPORTED;
    if (total_q == 0 && total_k == 0) return FA_OK;  // nothing to read or write
    const void *ptrs[] = {Q, K, V, O, dO};
    for (const void *q : ptrs)
        if (q == nullptr || !aligned16(q)) return FA_ERR_INVALID_ARG;
    // the gradients and the workspace take 32-byte vector stores
    const void *stored[] = {dQ, dK, dV, workspace};
    for (const void *q : stored)
        if (q == nullptr || !fa_host::aligned32(q)) return FA_ERR_INVALID_ARG;
    if (LSE == nullptr || !fa_host::aligned4(LSE)) return FA_ERR_INVALID_ARG;
    if (!cu_seqlens_q || !cu_seqlens_k || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
        return FA_ERR_INVALID_ARG;
    const VarlenBwdWorkspace wl = varlen_bwd_layout(B, H, total_q);
    if (workspace_bytes < wl.total) return FA_ERR_INVALID_ARG;
    if (H * wl.vstride > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    const size_t qb = static_cast<size_t>(total_q) * H * d * 2;
    const size_t kb = static_cast<size_t>(total_k) * H_kv * d * 2;
    const size_t lb = static_cast<size_t>(total_q) * H * sizeof(float);
    const size_t cb = static_cast<size_t>(B + 1) * sizeof(int32_t);
    const void *outs[] = {dQ, dK, dV, workspace};
    const size_t out_n[] = {qb, kb, kb, wl.total};
    const void *ins[] = {Q, K, V, O, dO, LSE, cu_seqlens_q, cu_seqlens_k};
    const size_t in_n[] = {qb, kb, kb, qb, qb, lb, cb, cb};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 8; ++b)
            if (overlaps(outs[a], out_n[a], ins[b], in_n[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_n[a], outs[b], out_n[b])) return FA_ERR_INVALID_ARG;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    const fa_host::DeviceInfo info = fa_host::device_info(dev);
    if (info.err != cudaSuccess) return FA_ERR_CUDA;
    if (!(info.cc_major == 10 && info.cc_minor == 3)) return FA_ERR_UNSUPPORTED;
    if (bwd_device_init(dev) != cudaSuccess) return FA_ERR_CUDA;
    for (const void *q : ptrs)
        if (!on_device(q, dev)) return FA_ERR_INVALID_ARG;
    if (!on_device(cu_seqlens_q, dev) || !on_device(cu_seqlens_k, dev)) return FA_ERR_INVALID_ARG;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // Gradients no query reaches (keys of sequences without queries, keys outside
    // every window, queries without keys) are zero: the kernels skip such blocks.
    if ((qb && cudaMemsetAsync(dQ, 0, qb, st) != cudaSuccess) ||
        (kb && cudaMemsetAsync(dK, 0, kb, st) != cudaSuccess) ||
        (kb && cudaMemsetAsync(dV, 0, kb, st) != cudaSuccess))
        return FA_ERR_CUDA;
    if (total_q == 0 || total_k == 0 || max_seqlen_q == 0 || max_seqlen_k == 0) return FA_OK;

    const bool bf16 = dtype == FA_DTYPE_BF16;
    CUtensorMap mq, mk, mv, mdo;
    if (!fa_host::make_map_tokens(&mq, Q, bf16, total_q, H, d) ||
        !fa_host::make_map_tokens(&mk, K, bf16, total_k, H_kv, d) ||
        !fa_host::make_map_tokens(&mv, V, bf16, total_k, H_kv, d) ||
        !fa_host::make_map_tokens(&mdo, dO, bf16, total_q, H, d))
        return FA_ERR_CUDA;

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    fa::bwd::PrepVarlenParams pp{};
    pp.O = O;
    pp.dO = dO;
    pp.LSE = LSE;
    pp.cu_q = cu_seqlens_q;
    pp.cu_pad = reinterpret_cast<int *>(ws + wl.pad);
    pp.Lw = reinterpret_cast<float *>(ws + wl.l);
    pp.Dw = reinterpret_cast<float *>(ws + wl.d);
    pp.B = static_cast<int>(B);
    pp.H = static_cast<int>(H);
    pp.total_q = static_cast<int>(total_q);
    pp.vstride = static_cast<int>(wl.vstride);

    fa::bwd::BwdParams p{};
    p.dQ = dQ;
    p.dK = dK;
    p.dV = dV;
    p.Lw = pp.Lw;
    p.Dw = pp.Dw;
    p.N = static_cast<int>(max_seqlen_q > max_seqlen_k ? max_seqlen_q : max_seqlen_k);
    p.H = static_cast<int>(H);
    p.Hkv = static_cast<int>(H_kv);
    p.group = static_cast<int>(H / H_kv);
    p.BH = static_cast<int>(B * H);
    p.BHkv = static_cast<int>(B * H_kv);
    const int64_t all = total_q + total_k;  // wider than any sequence's offsets
    int64_t wlv = all, wrv = all;
    if (mask_mode == FA_MASK_CAUSAL) wrv = 0;
    if (mask_mode == FA_MASK_WINDOW) {
        wlv = window_left < all ? window_left : all;
        wrv = window_right < all ? window_right : all;
    }
    p.wl = static_cast<int>(wlv);
    p.wr = static_cast<int>(wrv);
    p.scale = scale;
    p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    p.wait_budget_ns = fa_host::wait_budget();
    p.status = info.status;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.cu_pad = pp.cu_pad;
    p.total_q = static_cast<int>(total_q);
    p.total_k = static_cast<int>(total_k);
    p.vstride = static_cast<int>(wl.vstride);
    p.fault_unit = -1;
    fa::bwd::BwdParams pkv = p, pq = p;
    pkv.fault_unit = fa_host::take_fault_position();
    const int64_t nb_k = (max_seqlen_k + fa::bwd::kTile - 1) / fa::bwd::kTile;
    const int64_t nb_q = (max_seqlen_q + fa::bwd::kTile - 1) / fa::bwd::kTile;
    if (B * H_kv * nb_k > 0x7fffffffLL || B * H * nb_q > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    pkv.n_blk = static_cast<int>(nb_k);
    pkv.n_units = static_cast<int>(B * H_kv * nb_k);
    pq.n_blk = static_cast<int>(nb_q);
    pq.n_units = static_cast<int>(B * H * nb_q);
    pq.heavy_first = wrv < all ? 1 : 0;
    pkv.sched = fa_host::next_sched_slot(info.sched);
    pq.sched = fa_host::next_sched_slot(info.sched);

    if (d == 256) {
        CUtensorMap mq64, mk64, mv64, mdo64;
        if (!fa_host::make_map_tokens(&mq64, Q, bf16, total_q, H, d, 64) ||
            !fa_host::make_map_tokens(&mk64, K, bf16, total_k, H_kv, d, 64) ||
            !fa_host::make_map_tokens(&mv64, V, bf16, total_k, H_kv, d, 64) ||
            !fa_host::make_map_tokens(&mdo64, dO, bf16, total_q, H, d, 64))
            return FA_ERR_CUDA;
        fa::bwd256::Params b{};
        b.Lw = pp.Lw;
        b.Dw = pp.Dw;
        b.N = p.N;
        b.H = p.H;
        b.Hkv = p.Hkv;
        b.group = p.group;
        b.wl = p.wl;
        b.wr = p.wr;
        b.scale_log2 = p.scale_log2;
        b.wait_budget_ns = p.wait_budget_ns;
        b.status = p.status;
        b.fault_unit = -1;
        b.cu_q = cu_seqlens_q;
        b.cu_k = cu_seqlens_k;
        b.cu_pad = pp.cu_pad;
        b.total_q = p.total_q;
        b.total_k = p.total_k;
        b.vstride = p.vstride;
        fa::bwd256::Params pdq = b, pdk = b, pdv = b;
        pdq.out = dQ;
        pdq.res0 = Q;
        pdk.res0 = K;
        pdv.res0 = K;
        pdq.out_scale = scale;
        pdq.n_blk = pq.n_blk;                       // (sequence, query head, 128-query block)
        pdq.n_units = pq.n_units;
        pdk.out = dK;
        pdk.out_scale = scale;
        pdk.n_blk = pkv.n_blk;                      // (sequence, K/V head, 128-key block)
        pdk.n_units = pkv.n_units;
        pdv.out = dV;
        pdv.out_scale = 1.f;
        pdv.n_blk = pkv.n_blk;
        pdv.n_units = pkv.n_units;
        pdv.fault_unit = pkv.fault_unit;            // the hook applies to the first pass
        pdq.sched = pq.sched;
        pdk.sched = pkv.sched;
        pdv.sched = fa_host::next_sched_slot(info.sched);
        const cudaError_t e =
            bf16 ? launch_bwd256_varlen<true>(pp, mq, mdo, mk, mv, mq64, mdo64, mk64, mv64, pdq, pdk,
                                              pdv, info.sm_count, st)
                 : launch_bwd256_varlen<false>(pp, mq, mdo, mk, mv, mq64, mdo64, mk64, mv64, pdq,
                                               pdk, pdv, info.sm_count, st);
        if (e != cudaSuccess) return FA_ERR_CUDA;
        fa_host::count_launches(5);
        return FA_OK;
    }
    cudaError_t e;
    if (d == 32)
        e = bf16 ? launch_bwd_varlen<32, true>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st)
                 : launch_bwd_varlen<32, false>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st);
    else if (d == 64)
        e = bf16 ? launch_bwd_varlen<64, true>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st)
                 : launch_bwd_varlen<64, false>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st);
    else
        e = bf16 ? launch_bwd_varlen<128, true>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st)
                 : launch_bwd_varlen<128, false>(pp, mq, mk, mv, mdo, pkv, pq, info.sm_count, st);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    fa_host::count_launches(4);
    return FA_OK;
}

}  // extern "C"
