// fa_api.cu -- the C ABI declared in include/fa.h: argument checks, TMA tensor
// maps, launch of the sm_103a attention kernel, and the device status word.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <vector>

#include "fa.h"
#include "fa_combine.cuh"
#include "fa_fwd1t_kernel.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_host.h"

namespace {

// Device status word: [code, role, iteration, block]. Written by a kernel whose
// bounded wait ran out; read and cleared by fa_sync_status.
__device__ unsigned int g_fa_status[4];

// Work-unit counters of the persistent kernel: {next unit, finished CTAs} per
// launch. A launch takes slot (launch number mod kSchedSlots); its last CTA
// zeroes the slot again. Up to kSchedSlots launches may run concurrently.
constexpr int kSchedSlots = 64;
__device__ unsigned int g_fa_sched[kSchedSlots][2];

constexpr int kMaxDevices = 64;

// Scratch of fa_forward_splitkv_static: a fixed array in device memory for
// callers that cannot allocate. Every GPU that loads this library holds it
// until the process exits.
constexpr size_t kStaticScratchBytes = static_cast<size_t>(FA_SPLITKV_STATIC_SCRATCH_BYTES);
__device__ __align__(256) unsigned char g_fa_static_scratch[kStaticScratchBytes];

// Device address of g_fa_static_scratch, looked up once per device with that
// device current (in host code the symbol is only a host-side stand-in).
struct StaticScratch {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void *ptr = nullptr;
};
StaticScratch g_static_scratch[kMaxDevices];
constexpr uint64_t kDefaultBudgetNs = 2000000000ull;

std::atomic<int64_t> g_launches{0};
std::atomic<uint64_t> g_sched_next{0};
std::atomic<int> g_fault_pos{-1};
// Debug builds with bounds checks: rows added to every stored row of the next
// two-tile forward launch (fa_test_arm_row_shift); 0 = none.
std::atomic<long long> g_row_shift{0};
std::atomic<uint64_t> g_budget_ns{0};

struct DeviceState {
    std::once_flag once;
    cudaError_t init_err = cudaSuccess;
    int cc_major = 0, cc_minor = 0, sm_count = 0;
    unsigned int *status = nullptr;
    unsigned int *sched = nullptr;
};
DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

uint64_t wait_budget() {
    uint64_t b = g_budget_ns.load();
    if (b == 0) {
        b = kDefaultBudgetNs;
        if (const char *e = std::getenv("FA_WAIT_BUDGET_MS")) {
            char *end = nullptr;
            const double ms = std::strtod(e, &end);
            if (end != e && ms > 0 && ms < 1e9) b = static_cast<uint64_t>(ms * 1e6);
        }
        g_budget_ns.store(b);
    }
    return b;
}

// Opt in to the kernel's shared memory, and check that the registers a launch
// allocates cover the kernel's setmaxnreg split (a split above them would make
// setmaxnreg.inc wait forever).
template <int D, bool BF16, bool PACKED, bool VARLEN>
cudaError_t configure_one() {
    cudaFuncAttributes attr{};
    cudaError_t e = cudaFuncGetAttributes(&attr, fa::fa_fwd_kernel<D, BF16, PACKED, VARLEN>);
    if (e != cudaSuccess) return e;
    if (attr.numRegs * fa::kThreads < fa::kRegsNeeded) return cudaErrorInvalidConfiguration;
    return cudaFuncSetAttribute(fa::fa_fwd_kernel<D, BF16, PACKED, VARLEN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                fa::SmemLayout<D>::kAlloc);
}

template <int D, bool BF16>
cudaError_t configure_kernel() {
    cudaError_t e = configure_one<D, BF16, false, false>();
    if (e == cudaSuccess) e = configure_one<D, BF16, true, false>();
    return e != cudaSuccess ? e : configure_one<D, BF16, false, true>();
}

DeviceState *device_state(int dev) {
    if (dev < 0 || dev >= kMaxDevices) return nullptr;
    DeviceState &s = g_dev[dev];
    std::call_once(s.once, [&s, dev] {
        cudaError_t e = cudaDeviceGetAttribute(&s.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&s.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (e == cudaSuccess)
            e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess && s.cc_major == 10 && s.cc_minor == 3) {
            void *addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_fa_status);
            s.status = static_cast<unsigned int *>(addr);
            if (e == cudaSuccess) {
                e = cudaGetSymbolAddress(&addr, g_fa_sched);
                s.sched = static_cast<unsigned int *>(addr);
            }
            if (e == cudaSuccess) e = configure_kernel<32, false>();
            if (e == cudaSuccess) e = configure_kernel<32, true>();
            if (e == cudaSuccess) e = configure_kernel<64, false>();
            if (e == cudaSuccess) e = configure_kernel<64, true>();
            if (e == cudaSuccess) e = configure_kernel<128, false>();
            if (e == cudaSuccess) e = configure_kernel<128, true>();
        }
        s.init_err = e;
    });
    return &s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// Buffers the kernels write with 32-byte vector stores (O, the split scratch, and
// the gradients): a row starts on a 32-byte boundary only if the base does.
bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
// LSE is read and written one float at a time: float alignment is enough.
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool on_device(const void *p, int dev) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice) return a.device == dev;
    if (a.type == cudaMemoryTypeManaged) return true;
    return false;
}

// 3-D map over a contiguous BH x N x d 16-bit tensor, box = 64 columns x 128 rows,
// 128-byte swizzle; rows past N read as zero. Q is mapped by row space
// (n_spaces x R x d), K and V by head.
bool make_map(CUtensorMap *map, const void *base, bool bf16, int64_t BH, int64_t N, int64_t d,
              uint32_t box_rows = 128) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 2),
                                   static_cast<cuuint64_t>(N * d * 2)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(d < 64 ? d : 64), box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r =
        enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            d < 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, bool BF16>
cudaError_t launch(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                   const fa::FwdParams &p, bool packed, int64_t blocks, cudaStream_t stream,
                   bool varlen = false) {
    const unsigned g = static_cast<unsigned>(blocks);
    constexpr int smem = fa::SmemLayout<D>::kAlloc;
    if (varlen)
        fa::fa_fwd_kernel<D, BF16, false, true><<<g, fa::kThreads, smem, stream>>>(q, k, v, p);
    else if (packed)
        fa::fa_fwd_kernel<D, BF16, true, false><<<g, fa::kThreads, smem, stream>>>(q, k, v, p);
    else
        fa::fa_fwd_kernel<D, BF16, false, false><<<g, fa::kThreads, smem, stream>>>(q, k, v, p);
    return cudaGetLastError();
}

// 3-D map over a token-major (tokens x heads x d) 16-bit tensor, ordered (d, heads,
// tokens): box = 64 columns x 1 head x 128 tokens, 128-byte swizzle (the same
// shared-memory tile as make_map's); tokens past the end read as zero.
bool make_map_tokens(CUtensorMap *map, const void *base, bool bf16, int64_t tokens,
                     int64_t heads, int64_t d, uint32_t box_tokens = 128) {
    EncodeTiledFn enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                                static_cast<cuuint64_t>(tokens)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d * 2),
                                   static_cast<cuuint64_t>(heads * d * 2)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(d < 64 ? d : 64), 1, box_tokens};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r =
        enc(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
            const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            d < 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}


// ---- one forward launch (plus the split merge when the keys are split)
struct Call {
    const void *Q, *K, *V;
    void *O;
    float *LSE;
    int64_t B, H, H_kv, Nq, Nk, d;
    float scale;
    fa_mask_mode mask_mode;
    int64_t window_left, window_right;
    fa_dtype dtype;
    int64_t num_splits;
    void *workspace;
    size_t workspace_bytes;
    void *stream;
};

using fa_host::align256;

// Workspace of a key-split call: partial LSEs, then partial outputs, fp32.
size_t splitkv_bytes(int64_t rows, int64_t d, int64_t splits) {
    return align256(static_cast<size_t>(splits) * rows * sizeof(float)) +
           static_cast<size_t>(splits) * rows * d * sizeof(float);
}

// Query rows are packed per K/V head (all its query heads in one row space) when
// there are few queries per head and the heads are grouped.
bool pack_rows(int64_t H, int64_t H_kv, int64_t Nq) { return H_kv < H && Nq <= 64; }

// Splits that fill one wave: as many as fit on the SMs next to the unsplit
// units (measured on decode and chunked-prefill shapes, one wave beat both an
// underfilled grid and several waves of shorter units), each split keeping at
// least four 128-key tiles. 1 when the units alone fill the SMs.
int64_t default_splits(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int sms) {
    const bool packed = pack_rows(H, H_kv, Nq);
    const int64_t spaces = packed ? B * H_kv : B * H;
    const int64_t R = packed ? (H / H_kv) * Nq : Nq;
    const int64_t units = spaces * ((R + fa::kUnitRows - 1) / fa::kUnitRows);
    const int64_t tiles = (Nk + fa::kBN - 1) / fa::kBN;
    if (units >= sms) return 1;
    int64_t s = sms / units;
    const int64_t cap = tiles / 4 > 1 ? tiles / 4 : 1;
    if (s > cap) s = cap;
    if (s > 256) s = 256;
    return s < 1 ? 1 : s;
}

template <int D, bool BF16>
cudaError_t launch_combine(const fa::CombineParams &c, cudaStream_t stream) {
    const int64_t rows = static_cast<int64_t>(c.BH) * c.Nq;
    const int64_t blocks = (rows + fa::kCombineWarps - 1) / fa::kCombineWarps;
    fa::fa_combine_kernel<D, BF16><<<static_cast<unsigned>(blocks), fa::kCombineWarps * 32, 0,
                                     stream>>>(c);
    return cudaGetLastError();
}

// The one-tile kernel (fa_fwd1t_kernel.cuh), set up once per device.
struct OneTileState {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
};
OneTileState g_onetile[kMaxDevices];

template <int D, bool BF16, bool VARLEN = false>
cudaError_t onetile_attr() {
    return cudaFuncSetAttribute(fa::onetile::fa_fwd1t_kernel<D, BF16, VARLEN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                fa::onetile::Smem<D>::kAlloc);
}

template <int D, bool BF16, bool VARLEN = false>
cudaError_t launch_onetile(const CUtensorMap &q, const CUtensorMap &k, const CUtensorMap &v,
                           const fa::onetile::Params &p, unsigned blocks, cudaStream_t st) {
    fa::onetile::fa_fwd1t_kernel<D, BF16, VARLEN>
        <<<blocks, fa::onetile::kThreads, fa::onetile::Smem<D>::kAlloc, st>>>(q, k, v, p);
    return cudaGetLastError();
}

// The one-tile kernel runs d = 256; at d = 64 / 128 it runs row spaces of at most
// 128 rows (decode steps), and small unsplit problems: those whose 256-row units
// of the two-tile kernel would fill at most half of the SMs. There, twice as many
// 128-row units fill the GPU better, and three S buffers overlap a unit's
// softmax with its next products (measured on B1 H1 N256 d64: 8.8 -> 7.2 us per
// call; B1 H8 N1024 causal: 17.6 -> 12.0 us). Key splits (n_splits > 1) already
// spread a small problem over the SMs; they stay on the two-tile kernel.
bool use_onetile(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t d, int64_t n_splits,
                 int sms) {
    if (d == 256) return true;
    if (d != 64 && d != 128) return false;
    const bool packed = pack_rows(H, H_kv, Nq);
    const int64_t R = packed ? (H / H_kv) * Nq : Nq;
    if (R <= fa::onetile::kBM) return true;
    const int64_t spaces = packed ? B * H_kv : B * H;
    return n_splits == 1 && 2 * spaces * ((R + fa::kUnitRows - 1) / fa::kUnitRows) <= sms;
}

// Shared-memory opt-in of every one-tile kernel instance, once per device.
bool onetile_ready(int dev) {
    OneTileState &s = g_onetile[dev];
    std::call_once(s.once, [&s] {
        cudaError_t e = onetile_attr<64, false>();
        if (e == cudaSuccess) e = onetile_attr<64, true>();
        if (e == cudaSuccess) e = onetile_attr<128, false>();
        if (e == cudaSuccess) e = onetile_attr<128, true>();
        if (e == cudaSuccess) e = onetile_attr<256, false>();
        if (e == cudaSuccess) e = onetile_attr<256, true>();
        if (e == cudaSuccess) e = onetile_attr<256, false, true>();
        if (e == cudaSuccess) e = onetile_attr<256, true, true>();
        s.err = e;
    });
    return s.err == cudaSuccess;
}

// One 128-row Q tile per unit, bn(d)-key K/V tiles. The key splits are those of the
// two-tile path (split_tiles 128-key tiles each, so the workspace and the merge are
// the same); the kernel counts them in its own tiles.
fa_status run_forward_1t(const Call &c, DeviceState *ds, int dev, int64_t n_splits,
                         int64_t split_tiles) {
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    if (!onetile_ready(dev)) return FA_ERR_CUDA;
    const int64_t B = c.B, H = c.H, H_kv = c.H_kv, Nq = c.Nq, Nk = c.Nk, d = c.d;
    const bool bf16 = c.dtype == FA_DTYPE_BF16;
    // few queries with grouped heads: one row space per K/V head (its query heads'
    // rows in turn), so that each K/V tile is read once for all of them
    const bool packed = pack_rows(H, H_kv, Nq);
    const int64_t hps = packed ? H / H_kv : 1;
    const int64_t spaces = B * H / hps, R = hps * Nq;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, c.Q, bf16, spaces, R, d, fa::onetile::kBM) ||
        !make_map(&mk, c.K, bf16, B * H_kv, Nk, d, fa::onetile::bn(static_cast<int>(d))) ||
        !make_map(&mv, c.V, bf16, B * H_kv, Nk, d, fa::onetile::bn(static_cast<int>(d))))
        return FA_ERR_CUDA;
    const bool split = n_splits > 1;
    const int64_t BH = B * H;
    fa::onetile::Params p{};
    p.O = c.O;
    p.LSE = c.LSE;
    if (split) {
        p.part_LSE = static_cast<float *>(c.workspace);
        p.part_O = reinterpret_cast<float *>(static_cast<uint8_t *>(c.workspace) +
                                             align256(static_cast<size_t>(n_splits) * BH * Nq *
                                                      sizeof(float)));
    }
    p.Nq = static_cast<int>(Nq);
    p.Nk = static_cast<int>(Nk);
    p.q_off = static_cast<int>(Nk - Nq);
    p.BH = static_cast<int>(BH);
    p.kv_group = static_cast<int>(H / H_kv);
    p.hps = static_cast<int>(hps);
    p.R = static_cast<int>(R);
    const int64_t n_qb = (R + fa::onetile::kBM - 1) / fa::onetile::kBM;
    const int64_t n_units = spaces * n_qb * n_splits;
    if (n_units > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    p.n_units = static_cast<int>(n_units);
    p.n_qb = static_cast<int>(n_qb);
    p.n_splits = static_cast<int>(n_splits);
    p.split_tiles = static_cast<int>(split_tiles * (fa::kBN / fa::onetile::bn(static_cast<int>(d))));
    const int64_t all = Nq + Nk;
    int64_t wl = all, wr = all;
    if (c.mask_mode == FA_MASK_CAUSAL) wr = 0;
    if (c.mask_mode == FA_MASK_WINDOW) {
        wl = c.window_left < all ? c.window_left : all;
        wr = c.window_right < all ? c.window_right : all;
    }
    p.wl = static_cast<int>(wl);
    p.wr = static_cast<int>(wr);
    p.heavy_first = wr < Nk ? 1 : 0;
    p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634074);
    p.wait_budget_ns = wait_budget();
    p.status = ds->status;
    p.sched = ds->sched + 2 * (g_sched_next.fetch_add(1) % kSchedSlots);
    p.fault_skip_k = g_fault_pos.exchange(-1);
    const unsigned blocks = static_cast<unsigned>(n_units < ds->sm_count ? n_units : ds->sm_count);
    cudaStream_t st = static_cast<cudaStream_t>(c.stream);
    cudaError_t le;
    if (d == 64)
        le = bf16 ? launch_onetile<64, true>(mq, mk, mv, p, blocks, st)
                  : launch_onetile<64, false>(mq, mk, mv, p, blocks, st);
    else if (d == 128)
        le = bf16 ? launch_onetile<128, true>(mq, mk, mv, p, blocks, st)
                  : launch_onetile<128, false>(mq, mk, mv, p, blocks, st);
    else
        le = bf16 ? launch_onetile<256, true>(mq, mk, mv, p, blocks, st)
                  : launch_onetile<256, false>(mq, mk, mv, p, blocks, st);
    if (le != cudaSuccess) return FA_ERR_CUDA;
    g_launches.fetch_add(1);
    if (split) {
        fa::CombineParams cp{};
        cp.part_O = p.part_O;
        cp.part_LSE = p.part_LSE;
        cp.O = c.O;
        cp.LSE = c.LSE;
        cp.BH = p.BH;
        cp.Nq = p.Nq;
        cp.Nk = p.Nk;
        cp.q_off = p.q_off;
        cp.wl = p.wl;
        cp.wr = p.wr;
        cp.n_splits = p.n_splits;
        cp.split_keys = static_cast<int>(split_tiles * fa::kBN);
        cudaError_t e;
        if (d == 64)
            e = bf16 ? launch_combine<64, true>(cp, st) : launch_combine<64, false>(cp, st);
        else if (d == 128)
            e = bf16 ? launch_combine<128, true>(cp, st) : launch_combine<128, false>(cp, st);
        else
            e = bf16 ? launch_combine<256, true>(cp, st) : launch_combine<256, false>(cp, st);
        if (e != cudaSuccess) return FA_ERR_CUDA;
        g_launches.fetch_add(1);
    }
    return FA_OK;
}

// Row spaces per scheduling group of the heavy-first order (FwdParams::group).
// The launch-wide counter hands units to whichever CTA is free, so the launch
// ends when the last CTA finishes its last unit; with few units per CTA that
// tail is a large share. Grouping spaces puts the lightest units of many spaces
// at the end. The group size is chosen by simulating that greedy assignment on
// the units' K/V tile counts for a few sizes (cached per shape), among groups
// whose K and V stay well inside L2 (their units run concurrently and share it).
struct GroupKey {
    int v[12];
    bool operator==(const GroupKey &o) const {
        for (int i = 0; i < 12; ++i)
            if (v[i] != o.v[i]) return false;
        return true;
    }
};
std::mutex g_group_mu;
GroupKey g_group_keys[16];
int g_group_vals[16];
int g_group_n = 0;

int unit_group(const fa::FwdParams &p, int grid, size_t kv_head_bytes) {
    const int spaces = p.n_spaces;
    const int64_t n_units = static_cast<int64_t>(p.n_units);
    if (spaces < 2 || grid < 1 || n_units > 32 * static_cast<int64_t>(grid)) return 1;
    const GroupKey key{{p.n_qb, p.n_splits, spaces, p.split_tiles, p.wl, p.wr, p.R, p.Nk,
                        p.q_off, grid, p.kv_group, static_cast<int>(kv_head_bytes >> 10)}};
    {
        std::lock_guard<std::mutex> lk(g_group_mu);
        for (int i = 0; i < g_group_n && i < 16; ++i)
            if (g_group_keys[i] == key) return g_group_vals[i];
    }
    // Weight of unit (row block qb, split s): its MMA iterations (K/V tiles, plus one
    // to drain unless its two Q tiles pair one tile apart) and a fixed share for
    // the unit's start and epilogue. Same visibility rule as decode_unit.
    std::vector<int> w(static_cast<size_t>(p.n_qb) * p.n_splits, 0);
    for (int qb = 0; qb < p.n_qb; ++qb)
        for (int sp = 0; sp < p.n_splits; ++sp) {
            const int s_lo = sp * p.split_tiles, s_hi = s_lo + p.split_tiles - 1;
            int a[2] = {1, 1}, b[2] = {0, 0}, j0 = 0x7fffffff, j1 = -1;
            for (int t = 0; t < 2; ++t) {
                const int rt0 = qb * fa::kUnitRows + t * fa::kBM;
                if (rt0 >= p.R) continue;
                const int rl = std::min(rt0 + fa::kBM, p.R) - 1;
                const int64_t lo_key = static_cast<int64_t>(rt0) + p.q_off - p.wl;
                const int64_t hi_key = static_cast<int64_t>(rl) + p.q_off + p.wr;
                if (hi_key < 0 || lo_key > p.Nk - 1) continue;
                const int at = std::max(static_cast<int>(std::max<int64_t>(0, lo_key) / fa::kBN), s_lo);
                const int bt = std::min(static_cast<int>(std::min<int64_t>(p.Nk - 1, hi_key) / fa::kBN), s_hi);
                if (at > bt) continue;
                a[t] = at;
                b[t] = bt;
                j0 = std::min(j0, at);
                j1 = std::max(j1, bt);
            }
            if (j1 < j0) continue;
            const bool paired = a[0] <= b[0] && a[1] <= b[1] && a[1] == a[0] + 1;
            w[static_cast<size_t>(qb) * p.n_splits + sp] = (j1 - j0 + 1) + (paired ? 0 : 1) + 3;
        }
    const size_t l2_budget = size_t{48} << 20;
    const int cands[] = {1, 2, 4, 8, 12, 16, 24, 32, 48, 64};
    int best = 1;
    int64_t best_t = -1;
    std::vector<int64_t> heap(static_cast<size_t>(grid));
    for (int g : cands) {
        if (g > spaces) break;
        const size_t kv_heads = static_cast<size_t>((g + p.kv_group - 1) / p.kv_group + 1);
        if (g > 1 && kv_heads * kv_head_bytes > l2_budget) break;
        std::fill(heap.begin(), heap.end(), 0);  // a min-heap of the CTAs' finishing times
        for (int base = 0; base < spaces; base += g) {
            const int gs = std::min(g, spaces - base);
            for (int qbi = 0; qbi < p.n_qb; ++qbi) {
                const int qb = p.n_qb - 1 - qbi;
                for (int h = 0; h < gs; ++h)
                    for (int sp = 0; sp < p.n_splits; ++sp) {
                        const int wu = w[static_cast<size_t>(qb) * p.n_splits + sp];
                        if (wu == 0) continue;
                        std::pop_heap(heap.begin(), heap.end(), std::greater<int64_t>());
                        heap.back() += wu;
                        std::push_heap(heap.begin(), heap.end(), std::greater<int64_t>());
                    }
            }
        }
        const int64_t t = *std::max_element(heap.begin(), heap.end());
        if (best_t < 0 || t < best_t) {
            best_t = t;
            best = g;
        }
    }
    std::lock_guard<std::mutex> lk(g_group_mu);
    const int slot = g_group_n % 16;
    g_group_keys[slot] = key;
    g_group_vals[slot] = best;
    ++g_group_n;
    return best;
}

fa_status run_forward(const Call &c) {
    const void *Q = c.Q, *K = c.K, *V = c.V;
    void *O = c.O;
    float *LSE = c.LSE;
    const int64_t B = c.B, H = c.H, H_kv = c.H_kv, Nq = c.Nq, Nk = c.Nk, d = c.d;
    // ---- host-side checks: nothing is enqueued on failure
    if (!Q || !K || !V || !O || !LSE) return FA_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (c.dtype != FA_DTYPE_FP16 && c.dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
    const fa_mask_mode mask_mode = c.mask_mode;
    if (mask_mode != FA_MASK_NONE && mask_mode != FA_MASK_CAUSAL && mask_mode != FA_MASK_WINDOW)
        return FA_ERR_INVALID_ARG;
    if (mask_mode == FA_MASK_WINDOW && (c.window_left < 0 || c.window_right < 0))
        return FA_ERR_INVALID_ARG;
    // Masks place the queries at the last Nq key positions; more queries than keys
    // would leave rows with no visible key.
    if (mask_mode != FA_MASK_NONE && Nq > Nk) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(c.scale) || !(c.scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned32(O) || !aligned4(LSE))
        return FA_ERR_INVALID_ARG;
    if (c.num_splits < 1) return FA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    // Size limits of this implementation: 32-bit row indices and grid.
    if (Nq > (int64_t{1} << 29) || Nk > (int64_t{1} << 29) || B * H > (int64_t{1} << 31))
        return FA_ERR_UNSUPPORTED;
    const int64_t BH = B * H;
    const int64_t BHkv = B * H_kv;
    const bool packed = pack_rows(H, H_kv, Nq);
    const int64_t R = packed ? (H / H_kv) * Nq : Nq;
    const int64_t spaces = packed ? BHkv : BH;
    const int64_t n_qb = (R + fa::kUnitRows - 1) / fa::kUnitRows;
    const int64_t kv_tiles = (Nk + fa::kBN - 1) / fa::kBN;
    const int64_t splits = c.num_splits < kv_tiles ? c.num_splits : kv_tiles;
    const int64_t split_tiles = (kv_tiles + splits - 1) / splits;
    const int64_t n_splits = (kv_tiles + split_tiles - 1) / split_tiles;
    const int64_t n_units = spaces * n_qb * n_splits;
    if (n_units > 0x7fffffffLL || BH * Nq > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    const bool split = n_splits > 1;
    const size_t tbytes = static_cast<size_t>(BH) * Nq * d * 2;
    const size_t lbytes = static_cast<size_t>(BH) * Nq * sizeof(float);
    const size_t kvbytes = static_cast<size_t>(BHkv) * Nk * d * 2;
    if (overlaps(O, tbytes, Q, tbytes) || overlaps(O, tbytes, K, kvbytes) ||
        overlaps(O, tbytes, V, kvbytes) || overlaps(O, tbytes, LSE, lbytes) ||
        overlaps(LSE, lbytes, Q, tbytes) || overlaps(LSE, lbytes, K, kvbytes) ||
        overlaps(LSE, lbytes, V, kvbytes))
        return FA_ERR_INVALID_ARG;
    const size_t wbytes = split ? splitkv_bytes(BH * Nq, d, n_splits) : 0;
    if (split) {
        if (c.workspace == nullptr || c.workspace_bytes < wbytes) return FA_ERR_INVALID_ARG;
        const void *W = c.workspace;
        if (overlaps(W, wbytes, Q, tbytes) || overlaps(W, wbytes, K, kvbytes) ||
            overlaps(W, wbytes, V, kvbytes) || overlaps(W, wbytes, O, tbytes) ||
            overlaps(W, wbytes, LSE, lbytes))
            return FA_ERR_INVALID_ARG;
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    DeviceState *ds = device_state(dev);
    if (ds == nullptr) return FA_ERR_UNSUPPORTED;
    if (ds->init_err != cudaSuccess) return FA_ERR_CUDA;
    if (!(ds->cc_major == 10 && ds->cc_minor == 3)) return FA_ERR_UNSUPPORTED;
    if (!on_device(Q, dev) || !on_device(K, dev) || !on_device(V, dev) || !on_device(O, dev) ||
        !on_device(LSE, dev) || (split && !on_device(c.workspace, dev)))
        return FA_ERR_INVALID_ARG;
    if (use_onetile(B, H, H_kv, Nq, d, n_splits, ds->sm_count))
        return run_forward_1t(c, ds, dev, n_splits, split_tiles);

    const bool bf16 = c.dtype == FA_DTYPE_BF16;
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, Q, bf16, spaces, R, d) || !make_map(&mk, K, bf16, BHkv, Nk, d) ||
        !make_map(&mv, V, bf16, BHkv, Nk, d))
        return FA_ERR_CUDA;

    fa::FwdParams p{};
    p.O = O;
    p.LSE = LSE;
    float *part_LSE = nullptr, *part_O = nullptr;
    if (split) {
        part_LSE = static_cast<float *>(c.workspace);
        part_O = reinterpret_cast<float *>(static_cast<uint8_t *>(c.workspace) +
                                           align256(static_cast<size_t>(n_splits) * BH * Nq *
                                                    sizeof(float)));
    }
    p.part_O = part_O;
    p.part_LSE = part_LSE;
    p.Nq = static_cast<int>(Nq);
    p.Nk = static_cast<int>(Nk);
    p.q_off = static_cast<int>(Nk - Nq);
    p.H = static_cast<int>(H);
    p.BH = static_cast<int>(BH);
    p.kv_group = static_cast<int>(H / H_kv);
    p.R = static_cast<int>(R);
    p.n_units = static_cast<int>(n_units);
    p.n_qb = static_cast<int>(n_qb);
    p.n_splits = static_cast<int>(n_splits);
    p.split_tiles = static_cast<int>(split_tiles);
    // Visible keys of query i: [i + q_off - wl, i + q_off + wr]; "all keys" is a window
    // wider than any offset (values are clamped so the sums stay in 32 bits).
    const int64_t all = Nq + Nk;
    int64_t wl = all, wr = all;
    if (mask_mode == FA_MASK_CAUSAL) wr = 0;
    if (mask_mode == FA_MASK_WINDOW) {
        wl = c.window_left < all ? c.window_left : all;
        wr = c.window_right < all ? c.window_right : all;
    }
    p.wl = static_cast<int>(wl);
    p.wr = static_cast<int>(wr);
    p.heavy_first = wr < Nk ? 1 : 0;
    p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634074);
    p.wait_budget_ns = wait_budget();
    p.status = ds->status;
    p.fault_skip_k = g_fault_pos.exchange(-1);
    p.sched = ds->sched + 2 * (g_sched_next.fetch_add(1) % kSchedSlots);
    p.n_spaces = static_cast<int>(spaces);
    p.out_rows = static_cast<long long>(BH) * Nq;
    p.row_shift = g_row_shift.exchange(0);

    // Persistent grid: one CTA per SM (each holds the SM's whole tensor memory).
    const int64_t blocks = n_units < ds->sm_count ? n_units : ds->sm_count;
    p.group = p.heavy_first && !packed
                  ? unit_group(p, static_cast<int>(blocks),
                               static_cast<size_t>(Nk) * static_cast<size_t>(d) * 4)
                  : 1;
    cudaStream_t st = static_cast<cudaStream_t>(c.stream);
    cudaError_t e;
    if (d == 32)
        e = bf16 ? launch<32, true>(mq, mk, mv, p, packed, blocks, st)
                 : launch<32, false>(mq, mk, mv, p, packed, blocks, st);
    else if (d == 64)
        e = bf16 ? launch<64, true>(mq, mk, mv, p, packed, blocks, st)
                 : launch<64, false>(mq, mk, mv, p, packed, blocks, st);
    else
        e = bf16 ? launch<128, true>(mq, mk, mv, p, packed, blocks, st)
                 : launch<128, false>(mq, mk, mv, p, packed, blocks, st);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    g_launches.fetch_add(1);
    if (split) {
        fa::CombineParams cp{};
        cp.part_O = part_O;
        cp.part_LSE = part_LSE;
        cp.O = O;
        cp.LSE = LSE;
        cp.BH = p.BH;
        cp.Nq = p.Nq;
        cp.Nk = p.Nk;
        cp.q_off = p.q_off;
        cp.wl = p.wl;
        cp.wr = p.wr;
        cp.n_splits = p.n_splits;
        cp.split_keys = p.split_tiles * fa::kBN;
        if (d == 32)
            e = bf16 ? launch_combine<32, true>(cp, st) : launch_combine<32, false>(cp, st);
        else if (d == 64)
            e = bf16 ? launch_combine<64, true>(cp, st) : launch_combine<64, false>(cp, st);
        else
            e = bf16 ? launch_combine<128, true>(cp, st) : launch_combine<128, false>(cp, st);
        if (e != cudaSuccess) return FA_ERR_CUDA;
        g_launches.fetch_add(1);
    }
    return FA_OK;
}

struct VarlenCall {
    const void *Q, *K, *V;
    void *O;
    float *LSE;
    const int32_t *cu_q, *cu_k;
    int64_t B, H, H_kv, total_q, total_k, max_q, d;
    float scale;
    fa_mask_mode mask_mode;
    int64_t window_left, window_right;
    fa_dtype dtype;
    void *stream;
};

// Variable-length batch at d = 256: the one-tile kernel's VARLEN instance. Units are
// (sequence, head, 128-row block) of the longest sequence; K/V tiles hold 64 keys.
fa_status run_forward_varlen_1t(const VarlenCall &c, DeviceState *ds, int dev) {
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    if (!onetile_ready(dev)) return FA_ERR_CUDA;
    const int64_t B = c.B, H = c.H, H_kv = c.H_kv;
    constexpr int kD = 256;
    constexpr int kBn = fa::onetile::bn(kD);
    const bool bf16 = c.dtype == FA_DTYPE_BF16;
    CUtensorMap mq, mk, mv;
    if (!make_map_tokens(&mq, c.Q, bf16, c.total_q, H, kD, fa::onetile::kBM) ||
        !make_map_tokens(&mk, c.K, bf16, c.total_k, H_kv, kD, kBn) ||
        !make_map_tokens(&mv, c.V, bf16, c.total_k, H_kv, kD, kBn))
        return FA_ERR_CUDA;
    const int64_t BH = B * H;
    const int64_t n_qb = (c.max_q + fa::onetile::kBM - 1) / fa::onetile::kBM;
    const int64_t n_units = BH * n_qb;
    if (n_units > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    fa::onetile::Params p{};
    p.O = c.O;
    p.LSE = c.LSE;
    p.Nq = static_cast<int>(c.max_q);
    p.Nk = static_cast<int>(c.total_k);
    p.BH = static_cast<int>(BH);
    p.kv_group = static_cast<int>(H / H_kv);
    p.hps = 1;
    p.R = static_cast<int>(c.max_q);
    p.n_units = static_cast<int>(n_units);
    p.n_qb = static_cast<int>(n_qb);
    p.n_splits = 1;
    p.split_tiles = static_cast<int>((c.total_k + kBn - 1) / kBn);  // one split: every tile
    // Every sequence's query-key offset lies in [-total_q, total_k], so a window
    // of total_q + total_k stands for "all keys".
    const int64_t all = c.total_q + c.total_k;
    int64_t wl = all, wr = all;
    if (c.mask_mode == FA_MASK_CAUSAL) wr = 0;
    if (c.mask_mode == FA_MASK_WINDOW) {
        wl = c.window_left < all ? c.window_left : all;
        wr = c.window_right < all ? c.window_right : all;
    }
    p.wl = static_cast<int>(wl);
    p.wr = static_cast<int>(wr);
    p.heavy_first = wr < all ? 1 : 0;
    p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634074);
    p.wait_budget_ns = wait_budget();
    p.status = ds->status;
    p.sched = ds->sched + 2 * (g_sched_next.fetch_add(1) % kSchedSlots);
    p.fault_skip_k = g_fault_pos.exchange(-1);
    p.cu_q = c.cu_q;
    p.cu_k = c.cu_k;
    p.total_q = static_cast<int>(c.total_q);
    p.total_k = static_cast<int>(c.total_k);
    p.H = static_cast<int>(H);
    const unsigned blocks = static_cast<unsigned>(n_units < ds->sm_count ? n_units : ds->sm_count);
    cudaStream_t st = static_cast<cudaStream_t>(c.stream);
    const cudaError_t le = bf16 ? launch_onetile<kD, true, true>(mq, mk, mv, p, blocks, st)
                                : launch_onetile<kD, false, true>(mq, mk, mv, p, blocks, st);
    if (le != cudaSuccess) return FA_ERR_CUDA;
    g_launches.fetch_add(1);
    return FA_OK;
}

fa_status run_forward_varlen(const VarlenCall &c) {
    const int64_t B = c.B, H = c.H, H_kv = c.H_kv, d = c.d;
    // ---- host-side checks: nothing is enqueued on failure
    if (B < 1 || H < 1 || d < 1 || c.total_q < 0 || c.total_k < 0 || c.max_q < 0)
        return FA_ERR_INVALID_ARG;
    if (c.total_q == 0 || c.max_q == 0) return FA_OK;  // no query rows: nothing to do
    if (!c.Q || !c.K || !c.V || !c.O || !c.LSE || !c.cu_q || !c.cu_k) return FA_ERR_INVALID_ARG;
    if (H_kv < 1 || H % H_kv != 0) return FA_ERR_INVALID_ARG;
    if (c.dtype != FA_DTYPE_FP16 && c.dtype != FA_DTYPE_BF16) return FA_ERR_INVALID_ARG;
    if (c.mask_mode != FA_MASK_NONE && c.mask_mode != FA_MASK_CAUSAL &&
        c.mask_mode != FA_MASK_WINDOW)
        return FA_ERR_INVALID_ARG;
    if (c.mask_mode == FA_MASK_WINDOW && (c.window_left < 0 || c.window_right < 0))
        return FA_ERR_INVALID_ARG;
    if (!std::isfinite(c.scale) || !(c.scale > 0.f)) return FA_ERR_INVALID_ARG;
    if (!aligned16(c.Q) || !aligned16(c.K) || !aligned16(c.V) || !aligned32(c.O) ||
        !aligned4(c.LSE) || (reinterpret_cast<uintptr_t>(c.cu_q) & 3u) ||
        (reinterpret_cast<uintptr_t>(c.cu_k) & 3u))
        return FA_ERR_INVALID_ARG;
    if (d != 32 && d != 64 && d != 128 && d != 256) return FA_ERR_UNSUPPORTED;
    if (c.total_q > (int64_t{1} << 29) || c.total_k > (int64_t{1} << 29) || c.max_q > c.total_q ||
        B * H > (int64_t{1} << 31))
        return FA_ERR_UNSUPPORTED;
    if (c.total_k == 0) return FA_ERR_INVALID_ARG;  // rows without any key
    const int64_t BH = B * H;
    const int64_t n_qb = (c.max_q + fa::kUnitRows - 1) / fa::kUnitRows;
    const int64_t n_units = BH * n_qb;
    if (n_units > 0x7fffffffLL || c.total_q * H > 0x7fffffffLL) return FA_ERR_UNSUPPORTED;
    const size_t tbytes = static_cast<size_t>(c.total_q) * H * d * 2;
    const size_t lbytes = static_cast<size_t>(c.total_q) * H * sizeof(float);
    const size_t kvbytes = static_cast<size_t>(c.total_k) * H_kv * d * 2;
    const size_t cubytes = static_cast<size_t>(B + 1) * sizeof(int32_t);
    const void *O = c.O, *LSE = c.LSE;
    if (overlaps(O, tbytes, c.Q, tbytes) || overlaps(O, tbytes, c.K, kvbytes) ||
        overlaps(O, tbytes, c.V, kvbytes) || overlaps(O, tbytes, LSE, lbytes) ||
        overlaps(O, tbytes, c.cu_q, cubytes) || overlaps(O, tbytes, c.cu_k, cubytes) ||
        overlaps(LSE, lbytes, c.Q, tbytes) || overlaps(LSE, lbytes, c.K, kvbytes) ||
        overlaps(LSE, lbytes, c.V, kvbytes) || overlaps(LSE, lbytes, c.cu_q, cubytes) ||
        overlaps(LSE, lbytes, c.cu_k, cubytes))
        return FA_ERR_INVALID_ARG;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    DeviceState *ds = device_state(dev);
    if (ds == nullptr) return FA_ERR_UNSUPPORTED;
    if (ds->init_err != cudaSuccess) return FA_ERR_CUDA;
    if (!(ds->cc_major == 10 && ds->cc_minor == 3)) return FA_ERR_UNSUPPORTED;
    if (!on_device(c.Q, dev) || !on_device(c.K, dev) || !on_device(c.V, dev) ||
        !on_device(c.O, dev) || !on_device(c.LSE, dev) || !on_device(c.cu_q, dev) ||
        !on_device(c.cu_k, dev))
        return FA_ERR_INVALID_ARG;

    if (d == 256) return run_forward_varlen_1t(c, ds, dev);
    const bool bf16 = c.dtype == FA_DTYPE_BF16;
    CUtensorMap mq, mk, mv;
    if (!make_map_tokens(&mq, c.Q, bf16, c.total_q, H, d) ||
        !make_map_tokens(&mk, c.K, bf16, c.total_k, H_kv, d) ||
        !make_map_tokens(&mv, c.V, bf16, c.total_k, H_kv, d))
        return FA_ERR_CUDA;

    fa::FwdParams p{};
    p.O = c.O;
    p.LSE = c.LSE;
    p.Nq = static_cast<int>(c.max_q);
    p.Nk = static_cast<int>(c.total_k);
    p.H = static_cast<int>(H);
    p.BH = static_cast<int>(BH);
    p.kv_group = static_cast<int>(H / H_kv);
    p.R = static_cast<int>(c.max_q);
    p.n_units = static_cast<int>(n_units);
    p.n_qb = static_cast<int>(n_qb);
    p.n_splits = 1;
    p.split_tiles = static_cast<int>((c.total_k + fa::kBN - 1) / fa::kBN);
    // Every sequence's query-key offset lies in [-total_q, total_k], so a window
    // of total_q + total_k stands for "all keys".
    const int64_t all = c.total_q + c.total_k;
    int64_t wl = all, wr = all;
    if (c.mask_mode == FA_MASK_CAUSAL) wr = 0;
    if (c.mask_mode == FA_MASK_WINDOW) {
        wl = c.window_left < all ? c.window_left : all;
        wr = c.window_right < all ? c.window_right : all;
    }
    p.wl = static_cast<int>(wl);
    p.wr = static_cast<int>(wr);
    p.heavy_first = wr < all ? 1 : 0;
    p.scale_log2 = static_cast<float>(static_cast<double>(c.scale) * 1.4426950408889634074);
    p.wait_budget_ns = wait_budget();
    p.status = ds->status;
    p.fault_skip_k = g_fault_pos.exchange(-1);
    p.sched = ds->sched + 2 * (g_sched_next.fetch_add(1) % kSchedSlots);
    p.cu_q = c.cu_q;
    p.cu_k = c.cu_k;
    p.total_q = static_cast<int>(c.total_q);
    p.total_k = static_cast<int>(c.total_k);
    p.out_rows = static_cast<long long>(c.total_q) * H;
    p.row_shift = g_row_shift.exchange(0);

    const int64_t blocks = n_units < ds->sm_count ? n_units : ds->sm_count;
    // Causal / window: heaviest blocks first over groups of 16 row spaces (heads of one
    // sequence), so that the last units handed out are light ones. The lengths are on
    // the device, so the group is fixed rather than simulated as for dense calls
    // (16 measured best of 1-64 on the mixed-length causal workload, by under 1 %).
    p.n_spaces = static_cast<int>(BH);
    p.group = p.heavy_first ? 16 : 1;
    cudaStream_t st = static_cast<cudaStream_t>(c.stream);
    cudaError_t e;
    if (d == 32)
        e = bf16 ? launch<32, true>(mq, mk, mv, p, false, blocks, st, true)
                 : launch<32, false>(mq, mk, mv, p, false, blocks, st, true);
    else if (d == 64)
        e = bf16 ? launch<64, true>(mq, mk, mv, p, false, blocks, st, true)
                 : launch<64, false>(mq, mk, mv, p, false, blocks, st, true);
    else
        e = bf16 ? launch<128, true>(mq, mk, mv, p, false, blocks, st, true)
                 : launch<128, false>(mq, mk, mv, p, false, blocks, st, true);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    g_launches.fetch_add(1);
    return FA_OK;
}

}  // namespace

namespace fa_host {

DeviceInfo device_info(int dev) {
    DeviceInfo info{cudaErrorInvalidDevice, 0, 0, 0, nullptr, nullptr};
    DeviceState *s = device_state(dev);
    if (s == nullptr) return info;
    info.err = s->init_err;
    info.cc_major = s->cc_major;
    info.cc_minor = s->cc_minor;
    info.sm_count = s->sm_count;
    info.status = s->status;
    info.sched = s->sched;
    return info;
}
bool aligned16(const void *p) { return ::aligned16(p); }
bool aligned32(const void *p) { return ::aligned32(p); }
bool aligned4(const void *p) { return ::aligned4(p); }
bool overlaps(const void *a, size_t na, const void *b, size_t nb) { return ::overlaps(a, na, b, nb); }
bool on_device(const void *p, int dev) { return ::on_device(p, dev); }
bool make_map(CUtensorMap *map, const void *base, bool bf16, int64_t BH, int64_t N, int64_t d,
              uint32_t box_rows) {
    return ::make_map(map, base, bf16, BH, N, d, box_rows);
}
uint64_t wait_budget() { return ::wait_budget(); }
bool make_map_tokens(CUtensorMap *map, const void *base, bool bf16, int64_t tokens, int64_t heads,
                     int64_t d, uint32_t box_tokens) {
    return ::make_map_tokens(map, base, bf16, tokens, heads, d, box_tokens);
}
void count_launches(int64_t n) { g_launches += n; }
int take_fault_position() { return g_fault_pos.exchange(-1); }
unsigned int *next_sched_slot(unsigned int *base) {
    return base + 2 * (g_sched_next.fetch_add(1) % kSchedSlots);
}

}  // namespace fa_host

extern "C" {

const char *fa_status_string(fa_status s) {
    switch (s) {
        case FA_OK: return "FA_OK: success";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG: invalid argument";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED: not supported by this build or device";
        case FA_ERR_CUDA: return "FA_ERR_CUDA: a CUDA call failed";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT: a bounded in-kernel wait ran out";
        case FA_ERR_BOUNDS: return "FA_ERR_BOUNDS: a debug build's kernel refused an out-of-range store";
    }
    return "unknown fa_status";
}

void fa_set_wait_budget_ns(uint64_t ns) { g_budget_ns.store(ns); }

int64_t fa_launch_count(void) { return g_launches.load(); }

void fa_test_arm_fault(int32_t kv_position) { g_fault_pos.store(kv_position < 0 ? -1 : kv_position); }

void fa_test_arm_row_shift(int64_t rows) { g_row_shift.store(rows < 0 ? 0 : rows); }

int32_t fa_debug_flags(void) {
    return (fa::kDebugSerialize ? FA_DEBUG_SERIALIZE_FLAG : 0) |
           (fa::kDebugBounds ? FA_DEBUG_BOUNDS_FLAG : 0);
}

fa_status fa_forward_gqa(const void *Q, const void *K, const void *V, void *O, float *LSE,
                         int64_t B, int64_t H, int64_t H_kv, int64_t N, int64_t d, float scale,
                         fa_mask_mode mask_mode, int64_t window_left, int64_t window_right,
                         fa_dtype dtype, void *stream) {
    Call c{Q, K, V, O, LSE, B, H, H_kv, N, N, d, scale, mask_mode, window_left, window_right,
           dtype, 1, nullptr, 0, stream};
    return run_forward(c);
}

fa_status fa_forward(const void *Q, const void *K, const void *V, void *O, float *LSE, int64_t B,
                     int64_t H, int64_t N, int64_t d, float scale, fa_mask_mode mask_mode,
                     int64_t window_left, int64_t window_right, fa_dtype dtype, void *stream) {
    return fa_forward_gqa(Q, K, V, O, LSE, B, H, H, N, d, scale, mask_mode, window_left,
                          window_right, dtype, stream);
}

size_t fa_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t d,
                                  int64_t num_splits) {
    if (B < 1 || H < 1 || Nq < 1 || d < 1 || num_splits < 1) return 0;
    return splitkv_bytes(B * H * Nq, d, num_splits);
}

int64_t fa_splitkv_default_splits(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk) {
    if (B < 1 || H < 1 || H_kv < 1 || H % H_kv != 0 || Nq < 1 || Nk < 1) return 1;
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess)
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    else
        cudaGetLastError();
    return default_splits(B, H, H_kv, Nq, Nk, sms);
}

fa_status fa_forward_splitkv(const void *Q, const void *K, const void *V, void *O, float *LSE,
                             int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk,
                             int64_t d, float scale, fa_mask_mode mask_mode,
                             int64_t window_left, int64_t window_right, fa_dtype dtype,
                             int64_t num_splits, void *workspace, size_t workspace_bytes,
                             void *stream) {
    if (workspace != nullptr && !aligned32(workspace)) return FA_ERR_INVALID_ARG;
    Call c{Q, K, V, O, LSE, B, H, H_kv, Nq, Nk, d, scale, mask_mode, window_left, window_right,
           dtype, num_splits, workspace, workspace_bytes, stream};
    return run_forward(c);
}

fa_status fa_forward_splitkv_static(const void *Q, const void *K, const void *V, void *O,
                                    float *LSE, int64_t B, int64_t H, int64_t H_kv, int64_t Nq,
                                    int64_t Nk, int64_t d, float scale, fa_mask_mode mask_mode,
                                    int64_t window_left, int64_t window_right, fa_dtype dtype,
                                    int64_t num_splits, void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    StaticScratch &sc = g_static_scratch[dev];
    std::call_once(sc.once, [&sc] {
        void *ptr = nullptr;
        sc.err = cudaGetSymbolAddress(&ptr, g_fa_static_scratch);
        sc.ptr = ptr;
        if (sc.err != cudaSuccess) cudaGetLastError();
    });
    if (sc.err != cudaSuccess || sc.ptr == nullptr) return FA_ERR_CUDA;
    if (num_splits < 1) return FA_ERR_INVALID_ARG;
    if (B >= 1 && H >= 1 && Nq >= 1 && Nk >= 1 && d >= 1 && Nk <= (int64_t{1} << 29)) {
        // The split count the launch will use: at most one split per 128-key tile,
        // and no split left empty by rounding the tiles per split up.
        const int64_t kv_tiles = (Nk + fa::kBN - 1) / fa::kBN;
        const int64_t splits = num_splits < kv_tiles ? num_splits : kv_tiles;
        const int64_t split_tiles = (kv_tiles + splits - 1) / splits;
        const int64_t n_splits = (kv_tiles + split_tiles - 1) / split_tiles;
        if (fa_splitkv_workspace_bytes(B, H, Nq, d, n_splits) > kStaticScratchBytes)
            return FA_ERR_UNSUPPORTED;  // the request needs more than the fixed scratch
    }
    Call c{Q, K, V, O, LSE, B, H, H_kv, Nq, Nk, d, scale, mask_mode, window_left, window_right,
           dtype, num_splits, sc.ptr, kStaticScratchBytes, stream};
    return run_forward(c);
}

fa_status fa_forward_varlen(const void *Q, const void *K, const void *V, void *O, float *LSE,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int64_t B,
                            int64_t H, int64_t H_kv, int64_t total_q, int64_t total_k,
                            int64_t max_seqlen_q, int64_t d, float scale, fa_mask_mode mask_mode,
                            int64_t window_left, int64_t window_right, fa_dtype dtype,
                            void *stream) {
    VarlenCall c{Q, K, V, O, LSE, cu_seqlens_q, cu_seqlens_k, B, H, H_kv, total_q, total_k,
                 max_seqlen_q, d, scale, mask_mode, window_left, window_right, dtype, stream};
    return run_forward_varlen(c);
}

fa_status fa_sync_status(void *stream) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    unsigned int st[4] = {0, 0, 0, 0};
    if (cudaMemcpyFromSymbol(st, g_fa_status, sizeof(st)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    if (st[0] == 0) return FA_OK;
    const unsigned int zero[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_fa_status, zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_CUDA;
    }
    // The kernels store FA_ERR_TIMEOUT, FA_ERR_UNSUPPORTED for a shared-memory
    // layout they cannot use, or (debug builds with bounds checks) FA_ERR_BOUNDS.
    if (st[0] == static_cast<unsigned>(FA_ERR_UNSUPPORTED)) return FA_ERR_UNSUPPORTED;
    if (st[0] == static_cast<unsigned>(FA_ERR_BOUNDS)) return FA_ERR_BOUNDS;
    return FA_ERR_TIMEOUT;
}

}  // extern "C"
