/*
 * fa.h -- C ABI of the GB300 (sm_103a) attention forward library (libfa.so).
 *
 * The operation is the FlashAttention forward pass: for every batch b, head h
 * and query row i,
 *
 *     O[b,h,i,:] = sum_j softmax_j( scale * Q[b,h,i,:] . K[b,h,j,:] + mask(i,j) ) V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp( scale * Q[b,h,i,:] . K[b,h,j,:] + mask(i,j) )
 *
 * with mask(i,j) = 0 for a visible key and -inf for a hidden one. It follows
 * the definition S = QK^T/sqrt(d), P = softmax(S), O = PV of
 * "ai6s.net/6af30f4d40858c2d8819b6d5" §1 with the scale as a parameter, is
 * computed tile by tile with the online-softmax recurrence of §2.2-§2.3 of the
 * same page (running max m, running sum l, rescale of the output accumulator),
 * and writes the saved statistics of §2.4 as one log-sum-exp per row
 * (LSE = m + ln l, natural log, in units of the scaled logits). The three mask
 * variants are those of the (None | causal | (window_left, window_right))
 * attn_mask argument in "ai6s.net/6a0ed07b662f9a54cb761aa2", section
 * "使用：ops-transformer 怎么调 FlashAttention"; the B x H x S x D layout is the
 * one of "aicoding.csdn.net/6a69d3ff10ee7a33f2941f44", table "显存占用计算".
 *
 * All entry points are thread-safe for distinct streams and never throw.
 */
#ifndef TILED_ATTENTION_FA_H
#define TILED_ATTENTION_FA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* a null/misaligned/aliased pointer, a bad size or enum, a bad scale */
    FA_ERR_UNSUPPORTED = 2, /* a valid request this build does not implement (head dim, device) */
    FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed (launch, attribute, tensor map) */
    FA_ERR_TIMEOUT = 4,     /* a bounded in-kernel wait ran out (reported by fa_sync_status) */
    FA_ERR_BOUNDS = 5       /* debug builds only: a kernel refused an out-of-range store
                               (reported by fa_sync_status) */
} fa_status;

typedef enum {
    FA_MASK_NONE = 0,   /* every key 0..N-1 is visible */
    FA_MASK_CAUSAL = 1, /* key j visible to query i iff j <= i */
    FA_MASK_WINDOW = 2  /* key j visible to query i iff i - window_left <= j <= i + window_right */
} fa_mask_mode;

typedef enum { FA_DTYPE_FP16 = 0, FA_DTYPE_BF16 = 1 } fa_dtype;

/*
 * fa_forward -- enqueue one attention forward pass on `stream`.
 *
 * Q, K, V : device pointers, contiguous B x H x N x d tensors of `dtype`
 *           (row-major: d fastest, then N, then H, then B). Read only.
 * O       : device pointer, contiguous B x H x N x d of `dtype`. Written with
 *           O/l rounded to nearest-even. Must not overlap Q, K, V or LSE.
 * LSE     : device pointer, contiguous B x H x N float32. Written.
 * B, H, N : >= 1. Any N is accepted (no padding is required of the caller;
 *           rows and keys past N are handled inside the kernel).
 * d       : head dimension: 32, 64, 128 or 256 (else FA_ERR_UNSUPPORTED), in every
 *           forward call. d = 256 runs on a kernel with one 128-row Q tile per unit,
 *           as do d = 64 and 128 when a head's queries, or the queries of one K/V
 *           head's query heads, fit in one tile, and small unsplit problems (whose
 *           256-row units would fill at most half of the SMs). fa_backward takes
 *           32, 64, 128 and 256, and so does fa_backward_varlen.
 * scale   : multiplier of the logits, finite and > 0 (typically 1/sqrt(d)).
 * mask_mode, window_left, window_right : see fa_mask_mode. The window
 *           arguments are read only for FA_MASK_WINDOW and must then be >= 0
 *           (values >= N act as N). Every query sees at least itself.
 * dtype   : element type of Q, K, V and O; the products are exact and every
 *           sum, max, exponent and the accumulator are float32.
 * stream  : a cudaStream_t (NULL = the legacy default stream).
 *
 * Ownership: every pointer is owned by the caller; the library keeps none and
 * allocates no device memory per call. Q, K and V must be 16-byte aligned
 * (they are read by tensor-memory-access copies), O 32-byte aligned (each row is
 * written with 32-byte vector stores); LSE, accessed one float at a time, 4-byte
 * aligned. All on the current device; a pointer that breaks one of these rules is
 * FA_ERR_INVALID_ARG.
 *
 * Errors: arguments are checked before anything is enqueued; an invalid call
 * returns FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED and launches nothing. A
 * launch failure returns FA_ERR_CUDA. The call is asynchronous: a device-side
 * timeout of a bounded wait is reported by a later fa_sync_status().
 */
fa_status fa_forward(const void *Q, const void *K, const void *V, void *O, float *LSE,
                     int64_t B, int64_t H, int64_t N, int64_t d, float scale,
                     fa_mask_mode mask_mode, int64_t window_left, int64_t window_right,
                     fa_dtype dtype, void *stream);

/*
 * fa_forward_gqa -- fa_forward with grouped K/V heads (GQA; MQA when H_kv = 1),
 * the "GQA/MQA" adaptation that "ai6s.net/6af30f4d40858c2d8819b6d5" §5 lists
 * among the practical variants. K and V are contiguous B x H_kv x N x d; query
 * head h of batch b attends with K/V head h / (H / H_kv) of batch b. H_kv must
 * divide H (else FA_ERR_INVALID_ARG). Q, O, LSE, every other argument,
 * ownership and errors are as for fa_forward, which equals this call with
 * H_kv = H.
 */
fa_status fa_forward_gqa(const void *Q, const void *K, const void *V, void *O, float *LSE,
                         int64_t B, int64_t H, int64_t H_kv, int64_t N, int64_t d, float scale,
                         fa_mask_mode mask_mode, int64_t window_left, int64_t window_right,
                         fa_dtype dtype, void *stream);

/*
 * fa_forward_splitkv -- attention with the keys of every head cut into
 * `num_splits` contiguous chunks that are processed in parallel and merged
 * (the split variant of FlashAttention for few queries and many keys, the
 * "Flash Decoding" that "ai6s.net/6af30f4d40858c2d8819b6d5" §5 names). Each
 * chunk yields its own normalised output and log-sum-exp; the merge is
 * LSE = ln sum_s exp(LSE_s), O = sum_s exp(LSE_s - LSE) O_s.
 *
 * Q, O: contiguous B x H x Nq x d; K, V: contiguous B x H_kv x Nk x d; LSE:
 * B x H x Nq float32. Nq and Nk may differ: query i stands at key position
 * i + Nk - Nq (the queries are the last Nq positions, as when decoding), which
 * is what the causal and window masks refer to; masks require Nq <= Nk.
 * num_splits >= 1 (values above the number of 128-key tiles act as that
 * number; fa_splitkv_default_splits suggests one). The result equals
 * fa_forward_gqa's up to rounding.
 *
 * workspace: device memory owned by the caller, 32-byte aligned, at least
 * fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits) bytes, not overlapping
 * the other buffers; its contents are scratch (fp32 partial results) and are
 * overwritten. With num_splits = 1 it is not used (it may then be NULL).
 * Two kernels are enqueued: the split attention and the merge.
 * Errors as for fa_forward, plus FA_ERR_INVALID_ARG for a missing or short
 * workspace, num_splits < 1, or a mask with Nq > Nk.
 */
fa_status fa_forward_splitkv(const void *Q, const void *K, const void *V, void *O, float *LSE,
                             int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk,
                             int64_t d, float scale, fa_mask_mode mask_mode,
                             int64_t window_left, int64_t window_right, fa_dtype dtype,
                             int64_t num_splits, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Workspace bytes fa_forward_splitkv needs (0 for invalid sizes). */
size_t fa_splitkv_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t d,
                                  int64_t num_splits);

/* A split count that fills the current device in one wave: 1 when the query
 * blocks alone give at least one unit per SM, otherwise as many splits as the
 * SMs hold next to those units, each keeping at least four 128-key tiles
 * (1 for invalid sizes). */
int64_t fa_splitkv_default_splits(int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk);

/*
 * fa_forward_splitkv_static -- fa_forward_splitkv without a caller workspace,
 * for callers that cannot allocate device memory: runtimes that reserve all of
 * their device memory up front and forbid later allocations (to rule out
 * fragmentation or an out-of-memory failure in the middle of serving), and
 * plug-in hosts that give the library no allocator. The pages have no
 * counterpart: this is an interface choice of this library.
 *
 * The scratch is one fixed array of FA_SPLITKV_STATIC_SCRATCH_BYTES bytes in
 * device memory, part of the library: every GPU that loads the library holds
 * it until the process exits, and this call allocates nothing. Requests whose
 * fa_splitkv_workspace_bytes(B, H, Nq, d, n) exceeds that size are rejected
 * with FA_ERR_UNSUPPORTED before anything is enqueued (use fewer splits, or
 * fa_forward_splitkv with a workspace); n is the split count the call runs,
 * num_splits clamped to the number of 128-key tiles (and lowered further when
 * rounding the tiles per split up leaves a split empty). num_splits >= 1.
 *
 * All calls on a device share the one array and leave their partial results
 * in it; nothing in it needs to start at zero. Calls whose kernels overlap on
 * the GPU (for example on two streams at once) race on the array: order them
 * on one stream, or synchronise between them. The first call on each device
 * looks up the array's device address (with that device current); make that
 * first call before any stream capture. Everything else -- arguments, layout,
 * masks, results and errors -- is as for fa_forward_splitkv.
 */
#define FA_SPLITKV_STATIC_SCRATCH_BYTES (16u << 20)
fa_status fa_forward_splitkv_static(const void *Q, const void *K, const void *V, void *O,
                                    float *LSE, int64_t B, int64_t H, int64_t H_kv, int64_t Nq,
                                    int64_t Nk, int64_t d, float scale, fa_mask_mode mask_mode,
                                    int64_t window_left, int64_t window_right, fa_dtype dtype,
                                    int64_t num_splits, void *stream);

/*
 * fa_forward_varlen -- attention forward over a batch of sequences of different
 * lengths packed back to back (the variable-length batches that
 * "ai6s.net/6af30f4d40858c2d8819b6d5" §4.2 lists among the cases an
 * implementation has to handle). Sequence b owns query tokens
 * cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and keys cu_seqlens_k[b] ..
 * cu_seqlens_k[b+1]-1; each sequence is an independent fa_forward_gqa problem
 * whose L_q queries stand at its last L_q key positions (as in
 * fa_forward_splitkv), which is what the masks refer to.
 *
 * Layout (token-major): Q and O total_q x H x d, K and V total_k x H_kv x d, in
 * `dtype`; LSE total_q x H float32; cu_seqlens_q and cu_seqlens_k are B + 1
 * int32 on the device, non-decreasing from 0 to total_q / total_k. All on the
 * current device; Q, K, V 16-byte aligned, O 32-byte, LSE 4-byte. max_seqlen_q >= every L_q (rows
 * past it are not computed). With a mask, every sequence needs L_q <= L_k;
 * every sequence with queries needs L_k >= 1. The device arrays are read by
 * the kernel, not checked on the host; offsets are clamped to the tensors, so
 * inconsistent arrays give wrong results but no access outside them.
 *
 * Errors: as fa_forward. total_q = 0 or max_seqlen_q = 0 returns FA_OK with
 * nothing read, written or enqueued (the pointers may then be NULL).
 */
fa_status fa_forward_varlen(const void *Q, const void *K, const void *V, void *O, float *LSE,
                            const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int64_t B,
                            int64_t H, int64_t H_kv, int64_t total_q, int64_t total_k,
                            int64_t max_seqlen_q, int64_t d, float scale, fa_mask_mode mask_mode,
                            int64_t window_left, int64_t window_right, fa_dtype dtype,
                            void *stream);

/*
 * fa_forward_host -- the forward pass of fa_forward_splitkv over HOST buffers:
 * the inputs are copied to the device, processed and the results copied back,
 * in chunks (one batch entry and a range of K/V heads with their query heads,
 * about chunk_bytes of Q + K + V each; chunk_bytes <= 0 takes 64 MiB). The copy
 * in of chunk c+1, the kernel on chunk c and the copy out of chunk c-1 overlap:
 * the copies run on two streams of the library's own (created once per device),
 * the kernels on `stream`. So only the first copy in and the last copy out are
 * not hidden behind other work.
 *
 * Q, K, V, O, LSE: host memory (page-locked memory makes the copies
 * asynchronous; pageable memory works, with the host waiting on each copy), in
 * the layout of fa_forward_splitkv; O and LSE overlap no input. `workspace`:
 * device memory owned by the caller, 32-byte aligned, at least
 * fa_forward_host_workspace_bytes(...) bytes with the same sizes, num_splits and
 * chunk_bytes; it holds the device copies. num_splits: 0 runs Nq == Nk
 * unsplit and Nq < Nk with fa_splitkv_default_splits per chunk; n >= 1 runs
 * every chunk with n key splits.
 *
 * The call enqueues everything and returns; `stream` then waits for the last
 * copy out, so a stream synchronize (or fa_sync_status(stream)) means O and LSE
 * are in host memory. The host buffers must stay valid until then, and the
 * workspace must not be reused meanwhile. Calls on one device are enqueued one
 * at a time (a lock), so concurrent callers stay correct.
 *
 * Errors: every argument is checked before anything is enqueued (as fa_forward,
 * plus: a device pointer among Q, K, V, O, LSE, or a workspace that is not
 * device memory or is too small, is FA_ERR_INVALID_ARG). A CUDA failure while
 * enqueueing returns FA_ERR_CUDA.
 */
size_t fa_forward_host_workspace_bytes(int64_t B, int64_t H, int64_t H_kv, int64_t Nq,
                                       int64_t Nk, int64_t d, int64_t num_splits,
                                       int64_t chunk_bytes);
fa_status fa_forward_host(const void *Q, const void *K, const void *V, void *O, float *LSE,
                          int64_t B, int64_t H, int64_t H_kv, int64_t Nq, int64_t Nk, int64_t d,
                          float scale, fa_mask_mode mask_mode, int64_t window_left,
                          int64_t window_right, fa_dtype dtype, int64_t num_splits,
                          int64_t chunk_bytes, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * fa_backward -- gradients of the forward pass: given Q, K, V, the forward's
 * O and LSE (as fa_forward / fa_forward_gqa wrote them) and dO, the gradient
 * of a loss with respect to O, writes dQ, dK and dV. The forward keeps only O
 * and the row statistics; like the method of "ai6s.net/6af30f4d40858c2d8819b6d5"
 * §2.4 ("重计算(Recomputation)与反向传播"), this call recomputes the scores and
 * probabilities tile by tile from them instead of storing P. With
 * D_i = sum_c dO_ic O_ic and P_ij = exp(scale q_i.k_j - LSE_i) on visible keys:
 *   dV_j = sum_i P_ij dO_i,  dS_ij = P_ij (dO_i . V_j - D_i),
 *   dQ_i = scale sum_j dS_ij K_j,  dK_j = scale sum_i dS_ij Q_i,
 * dK and dV of a K/V head summing over every query head that reads it.
 *
 * Layout: Q, O, dO and dQ are contiguous B x H x N x d; K, V, dK and dV are
 * B x H_kv x N x d (H_kv divides H); LSE is B x H x N float32; all in `dtype`
 * except LSE, on the current device; Q, K, V, O and dO 16-byte aligned, dQ, dK and
 * dV 32-byte aligned (32-byte vector stores), LSE 4-byte. Queries and keys share
 * positions (as in fa_forward); the mask arguments are those of fa_forward.
 * `workspace` is caller-owned device memory of at least
 * fa_backward_workspace_bytes(B, H, N, d) bytes (two fp32 row terms per query
 * row), 32-byte aligned; its contents on entry do not matter. dQ, dK, dV and
 * the workspace overlap no input and no other output. The results are
 * deterministic: no atomics, fixed summation order.
 *
 * d is 32, 64, 128 or 256. At d = 256 each gradient has its own pass (a 128 x 256
 * tile of each operand and both accumulators do not fit one SM's shared and
 * tensor memory): four launches (row terms, dV, dK, dQ) instead of three.
 *
 * Errors: as fa_forward, plus FA_ERR_INVALID_ARG for a missing or small
 * workspace. Asynchronous on `stream` (three kernel launches: row terms, dK/dV,
 * dQ; four at d = 256); timeouts are reported by fa_sync_status.
 */
fa_status fa_backward(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                      const float *LSE, void *dQ, void *dK, void *dV, int64_t B, int64_t H,
                      int64_t H_kv, int64_t N, int64_t d, float scale, fa_mask_mode mask_mode,
                      int64_t window_left, int64_t window_right, fa_dtype dtype, void *workspace,
                      size_t workspace_bytes, void *stream);

/* Workspace bytes fa_backward needs (0 for invalid sizes). */
size_t fa_backward_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t d);

/*
 * fa_backward_varlen -- fa_backward for a variable-length batch laid out as in
 * fa_forward_varlen (token-major; sequence b owns query tokens cu_seqlens_q[b]
 * .. cu_seqlens_q[b+1]-1 and keys cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1, its
 * queries at its last key positions). O and LSE are fa_forward_varlen's
 * outputs; dO and dQ are total_q x H x d, dK and dV total_k x H_kv x d.
 * max_seqlen_q / max_seqlen_k bound every sequence's lengths. Gradients of
 * keys that no query sees, and of queries that see no key, are zero.
 * `workspace`: fa_backward_varlen_workspace_bytes(B, H, total_q) bytes, 32-byte
 * aligned; pointer alignment as in fa_backward. d is 32, 64, 128 or 256.
 * Deterministic. Errors as fa_backward; the device arrays are clamped to the
 * tensors, as in fa_forward_varlen. Asynchronous on `stream`: three zero-fills
 * of dQ, dK and dV, then four kernel launches (padded row offsets, row terms,
 * dK/dV, dQ), five at d = 256 (one pass per gradient).
 */
fa_status fa_backward_varlen(const void *Q, const void *K, const void *V, const void *O,
                             const void *dO, const float *LSE, const int32_t *cu_seqlens_q,
                             const int32_t *cu_seqlens_k, void *dQ, void *dK, void *dV, int64_t B,
                             int64_t H, int64_t H_kv, int64_t total_q, int64_t total_k,
                             int64_t max_seqlen_q, int64_t max_seqlen_k, int64_t d, float scale,
                             fa_mask_mode mask_mode, int64_t window_left, int64_t window_right,
                             fa_dtype dtype, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Workspace bytes fa_backward_varlen needs (0 for invalid sizes). */
size_t fa_backward_varlen_workspace_bytes(int64_t B, int64_t H, int64_t total_q);

/* Static, NUL-terminated description of a status code. Never NULL. */
const char *fa_status_string(fa_status status);

/*
 * fa_sync_status -- synchronise `stream`, then read and clear the device
 * status word of the current device. Returns FA_ERR_TIMEOUT if any kernel
 * since the last call gave up on a bounded wait, FA_ERR_UNSUPPORTED if a
 * kernel reported a shared-memory layout it cannot use (it then did
 * nothing), FA_ERR_CUDA if the synchronisation itself failed, else FA_OK.
 */
fa_status fa_sync_status(void *stream);

/*
 * fa_set_wait_budget_ns -- upper bound, in nanoseconds of GPU global time, of
 * every in-kernel wait of later launches (default 2e9, or the value of the
 * environment variable FA_WAIT_BUDGET_MS read at the first call). 0 restores
 * the default. Process-wide.
 */
void fa_set_wait_budget_ns(uint64_t ns);

/* Number of kernels this library has launched in this process. */
int64_t fa_launch_count(void);

/*
 * fa_test_arm_fault -- test hook for the failure path. The next launch of this
 * process (only that one) makes every CTA skip the TMA load of K at its K/V
 * ring position `kv_position` (counted from 0 over that CTA's work; position 0
 * exists in every CTA that gets any work). Its MMA warp then waits for data
 * that never arrives: the wait runs out after the wait budget, every role of
 * the kernel gives up, drains its copies and MMAs, frees its tensor memory and
 * returns, and fa_sync_status reports FA_ERR_TIMEOUT. The GPU context stays
 * usable. A negative position disarms the hook. When the next call is
 * fa_backward or fa_backward_varlen, the position counts units instead: every
 * CTA of its dK/dV kernel skips the K/V load of its unit number
 * `kv_position`, with the same outcome.
 */
void fa_test_arm_fault(int32_t kv_position);

/*
 * Debug builds. The library can be compiled with two checks that release builds
 * leave out (tiled_attention_03_gb300/build.py, debug="serialize" / "bounds"); the
 * pages have no counterpart, they are aids for changing the kernels. They apply
 * to the two-tile forward kernel (every forward at d = 32, and at d = 64 / 128
 * unless the one-tile kernel runs it).
 *  - FA_DEBUG_SERIALIZE: the kernel runs with the least overlap its protocol
 *    allows (K/V rings two deep, the next unit claimed with the current unit's
 *    last K/V tile, every group of matrix products completed before the next is
 *    issued), so that an ordering mistake shows as a wrong result or a timeout.
 *  - FA_DEBUG_BOUNDS: every store of O, LSE and the split buffers is checked
 *    against the output first; an out-of-range row is not stored, and the first
 *    one is recorded in the status word, which fa_sync_status then reports as
 *    FA_ERR_BOUNDS, instead of a memory fault.
 * fa_debug_flags returns which checks the loaded library has (0 in release builds).
 * fa_test_arm_row_shift(rows) is the test hook of the bounds check: the next
 * two-tile forward launch adds `rows` to every row it stores, so that rows at or
 * past the end of the output are refused and reported. Release builds ignore the
 * shift.
 */
#define FA_DEBUG_SERIALIZE_FLAG 1
#define FA_DEBUG_BOUNDS_FLAG 2
int32_t fa_debug_flags(void);
void fa_test_arm_row_shift(int64_t rows);

#ifdef __cplusplus
}
#endif

#endif /* TILED_ATTENTION_FA_H */
