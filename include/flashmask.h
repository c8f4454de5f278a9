/*
 * flashmask.h -- C ABI of libflashmask: exact masked attention with a
 * column-wise sparse mask, forward and backward, on one sm_103a GPU.
 *
 * Method (FlashMask README, "Formulation"):
 *     O = softmax(Q K^T * scale + M) V,      scale = 1/sqrt(d) by default,
 * d is the head dim of Q and K; V may have its own head dim dv.
 *
 * Mask (FlashMask README, "Overview"; FlashMask-3 abstract): for every key
 * column j, four int32 query-row boundaries LTS_j, LTE_j, UTS_j, UTE_j.
 * Query row i is masked in column j (M_ij = -inf) when
 *     LTS_j <= i < LTE_j   or   UTS_j <= i < UTE_j   or   (causal and i < j).
 * Boundaries are clamped to [0, N], which does not change the mask; start >= end
 * is an empty interval.  A NULL pair (both pointers NULL) is an empty interval;
 * exactly one NULL pointer of a pair is an error.
 *
 * Sparsity skipping ("FlashMask: Efficient and Rich Mask Extension of
 * FlashAttention", abstract): 128 x 128 tiles whose elements are all masked are
 * never computed, and the result is exact.
 *
 * Conventions shared by every entry point:
 *   - Device pointers are owned by the caller.  The library never allocates,
 *     frees or synchronises, except flashmask_get_error, which synchronises
 *     its stream.
 *   - An entry point makes the device that owns the caller's memory current
 *     for its own launches (flashmask_get_error: the stream's device) and,
 *     before it returns, makes the calling thread's previous context current
 *     again: the caller's current device is unchanged.
 *   - Work is enqueued on `stream` (a cudaStream_t, NULL = legacy default
 *     stream), and the call returns at once.
 *   - Errors are returned as fm_status; nothing is thrown and nothing is
 *     printed.
 *   - Layouts, row-major and contiguous:
 *       q, k: [B, N, H, d] bf16;  v, o, dout, dv: [B, N, H, dv] bf16;
 *       dq, dk: [B, N, H, d] bf16;  lse: [B, H, N] fp32 (natural log);
 *       mask vectors: [B, Hm, N] int32 with Hm in {1, H}.  Hm = 1 shares one
 *       mask among all heads; otherwise head h uses mask head h.
 *   - Pointers must be 16-byte aligned.
 *   - Rows whose every key is masked give O = 0 and LSE = -inf, and they add
 *     nothing to any gradient.
 *   - Supported (d, dv): (64, 64), (128, 128), (192, 128), (256, 256).
 *   - Nq = Nk = N.  1 <= N <= 2^24.
 */
#ifndef FLASHMASK_H
#define FLASHMASK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FM_OK = 0,
    FM_ERR_INVALID_ARG = 1,     /* NULL/unaligned pointer, bad size or flag        */
    FM_ERR_UNSUPPORTED = 2,     /* (d, dv) pair or device not supported            */
    FM_ERR_WORKSPACE = 3,       /* workspace NULL, unaligned or smaller than needed */
    FM_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed               */
    FM_ERR_DEVICE_TIMEOUT = 5,  /* a kernel gave up on a bounded wait              */
    FM_ERR_DEVICE_BOUNDS = 6    /* debug_bounds: a kernel found its work list out of
                                 * range (for example a stale reused tile map)     */
} fm_status;

/* Problem shape.  scale <= 0 selects the default 1/sqrt(d). */
typedef struct {
    int B, H, Hm, N, d, dv;
    float scale;
    int causal;
} fm_problem;

/* Options.  deterministic: the backward adds every partial sum in a fixed
 * order, so dQ/dK/dV are bit-identical from run to run (without it, at
 * d = dv <= 128, dQ is summed over key tiles with fp32 reductions whose order
 * varies, and its last bits with it).  wait_timeout_ns
 * bounds every wait on the device; 0 selects 1 s.
 * debug_bounds (0 or 1): before the attention kernels, a check kernel reads
 * every work list in the workspace: each list's length must lie in [0, T]
 * and each of its tile indices in [0, T), T = ceil(N / 128), and each entry
 * of the forward's pair order in [0, ceil(T / 2)).  A list that fails is
 * emptied (length 0) and an order entry that fails is replaced by a valid
 * one, so no kernel after it reads out of range; flashmask_get_error then
 * returns FM_ERR_DEVICE_BOUNDS, and the outputs are not meaningful.  The
 * lists the library builds itself always pass (results are bit-identical
 * with and without the check); it is meant for workspaces reused with
 * reuse_tile_map.  kernel_events do not record the check kernel.
 * sink (optional, may be NULL): per-head attention-sink logits, [H] fp32 on
 * the device (FlashMask README, "News", names sink bias without a formula;
 * reading taken): head h's logit joins every row's softmax denominator as a
 * term exp(sink[h]) that carries no value, so
 *     O_i = sum_j exp(s_ij) v_j / (exp(sink[h]) + sum_j exp(s_ij)),
 *     LSE_i = log(exp(sink[h]) + sum_j exp(s_ij));
 * a row whose keys are all masked gets O = 0 and LSE = sink[h].  Pass the same
 * logits to flashmask_fwd and flashmask_bwd.
 * dsink (optional, flashmask_bwd only, may be NULL): [H] fp32 on the device,
 * receives the gradient of the sink logits, -sum_i exp(sink[h] - LSE_i) D_i
 * over the batch and rows of head h (D_i = sum_c dO_ic O_ic), summed in a
 * fixed order.  With a sink, a sink-gradient kernel runs after the preprocess
 * kernel; kernel_events do not record it.
 * reuse_tile_map (0 or 1): the workspace already holds the tile map and tile
 * lists of this very problem and mask, written by an earlier flashmask_fwd or
 * flashmask_bwd on the same workspace (every call writes all of them), and
 * the call skips the classify and lists kernels (kernel_events then start at
 * the next kernel).  A forward and the backward of one layer, or layers that
 * share one mask, can share them this way; the workspace must then be sized
 * for the backward (is_bwd = 1) in every call, since the backward's own parts
 * follow the shared ones.  The library cannot check that the contents match:
 * stale contents give wrong results.
 * kernel_events (optional, may be NULL): an array of n_kernel_events
 * cudaEvent_t handles owned by the caller.  The call records
 * kernel_events[2i] on `stream` just before its i-th kernel launch and
 * kernel_events[2i+1] just after it.  Events beyond the array are skipped.
 * Kernel order: fwd = classify, lists, attention.  bwd = classify, lists,
 * the preprocess step, then: without the deterministic mode at d = dv <= 128,
 * the one-pass gradient kernel (dK, dV, and dQ sums in fp32) and the dQ
 * conversion; otherwise one launch of the key-side and query-side gradient
 * kernels (at d = dv = 256 after a separate dV pass of the key side).  The
 * preprocess step is three launches under one event pair: the largest |dO|
 * and |V| per row tile, their per-(batch, head) scales, then D, the log2 LSE
 * and the scaled fp16 copies of dO (and of V for the split kernels).
 * accumulate_f32 (0 or 1, flashmask_bwd only): dq, dk and dv are fp32 arrays
 * of the same shapes ([B,N,H,d], [B,N,H,d], [B,N,H,dv]), and the backward adds
 * its gradients to them in fp32 instead of writing bf16 (each element is
 * read and written once, by one thread; no atomics).  Partial gradients of
 * several calls, such as the (query chunk, key chunk) pairs of a context-
 * parallel run, are then summed before a single rounding to bf16.
 * debug_drop_load (>= 0; 0 = off; failure-detection tests only): with k > 0
 * the forward kernel at d <= 128 never issues the k-th key-tile load of each
 * CTA, so the waits for it run out after wait_timeout_ns: the CTA stops, waits
 * for its own loads and MMAs already in flight, frees its tensor memory and
 * returns; flashmask_get_error then reports FM_ERR_DEVICE_TIMEOUT and the
 * outputs are not meaningful.  No memory is touched out of place.
 * A NULL options pointer selects all defaults. */
typedef struct {
    int deterministic;
    int debug_bounds;
    unsigned long long wait_timeout_ns;
    void **kernel_events;
    int n_kernel_events;
    const float *sink;
    float *dsink;
    int reuse_tile_map;
    int accumulate_f32;
    int debug_drop_load;
} fm_options;

/* Tile classes written by flashmask_classify (128 x 128 tiles). */
#define FM_TILE_SKIP 0      /* every in-range element masked */
#define FM_TILE_PARTIAL 1   /* some, not all, masked         */
#define FM_TILE_UNMASKED 2  /* no element masked             */

/*
 * Bytes of device workspace that flashmask_fwd (is_bwd = 0),
 * flashmask_bwd (is_bwd = 1), flashmask_classify and flashmask_count_unmasked
 * need for this problem.  Returns 0 for an invalid problem.
 * The workspace must be 256-byte aligned.
 */
size_t flashmask_workspace_size(const fm_problem *p, const fm_options *opt, int is_bwd);

/*
 * Forward (FlashMask README, "Formulation").  Writes o [B,N,H,dv] bf16 and
 * lse [B,H,N] fp32, with LSE_i = log sum_j exp(scale q_i.k_j + M_ij).
 * Tiles that are fully masked are skipped, and the mask is applied only on
 * partial tiles.
 */
fm_status flashmask_fwd(const fm_problem *p, const fm_options *opt,
                        const void *q, const void *k, const void *v,
                        const int32_t *lts, const int32_t *lte,
                        const int32_t *uts, const int32_t *ute,
                        void *o, float *lse,
                        void *workspace, size_t ws_bytes, void *stream);

/*
 * Backward, the derivative of the forward above.  P is rebuilt from lse.
 * o and lse must be the forward's outputs for the same inputs.  dout has the
 * layout of o.  Writes dq, dk [B,N,H,d] and dv [B,N,H,dv] bf16.  These are the
 * gradients of sum(dout * O) with respect to q, k and v (with
 * fm_options.accumulate_f32: fp32 arrays that the gradients are added to).
 * Accuracy holds over the whole bf16 range of dout and v: the products with
 * dout and v run in fp16 (more mantissa than bf16) on copies scaled by a power
 * of two per (batch, head) that puts the largest magnitude in [2^14, 2^15),
 * and the scales are undone in fp32.  Scales are limited to 2^-63 .. 2^63, so
 * magnitudes below about 2^-49 lose fp16 precision; products and sums are
 * formed in fp32.
 */
fm_status flashmask_bwd(const fm_problem *p, const fm_options *opt,
                        const void *q, const void *k, const void *v,
                        const void *o, const float *lse, const void *dout,
                        const int32_t *lts, const int32_t *lte,
                        const int32_t *uts, const int32_t *ute,
                        void *dq, void *dk, void *dv,
                        void *workspace, size_t ws_bytes, void *stream);

/*
 * Tile map (the sparsity-skipping step of the FlashMask abstract).  Writes
 * tile_class [B*Hm, T, T] uint8 with T = ceil(N/128).  Entry [bm, qt, kt]
 * gives the class of query rows [128 qt, 128 qt + 128) and key columns
 * [128 kt, 128 kt + 128), counting only elements inside [0, N).
 */
fm_status flashmask_classify(const fm_problem *p,
                             const int32_t *lts, const int32_t *lte,
                             const int32_t *uts, const int32_t *ute,
                             uint8_t *tile_class,
                             void *workspace, size_t ws_bytes, void *stream);

/*
 * Number of unmasked (i, j) pairs of each mask head, summed over all columns.
 * Writes counts [B*Hm] uint64 (device memory).  This is the work the
 * effective-FLOP figures count.
 */
fm_status flashmask_count_unmasked(const fm_problem *p,
                                   const int32_t *lts, const int32_t *lte,
                                   const int32_t *uts, const int32_t *ute,
                                   unsigned long long *counts, void *stream);

/*
 * Synchronises `stream`, then reads and clears the library's device error
 * words.  Since the last call: FM_ERR_DEVICE_BOUNDS if a kernel found its
 * work list out of range (debug_bounds), else FM_ERR_DEVICE_TIMEOUT if a
 * kernel gave up on a bounded wait.  FM_ERR_CUDA if the stream itself
 * failed, else FM_OK.
 */
fm_status flashmask_get_error(void *stream);

/*
 * Failure-detection self-test.  Enqueues on `stream` a one-thread kernel that
 * waits, through the same bounded wait every kernel of the library uses, on
 * an mbarrier phase that nothing completes.  After timeout_ns nanoseconds the
 * wait gives up, records a timeout in the device error word and the kernel
 * returns, so the next flashmask_get_error reports FM_ERR_DEVICE_TIMEOUT and
 * the context stays usable.  0 < timeout_ns <= 10 s, else FM_ERR_INVALID_ARG.
 */
fm_status flashmask_selftest_wait(unsigned long long timeout_ns, void *stream);

/*
 * Forward without a workspace, for callers that cannot allocate device memory
 * (a host that only hands out its own tensors, code where cudaMalloc is not
 * allowed or would stall, an embedding with no allocator).  It computes
 * exactly what flashmask_fwd computes; the paper has no counterpart of this
 * entry point.  Its scratch is a fixed array of FM_NOALLOC_SCRATCH_BYTES
 * inside the library, held by every GPU that loads it until the process exits.
 *  - Problems whose forward workspace (flashmask_workspace_size, is_bwd = 0)
 *    exceeds FM_NOALLOC_SCRATCH_BYTES are rejected with FM_ERR_WORKSPACE, and
 *    flashmask_last_error_detail says why.
 *  - fm_options.reuse_tile_map must be 0 (else FM_ERR_INVALID_ARG, before any
 *    CUDA call): the array may hold the tile map of another problem.  The
 *    other options (deterministic, debug_bounds, wait_timeout_ns,
 *    kernel_events, sink) act as in flashmask_fwd.
 *  - The first call on a device looks up the array's device address (a
 *    cudaGetSymbolAddress with that device current), and so does the first
 *    call after a cudaDeviceReset of it; make that first call before any
 *    stream capture.  A failed lookup returns FM_ERR_CUDA and is retried on
 *    the next call.
 *  - All calls on a device share the array.  Calls that overlap on the GPU
 *    race and give wrong results; order them on one stream.  Every call
 *    rewrites what it reads, so nothing in the array needs clearing.
 *  - The device is the one that owns q.  Allocates nothing and frees nothing.
 */
#define FM_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
fm_status flashmask_fwd_noalloc(const fm_problem *p, const fm_options *opt,
                                const void *q, const void *k, const void *v,
                                const int32_t *lts, const int32_t *lte,
                                const int32_t *uts, const int32_t *ute,
                                void *o, float *lse, void *stream);

/*
 * Context-parallel chunks on one GPU ("FlashMask-3: Efficient and Expressive
 * Mask-Aware Distributed Attention", abstract: under any multi-chunk
 * context-parallel assignment, per-rank mask localization is a
 * zero-communication clip-shift-max on the boundary vectors, compatible with
 * the single-GPU kernel).  The sequence is cut into chunks of `len` rows and
 * keys starting at multiples of `len`; every (query chunk, key chunk) pair is
 * a local problem of size len that runs through flashmask_fwd / flashmask_bwd,
 * and a query chunk's partial results are merged by log-sum-exp.
 */

/*
 * Local boundary vectors of the pair (query chunk at row q0, key chunk at key
 * k0): for local key j' = j - k0, every boundary x of column j, clamped to
 * [0, N], becomes  x' = max(min(x, q0 + len) - q0, 0)  (clip to the query
 * chunk, shift by its start, max with 0).  *local_causal receives the causal
 * flag of the local problem: 1 on the diagonal pair (q0 == k0) of a causal
 * mask, 0 when the mask is not causal or the key chunk lies before the query
 * chunk, and -1 when it is causal and the key chunk lies after the query chunk:
 * then every element is masked, the pair is to be skipped and nothing is
 * written or enqueued.
 *  - In: the problem's B, Hm, H, N and causal (other fields unused); global
 *    vectors [B, Hm, N] int32 (a NULL pair is an empty interval).
 *  - Out: four [B, Hm, len] int32 device arrays (absent intervals are written
 *    empty).  Requires 1 <= len, 0 <= q0, k0 <= N - len, (q0 - k0) % len == 0;
 *    else FM_ERR_INVALID_ARG.
 */
fm_status flashmask_localize(const fm_problem *p, const int32_t *lts, const int32_t *lte,
                             const int32_t *uts, const int32_t *ute, int q0, int k0, int len,
                             int32_t *out_lts, int32_t *out_lte, int32_t *out_uts,
                             int32_t *out_ute, int *local_causal, void *stream);

/*
 * Log-sum-exp merge of one query chunk's partial results.  A chunk of one
 * batch: O [L, H, dv] (the rows q0 .. q0 + L - 1 of a [1, N, H, dv] tensor, or a
 * local problem's output), LSE [H, L]; running values o_acc [L, H, dv] fp32
 * and lse_acc [H, L] fp32.  dv a multiple of 8; O pointers 16-byte aligned.
 *  - merge_init: o_acc = 0, lse_acc = -inf.
 *  - merge: lse = log(exp(lse_acc) + exp(lse_part)),
 *           o_acc = o_acc * exp(lse_acc - lse) + o_part * exp(lse_part - lse)
 *    (rows where both are -inf stay O = 0, LSE = -inf).
 *  - merge_finish: o_out [L, H, dv] bf16 = o_acc (round to nearest even), and
 *    head h's LSE to lse_out + h * lse_stride (lse_stride >= L; N for the
 *    chunk's rows inside a [1, H, N] LSE).
 */
fm_status flashmask_merge_init(int L, int H, int dv, float *o_acc, float *lse_acc,
                               void *stream);
fm_status flashmask_merge(int L, int H, int dv, const void *o_part, const float *lse_part,
                          float *o_acc, float *lse_acc, void *stream);
fm_status flashmask_merge_finish(int L, int H, int dv, const float *o_acc, const float *lse_acc,
                                 void *o_out, float *lse_out, long long lse_stride,
                                 void *stream);

/*
 * Sums of partial gradients over chunk pairs: acc[i] += part[i] (n bf16 values
 * into fp32), and dst = bf16(src) (round to nearest even).  n a multiple of 8,
 * pointers 16-byte aligned.
 */
fm_status flashmask_accumulate(long long n, const void *part, float *acc, void *stream);
fm_status flashmask_to_bf16(long long n, const float *src, void *dst, void *stream);

/* Static text for a status code. */
const char *flashmask_error_string(fm_status s);

/* Text of the last FM_ERR_CUDA raised on the calling host thread: the failed
 * step and the CUDA error string.  Empty if none.  Valid until the next call
 * on the same thread. */
const char *flashmask_last_error_detail(void);

#ifdef __cplusplus
}
#endif

#endif /* FLASHMASK_H */
