/*
 * kdkl.h — C ABI of libkdkl.so: an offline top-K teacher cache and a fused,
 * chunked KL(p_teacher || q_student) distillation loss for one GB300 (sm_103a).
 *
 * The method is the one described in "Efficient Knowledge Distillation for
 * LLMs: Offline Top-K Logits and a Fused Chunked KL Loss" (Multiverse Computing,
 * Hugging Face blog, 10 Aug 2026), as reported by:
 *   [ART] aiexpert.news, "Making knowledge distillation cheap enough to run in
 *         production" — the offline top-K cache, the three loss formulations
 *         (dense, forward-chunked, fused chunked) and the top-K limitation;
 *   [DAI] dailyai.com.br launch report, section "As duas inovações";
 *   [EPO] epoka.news, sections "Adónde se va la memoria" and "Los dos cambios
 *         propuestos".
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is DEVICE memory owned by the caller, unless the
 *     argument says otherwise.  The library allocates no device memory: scratch
 *     space is the caller's workspace `ws` of at least the size that the matching
 *     *_workspace() query returns, 256-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every call
 *     only enqueues work on it and returns without synchronising.
 *   - Matrices are row-major.  bf16 is IEEE binary32 with the low 16 bits
 *     dropped (the raw uint16 pattern).  Token rows are the flattened B*T
 *     positions.
 *   - Argument errors are detected on the host, before anything is enqueued,
 *     and returned as KD_ERR_INVALID_ARG / KD_ERR_WORKSPACE / KD_ERR_UNSUPPORTED;
 *     no CUDA call is made in that case.  A failed launch returns KD_ERR_CUDA.
 *     Conditions that only the device can see (a teacher id outside [0, V), a
 *     bounded wait inside a kernel that ran out) are recorded in an error word
 *     inside the workspace and read with kd_get_device_error().
 *   - Calls that share a workspace must be ordered (same stream, or events).
 */
#ifndef KDKL_H_
#define KDKL_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KD_API __attribute__((visibility("default")))
#else
#define KD_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KD_OK = 0,
  KD_ERR_INVALID_ARG = 1,   /* a size, pointer, alignment or K out of range     */
  KD_ERR_UNSUPPORTED = 2,   /* no sm_103a device, or a shape the kernels refuse */
  KD_ERR_WORKSPACE = 3,     /* ws is NULL, misaligned or smaller than required  */
  KD_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed      */
  KD_ERR_TIMEOUT = 5,       /* device: a bounded wait inside a kernel ran out   */
  KD_ERR_DEVICE = 6,        /* device: an input value out of range (teacher id) */
  KD_ERR_IO = 7             /* cache file: open/read/write failed, truncated or corrupt */
} kd_status;

#define KD_MAX_K 1024

/* Human-readable name of a kd_status value (static string, never NULL). */
KD_API const char* kd_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
KD_API int kd_version(void);

/* ------------------------------------------------------------------------ *
 * Offline top-K teacher cache.
 * [ART] paragraph on the first fix (offline distillation); [DAI] "As duas
 * inovações" item 1; [EPO] "Los dos cambios propuestos", first item: the
 * teacher runs once and only its K highest logits per position, with their
 * token ids, are kept and reused.
 * ------------------------------------------------------------------------ */

/* Workspace bytes kd_topk_cache needs (>= 256; it holds the control block: the error
 * word read by kd_get_device_error, and as its third uint32 (byte offset 8) a count, which
 * the caller may read and reset, of rows selected a second time, see below). */
KD_API size_t kd_topk_cache_workspace(int64_t N, int64_t V, int K);

/*
 * For each of the N rows of a dense bf16 teacher-logits matrix, the K largest
 * logits and their column (token) ids.
 *   logits_bf16 : [N, ld] bf16, row r at logits_bf16 + r*ld; columns [0, V) are
 *                 read.  16-byte aligned; ld >= V and ld*2 a multiple of 16.
 *   K           : 1 <= K <= min(V, KD_MAX_K).
 *   ids_out     : [N, K] int32, written.   vals_out: [N, K] fp32, written.
 *   lse_out     : [N] fp32 or NULL.  If given, also the full-row logsumexp of the
 *                 logits (fp32 running max and sum of exponentials).
 *   dropped_out : [N] fp32 or NULL.  If given, the teacher probability the cache
 *                 drops per row, 1 - sum_k exp(vals_k - lse) (the softmax of the
 *                 full row outside its K kept logits, [ART] paragraph on the top-K
 *                 limitation: the cache loses the teacher's tail), computed in the
 *                 same pass (fp32, compensated sum; NaN where lse is not finite).
 * Each output row is ordered by value, highest first; equal values are ordered
 * by ascending id and the cut at K keeps the lowest ids; -0.0 equals +0.0.
 * Values are the bf16 inputs widened exactly.  NaN inputs take their place in
 * the IEEE 754 totalOrder (positive NaNs above +inf, negative NaNs below -inf,
 * a larger payload further out); apart from the zeros, that is the order.
 * Performance note: each row is streamed once by one warp.  Its selection starts
 * from a threshold taken from the row's first 4096 values, extrapolated into its
 * upper tail (invariant to the row's offset and scale); when fewer than K values
 * reach it (rows whose first 4096 values are far above the rest, for instance),
 * the row is read and selected a second time from an exact bound, the count in
 * the control block's third word goes up, and that warp stops extrapolating for
 * the rest of the call.  The result never depends on the start.
 */
KD_API int kd_topk_cache(const void* logits_bf16, int64_t N, int64_t V, int64_t ld, int K,
                  int32_t* ids_out, float* vals_out, float* lse_out, float* dropped_out,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * The teacher's single pass fused with the cache extraction: for N positions of
 * teacher hidden states Ht [N, dt] bf16 and the teacher's LM-head Wt [V, dt] bf16,
 * the logits Ht Wt^T are formed on the tensor cores `chunk` positions at a time
 * (fp32 accumulation, rounded once to bf16 as a bf16 teacher would emit them) into a
 * [chunk, V] workspace buffer and reduced to their top K right away, so the dense
 * [N, V] teacher logits never exist.  Outputs as kd_topk_cache (ids, vals, optional
 * row logsumexp and dropped mass).  dt % 8 == 0; chunk a multiple of 128.  The
 * workspace holds the [chunk, V] bf16 logits and, per row and 256-column tile, the
 * tile's largest logit, which the projection's epilogue emits: with at least K
 * tiles, their K-th largest is an exact start for the row's selection.  When the
 * row logsumexp or the dropped mass is asked for (K <= 256), the epilogue also
 * emits per row and tile the sum of exp(z - tile max) over the tile's stored
 * (bf16) logits; the row logsumexp is combined from those, and the selection runs
 * without computing it.
 */
KD_API size_t kd_teacher_topk_workspace(int64_t N, int64_t dt, int64_t V, int K, int64_t chunk);
KD_API int kd_teacher_topk(const void* Ht_bf16, const void* Wt_bf16, int64_t N, int64_t dt, int64_t V, int K,
                           int64_t chunk, int32_t* ids_out, float* vals_out, float* lse_out, float* dropped_out,
                           void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ *
 * Fused chunked KL loss.
 * [ART] paragraph on the second fix; [DAI] "As duas inovações" item 2; [EPO]
 * "Los dos cambios propuestos", second item.  Per position t (reading: forward
 * KL, teacher renormalised over its K cached logits, student normalised over
 * the full vocabulary):
 *   z_t   = H_t W^T / tau                            (never stored)
 *   p_t,k = softmax_k(t_logits_t,k / tau)
 *   KL_t  = sum_k p_t,k (log p_t,k - z_t,id_k + logsumexp_v z_t,v)
 *   loss  = sum over valid t of KL_t / N_valid       (0 when N_valid == 0)
 * The positions are processed `chunk` rows at a time; the [chunk, V] logits
 * live only in tensor memory, tile by tile.
 * ------------------------------------------------------------------------ */

/* Workspace bytes for kd_fused_kl_fwd and kd_fused_kl_bwd with these sizes
 * (one query covers both calls).  Grows with chunk*V, not with N*V. */
KD_API size_t kd_fused_kl_workspace(int64_t N, int64_t d, int64_t V, int K, int64_t chunk);

/*
 * Forward pass.
 *   H_bf16   : [N, d] bf16 student hidden states (16-byte aligned rows: d % 8 == 0).
 *   W_bf16   : [V, d] bf16 LM-head (output projection) weight.
 *   t_ids    : [N, K] int32 cached teacher token ids, distinct within a row.
 *   t_logits : [N, K] fp32 cached teacher logits (any order).
 *   mask     : [N] uint8, 1 = valid position, 0 = padding; NULL = all valid.
 *   chunk    : positions per chunk, a multiple of 128 (the last chunk may be short).
 *   tau      : temperature > 0, divides both teacher and student logits.
 *   loss_out : device fp32 scalar, written.
 *   lse_out  : [N] fp32, logsumexp_v z_t,v, written; keep it for the backward.
 *   kl_per_token_out : [N] fp32 KL_t (also for padding rows) or NULL.
 */
KD_API int kd_fused_kl_fwd(const void* H_bf16, const void* W_bf16,
                    const int32_t* t_ids, const float* t_logits, const uint8_t* mask,
                    int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    float* loss_out, float* lse_out, float* kl_per_token_out,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * Backward pass: recomputes each chunk's logits from H and W ([ART], the
 * backward recomputes every chunk instead of storing it) and forms
 *   dZ_t = grad_loss * mask_t / (N_valid * tau) * (softmax(z_t) - p_t scattered to its ids)
 *   grad_H = dZ W            (overwritten; bf16, or fp32 if grad_H_is_fp32)
 *   grad_W += dZ^T H         (fp32, ACCUMULATED into what the caller passes)
 * with fp32 tensor-core accumulation; dZ is rounded to bf16 before the two
 * gradient products.  Inputs as in kd_fused_kl_fwd, plus
 *   lse       : [N] fp32 from the forward pass with the same inputs.
 *   grad_loss : device fp32 scalar, the upstream gradient of the loss.
 *   grad_H    : [N, d] bf16 or fp32.   grad_W : [V, d] fp32.
 */
KD_API int kd_fused_kl_bwd(const void* H_bf16, const void* W_bf16,
                    const int32_t* t_ids, const float* t_logits, const uint8_t* mask,
                    int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    const float* lse, const float* grad_loss,
                    void* grad_H, int grad_H_is_fp32, float* grad_W,
                    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ *
 * Forward-chunked KL: the same loss, keeping each chunk's student logits.
 * [ART] fused-loss paragraph, second formulation: the teacher stays sparse and
 * the loss is taken one chunk at a time, but the full student logits are kept
 * for the backward pass (so memory grows with sequence x vocabulary), which
 * saves the backward recompute; the page calls it the fastest of the three.
 * z_store holds the raw logits H W^T (bf16, before 1/tau) in a blocked layout:
 * element (t, v) at ((v / 64) * N + t) * 64 + v % 64, i.e.
 * kd_chunked_kl_logits_bytes(N, V) = ceil(V / 64) * N * 128 bytes, 16-byte
 * aligned, owned by the caller; the forward writes it, the backward only reads
 * it.  Everything else (arguments, workspace, outputs, errors) is as for
 * kd_fused_kl_fwd / kd_fused_kl_bwd; the backward uses the bf16-rounded
 * logits, so its gradients differ from the fused ones by that rounding.
 * ------------------------------------------------------------------------ */

KD_API size_t kd_chunked_kl_logits_bytes(int64_t N, int64_t V);

KD_API int kd_chunked_kl_fwd(const void* H_bf16, const void* W_bf16,
                    const int32_t* t_ids, const float* t_logits, const uint8_t* mask,
                    int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    float* loss_out, float* lse_out, float* kl_per_token_out,
                    void* z_store, size_t z_bytes, void* ws, size_t ws_bytes, void* stream);

KD_API int kd_chunked_kl_bwd(const void* H_bf16, const void* W_bf16,
                    const int32_t* t_ids, const float* t_logits, const uint8_t* mask,
                    int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    const float* lse, const float* grad_loss, const void* z_store, size_t z_bytes,
                    void* grad_H, int grad_H_is_fp32, float* grad_W,
                    void* ws, size_t ws_bytes, void* stream);

/*
 * Forward pass without a caller workspace, for callers that cannot allocate
 * device memory (no counterpart in the paper: it is an integration variant).
 * Some callers may not call cudaMalloc: plugins whose host framework owns all
 * device memory through its own pre-sized pool, and latency-critical paths that
 * cannot take the device-wide synchronisation cudaMalloc/cudaFree may cause;
 * they cannot provide the workspace kd_fused_kl_fwd needs either.  This call
 * computes exactly what kd_fused_kl_fwd computes (same arguments minus ws,
 * ws_bytes), using a scratch array of KD_STATIC_SCRATCH_BYTES compiled into
 * the library instead of a workspace:
 *   - every GPU that loads the library holds that array until the process exits;
 *   - the array's device address is looked up on the first call made with a
 *     given device current, so make that first call before any stream capture
 *     (it is looked up again after a device reset gives the device a new context);
 *   - it returns KD_ERR_WORKSPACE, before any launch, when the problem needs more
 *     than the array holds, i.e. when kd_fused_kl_workspace(N, d, V, K, chunk)
 *     exceeds KD_STATIC_SCRATCH_BYTES;
 *   - it allocates nothing; all calls share the one array, which keeps the last
 *     call's contents (its control block is cleared at the start of each call),
 *     so calls whose GPU work overlaps (other streams or host threads) race and
 *     must be serialised by the caller;
 *   - device-side conditions (a teacher id out of range) are recorded in the
 *     shared array's error word: kd_get_device_error(NULL, stream, &detail)
 *     reads and clears it.
 * Argument errors that kd_fused_kl_fwd detects are returned as there; the
 * scratch set-up and the clearing of its control block may already have been
 * enqueued when an alignment or shape check fails.
 */
#define KD_STATIC_SCRATCH_BYTES (32u * 1024u * 1024u)
KD_API int kd_fused_kl_fwd_static(const void* H_bf16, const void* W_bf16,
                    const int32_t* t_ids, const float* t_logits, const uint8_t* mask,
                    int64_t N, int64_t d, int64_t V, int K, int64_t chunk, float tau,
                    float* loss_out, float* lse_out, float* kl_per_token_out, void* stream);

/*
 * Reads (synchronising `stream`) and clears the device error word of a
 * workspace used by the calls above; ws == NULL names the scratch array of
 * kd_fused_kl_fwd_static on the current device.  Returns KD_OK, KD_ERR_TIMEOUT or
 * KD_ERR_DEVICE; *detail_out (may be NULL) receives a call-specific detail
 * (for a bad teacher id: the first offending row).  A library built with
 * KD_DEBUG (libkdkl_debug.so) also checks the indices its kernels compute and
 * reports one out of range as KD_ERR_DEVICE with the place of the check as the
 * detail (0x7xxx: top-K), after skipping the access.
 */
KD_API int kd_get_device_error(void* ws, void* stream, int64_t* detail_out);

/* ------------------------------------------------------------------------ *
 * On-disk teacher cache ([ART] paragraph on the first fix: run the teacher once,
 * keep its top-K logits per position on disk, reuse them across experiments).
 * HOST memory and host files only; no CUDA call.  One file per contiguous range
 * of positions (a shard): a 64-byte header (magic, version, K, V, N, row0,
 * logits type, flags, FNV-1a 64 checksum of the payload), then ids int32 [N, K],
 * logits fp32 or bf16 [N, K] and optionally the teacher's full-row logsumexp
 * fp32 [N].  bf16 logits round to nearest even (exact for caches extracted from
 * bf16 teacher logits) and are widened back to fp32 on reading.
 * ------------------------------------------------------------------------ */

/* Write a shard atomically (temporary file + rename).  lse may be NULL. */
KD_API int kd_cache_write(const char* path, const int32_t* ids, const float* logits, const float* lse,
                          int64_t N, int K, int64_t V, int64_t row0, int logits_bf16);
/* Header fields of a shard (any out pointer may be NULL); checks the file size. */
KD_API int kd_cache_info(const char* path, int64_t* N, int* K, int64_t* V, int64_t* row0,
                         int* logits_bf16, int* has_lse);
/* Recompute the payload checksum: KD_OK, or KD_ERR_IO if the file is corrupt or truncated. */
KD_API int kd_cache_verify(const char* path);
/* Read positions [first, first + count) into host buffers ids_out [count, K] and
 * logits_out [count, K] (fp32); lse_out [count] or NULL. */
KD_API int kd_cache_read(const char* path, int64_t first, int64_t count, int32_t* ids_out,
                         float* logits_out, float* lse_out);
/* Streaming reader: batches of up to rows_per_batch consecutive positions; the next
 * batch is read on a background thread while the caller uses the current one.
 * kd_cache_reader_next copies one batch into host buffers (rows_out = 0 at the end). */
KD_API int kd_cache_reader_open(const char* path, int64_t rows_per_batch, void** handle);
KD_API int kd_cache_reader_next(void* handle, int32_t* ids_out, float* logits_out, int64_t* rows_out);
KD_API int kd_cache_reader_close(void* handle);

/* ------------------------------------------------------------------------ *
 * Building blocks, exposed for testing and profiling.  No page describes these
 * separately; they are the pieces the calls above are made of.
 * ------------------------------------------------------------------------ */

/*
 * C[M, N] (op)= A · B^T-or-B with bf16 inputs and fp32 tensor-core accumulation,
 * the projection engine shared by the loss kernels.
 *   a_mn_major = 0: A is [M, K] row-major (K contiguous); 1: A is [K, M] (M contiguous).
 *   b_mn_major = 0: B is [N, K] row-major;                 1: B is [K, N].
 *   C is [M, N] fp32 row-major; accumulate != 0 adds into C.
 * All leading dimensions are the contiguous extents above; K % 8 == 0 for
 * K-major operands and M % 8 / N % 8 == 0 for MN-major ones.
 */
KD_API int kd_gemm_bf16(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                 int a_mn_major, int b_mn_major, int accumulate,
                 void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for kd_gemm_bf16. */
KD_API size_t kd_gemm_workspace(void);

/*
 * Self-check of the bounded waits every kernel uses: launches one block that
 * waits on a shared-memory barrier nothing arrives at, with a limit of
 * `limit_ns` (1 us .. 1 s) instead of the kernels' 2 s.  The wait gives up, the
 * kernel records a timeout in the error word of `ws` and exits normally, so
 * kd_get_device_error(ws) then returns KD_ERR_TIMEOUT and the CUDA context
 * stays usable.
 */
KD_API int kd_check_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_ns, void* stream);

/*
 * Per-launch timing of this library's kernels, for profiling.  While enabled,
 * each launch on `stream` is bracketed by two CUDA events (at most `capacity`
 * launches are recorded).  kd_profile_read synchronises, then fills up to `n`
 * entries of names[] (static strings), ms[] and returns how many launches were
 * recorded since kd_profile_begin.  Host-side state; not thread-safe.
 */
KD_API int kd_profile_begin(int capacity);
KD_API int kd_profile_end(void);
KD_API int kd_profile_read(const char** names, float* ms, int n);

#ifdef __cplusplus
}
#endif
#endif /* KDKL_H_ */
