/*
 * attn_fwd.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * Operation (all entry points):
 *   O[b, h, i, :] = sum_j P[i, j] V[b, h, j, :],
 *   P[i, :] = softmax_j(scale * Q[b, h, i, :] . K[b, h, j, :]  [+ causal mask])
 *   LSE[b, h, i] = ln sum_j exp(scale * Q[b, h, i, :] . K[b, h, j, :])   (visible j)
 * This is the attention formula of "flash-attn 实现 prefill 阶段" (问题分析),
 * over [b, h, s, d] tensors as laid out there, with the scale applied after
 * the dot product and a natural-exponent softmax as in flash-attention-minimal
 * forward_kernel; it is computed with the online-softmax recurrence of that
 * kernel (running row max m and row sum l, O rescaled as K/V tiles arrive),
 * so S and P never reach memory.
 *
 * Causal mask ("05 · kernel 工程与四代演化", 2.1 names `causal` without
 * defining it): bottom-right aligned -- key j is visible to query i iff
 * j <= i + (sk - sq); for sq == sk this is j <= i.  A query row that sees no
 * key gets O = 0 and LSE = -inf.
 *
 * Layout: Q and O are contiguous [b, h, sq, d]; K and V are contiguous
 * [b, h, sk, d]; all four have the element type `dtype` (fp16 or bf16).
 * LSE is contiguous fp32 [b, h, sq].  d must be 64 or 128.
 *
 * Ownership: every pointer is owned by the caller.  attn_fwd allocates
 * nothing and keeps no reference after it returns.
 *
 * Execution: attn_fwd enqueues its work on `stream` (a cudaStream_t, NULL =
 * legacy default stream) of the current device and returns without
 * synchronising; results are ready when the stream reaches that point.  It
 * may be called from several host threads on different streams.
 *
 * Errors: a negative return code, never an exception or abort.  The message
 * of the last failing call on the calling thread is given by
 * attn_last_error().  Argument errors are detected before anything is
 * enqueued.  Precision: fp32 accumulation and statistics; P is rounded to
 * `dtype` before the P.V product; O is rounded to nearest-even into `dtype`.
 *
 * Argument types: sizes are int64_t (so that b*h*s*d products of large
 * problems are formed without overflow on either side of the call) and
 * `stream` is a void* holding a cudaStream_t, so that this header needs no
 * CUDA header.  The device watchdog word is read with attn_fwd_status (all
 * four words) or attn_fwd_debug_status (the code only).
 *
 * Device state: the library keeps, per device, a status word, the counter
 * slots of the dynamic schedule and a scratch array (attn_fwd_splitkv_noalloc),
 * whose device addresses it looks up on the first call on that device and
 * keeps for the life of the process.  cudaDeviceReset, or anything else that
 * destroys the device's primary context, invalidates them: the library must
 * not be used on that device afterwards.
 */
#ifndef ATTN_FWD_H
#define ATTN_FWD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { ATTN_FP16 = 0, ATTN_BF16 = 1 } attn_dtype_t;

enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = -1,    /* a required pointer is NULL                       */
    ATTN_ERR_SHAPE = -2,   /* negative or too large b, h, sq, sk               */
    ATTN_ERR_HEADDIM = -3, /* d is not 64 or 128                               */
    ATTN_ERR_DTYPE = -4,   /* dtype is not ATTN_FP16 / ATTN_BF16               */
    ATTN_ERR_SCALE = -5,   /* scale is NaN or infinite                         */
    ATTN_ERR_ALIGN = -6,   /* q/k/v/o not 16-byte aligned, lse not 4-byte     */
    ATTN_ERR_ARCH = -7,    /* current device is not compute capability 10.3   */
    ATTN_ERR_CUDA = -8,    /* a CUDA runtime/driver call failed                */
    ATTN_ERR_WATCHDOG = -9, /* a device-side wait gave up (see attn_fwd_status) */
    ATTN_ERR_BUILD = -10    /* the entry point needs the checked build          */
};

/*
 * attn_fwd: the fused forward.
 *   q, k, v : device pointers, layout above, 16-byte aligned.
 *   o       : device pointer, [b, h, sq, d] of dtype, 16-byte aligned.
 *   lse     : device pointer to fp32 [b, h, sq], 4-byte aligned, or NULL to
 *             skip writing it.
 *   b, h    : batch and heads (>= 0, b*h < 2^31).  sq, sk : query / key
 *             lengths (0 .. 2^30).  d : head dimension, 64 or 128.
 *   causal  : 0 = no mask, nonzero = bottom-right causal mask.
 *   scale   : finite multiplier of Q.K (1/sqrt(d) in the pages' formula).
 *   dtype   : attn_dtype_t of q, k, v, o.
 *   stream  : cudaStream_t to enqueue on.
 * b*h*sq == 0 returns ATTN_OK with nothing enqueued; sk == 0 writes O = 0 and
 * LSE = -inf.  Returns ATTN_OK or a negative ATTN_ERR_* code.
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
             int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d,
             int causal, float scale, int dtype, void *stream);

/*
 * attn_fwd_host: attn_fwd for inputs and outputs in HOST memory: copies
 * q_host/k_host/v_host into the caller's device buffers q_dev/k_dev/v_dev,
 * runs attn_fwd into o_dev/lse_dev, then copies O (and LSE when both lse
 * pointers are non-NULL) back into o_host/lse_host.  All buffers are
 * caller-owned with the layouts of attn_fwd; host buffers should be
 * page-locked for the copies to be asynchronous.  Problems of 64 MB and more
 * are cut into up to 8 chunks of whole heads, and the copies in of one chunk
 * and out of another overlap the forward of a third: the copies run on two
 * streams the library creates once per device, the forwards on `stream`,
 * ordered by events so that the whole operation comes after earlier work on
 * `stream` and later work on `stream` comes after it.  The call returns once
 * everything is enqueued; the host outputs are valid after `stream` is
 * synchronised.  Same error codes as attn_fwd (copy failures give
 * ATTN_ERR_CUDA).
 */
int attn_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                  void *o_host, float *lse_host,
                  void *q_dev, void *k_dev, void *v_dev, void *o_dev,
                  float *lse_dev,
                  int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d,
                  int causal, float scale, int dtype, void *stream);

/*
 * Split-KV forward.  "05 · kernel 工程与四代演化" 2.1 lists split-KV kernels
 * beside the forward and backward ones.  The key range of every (b, h,
 * 256-row block) -- the keys that block sees -- is cut into `num_splits`
 * near-equal ranges of whole 128-key tiles, processed by separate CTAs
 * (this fills the GPU when b*h*ceil(sq/256) is small, as in decoding).
 * Each range yields a partial softmax: O normalised
 * by its own row sum plus the range's log-sum-exp.  A second kernel merges
 * the ranges with the rescale-and-add step of the online recurrence
 * (flash-attention-minimal forward_kernel: m_new = max, l_new = sum of
 * e^(m - m_new) l, O weighted accordingly).  Result and semantics are those
 * of attn_fwd.
 *
 *   num_splits : 1..min(1024, ceil(sk / 128)); 1 runs attn_fwd directly.
 *   workspace  : caller-owned device scratch, 16-byte aligned, at least
 *                attn_fwd_splitkv_workspace_bytes(b, h, sq, d, num_splits)
 *                bytes (fp32 partial O [num_splits, b, h, sq, d] followed by
 *                2 fp32 log-sum-exps per partial row).  Its contents on
 *                entry do not matter; calls on different streams need
 *                different workspaces.
 * Returns ATTN_OK or a negative ATTN_ERR_* code (ATTN_ERR_SHAPE for a bad
 * split count or a too small workspace, ATTN_ERR_NULL for a missing one).
 */
int attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o,
                     float *lse, int64_t b, int64_t h, int64_t sq, int64_t sk,
                     int64_t d, int causal, float scale, int dtype,
                     int num_splits, void *workspace, int64_t workspace_bytes,
                     void *stream);

/*
 * Variable-length (packed) forward.  "05 · kernel 工程与四代演化" 6.1 lists
 * varlen_fwd among the exported entry points; the operation is attn_fwd
 * applied to each sequence of a batch of different lengths, with the
 * sequences concatenated along the token axis.
 *
 *   q, o          : [total_q, h, d] of dtype (token-major, heads inside),
 *                   16-byte aligned.
 *   k, v          : [total_k, h, d] of dtype, 16-byte aligned.
 *   lse           : fp32 [h, total_q], or NULL.
 *   cu_seqlens_q  : device int32 [batch + 1]: sequence s owns query tokens
 *                   cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1 (non-decreasing,
 *                   cu_seqlens_q[0] = 0, cu_seqlens_q[batch] = total_q).
 *   cu_seqlens_k  : the same for keys/values (total_k).
 *   max_seqlen_q/k: upper bounds of the per-sequence lengths (they size the
 *                   work grid; the host never reads the offsets).
 * The causal mask is bottom-right per sequence.  A sequence whose offsets
 * fall outside the totals is skipped (its outputs are not written).  Same
 * error codes as attn_fwd.
 * Work units of unequal size are handed out through one of 256 device
 * counter slots that launches of this entry point and of attn_fwd_kvcache
 * take in turn, each launch tagged with its own generation number (each
 * launch leaves its slot free when it ends), so at most 256 such launches may
 * be in flight on one device at a time.  A launch that finds its slot still
 * held by another launch does not share its counters: the CTAs that find it
 * so take no work and record ATTN_STATUS_SCHED_COLLISION in the status word
 * (attn_fwd_status); the outputs of that launch are then not to be trusted,
 * and the slot stays held until attn_fwd_status_clear.  A CUDA graph that
 * holds such a launch must not be replayed concurrently with itself (both
 * replays carry the same generation).
 */
int attn_fwd_varlen(const void *q, const void *k, const void *v, void *o,
                    float *lse, const int32_t *cu_seqlens_q,
                    const int32_t *cu_seqlens_k, int64_t batch, int64_t h,
                    int64_t total_q, int64_t total_k, int64_t max_seqlen_q,
                    int64_t max_seqlen_k, int64_t d, int causal, float scale,
                    int dtype, void *stream);

/*
 * FP8 forward.  "05 · kernel 工程与四代演化" 4.4 describes an FP8 forward that
 * subtracts an extra 8 from the softmax maximum so that exp2 lands in
 * [0, 256] and uses more of the 8-bit range.  Here q, k, v are e4m3 (1 byte
 * per element, [b, h, s, d] contiguous, 16-byte aligned) with per-tensor
 * descale factors, so the operation is attn_fwd on the real-valued inputs
 * Q = descale_q*q, K = descale_k*k, V = descale_v*v:
 *   O = softmax(scale * descale_q * descale_k * q.k^T [+ causal]) (descale_v * v)
 * Both products run on the 8-bit tensor cores; P is rounded to e4m3 (its
 * reference sits 8 below the row maximum, so P <= 2^8.5 < 448) and O is
 * written as bf16 [b, h, sq, d]; LSE as for attn_fwd.  d must be 64 or 128
 * (64: the 64-byte rows are read with the 64-byte swizzle).
 * Returns ATTN_OK or a negative ATTN_ERR_* code.
 */
int attn_fwd_fp8(const void *q, const void *k, const void *v, void *o,
                 float *lse, int64_t b, int64_t h, int64_t sq, int64_t sk,
                 int64_t d, int causal, float scale, float descale_q,
                 float descale_k, float descale_v, void *stream);

/* Bytes of workspace attn_fwd_splitkv needs (0 when num_splits == 1), or a
 * negative ATTN_ERR_* code for invalid sizes. */
int64_t attn_fwd_splitkv_workspace_bytes(int64_t b, int64_t h, int64_t sq,
                                         int64_t d, int num_splits);

/* A split count for the current device: 1 when the problem has more than
 * 64 query rows and at least one work unit per SM; otherwise the count
 * whose units (b*h*ceil(sq/256)*splits) fill whole waves of the SMs best,
 * less 1% per wave, keeping at least two key tiles per split.  A negative
 * ATTN_ERR_* code for invalid sizes. */
int attn_fwd_splitkv_default_splits(int64_t b, int64_t h, int64_t sq,
                                    int64_t sk, int64_t d, int causal);

/*
 * attn_fwd_splitkv_noalloc: attn_fwd_splitkv for callers that cannot
 * allocate device memory.  The pages have no counterpart to this entry
 * point.  Some callers have no workspace to pass and may not call cudaMalloc
 * themselves: for example a plugin whose host program's memory planner owns
 * every device allocation, or latency-critical code that must not pay the
 * implicit device synchronisation of an allocation.  This entry point keeps
 * the split partials in a fixed scratch array of ATTN_NOALLOC_SCRATCH_BYTES
 * (16 MiB) compiled into the library; every GPU that loads the library holds
 * that array until the process exits.  The caller still passes the inputs
 * and outputs, with the layouts and semantics of attn_fwd.  It allocates
 * nothing.
 *
 *   num_splits : 1..min(1024, ceil(sk / 128)), as for attn_fwd_splitkv.
 *                With num_splits == 1 or sk == 0 the scratch is not
 *                touched, and such calls do not race with others.  Sizes
 *                whose partials need more than ATTN_NOALLOC_SCRATCH_BYTES
 *                (see attn_fwd_splitkv_workspace_bytes) are rejected with
 *                ATTN_ERR_SHAPE and a message saying how much they need;
 *                other argument errors give the codes of attn_fwd_splitkv.
 *
 * The first call on each device looks up the array's device address on that
 * device (make that first call before any stream capture); the address is
 * kept for the life of the process, so a device reset invalidates it (see
 * "Device state" above).  All calls on a device share the one array, and it
 * keeps the last call's contents (nothing in it needs to start at zero: each
 * call writes what it reads).  Calls that overlap on the GPU -- on different
 * streams, or from different host threads -- race on the array; serialise
 * them.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
int attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v,
                             void *o, float *lse, int64_t b, int64_t h,
                             int64_t sq, int64_t sk, int64_t d, int causal,
                             float scale, int dtype, int num_splits,
                             void *stream);

/*
 * KV-cache forward (decoding).  "05 · kernel 工程与四代演化" 6.1 lists
 * fwd_kvcache among the exported entry points without defining it; the
 * reading here is the plainest one: attention of the new queries against a
 * cache whose batch elements hold different numbers of valid tokens, after
 * the new tokens' keys and values have been written into the cache.
 *
 *   q          : [b, h, sq, d] of dtype, contiguous, 16-byte aligned.
 *   k_cache,
 *   v_cache    : [b, h, s_cache, d] of dtype, contiguous, 16-byte aligned;
 *                s_cache is the capacity.  Written when k_new is given.
 *   k_new,
 *   v_new      : [b, h, s_new, d] of dtype, contiguous, 16-byte aligned,
 *                or both NULL (then s_new must be 0).  They must not
 *                overlap the caches (ATTN_ERR_SHAPE).
 *   cache_seqlens : device int32 [b], the number of valid cached tokens of
 *                each batch element before this call (read, not updated).
 *                Values are clamped to [0, s_cache].
 * With L0 = clamp(cache_seqlens[b], 0, s_cache):
 *   1. row t of k_new / v_new is written to position L0 + t of the cache;
 *      rows that would land at or past s_cache are dropped;
 *   2. batch element b attends to its first L = min(L0 + s_new, s_cache)
 *      cached keys: attn_fwd on q[b] and k/v_cache[b, :, :L], with the
 *      causal mask bottom-right aligned to L (query i sees keys
 *      j <= i + L - sq), O = 0 and LSE = -inf for a row that sees no key.
 * Cache slots at or past L are never read into the result (they may hold
 * anything, NaN included).  num_splits, workspace and workspace_bytes are
 * those of attn_fwd_splitkv with sk = s_cache (num_splits 1: no workspace).
 * o, lse, d, causal, scale, dtype, stream as for attn_fwd.  Asynchronous;
 * the cache write precedes the attention on `stream`.  The schedule
 * counters of attn_fwd_varlen are used here too (same limit of 256 launches
 * in flight per device).
 * Returns ATTN_OK or a negative ATTN_ERR_* code.
 */
int attn_fwd_kvcache(const void *q, void *k_cache, void *v_cache,
                     const void *k_new, const void *v_new,
                     const int32_t *cache_seqlens, void *o, float *lse,
                     int64_t b, int64_t h, int64_t sq, int64_t s_cache,
                     int64_t s_new, int64_t d, int causal, float scale,
                     int dtype, int num_splits, void *workspace,
                     int64_t workspace_bytes, void *stream);

/*
 * attn_fwd_kvcache over a paged cache: the same operation, with each batch
 * element's cache made of fixed-size pages of a shared pool, as a decoder
 * that allocates its cache page by page keeps it.
 *
 *   k_pool,
 *   v_pool     : [num_pages, page_size, h, d] of dtype (token-major within a
 *                page, heads inside), 16-byte aligned; written when k_new is
 *                given.
 *   block_table: device int32 [b, pages_per_seq]: logical page p of batch
 *                element b is pool page block_table[b * pages_per_seq + p].
 *                Pages of different elements must be distinct; a page index
 *                outside [0, num_pages) reads as zeros and is not written.
 *   page_size  : a positive multiple of 128 (a key tile never straddles two
 *                pages).  The capacity of each element is
 *                pages_per_seq * page_size (at most 2^30), the pool at most
 *                2^31-1 tokens.
 * Logical key r of element b is row r % page_size of page
 * block_table[b, r / page_size]; everything else (q, k_new, v_new,
 * cache_seqlens, the write, the lengths, the mask, num_splits with
 * sk = pages_per_seq * page_size, o, lse) is as for attn_fwd_kvcache.
 * Returns ATTN_OK or a negative ATTN_ERR_* code.
 */
int attn_fwd_kvcache_paged(const void *q, void *k_pool, void *v_pool,
                           const void *k_new, const void *v_new,
                           const int32_t *cache_seqlens,
                           const int32_t *block_table, void *o, float *lse,
                           int64_t b, int64_t h, int64_t sq,
                           int64_t num_pages, int64_t page_size,
                           int64_t pages_per_seq, int64_t s_new, int64_t d,
                           int causal, float scale, int dtype, int num_splits,
                           void *workspace, int64_t workspace_bytes,
                           void *stream);

/*
 * Backward pass: the gradients of attn_fwd.  "05 · kernel 工程与四代演化" 6.1
 * lists bwd among the exported entry points (and chapter 04 of that series
 * as its implementation, which is not among the pages); the operation is the
 * chain rule through attn_fwd's definition.  For the loss gradient dO:
 *   P  = softmax(scale * Q K^T [+ causal])   recomputed from LSE:
 *        P[i, j] = exp(scale * q_i . k_j - lse[i])
 *   dV = P^T dO
 *   dS = P * (dO V^T - D),  D[i] = sum_c dO[i, c] * O[i, c]
 *   dQ = scale * dS K,      dK = scale * dS^T Q
 * with the causal mask of attn_fwd (bottom-right aligned).
 *
 *   q, o, dout, dq : [b, h, sq, d] of dtype, contiguous, 16-byte aligned.
 *   k, v, dk, dv   : [b, h, sk, d] of dtype, contiguous, 16-byte aligned.
 *   lse            : fp32 [b, h, sq] as written by attn_fwd (natural log;
 *                    -inf for a row that sees no key).
 *   o, lse         : the forward's outputs for these q, k, v; D is computed
 *                    from o (so an o rounded to dtype carries that rounding
 *                    into D).
 *   d              : 64 or 128 (ATTN_ERR_HEADDIM otherwise).
 *   workspace      : caller-owned device scratch, 16-byte aligned, of at
 *                    least attn_bwd_workspace_bytes(b, h, sq, d) bytes (an
 *                    fp32 dQ accumulator, two fp32 values per query row
 *                    and a work counter); its contents on entry do not
 *                    matter.  Calls on different streams need different
 *                    workspaces.
 * Outputs dq, dk, dv are written in full (zeros where the gradient is zero,
 * e.g. dq of rows that see no key, or everything when sq or sk is 0).
 * Three kernels run on `stream`, asynchronously; the library allocates
 * nothing.  Returns ATTN_OK or a negative ATTN_ERR_* code.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o,
             const void *dout, const float *lse, void *dq, void *dk, void *dv,
             int64_t b, int64_t h, int64_t sq, int64_t sk, int64_t d,
             int causal, float scale, int dtype, void *workspace,
             int64_t workspace_bytes, void *stream);

/* Bytes of workspace attn_bwd needs, or a negative ATTN_ERR_* code. */
int64_t attn_bwd_workspace_bytes(int64_t b, int64_t h, int64_t sq, int64_t d);

/*
 * Variable-length (packed) backward: attn_bwd applied to each sequence of a
 * packed batch ("05 · kernel 工程与四代演化" 6.1 lists varlen_bwd beside
 * varlen_fwd), with the layouts of attn_fwd_varlen:
 *   q, o, dout, dq : [total_q, h, d] of dtype, 16-byte aligned.
 *   k, v, dk, dv   : [total_k, h, d] of dtype, 16-byte aligned.
 *   lse            : fp32 [h, total_q], as written by attn_fwd_varlen.
 *   cu_seqlens_q/k : device int32 [batch + 1] offsets, as for
 *                    attn_fwd_varlen; max_seqlen_q/k bound the lengths.
 *   workspace      : caller-owned device scratch, 16-byte aligned, of at
 *                    least attn_bwd_varlen_workspace_bytes(batch, h,
 *                    total_q, max_seqlen_q, d) bytes.
 * The causal mask is bottom-right per sequence.  A sequence whose offsets
 * fall outside the totals is skipped (its gradients are not written).  d is
 * 64 or 128.  Same error codes and asynchrony as attn_bwd.
 */
int attn_bwd_varlen(const void *q, const void *k, const void *v,
                    const void *o, const void *dout, const float *lse,
                    void *dq, void *dk, void *dv,
                    const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k,
                    int64_t batch, int64_t h, int64_t total_q,
                    int64_t total_k, int64_t max_seqlen_q,
                    int64_t max_seqlen_k, int64_t d, int causal, float scale,
                    int dtype, void *workspace, int64_t workspace_bytes,
                    void *stream);

/* Bytes of workspace attn_bwd_varlen needs, or a negative ATTN_ERR_* code. */
int64_t attn_bwd_varlen_workspace_bytes(int64_t batch, int64_t h,
                                        int64_t total_q, int64_t max_seqlen_q,
                                        int64_t d);

/* Thread-local message describing the last non-OK return on this thread
 * ("" if none).  The pointer stays valid until the next call on the thread. */
const char *attn_last_error(void);

/*
 * Device watchdog.  Every wait inside the kernels is bounded; a wait that
 * runs out records a nonzero code in a per-device status word and the kernel
 * winds down (waits for its own copies and MMAs, frees tensor memory) and
 * returns instead of hanging.  The first failure is kept until cleared:
 *   code ATTN_STATUS_TIMEOUT (1)         a wait ran out;
 *   code ATTN_STATUS_SCHED_COLLISION (2) a launch found its schedule slot
 *                                        held by another (attn_fwd_varlen);
 *   code ATTN_STATUS_BOUNDS (3)          checked build: a computed index was
 *                                        outside its bounds (see below).
 * attn_fwd_status synchronises the current device, copies the status into
 * out[0..3] = {code, block, warp, site} (out may be NULL) and returns code
 * (0 = nothing recorded, <0 = CUDA error while reading).
 * attn_fwd_status_clear synchronises the device, then zeroes the status word
 * and frees every schedule slot; call it with no forward in flight on the
 * device (from any thread).
 * attn_fwd_debug_status is attn_fwd_status(NULL): the code alone.
 */
#define ATTN_STATUS_TIMEOUT 1
#define ATTN_STATUS_SCHED_COLLISION 2
#define ATTN_STATUS_BOUNDS 3
int attn_fwd_status(uint32_t *out);
int attn_fwd_status_clear(void);
int attn_fwd_debug_status(void);

/*
 * Testing hook: make every later launch of the dynamic schedule on the
 * current device take counter slot `slot` (0..255) instead of the next one
 * in turn; -1 restores the turn.  It exists so that a test can put two
 * launches on one slot and check that the collision is reported.  Returns
 * ATTN_OK or ATTN_ERR_SHAPE for a slot outside -1..255.
 */
int attn_fwd_sched_pin_slot(int slot);

/*
 * attn_fwd_watchdog_selftest: launches the forward on tiny caller-provided
 * buffers (same contract as attn_fwd) with the key/value load number
 * `withheld_load` deliberately never issued and the wait limit set to
 * `timeout_ms`, so that the waits run out.  It synchronises and returns the
 * status code the kernel recorded (expected nonzero), or a negative error.
 * Exists only to test the watchdog without faulting or hanging the GPU.
 */
int attn_fwd_watchdog_selftest(const void *q, const void *k, const void *v,
                               void *o, float *lse, int64_t b, int64_t h,
                               int64_t sq, int64_t sk, int64_t d, int causal,
                               float scale, int dtype, int withheld_load,
                               int timeout_ms, void *stream);

/*
 * attn_bwd_watchdog_selftest: the same for the backward -- attn_bwd on tiny
 * caller buffers (contract of attn_bwd, b*h*sq <= 4096, 1 <= sk <= 1024)
 * with the query-tile load number `withheld_load` of every CTA never issued
 * and the wait limit set to `timeout_ms`; synchronises and returns the
 * recorded status code (expected ATTN_STATUS_TIMEOUT), or a negative error.
 * The gradients of that call are not meaningful.  The backward's waits are
 * the same code in both builds; the knob that withholds the load exists in
 * the checked build only (in the normal one it would cost the kernel time),
 * so the normal build returns ATTN_ERR_BUILD.
 */
int attn_bwd_watchdog_selftest(const void *q, const void *k, const void *v,
                               const void *o, const void *dout,
                               const float *lse, void *dq, void *dk, void *dv,
                               int64_t b, int64_t h, int64_t sq, int64_t sk,
                               int64_t d, int causal, float scale, int dtype,
                               void *workspace, int64_t workspace_bytes,
                               int withheld_load, int timeout_ms,
                               void *stream);

/*
 * Checked build.  libattn_fwd_checked.so exports this same interface from
 * the same sources compiled with every computed index of the forward and
 * backward kernels checked.  Forward: copy coordinates of Q, K, V (page
 * lookups included) and of the O stores, thread-written O, LSE and
 * split-partial offsets, the decoded work units, the tensor-memory
 * allocation and the shared-memory window.  Backward: the claimed and
 * decoded units, the copy coordinates of K, V, Q and dO and the rows of the
 * LSE / D vectors, the dQ reduce-add coordinates, the thread-written dK / dV
 * rows, the prep kernel's O / dO / accumulator / LSE offsets, the
 * tensor-memory allocation and the shared-memory window.  An index outside
 * its bounds is not used: the kernel records {ATTN_STATUS_BOUNDS, block,
 * warp, site} in the status word and the CTA winds down as after a wait
 * that ran out.  It stands in for a memory checker, which is not available
 * on every machine, and is slower than the normal build.  (In every build,
 * a backward launch whose shared-memory window is not 1 KiB aligned records
 * ATTN_STATUS_BOUNDS and does nothing.)
 *
 * attn_fwd_bounds_selftest runs attn_fwd on tiny caller buffers (contract of
 * attn_fwd, no mask, b*h*sq <= 4096, 1 <= sk <= 1024) with one work unit past
 * the end of the problem, whose head plane is out of range, synchronises and
 * returns the recorded status code (expected ATTN_STATUS_BOUNDS).  The
 * normal build returns ATTN_ERR_BUILD.
 */
int attn_fwd_bounds_selftest(const void *q, const void *k, const void *v,
                             void *o, float *lse, int64_t b, int64_t h,
                             int64_t sq, int64_t sk, int64_t d, float scale,
                             int dtype, void *stream);

/*
 * attn_bwd_bounds_selftest: the same for the backward -- attn_bwd on tiny
 * caller buffers (contract of attn_bwd, no mask, b*h*sq <= 4096, 1 <= sk <=
 * 1024) with one work unit past the end of the problem, whose index every
 * warp role checks before decoding it; synchronises and returns the
 * recorded status code (expected ATTN_STATUS_BOUNDS).  The normal build
 * returns ATTN_ERR_BUILD.
 */
int attn_bwd_bounds_selftest(const void *q, const void *k, const void *v,
                             const void *o, const void *dout,
                             const float *lse, void *dq, void *dk, void *dv,
                             int64_t b, int64_t h, int64_t sq, int64_t sk,
                             int64_t d, float scale, int dtype,
                             void *workspace, int64_t workspace_bytes,
                             void *stream);

/* Library version string. */
const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_FWD_H */
