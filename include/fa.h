/*
 * fa.h -- C ABI of the exact tiled attention library for NVIDIA GB300 (sm_103a).
 *
 * Two operations, as the source pages define them:
 *
 *  fa_fwd             exact attention forward, O = softmax(scale * Q K^T [+ causal mask]) V,
 *                     plus the per-row log-sum-exp.  Page "flash-attention-v100", section
 *                     "How to use FlashAttention" (flash_attn_func: tensors
 *                     (batch, seqlen, nheads, headdim), grouped-query heads, default scale
 *                     1/sqrt(headdim)); section "Changelog", "2.1: Change behavior of causal
 *                     flag" (bottom-right aligned mask, all-masked rows give zero output);
 *                     page "ampere_flash_attention_from_scratch" (the FlashAttention-2 forward
 *                     that tiles Q row blocks over thread blocks and streams K/V tiles).
 *
 *  fa_decode_splitkv  single-token decode over a KV cache with per-sequence lengths, the KV
 *                     range cut into pieces processed by different thread blocks, each
 *                     writing a partial output and its log-sum-exp, then merged by a
 *                     separate kernel.  Page "flash-attention-v100", "Changelog",
 *                     "2.2: Optimize for inference" and flash_attn_with_kvcache
 *                     (cache_seqlens); page "flash attention-2 github" (Flash-Decoding,
 *                     steps 1-3).
 *
 * Conventions for every entry point:
 *  - Tensors are contiguous, row-major, 16-bit (bf16 or fp16 as `dtype` says):
 *    Q [B, Sq, Hq, D], K and V [B, Sk, Hkv, D], O [B, Sq, Hq, D]; LSE is fp32 [B, Hq, Sq].
 *    Hq must be a multiple of Hkv; Q head h reads K/V head h / (Hq / Hkv).
 *  - All pointers are device memory owned by the caller and must be 16-byte aligned.
 *    The library allocates nothing on these paths; the decode workspace is sized by
 *    fa_decode_workspace_bytes() and passed in.
 *  - Work is enqueued on `stream` and runs asynchronously; no entry point synchronises.
 *    Arguments are validated before anything is enqueued: a bad argument returns an error
 *    and enqueues nothing.  FA_ERR_CUDA reports a launch failure (cudaGetLastError).
 *  - Kernel-side waits are bounded: a wait that exceeds its limit makes the kernel unwind
 *    and records FA_ERR_TIMEOUT, read back with fa_last_device_status().
 *  - No C++ exception crosses this interface.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *fa_stream_t;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, non-positive size, Hq % Hkv != 0 */
    FA_ERR_UNSUPPORTED = 2, /* head dim not in {64, 96, 128, 256}, unknown dtype */
    FA_ERR_WORKSPACE = 3,   /* decode workspace missing or smaller than required */
    FA_ERR_CUDA = 4,        /* a CUDA runtime / driver call failed */
    FA_ERR_TIMEOUT = 5      /* a kernel gave up on a bounded wait (see fa_last_device_status) */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP16 = 1 } fa_dtype;

/*
 * Exact attention forward (FlashAttention-2 style: Q row blocks in parallel, K/V tiles
 * streamed, online softmax, the Sq x Sk score matrix never stored).
 *   q     [B, Sq, Hq, D]    k, v  [B, Sk, Hkv, D]    o  [B, Sq, Hq, D]  (dtype)
 *   lse   [B, Hq, Sq] fp32, natural log of sum_j exp(scale * q_i . k_j) over the visible
 *         keys; -inf for a row with no visible key (whose output row is 0).  May be NULL.
 *   scale softmax scale (the pages' default is 1/sqrt(D); the caller passes it).
 *   causal nonzero: key j is visible to query i iff j <= i + Sk - Sq.
 * Sizes: B, Sq, Sk, Hq, Hkv >= 1; D in {64, 96, 128, 256}; Hq % Hkv == 0.
 * Accumulation is fp32; P is rounded to the input dtype before the P.V product; O is
 * rounded once (round-to-nearest-even).  Deterministic: the same inputs give the same bits.
 */
FA_API fa_status fa_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Sq,
                 int Sk, int Hq, int Hkv, int D, float scale, int causal, fa_dtype dtype,
                 fa_stream_t stream);

/*
 * fa_fwd restricted to a sliding window (local attention; page "flash-attention-v100",
 * flash_attn_func window_size, and "Changelog", "2.3: Local (i.e., sliding window)
 * attention"): query i attends only to keys j with
 *     i + Sk - Sq - window_left <= j <= i + Sk - Sq + window_right,
 * where -1 leaves that side unbounded; with causal != 0 the right bound is additionally
 * j <= i + Sk - Sq.  K/V blocks outside every row's window are skipped, not masked.  A row
 * whose window holds no key gets O = 0 and LSE = -inf.  window_left/right >= -1, else
 * FA_ERR_INVALID_ARG; everything else as fa_fwd (which equals window (-1, -1)).
 */
FA_API fa_status fa_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse,
                               int B, int Sq, int Sk, int Hq, int Hkv, int D, float scale,
                               int causal, int window_left, int window_right, fa_dtype dtype,
                               fa_stream_t stream);

/*
 * Variable-length batch (page "flash-attention-v100", "Changelog", "2.0",
 * flash_attn_varlen_func): the B sequences are packed along the rows.
 *   q, o          [total_q, Hq, D]     k, v  [total_k, Hkv, D]      (dtype)
 *   cu_seqlens_q  device int32 [B + 1]: sequence b owns query rows
 *                 [cu_seqlens_q[b], cu_seqlens_q[b + 1]); cu_seqlens_k likewise for keys;
 *                 both non-decreasing, from 0, ending at most at total_q / total_k.
 *   lse           [Hq, total_q] fp32 (may be NULL).
 * Within a sequence everything is as fa_fwd_window: the causal mask is aligned to that
 * sequence's bottom-right corner.  A sequence with no keys gets O = 0 and LSE = -inf.
 * B <= 1024.  The offsets are read on the device; rows they place outside [0, total_q)
 * are not written, and keys outside [0, total_k) read as zero.
 */
FA_API fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                               const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int B,
                               int total_q, int total_k, int Hq, int Hkv, int D, float scale,
                               int causal, int window_left, int window_right, fa_dtype dtype,
                               fa_stream_t stream);

/*
 * Bytes of decode workspace fa_decode_splitkv needs for these sizes and `num_splits`
 * (the partial outputs [B, Hq, num_splits, D] fp32 and their log-sum-exps
 * [B, Hq, num_splits] fp32, each region 256-byte aligned).  0 for invalid sizes.
 * Host-only; needs no GPU.
 */
FA_API size_t fa_decode_workspace_bytes(int B, int Hq, int D, int num_splits);

/*
 * The split count fa_decode_splitkv uses when given num_splits <= 0: about eight partials
 * per SM over the B * Hkv (sequence, kv head) pairs, and no more than one per 256 keys of
 * max_kv_len.  It bounds how finely a pair may be cut (see num_splits below).  max_kv_len
 * is an upper bound on the KV lengths (the cache capacity Smax will do).  num_sms <= 0
 * queries the current device.  Returns >= 1, or -1 on an invalid argument or when no
 * device can be queried.
 */
FA_API int fa_decode_default_splits(int B, int Hkv, int max_kv_len, int num_sms);

/*
 * Split-KV decode for one query token per sequence.
 *   q        [B, 1, Hq, D]   k_cache, v_cache [B, Smax, Hkv, D]   (dtype)
 *   kv_lens  device int32 [B], 0 <= kv_lens[b] <= Smax: sequence b attends to cache
 *            positions [0, kv_lens[b]).  kv_lens[b] == 0 gives o = 0, lse = -inf.
 *   o        [B, 1, Hq, D] (dtype)      lse [B, Hq] fp32 (may be NULL)
 *   num_splits  the most pieces any (sequence, kv head) pair is cut into (<= 0: the
 *            default above).  The keys of all pairs, in 128-key tiles, are laid end to end
 *            in (b, kv head) order and cut into one equal range of W tiles per SM, W at
 *            least ceil(T / (num_splits - 1)) for the longest pair's T tiles (with
 *            num_splits == 1 no pair is cut).  Each piece of a pair writes a partial
 *            output and log-sum-exp, and a second kernel merges each pair's pieces.
 *            The kv heads are laid out in groups of g adjacent heads, g the largest of
 *            8, 4 and 2 that divides Hkv (else 1): a group is one entry, whose tiles count
 *            once, and the ranges go one per g SMs (the SM count rounded down to a
 *            multiple of g), one SM per head, so that the heads of a group get the same
 *            pieces and read the rows that sit side by side in the cache together.
 *   workspace   device memory of at least fa_decode_workspace_bytes(B, Hq, D, num_splits)
 *            bytes (after the default is applied); its contents need no initialisation.
 * Sizes: B, Hq, Hkv, Smax >= 1; B <= 1024; D in {64, 96, 128, 256}; Hq % Hkv == 0;
 * Hq / Hkv <= 16.
 * The result does not depend on num_splits beyond fp32 rounding.  Values of kv_lens
 * outside [0, Smax] are the caller's error and are clamped on the device.
 */
FA_API fa_status fa_decode_splitkv(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *kv_lens, void *o, float *lse, int B, int Hq, int Hkv,
                            int D, int Smax, float scale, int num_splits, void *workspace,
                            size_t workspace_bytes, fa_dtype dtype, fa_stream_t stream);

/*
 * Split-KV decode with Sq >= 1 query tokens per sequence (speculative or chunked decoding;
 * page "flash-attention-v100", flash_attn_with_kvcache with seqlen_q > 1 and the causal
 * flag of "Changelog", "2.1").
 *   q, o      [B, Sq, Hq, D] (dtype)     lse [B, Hq, Sq] fp32 (may be NULL)
 *   causal    nonzero: token s of sequence b sees cache keys j <= kv_lens[b] - Sq + s
 *             (the bottom-right aligned mask); zero: every token sees [0, kv_lens[b]).
 * (Hq / Hkv) * Sq <= 16.  The workspace is fa_decode_workspace_bytes(B * Sq, Hq, D,
 * num_splits).  A token that sees no key gets O = 0 and LSE = -inf.  Everything else as
 * fa_decode_splitkv, which is the Sq = 1 case.
 */
FA_API fa_status fa_decode_splitkv_multi(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *kv_lens, void *o, float *lse, int B,
                                         int Sq, int Hq, int Hkv, int D, int Smax, float scale,
                                         int causal, int num_splits, void *workspace,
                                         size_t workspace_bytes, fa_dtype dtype,
                                         fa_stream_t stream);

/*
 * fa_decode_splitkv over a paged KV cache (page "flash-attention-v100",
 * flash_attn_with_kvcache with block_table; "Changelog", "2.5: Paged KV cache").
 *   k_pages, v_pages   [num_pages, page_size, Hkv, D] (dtype): a pool of pages
 *   block_table        device int32 [B, max_pages_per_seq]: key r of sequence b is row
 *                      r % page_size of page block_table[b][r / page_size]
 *   kv_lens            device int32 [B], 0 <= kv_lens[b] <= page_size * max_pages_per_seq
 * page_size must be a multiple of 128 (the pages ask for multiples of 256, which are
 * accepted).  Table entries outside [0, num_pages) for pages a sequence uses are the
 * caller's error: those keys read as zeros, never outside the pool.  Everything else,
 * including the workspace (fa_decode_workspace_bytes(B, Hq, D, num_splits)) and the
 * split into pieces, is as fa_decode_splitkv with Smax = page_size * max_pages_per_seq.
 */
FA_API fa_status fa_decode_splitkv_paged(const void *q, const void *k_pages, const void *v_pages,
                                         const int32_t *block_table, const int32_t *kv_lens,
                                         void *o, float *lse, int B, int Hq, int Hkv, int D,
                                         int num_pages, int page_size, int max_pages_per_seq,
                                         float scale, int num_splits, void *workspace,
                                         size_t workspace_bytes, fa_dtype dtype,
                                         fa_stream_t stream);

/*
 * Split-KV decode for callers that cannot allocate device memory -- for example a plugin
 * running inside a host runtime that owns every device allocation, or a latency-critical
 * serving loop that must never call cudaMalloc (which may synchronise the device).  The
 * source pages have no counterpart to this entry point; it exists for those callers.
 *
 * Same arguments and results as fa_decode_splitkv, minus the workspace: the partial
 * results go to a fixed scratch array of FA_DECODE_NOALLOC_SCRATCH_BYTES that lives in
 * the library's device image (every GPU that loads the library holds it until the process
 * exits).  The call allocates nothing and calls no allocating routine.
 *  - Limit: sizes whose workspace, fa_decode_workspace_bytes(B, Hq, D, num_splits) after
 *    the default split count is applied, exceeds FA_DECODE_NOALLOC_SCRATCH_BYTES are
 *    rejected with FA_ERR_WORKSPACE before anything is enqueued.
 *  - Set-up: the first call on each device (with that device current) looks up the
 *    array's device address once and keeps it; later calls reuse it.
 *  - Sharing: every call on a device uses the same array and leaves its contents behind.
 *    Nothing in it needs to start at zero (each call writes every partial it reads), but
 *    calls whose kernels overlap on the GPU (e.g. on two streams at once) race on it.
 */
#define FA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

FA_API fa_status fa_decode_splitkv_noalloc(const void *q, const void *k_cache,
                                           const void *v_cache, const int32_t *kv_lens, void *o,
                                           float *lse, int B, int Hq, int Hkv, int D, int Smax,
                                           float scale, int num_splits, fa_dtype dtype,
                                           fa_stream_t stream);

/* Static, human-readable name of a status code. */
FA_API const char *fa_status_string(fa_status s);

/*
 * Reads and clears the sticky device status word of the current device that kernels
 * write when a bounded wait gives up (FA_ERR_TIMEOUT); FA_OK if none did.  Synchronises
 * the current device.  FA_ERR_CUDA if the device cannot be queried.
 */
FA_API fa_status fa_last_device_status(void);

/*
 * Self-test of the bounded-wait path that every kernel's barrier waits use.  Enqueues one
 * CTA of two warps on `stream`.  Warp 0 waits on an mbarrier phase that no thread
 * completes.  After the wait limit (2 s of GPU time) it gives up, records FA_ERR_TIMEOUT in
 * the device status word and raises the CTA's abort flag.  Warp 1 starts the same kind of
 * wait 0.5 s later and leaves when it sees the flag.  Nothing faults: every wait ends by
 * itself, and the context stays usable.
 *   result  device int32[3], caller-owned, 16-byte aligned.  It receives:
 *           [0] 1 if warp 0's wait gave up;
 *           [1] 1 if warp 1 left on the abort flag before its own limit;
 *           [2] warp 0's wait in milliseconds.
 * Read the status afterwards with fa_last_device_status(), which also clears it.
 * FA_ERR_INVALID_ARG for a null or misaligned result; FA_ERR_CUDA if the launch failed.
 */
FA_API fa_status fa_selftest_bounded_wait(int *result, fa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
