/*
 * fa.h -- C ABI of the GB300 (sm_103a) exact-attention forward library, libfa.so.
 *
 * The library computes exact scaled-dot-product attention and the per-row
 * log-sum-exp:
 *     O   = softmax(scale * Q K^T) V
 *     LSE = ln( sum_j exp(scale * q . k_j) )       (natural log, one value per query row)
 * ("FlashAttention 1-4 详解" (pinghaoyang.com.cn), section 原算法 for the definition;
 *  "flash-attention" (ai-reference-codex.pages.dev), sections 2.1 and 2.3 for the
 *  out + softmax_lse pair written by the fused forward kernel.)
 * It never materialises the N x N score or probability matrices: every call runs a
 * fused kernel that keeps the online-softmax state (running max m, running sum l,
 * rescaled output accumulator; "FlashAttention 1-4 详解", section Online Softmax
 * 数学推导) on chip.
 *
 * Conventions shared by every call
 *   - Element type: Q, K, V and O are all bf16 or all fp16 (fa_dtype, "flash-attention"
 *     section 5: fp16 / bf16 only); LSE is fp32.  S, l and O accumulate in fp32.
 *   - Head dimension d: a multiple of 8 from 8 to 256 for the forward and decode calls, to
 *     128 for the backward (the upstream limit is "d <= 256 and a multiple of 8" --
 *     "flash-attention", section 5).  The kernels run at width 64 (d <= 64), 128 or 256;
 *     the columns past d are read as zeros and never written.
 *   - Grouped-query attention: Hkv must divide Hq; query head h reads key/value head
 *     h / (Hq / Hkv) ("flash-attention", capabilities table, MQA / GQA row).
 *   - Causal masking is aligned bottom-right: query i of Nq sees key j of Nk when
 *     j <= i + (Nk - Nq).  Rows that see no key produce O = 0 and LSE = -inf.
 *   - All pointers are caller-owned DEVICE memory (unless stated otherwise).  The library
 *     does not allocate, free or synchronise: it validates, then enqueues kernels on the
 *     caller's stream and returns.  Outputs are valid once that stream reaches them.
 *   - Alignment (TMA): q, k, v, k_cache and v_cache must be 16-byte aligned and every
 *     stride a multiple of 8 elements; o must be 16-byte aligned with strides a
 *     multiple of 8 elements; lse 4-byte aligned.
 *   - Errors: arguments are validated on the host before any CUDA call; an invalid call
 *     returns a non-zero fa_status and enqueues nothing.  FA_ERR_CUDA means a CUDA call
 *     failed; fa_last_cuda_error() gives its text.  Faults detected on the device (a
 *     bounded wait that ran out, an out-of-range sequence length) are recorded in a
 *     per-device error word that fa_get_last_device_error() reads.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O. */
typedef enum fa_dtype {
    FA_BF16 = 0, /* bfloat16 */
    FA_FP16 = 1, /* IEEE binary16 */
    FA_E4M3 = 2  /* 8-bit float E4M3 (torch.float8_e4m3fn): the inputs of fa_fwd_fp8, the
                    caches of fa_fwd_kvcache_fp8 */
} fa_dtype;

typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, bad size, Hq % Hkv != 0, misaligned pointer/stride */
    FA_ERR_UNSUPPORTED = 2, /* d not a multiple of 8 in [8, 256] (forward and decode calls)
                               or [8, 128] (backward), dtype not a fa_dtype, or the current
                               device is not an sm_103 GPU */
    FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed: see fa_last_cuda_error() */
    FA_ERR_WORKSPACE = 4,   /* workspace pointer null or smaller than required */
    FA_ERR_TIMEOUT = 5,     /* a device-side wait gave up (reported by fa_get_last_device_error) */
    FA_ERR_CONCURRENT = 6   /* reported by fa_get_last_device_error: a forward or decode launch
                               found its work-ticket counter shared with another launch running
                               at the same time (see "Work tickets" below); its outputs are not
                               valid */
} fa_status;

/*
 * Work tickets.  The forward (fa_fwd, fa_fwd_varlen, fa_fwd_fp8, fa_fwd_host) and decode
 * (fa_fwd_kvcache*, fa_fwd_kvcache_noalloc) kernels hand out their work tiles dynamically:
 * the CTAs of a launch take tickets from a counter in a 256-entry table compiled into the
 * library, one table per call kind, and the host gives each launch the next entry in turn
 * (the entry is fixed when the call is made, so a captured CUDA graph replays with the
 * entry it was captured with).  Two launches that use the same entry must not run at the
 * same time: do not replay one captured call concurrently with itself (on two streams, or
 * from two graphs running at once), and keep fewer than 256 forward (or decode) launches in
 * flight at once.  Launches on one stream never overlap.  A launch that finds its counter
 * disturbed by another sets FA_ERR_CONCURRENT in the device error word (a check made when
 * its last CTA finishes; it catches a shared entry in most cases, not in every case).
 */

/*
 * Score modifiers: the sliding window, softcap and ALiBi variants named in the
 * capabilities table of "flash-attention" (causal / sliding window / ALiBi / softcap).
 * The pages give no formulas; this library reads them as follows.  With
 * pos = i + (Nk - Nq) the bottom-right position of query i (for decode, the query is the
 * last of cache_seqlens[b] tokens: pos = cache_seqlens[b] - 1):
 *   - window: key j is visible when pos - window_left <= j <= pos + window_right; a
 *     negative bound is unbounded.  causal != 0 forces window_right = 0.  Used only when
 *     use_window != 0 (so a zero-filled struct changes nothing).
 *   - softcap > 0: the scaled score z = scale * q . k_j becomes softcap * tanh(z / softcap).
 *     0 disables it; negative or non-finite values are rejected (FA_ERR_INVALID_ARG).
 *   - alibi_slopes: NULL, or DEVICE fp32 slopes, slope of (batch b, query head h) at
 *     alibi_slopes[b * alibi_batch_stride + h] (stride 0 shares one row of Hq slopes).
 *     The score (after the softcap) gets -slope * |pos - j| added.  4-byte aligned;
 *     alibi_batch_stride >= 0.
 * The softmax and the LSE are then taken over the modified scores of the visible keys;
 * rows that see no key give O = 0 and LSE = -inf.  A NULL fa_score_mod pointer (or a
 * zero-filled struct) means no modifier.
 */
typedef struct fa_score_mod {
    int use_window;
    int window_left;
    int window_right;
    float softcap;
    const float *alibi_slopes;
    int64_t alibi_batch_stride;
} fa_score_mod;

/*
 * Dense batched attention, the flash_attn_func call of "flash-attention" section 1:
 * q/k/v in the (batch, seqlen, nheads, headdim) layout; element type `dtype` (fa_dtype).
 *   q   : [B, Nq, Hq,  d], element (b,n,h,c) at q + b*q_strides[0] + n*q_strides[1]
 *                                                    + h*q_strides[2] + c
 *   k, v: [B, Nk, Hkv, d] bf16, same convention with k_strides / v_strides
 *   o   : [B, Nq, Hq,  d] bf16 output, same convention with o_strides
 *   lse : [B, Hq, Nq] fp32 output, contiguous
 * Strides are in elements; the head dimension has unit stride.  d: a multiple of 8 up to
 * 256 (the capabilities table of "flash-attention": head_dim <= 256, multiple of 8).
 * scale multiplies the scores before the softmax (usually 1/sqrt(d)); causal != 0
 * applies the bottom-right causal mask; mod holds the score modifiers (zero-filled = none).
 * Nk = 0 is allowed (O = 0, LSE = -inf); B = 0 or Nq = 0 is a no-op.
 */
typedef struct fa_fwd_params {
    const void *q;
    const void *k;
    const void *v;
    void *o;
    float *lse;
    int B, Nq, Nk, Hq, Hkv, d;
    int64_t q_strides[3], k_strides[3], v_strides[3], o_strides[3]; /* (b, n, h) */
    float scale;
    int causal;
    int dtype; /* fa_dtype of q, k, v and o */
    fa_score_mod mod;
} fa_fwd_params;

fa_status fa_fwd(const fa_fwd_params *p, cudaStream_t stream);

/*
 * fa_fwd with the tensors in host memory: p->q, k, v, o and lse are HOST pointers (page-
 * locked, so that the copies run asynchronously), in the contiguous layouts [B, Nq, Hq, d],
 * [B, Nk, Hkv, d] and [B, Hq, Nq] (the strides in p must be those); dev_q, dev_k, dev_v,
 * dev_o, dev_lse are caller-owned DEVICE buffers of the same shapes, overwritten by the
 * call.  Enqueues the copies in, the computation and the copies out, ordered after earlier
 * work on `stream`; later work on `stream` sees O and LSE in host memory.  The query rows
 * of each batch entry are split into up to `chunks` ranges (1..64) so that copying one
 * range overlaps computing the previous one: when no row sees keys past its own position
 * (causal, or a right window bound of 0) a range needs only the key prefix up to its last
 * row, so K and V travel range by range too, and each range is computed as its own
 * bottom-right-aligned problem over that prefix (the same rows and LSE as the whole call);
 * otherwise the ranges are whole batch entries.  B x ranges <= 128.  The library keeps two
 * copy streams and their events per device for these calls (created on first use).
 * Errors as fa_fwd; FA_ERR_INVALID_ARG also for other strides or too many ranges.
 */
fa_status fa_fwd_host(const fa_fwd_params *p, void *dev_q, void *dev_k, void *dev_v,
                      void *dev_o, float *dev_lse, int chunks, cudaStream_t stream);

/*
 * Packed variable-length batch, the flash_attn_varlen_func call of "flash-attention"
 * section 1 (capabilities table, varlen row: sequences packed by cu_seqlens).
 *   q   : [total_q, Hq,  d] bf16, contiguous
 *   k, v: [total_k, Hkv, d] bf16, contiguous
 *   cu_seqlens_q, cu_seqlens_k: DEVICE int32 [B+1] prefix sums; sequence b owns query
 *         tokens [cu_seqlens_q[b], cu_seqlens_q[b+1]) and key tokens likewise.  They must
 *         start at 0, be non-decreasing and end at most at total_q / total_k; sequence
 *         b's query length must not exceed max_seqlen_q.  A sequence that breaks this is
 *         skipped and flagged in the device error word (FA_ERR_INVALID_ARG from
 *         fa_get_last_device_error).
 *   o   : [total_q, Hq, d] bf16 output, contiguous
 *   lse : [Hq, total_q] fp32 output, contiguous
 * Each sequence is attended on its own; causal and window alignment is per sequence.
 * dtype is the fa_dtype of q, k, v and o; mod the score modifiers (NULL = none; host
 * memory, read during the call).
 */
fa_status fa_fwd_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                        const int *cu_seqlens_q, const int *cu_seqlens_k, int B,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, float scale, int causal, int dtype,
                        const fa_score_mod *mod, cudaStream_t stream);

/*
 * Single-query decode against a padded KV cache, the flash_attn_with_kvcache call of
 * "flash-attention" section 1, computed with split-KV: the keys of each sequence are cut
 * into chunks, every (batch, kv head, chunk) writes a partial (O_s, LSE_s) to the
 * workspace, and a combine kernel merges them with weights exp(LSE_s - LSE)
 * ("flash-attention", code map: combine_attn_seqk_parallel; section 4 on folding the
 * query heads of one GQA group into one work unit).
 *   q            : [B, 1, Hq, d] bf16, contiguous
 *   k_cache/v_cache: [B, Lmax, Hkv, d] bf16 with element strides cache_strides (b, n, h)
 *                  (host array of 3), shared by both caches
 *   cache_seqlens: DEVICE int32 [B]; query b sees cache rows [0, cache_seqlens[b]).
 *                  Rows at or past that length are never read into the result.  A length
 *                  outside [0, Lmax] is clamped and flagged in the device error word.
 *   num_splits   : 0 picks the chunk length automatically; n > 0 uses chunks of
 *                  ceil(Lmax / n) keys rounded up to a multiple of 128.
 *   workspace    : DEVICE scratch of at least fa_fwd_kvcache_workspace_size(...) bytes,
 *                  256-byte aligned; owned by the caller, overwritten by the call.
 *   o            : [B, 1, Hq, d] bf16 output, contiguous
 *   lse          : [B, Hq] fp32 output, contiguous
 * Hkv must divide Hq (any group size: the query heads of one kv head are evaluated
 * together in work items of up to 8 heads, 4 at d > 128, that share the K/V stream).
 * dtype is the fa_dtype of q, the caches and o.
 * mod: score modifiers (NULL = none; host memory, read during the call).  Only the left
 * window bound can hide a cached key (the query is the last position); cache rows before
 * the window start take no part in the result.  ex: append / rotary / paged cache
 * (fa_kvcache_extras below; NULL = none; host memory, read during the call).
 */
size_t fa_fwd_kvcache_workspace_size(int B, int Hq, int Lmax, int d, int num_splits);

/*
 * Decode-step extras of fa_fwd_kvcache ("flash-attention", section 1: the decode call
 * updates the KV cache in place and applies rotary in the same step; capabilities table,
 * KV cache row: in-place append, paged KV).  The pages give no formulas; this library
 * reads them as follows.  A NULL pointer (or a zero-filled struct) means none of them.
 *
 * In-place append (k_new, v_new non-NULL): one new token per sequence.  Its key and value
 * ([B, 1, Hkv, d], element strides new_strides (b, n, h), the type of the cache) are
 * written to logical cache row cache_seqlens[b] BEFORE the attention, which then covers
 * cache_seqlens[b] + 1 keys.  cache_seqlens itself is not modified.  A sequence whose row
 * would fall outside the cache (cache_seqlens[b] >= Lmax, or a block-table entry outside
 * [0, num_pages)) is not written and is flagged in the device error word.
 *
 * Rotary (rotary_cos, rotary_sin non-NULL; only with an append): DEVICE fp32 tables
 * [rotary_positions, rotary_dim / 2].  The query and the new key are turned by the angle
 * of position p = cache_seqlens[b]: dimension pairs (a, b) of the first rotary_dim
 * dimensions -- (i, i + rotary_dim/2), or (2i, 2i+1) with rotary_interleaved -- become
 *     y_a = x_a cos[p][i] - x_b sin[p][i],   y_b = x_a sin[p][i] + x_b cos[p][i],
 * evaluated in fp32 (one fused multiply-add per output) and rounded to the element type
 * (nearest even); the other dimensions are copied.  The rotated key is what the cache
 * keeps.  The rotated query is staged in `o` (which the call overwrites with the result
 * at the end), so o must not alias q.  rotary_dim is even, 2 <= rotary_dim <= d;
 * cache_seqlens[b] < rotary_positions (a sequence breaking this is flagged and not
 * appended).
 *
 * Paged cache (block_table non-NULL): k_cache / v_cache are [num_pages, page_size, Hkv, d]
 * with element strides cache_strides (page, row, head); logical row r of sequence b is
 * row r % page_size of page block_table[b * block_table_stride + r / page_size].  Lmax
 * is the logical maximum length, at most block_table_stride * page_size.  page_size is a
 * multiple of 128; entries outside [0, num_pages) are flagged (their rows read as 0).
 */
typedef struct fa_kvcache_extras {
    const void *k_new;
    const void *v_new;
    int64_t new_strides[3];
    const float *rotary_cos;
    const float *rotary_sin;
    int rotary_dim;
    int rotary_positions;
    int rotary_interleaved;
    const int *block_table;
    int block_table_stride;
    int page_size;
    int num_pages;
} fa_kvcache_extras;

fa_status fa_fwd_kvcache(const void *q, const void *k_cache, const void *v_cache,
                         const int *cache_seqlens, int B, int Lmax, int Hq, int Hkv, int d,
                         const int64_t cache_strides[3], float scale, int num_splits,
                         void *workspace, size_t workspace_bytes, void *o, float *lse,
                         int dtype, const fa_score_mod *mod, const fa_kvcache_extras *ex,
                         cudaStream_t stream);

/*
 * Single-query decode over an FP8 KV cache: fa_fwd_kvcache with k_cache / v_cache in E4M3
 * (torch.float8_e4m3fn bytes, the FP8 format of the FP8 forward pass the capabilities table
 * of "flash-attention" names) and a bf16 query and output.  Attended values are
 * k_descale[b * Hkv + g] * K and v_descale[b * Hkv + g] * V for kv head g of sequence b
 * (DEVICE fp32 [B, Hkv], 4-byte aligned; NULL means 1).  Scores, softmax and O accumulate in
 * fp32, as in fa_fwd_kvcache; E4M3 values are decoded exactly (a NaN code decodes to NaN).
 * d: a multiple of 16 from 16 to 256; cache strides (elements = bytes) multiples of 16.
 * Windows, softcap, ALiBi and paged caches (ex->block_table) apply as in fa_fwd_kvcache;
 * an append (ex->k_new) or rotary is FA_ERR_UNSUPPORTED.  Workspace: as fa_fwd_kvcache,
 * fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, num_splits) bytes.  Errors as
 * fa_fwd_kvcache.
 */
fa_status fa_fwd_kvcache_fp8(const void *q, const void *k_cache, const void *v_cache,
                             const int *cache_seqlens, int B, int Lmax, int Hq, int Hkv, int d,
                             const int64_t cache_strides[3], float scale, int num_splits,
                             const float *k_descale, const float *v_descale, void *workspace,
                             size_t workspace_bytes, void *o, float *lse,
                             const fa_score_mod *mod, const fa_kvcache_extras *ex,
                             cudaStream_t stream);

/*
 * Split-KV decode that allocates nothing.  Same computation, arguments, outputs and limits
 * (head dimensions 8..256, every group size fa_fwd_kvcache takes) as fa_fwd_kvcache with
 * bf16 inputs and no score modifiers or extras, minus the workspace; with the same
 * num_splits the two calls return the same bits.  (The paper has no counterpart: this
 * entry point exists for callers of this library, not for the method.)
 *
 * Some callers cannot allocate device memory at call time and have no buffer set aside
 * to pass as a workspace -- for example code running as a plugin inside another runtime
 * that hands it no workspace, or a serving loop that keeps cudaMalloc (which can
 * synchronise the whole device) out of its decode step.  This call writes the split
 * partials to a scratch array compiled into the library instead: a file-scope __device__
 * array of FA_NOALLOC_SCRATCH_BYTES (64 MiB) that every GPU which loads the library holds
 * until the process exits.  It calls no cudaMalloc, cudaFree or other allocating routine.
 *   - A call whose partials need more than FA_NOALLOC_SCRATCH_BYTES
 *     (fa_fwd_kvcache_workspace_size(B, Hq, Lmax, d, num_splits) > the maximum) is
 *     rejected with FA_ERR_WORKSPACE before anything is enqueued; use fa_fwd_kvcache with
 *     your own workspace for it, or fewer splits (num_splits > 0).
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and caches it; make that first call
 *     before any stream capture.
 *   - All calls on a device share the one array, which keeps the last call's contents.
 *     Nothing in it needs to start at zero (each partial is written before it is read),
 *     but calls that overlap on the GPU -- on different streams, or from graphs running at
 *     the same time -- race on it; the caller must keep them from overlapping.
 */
#define FA_NOALLOC_SCRATCH_BYTES (64u << 20)

fa_status fa_fwd_kvcache_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                 const int *cache_seqlens, int B, int Lmax, int Hq, int Hkv,
                                 int d, const int64_t cache_strides[3], float scale,
                                 int num_splits, void *o, float *lse, cudaStream_t stream);

/*
 * Backward pass of fa_fwd (dense batched attention, causal or not, GQA), the gradients the
 * flash-attention page describes (sections 2.3 and 4): the forward keeps q, k, v, out and
 * softmax_lse; the backward recomputes P = exp(S * scale - LSE) block by block instead of
 * storing it, runs parallel over key blocks with dK and dV kept on chip, and accumulates
 * dQ across key blocks (in fp32, in the workspace).  For an upstream gradient dO:
 *     D_i = rowsum(dO_i * O_i),  dS = P * (dO V^T - D),
 *     dV = P^T dO,  dK = scale dS^T Q,  dQ = scale dS K
 * (GQA: dK and dV of a key/value head sum over the query heads that read it).
 *   q, o, dout, dq : [B, Nq, Hq, d] (strides as in fa_fwd_params)
 *   k, v, dk, dv   : [B, Nk, Hkv, d]
 *   d              : a multiple of 8 from 8 to 256 (above 128 the work of a key block runs
 *                    as two units, one per half of d, over 64-query steps, with the dQ
 *                    accumulator stored transposed; fa_bwd_workspace_size accounts for it)
 *   lse            : [B, Hq, Nq] fp32, the LSE fa_fwd wrote for the same q, k, v
 *   workspace      : DEVICE, fa_bwd_workspace_size(B, Nq, Hq, d) bytes, 256-byte aligned,
 *                    owned by the caller (the fp32 dQ accumulator, the D vector and the
 *                    counters that order the dQ additions in deterministic mode)
 * All 16-bit tensors share the element type `dtype`; P and dS enter the tensor cores as
 * 16-bit values, every product is accumulated in fp32.  dQ sums the key blocks' parts in
 * an unspecified order (two calls may differ in the last bits of dQ) unless
 * deterministic != 0, which fixes the order (key block 0, 1, 2, ...) at some cost in
 * speed ("flash-attention" section 5: deterministic backward, slower); dK and dV are
 * always deterministic.
 * With score modifiers (mod, the same as the forward call's) the gradients pass through
 * them: the window and the ALiBi bias change which pairs count and P, a softcap c
 * multiplies dS by 1 - tanh^2(s / c).  Nk = 0 gives dQ = 0; Nq = 0 gives dK = dV = 0;
 * B = 0 is a no-op.
 */
typedef struct fa_bwd_params {
    const void *q, *k, *v, *o, *dout;
    const float *lse;
    void *dq, *dk, *dv;
    int B, Nq, Nk, Hq, Hkv, d;
    int64_t q_strides[3], k_strides[3], v_strides[3], o_strides[3], do_strides[3];
    int64_t dq_strides[3], dk_strides[3], dv_strides[3];
    float scale;
    int causal;
    int dtype;
    void *workspace;
    size_t workspace_bytes;
    int deterministic;
    fa_score_mod mod; /* the forward call's score modifiers (zero-filled = none) */
} fa_bwd_params;

size_t fa_bwd_workspace_size(int B, int Nq, int Hq, int d);

fa_status fa_bwd(const fa_bwd_params *p, cudaStream_t stream);

/*
 * Backward of fa_fwd_varlen (packed sequences delimited by cu_seqlens): the same gradients,
 * per sequence.  q, o, dout, dq: [total_q, Hq, d]; k, v, dk, dv: [total_k, Hkv, d], all
 * contiguous; lse: [Hq, total_q] fp32 from fa_fwd_varlen; cu_seqlens_q / _k: DEVICE int32
 * [B+1] as for fa_fwd_varlen (a sequence that breaks their rules is skipped and flagged in
 * the device error word).  workspace: fa_bwd_workspace_size(B, max_seqlen_q, Hq, d) bytes.
 * deterministic as in fa_bwd_params; mod: the forward call's score modifiers (NULL = none).
 */
fa_status fa_bwd_varlen(const void *q, const void *k, const void *v, const void *o,
                        const void *dout, const float *lse, void *dq, void *dk, void *dv,
                        const int *cu_seqlens_q, const int *cu_seqlens_k, int B,
                        int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                        int Hkv, int d, float scale, int causal, int dtype, void *workspace,
                        size_t workspace_bytes, int deterministic, const fa_score_mod *mod,
                        cudaStream_t stream);

/* sizeof(fa_bwd_params), for bindings that check their struct layout. */
size_t fa_bwd_params_size(void);

/*
 * Synchronises `stream`, then reads and clears the current device's error word.
 * Returns FA_OK when no kernel recorded a fault since the last read, FA_ERR_TIMEOUT when a
 * bounded device-side wait gave up (the kernel then stopped early and its outputs are
 * not valid), FA_ERR_INVALID_ARG when a device-resident argument (cu_seqlens,
 * cache_seqlens) was out of range, FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_get_last_device_error(cudaStream_t stream);

/* sizeof(fa_fwd_params), so that foreign-language bindings can check their struct layout. */
size_t fa_fwd_params_size(void);

/*
 * FP8 forward ("FlashAttention 1-4 详解", FlashAttention 3 engineering notes: FP8 tensor
 * cores in the forward pass).  p is read as for fa_fwd, with p->dtype = FA_E4M3: q, k, v
 * hold E4M3 bytes (strides in elements = bytes, multiples of 16 except where the extent is
 * 1), o is bf16 (o_strides in bf16 elements), lse fp32.  The attended values are
 * q_descale * Q, k_descale * K and v_descale * V with one factor per (batch, kv head):
 * fp32 device arrays [B, Hkv] (contiguous), each may be NULL (= 1).  So S = scale *
 * (dq dk) Q K^T and O = dv softmax(S) V.  P is rounded to E4M3 for the P V product; the
 * row sums and the LSE use the unrounded fp32 P.  The score modifiers (p->mod) and causal
 * apply as in fa_fwd.  d: a multiple of 16 up to 128.  Dense inputs (packed sequences:
 * fa_fwd_varlen_fp8).
 * workspace: device memory of at least fa_fwd_fp8_workspace_size(B, Nk, Hkv, d) bytes,
 * 256-byte aligned, for the transposed V (written by the call, no content needed).
 * Errors as fa_fwd; FA_ERR_WORKSPACE when the workspace is missing or too small.
 */
size_t fa_fwd_fp8_workspace_size(int B, int Nk, int Hkv, int d);
fa_status fa_fwd_fp8(const fa_fwd_params *p, const float *q_descale, const float *k_descale,
                     const float *v_descale, void *workspace, size_t workspace_bytes,
                     cudaStream_t stream);

/*
 * FP8 forward over packed sequences: the computation of fa_fwd_fp8 with the layout and the
 * sequence handling of fa_fwd_varlen.  q [total_q, Hq, d], k, v [total_k, Hkv, d], E4M3,
 * contiguous; o [total_q, Hq, d] bf16 and lse [Hq, total_q] fp32 as in fa_fwd_varlen;
 * cu_seqlens_q / cu_seqlens_k, B, max_seqlen_q / max_seqlen_k, causal (bottom-right aligned
 * per sequence) and mod as in fa_fwd_varlen.  q/k/v_descale: fp32 device arrays [B, Hkv],
 * one factor per (sequence, kv head), each may be NULL (= 1).  d: a multiple of 16 up to
 * 128; B <= 65535.
 * workspace: device memory of at least fa_fwd_varlen_fp8_workspace_size(B, total_k, Hkv, d)
 * bytes, 256-byte aligned, for the transposed V (each sequence's keys from a 16-aligned
 * column; written by the call, no content needed).
 * Errors as fa_fwd_varlen; FA_ERR_WORKSPACE when the workspace is missing or too small.
 */
size_t fa_fwd_varlen_fp8_workspace_size(int B, int total_k, int Hkv, int d);
fa_status fa_fwd_varlen_fp8(const void *q, const void *k, const void *v, void *o, float *lse,
                            const int *cu_seqlens_q, const int *cu_seqlens_k, int B,
                            int max_seqlen_q, int max_seqlen_k, int total_q, int total_k, int Hq,
                            int Hkv, int d, float scale, int causal, const fa_score_mod *mod,
                            const float *q_descale, const float *k_descale,
                            const float *v_descale, void *workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/* Static text for a status code. */
const char *fa_status_string(fa_status s);

/* Text of the last CUDA error seen by this thread inside the library ("" if none). */
const char *fa_last_cuda_error(void);

/*
 * Limit, in nanoseconds, on every device-side wait of the kernels launched after this
 * call (process-wide).  0 restores the default (10 s).  Testing aid: a very small value
 * makes the waits give up and return FA_ERR_TIMEOUT through fa_get_last_device_error
 * instead of computing, without faulting the GPU.
 */
void fa_set_wait_timeout_ns(unsigned long long ns);

/*
 * Failure injection, a testing aid (process-wide, for kernels launched after the call):
 * with withhold_loads != 0 the producer role of every attention kernel issues no load, so
 * the other roles' first waits cannot complete and run into the wait limit (set a short
 * one with fa_set_wait_timeout_ns); the call then reports FA_ERR_TIMEOUT through
 * fa_get_last_device_error and its outputs are unspecified.  Nothing faults and the
 * context stays usable.  0 (the default) turns it off.
 */
void fa_set_fault_injection(int withhold_loads);

/*
 * Forward kernel selection (process-wide, for calls made after it).  With enable != 0 the
 * 16-bit forward calls at head dimensions 72..128 (fa_fwd, fa_fwd_varlen, fa_fwd_host) run
 * on CTA pairs: clusters of two CTAs that compute each 256-row query sub-tile as one product
 * over both SMs' tensor cores (tcgen05 cta_group::2, the 2-CTA MMA mode of "FlashAttention
 * 1-4 详解", FlashAttention 4 section), each CTA loading half of every K and V tile.
 * enable = 0 (the default) selects the single-CTA kernel, which measures faster on the
 * causal and dense workloads.  Both give the same results (bit for bit in every case
 * tested; each call is deterministic).
 */
void fa_set_cta_pairs(int enable);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
