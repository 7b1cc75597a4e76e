/*
 * attn.h -- C ABI of libattn.so: varlen causal attention over a paged KV
 * cache on one GB300 (sm_103a).
 *
 * The operations follow two pages:
 *  [vLLM-FA]  "FlashAttention deep dive" (vLLM V1 FlashAttention backend):
 *             flash_attn_varlen_func and its argument table, the KV cache
 *             shape (2, num_blocks, block_size, num_kv_heads, head_size),
 *             reshape_and_cache_flash, cascade attention and
 *             merge_attn_states, the FP8 KV cache.
 *  [MR]       "vLLM 中 Attention Kernel 如何并行处理多个请求": packed requests
 *             (sec. 1, 5), tile classification (sec. 3-4), online softmax
 *             (sec. 7), decode (sec. 9), bottom-right causal alignment
 *             (sec. 10), paged lookup (sec. 11), split-KV segments merged by a
 *             second reduction kernel (sec. 12).
 *
 * Conventions shared by every entry point
 *  - All tensor pointers are DEVICE pointers owned by the caller.  No call
 *    allocates or frees device memory, and none keeps a caller's pointer
 *    after it returns.  Scratch space comes from the caller through
 *    (workspace, ws_bytes).  The library itself holds two fixed device
 *    arrays, loaded with it on every GPU that uses it: the error word
 *    (4 bytes) and the 8 MiB scratch of attn_paged_decode_noalloc.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *    does no host synchronisation, so a call can be captured in a CUDA graph
 *    when its pointers and host scalars stay fixed.
 *  - A call's workspace is its own while the call runs: calls that may run
 *    at the same time (other streams, other host threads, graph replays)
 *    need separate workspaces.  Nothing else is shared between calls: the
 *    tensor-core kernel's work counter lives in the call's workspace and is
 *    zeroed by the call itself.
 *  - Arguments are validated on the host before anything is launched.  On a
 *    non-zero status nothing was launched and no memory was touched.
 *  - Block ids and slots are also checked inside the kernels: an id outside
 *    [0, num_blocks) or a slot outside [0, num_blocks * block_size) is never
 *    dereferenced and the device error word read by attn_device_error_flag()
 *    is raised.  KV write: the token is skipped.  Attention: the result of
 *    the affected request is unspecified (the rows-light kernel reads zero K
 *    and V for that block, the tensor-core kernel reads block 0 instead);
 *    every other request is unaffected.
 *  - Layouts are row-major with the last dimension contiguous:
 *      q, out      [T, Hq, D]        token stride given in elements
 *      lse         [T, Hq] fp32      natural-log log-sum-exp per query head
 *      k/v cache   [num_blocks, block_size, Hkv, D] each; the two halves of
 *                  the [vLLM-FA] cache tensor (kv_cache.unbind(0)) are passed
 *                  as separate pointers
 *      block_table [B, >= ceil(kv_len / block_size)] int32, row stride given
 *                  in elements; a pointer offset into a row (cascade suffix
 *                  view block_table[:, n:]) is allowed
 *  - Head size D is 64 or 128, Hq % Hkv == 0 (GQA: query head h reads KV
 *    head h / (Hq / Hkv)), block_size is a positive multiple of 16, and
 *    B and Hq are at most 65535 (ATTN_ERR_SHAPE otherwise).
 *  - Pointers must be 16-byte aligned and token strides multiples of 8
 *    elements (16 bytes for 16-bit types).
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *attn_stream_t; /* same type as cudaStream_t */

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_NULL = 1,        /* a required pointer is NULL */
    ATTN_ERR_SHAPE = 2,       /* inconsistent sizes, strides or counts */
    ATTN_ERR_DTYPE = 3,       /* unsupported dtype or dtype combination */
    ATTN_ERR_ALIGN = 4,       /* pointer / stride not 16-byte aligned */
    ATTN_ERR_BLOCK_SIZE = 5,  /* block_size not a positive multiple of 16 */
    ATTN_ERR_HEAD_SIZE = 6,   /* head size not 64 or 128 */
    ATTN_ERR_WORKSPACE = 7,   /* workspace NULL or smaller than required */
    ATTN_ERR_CUDA = 8,        /* a CUDA runtime call failed (no device, launch error) */
    ATTN_ERR_DEVICE = 9,      /* the current device is not an sm_103 GPU */
    ATTN_ERR_TABLE = 10       /* ATTN_DEBUG_VALIDATE=1 or attn_validate_*: an
                                 integer table breaks the contract */
} attn_status;

typedef enum {
    ATTN_BF16 = 0,
    ATTN_FP16 = 1,
    ATTN_FP8_E4M3 = 2,        /* float8 e4m3 "fn": bias 7, no inf, max 448 */
    ATTN_FP32 = 3
} attn_dtype;

/*
 * attn_varlen_prefill -- [vLLM-FA] flash_attn_varlen_func over a paged cache
 * (argument table: q, k = key_cache, v = value_cache, out, cu_seqlens_q,
 * max_seqlen_q, seqused_k, max_seqlen_k, softmax_scale, causal,
 * block_table, k/v descale, num_splits, return of the softmax lse).
 *
 * For request r in [0, B): its query tokens are rows
 * [cu_seqlens_q[r], cu_seqlens_q[r+1]) of q; it has kv_len = seqused_k[r]
 * cached keys (the new tokens' keys included, written beforehand with
 * kv_cache_write).  Query i of the request sits at absolute position
 * ctx + i, ctx = kv_len - q_len ([MR] sec. 10), and with causal != 0 sees
 * keys j <= ctx + i; otherwise all kv_len keys.  Key j is read from block
 * block_table[r * bt_row_stride + j / block_size], row j % block_size
 * ([MR] sec. 11).
 *
 *   out[t, h, :] = softmax_j(softmax_scale * k_descale * q[t,h,:] . K_j)
 *                  @ (v_descale * V_j)
 *   lse_out[t, h] = log sum_j exp(softmax_scale * k_descale * q . K_j)
 *
 * A query with no visible key gets out = 0 and lse = -inf.
 *
 * q_dtype: ATTN_BF16 or ATTN_FP16 (out has the same type).
 * kv_dtype: q_dtype, or ATTN_FP8_E4M3 (k/v_descale multiply the stored
 *   values; pass 1.0 for 16-bit caches).  The kernels widen e4m3 by placing
 *   its fields into fp16 (exact for every finite code); the NaN code
 *   S.1111.111, which kv_cache_write stores only for NaN input, reads as
 *   +-480.
 * max_seqlen_q / max_seqlen_k: upper bounds of q_len / kv_len over the batch
 *   (host scalars used to size the launch; values larger than the truth are
 *   safe, smaller ones are an error the kernels cannot detect).
 * total_q: number of rows of q (= cu_seqlens_q[B]).
 * num_splits: number of KV segments per (request, KV head) for split-KV
 *   ([MR] sec. 12): 0 = choose automatically, 1 = no split.  Partial
 *   results go to the workspace and a second kernel merges them.
 * lse_out may be NULL.
 * workspace: device scratch (16-byte aligned) of at least
 *   attn_workspace_size(total_q, Hq, D, splits) bytes for the split count the
 *   call ends up using; with num_splits = 0 the automatic choice is capped
 *   to what fits in ws_bytes.  Its first 256 bytes hold the work counter of
 *   the tensor-core kernel, which takes requests of more than 64 packed rows
 *   (q_len * Hq / Hkv, head size 128): a call with
 *   max_seqlen_q * Hq / Hkv > 64 (and head size 128) needs those 256 bytes
 *   even with num_splits = 1, and returns ATTN_ERR_WORKSPACE without them.
 *   Other calls may pass workspace = NULL and ws_bytes = 0, which disables
 *   splitting.  The contents need no initial value and are scratch after
 *   the call.
 */
attn_status attn_varlen_prefill(
    const void *q, int64_t q_stride_tok,
    const void *k_cache, const void *v_cache,
    void *out, int64_t out_stride_tok, float *lse_out,
    const int32_t *cu_seqlens_q, const int32_t *seqused_k,
    const int32_t *block_table, int64_t bt_row_stride,
    int B, int total_q, int max_seqlen_q, int max_seqlen_k,
    int Hq, int Hkv, int D, int block_size, int num_blocks,
    attn_dtype q_dtype, attn_dtype kv_dtype,
    float softmax_scale, int causal, float k_descale, float v_descale,
    int num_splits, void *workspace, size_t ws_bytes, attn_stream_t stream);

/*
 * attn_varlen_prefill_ext -- attn_varlen_prefill with the attention
 * variants of [vLLM-FA]'s argument table and variant list (window_size,
 * softcap, s_aux: sliding window, soft cap on the logits, attention sinks).
 * The page names them without formulas; the readings are:
 *   window_left, window_right: query i at absolute position p = ctx + i
 *     sees keys j with p - window_left <= j <= p + window_right, on top of
 *     the causal rule and j < kv_len; -1 leaves that side unlimited.
 *   softcap > 0: each logit s = softmax_scale * k_descale * q . K_j
 *     becomes softcap * tanh(s / softcap) before the softmax; 0 = off.
 *   sinks: NULL, or a DEVICE array of Hq fp32 logits (natural-log units);
 *     the sink z_h of query head h joins the normalisation with a zero
 *     value vector:
 *       out = sum_j e^{s_j} V_j / (e^{z_h} + sum_j e^{s_j}),
 *       lse = log(e^{z_h} + sum_j e^{s_j})
 *     (a query with no visible key then gets out = 0, lse = z_h).
 * fp8 queries ([vLLM-FA] FA3 FP8 support, q_descale): q_dtype may be
 *   ATTN_FP8_E4M3 when kv_dtype is ATTN_FP8_E4M3 and D is 128; a query
 *   element's value is then code * q_descale, QK^T runs on e4m3 operands
 *   (K codes as stored: a NaN code in K or q gives NaN scores, unlike the
 *   widened +-480 above), out is bf16, and q_stride_tok must be a multiple
 *   of 16 elements.  For 16-bit queries pass q_descale = 1.
 * Errors as attn_varlen_prefill, plus ATTN_ERR_SHAPE for a window bound
 * below -1 or a negative or NaN softcap.  attn_varlen_prefill is this call
 * with q_descale 1, window (-1, -1), softcap 0 and no sinks.
 */
attn_status attn_varlen_prefill_ext(
    const void *q, int64_t q_stride_tok,
    const void *k_cache, const void *v_cache,
    void *out, int64_t out_stride_tok, float *lse_out,
    const int32_t *cu_seqlens_q, const int32_t *seqused_k,
    const int32_t *block_table, int64_t bt_row_stride,
    int B, int total_q, int max_seqlen_q, int max_seqlen_k,
    int Hq, int Hkv, int D, int block_size, int num_blocks,
    attn_dtype q_dtype, attn_dtype kv_dtype,
    float softmax_scale, int causal, float q_descale, float k_descale, float v_descale,
    int window_left, int window_right, float softcap, const float *sinks,
    int num_splits, void *workspace, size_t ws_bytes, attn_stream_t stream);

/*
 * attn_paged_decode -- one query token per request ([MR] sec. 9: the decode
 * row is the last row of the causal matrix, so all kv_len = seq_lens[r]
 * keys are visible).  q and out are [B, Hq, D] contiguous, lse_out [B, Hq].
 * Same as attn_varlen_prefill with cu_seqlens_q = [0, 1, ..., B] and
 * seqused_k = seq_lens; split-KV is on by default (num_splits 0).
 */
attn_status attn_paged_decode(
    const void *q, const void *k_cache, const void *v_cache,
    void *out, float *lse_out,
    const int32_t *seq_lens, const int32_t *block_table, int64_t bt_row_stride,
    int B, int max_seq_len, int Hq, int Hkv, int D, int block_size, int num_blocks,
    attn_dtype q_dtype, attn_dtype kv_dtype,
    float softmax_scale, float k_descale, float v_descale,
    int num_splits, void *workspace, size_t ws_bytes, attn_stream_t stream);

/*
 * attn_paged_decode_noalloc -- attn_paged_decode for callers that cannot
 * allocate device memory.  (The source pages have no counterpart: this is a
 * deployment convenience, not part of the method.)
 *
 * Who needs it: code that may not call cudaMalloc or an allocating library
 * routine -- for instance a plugin inside a host framework that owns every
 * device allocation, or a latency-critical serving loop where cudaMalloc /
 * cudaFree can synchronise the device and stall other work.  The caller
 * still passes q, the caches, out, lse_out and the tables; only the split-KV
 * scratch (per-segment partial outputs) is taken from a fixed array of
 * ATTN_NOALLOC_SCRATCH_BYTES that the library keeps in device memory.
 *
 * Arguments and results are those of attn_paged_decode without the
 * workspace.  num_splits = 0 picks the split count automatically and caps it
 * to what fits in the array; an explicit num_splits whose scratch
 * (attn_workspace_size(B, Hq, D, n) for the count n the call uses, which is
 * num_splits clamped to 256) exceeds ATTN_NOALLOC_SCRATCH_BYTES returns
 * ATTN_ERR_WORKSPACE and launches nothing.
 *
 * Notes for callers:
 *  - Every GPU that loads the library holds the array until the process
 *    exits, whether or not this entry point is used.
 *  - The first call on a device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and caches it; make that
 *    first call before any stream capture.
 *  - All calls on a device share the one array and it keeps whatever the
 *    last call left in it.  Nothing in it needs to start at zero (every slot
 *    read is written earlier in the same call), but calls whose execution
 *    overlaps on the GPU (different streams, or different host threads)
 *    race on it: serialise them.
 *  - Allocates nothing and calls no allocating routine.
 */
#define ATTN_NOALLOC_SCRATCH_BYTES (8u << 20)
attn_status attn_paged_decode_noalloc(
    const void *q, const void *k_cache, const void *v_cache,
    void *out, float *lse_out,
    const int32_t *seq_lens, const int32_t *block_table, int64_t bt_row_stride,
    int B, int max_seq_len, int Hq, int Hkv, int D, int block_size, int num_blocks,
    attn_dtype q_dtype, attn_dtype kv_dtype,
    float softmax_scale, float k_descale, float v_descale,
    int num_splits, attn_stream_t stream);

/*
 * attn_merge_states -- [vLLM-FA] merge_attn_states: combine two attention
 * results over disjoint key sets (cascade prefix and suffix):
 *   lse = log(exp(lse1) + exp(lse2)),
 *   out = exp(lse1 - lse) * o1 + exp(lse2 - lse) * o2.
 * o1, o2, out: [T, Hq, D] contiguous, all of `dtype` (bf16, fp16 or fp32);
 * lse1, lse2: [T, Hq] fp32; lse_out may be NULL.  A side with lse = -inf
 * has weight 0; both -inf gives out = 0, lse = -inf.  out may alias o1 or o2.
 */
attn_status attn_merge_states(
    void *out, float *lse_out,
    const void *o1, const float *lse1, const void *o2, const float *lse2,
    int T, int Hq, int D, attn_dtype dtype, attn_stream_t stream);

/*
 * kv_cache_write -- [vLLM-FA] reshape_and_cache_flash: token t of
 * key/value [T, Hkv, D] (token strides in elements) is stored at block
 * slot_mapping[t] / block_size, row slot_mapping[t] % block_size of both
 * caches.  slot_mapping[t] < 0 skips the token (padding).
 * src_dtype: ATTN_BF16 or ATTN_FP16.  kv_dtype: src_dtype (bit copy) or
 * ATTN_FP8_E4M3: each value x is stored as e4m3(x / scale) with the
 * division in fp32, round to nearest even, saturating at +-448
 * (k_scale for keys, v_scale for values).
 */
attn_status kv_cache_write(
    const void *key, int64_t key_stride_tok, const void *value, int64_t value_stride_tok,
    void *k_cache, void *v_cache, const int64_t *slot_mapping,
    int T, int Hkv, int D, int block_size, int num_blocks,
    attn_dtype src_dtype, attn_dtype kv_dtype, float k_scale, float v_scale,
    attn_stream_t stream);

/*
 * attn_workspace_size -- bytes of scratch attn_varlen_prefill /
 * attn_paged_decode need for `num_splits` KV segments: 256 bytes for the
 * tensor-core kernel's work counter, then fp32 partial outputs and
 * log-sum-exps for every (token, query head, segment).  256 when
 * num_splits <= 1.
 */
size_t attn_workspace_size(int total_q, int Hq, int D, int num_splits);

/*
 * attn_num_splits -- the split count attn_varlen_prefill(num_splits = 0)
 * would choose for these host scalars with bf16 query and cache at head
 * size 128 (attn_num_splits_typed: any head size and dtypes) (the decode
 * rule: enough segments to fill every SM a few times over, each segment at
 * least a few K/V tiles long).  Exposed for planning and tests.
 */
int attn_num_splits(int B, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int num_sms);

/*
 * attn_num_splits_typed -- the same choice for a given head size and query /
 * cache dtypes (the request classes and their kernels depend on them: an
 * e4m3 cache at head size 128 runs decode rows on its own kernel with its
 * own split target).  attn_num_splits is this call with D = 128 and bf16
 * query and cache.  Size a workspace with it for num_splits = 0 calls on
 * other dtypes.  Returns 1 for invalid head counts.
 */
int attn_num_splits_typed(int B, int max_seqlen_q, int max_seqlen_k, int Hq, int Hkv, int D, attn_dtype q_dtype,
                          attn_dtype kv_dtype, int num_sms);

/*
 * attn_tile_kind -- [MR] sec. 4 tile classification for a query tile holding
 * local positions [q_lo, q_hi) of a request with cached context ctx against
 * keys [k_lo, k_hi): 0 = skip (every key in the future of every query),
 * 1 = full (every key visible to every query), 2 = diagonal (needs the
 * element mask).  Host mirror of the rule the kernels apply.
 */
int attn_tile_kind(int q_lo, int q_hi, int k_lo, int k_hi, int ctx);

/*
 * attn_cascade -- [vLLM-FA] Cascade Attention in one call: every query
 * token attends to a prefix of keys shared by all requests and to its own
 * request's suffix, and the two states are merged by log-sum-exp
 * (merge_attn_states).  The result equals attn_varlen_prefill over the
 * concatenated block rows (prefix blocks, then the request's own), causal.
 *
 * Prefix half (the pages' cu_prefix_query_lens / prefix_kv_lens form):
 *   cu_prefix_query_lens  device int32 [2] = {0, total_q}
 *   prefix_kv_lens        device int32 [1] = {prefix_len}
 *   prefix_block_table    device int32, ceil(prefix_len / block_size) ids
 *   prefix_len            host copy of prefix_kv_lens[0]; a multiple of
 *                         block_size (ATTN_ERR_SHAPE otherwise), may be 0
 *   Every prefix key precedes every query: no mask.
 * Suffix half: cu_seqlens_q, suffix_kv_lens (the request's keys after the
 *   prefix, its new tokens' keys included), suffix_block_table (row stride
 *   bt_row_stride; a view block_table[:, prefix_len / block_size:] of the
 *   full table is allowed), max_seqlen_q, max_suffix_len: as in
 *   attn_varlen_prefill, causal with bottom-right alignment within the suffix.
 * Both halves write the partial states of their KV segments into one
 *   workspace array and a single combine writes out / lse_out (lse_out may
 *   be NULL): three launches instead of the five of two split calls and a
 *   merge.  prefix_splits / suffix_splits: segments of each half, 0 = the
 *   library's choice for the two halves running side by side
 *   (attn_cascade_splits).
 * workspace: at least attn_workspace_size(total_q, Hq, D, ns_p + ns_s) bytes
 *   (16-byte aligned) for the counts the call uses; ATTN_ERR_WORKSPACE
 *   otherwise.
 * aux_stream: a second stream for the prefix half, forked from `stream`
 *   after the work already queued there and joined before the combine (the
 *   library records two events it owns per host thread and device); NULL or
 *   equal to `stream`: both halves on `stream`.  Capturable in a CUDA graph
 *   (fork and join become graph edges).
 * Types, head sizes, alignment and errors as attn_varlen_prefill, with
 * 16-bit q (out in q's type) over a cache of q's type or e4m3.
 */
attn_status attn_cascade(
    const void *q, int64_t q_stride_tok, const void *k_cache, const void *v_cache,
    void *out, int64_t out_stride_tok, float *lse_out,
    const int32_t *cu_prefix_query_lens, const int32_t *prefix_kv_lens,
    const int32_t *prefix_block_table, int prefix_len,
    const int32_t *cu_seqlens_q, const int32_t *suffix_kv_lens,
    const int32_t *suffix_block_table, int64_t bt_row_stride,
    int B, int total_q, int max_seqlen_q, int max_suffix_len,
    int Hq, int Hkv, int D, int block_size, int num_blocks,
    attn_dtype q_dtype, attn_dtype kv_dtype, float softmax_scale,
    float k_descale, float v_descale, int prefix_splits, int suffix_splits,
    void *workspace, size_t ws_bytes, attn_stream_t stream, attn_stream_t aux_stream);

/*
 * attn_cascade_splits -- the segment counts attn_cascade(prefix_splits = 0,
 * suffix_splits = 0) chooses for these host scalars on num_sms SMs: each
 * half gets a share of the SMs in proportion to its estimated time alone
 * (the prefix's tensor-core work, the suffix's cache bytes) and enough
 * segments to fill it.  Returns 0, or -1 for invalid sizes.
 */
int attn_cascade_splits(int B, int total_q, int max_seqlen_q, int prefix_len, int max_suffix_len, int Hq,
                        int Hkv, int D, int q_dtype, int kv_dtype, int num_sms, int *prefix_splits,
                        int *suffix_splits);

/*
 * Debug validation of the integer tables ("FlashAttention deep dive",
 * flash_attn_varlen_func argument table; [MR] sec. 10-11).
 *
 * With ATTN_DEBUG_VALIDATE set to a non-empty value other than "0" in the
 * environment, attn_varlen_prefill(_ext), attn_paged_decode(_noalloc) and
 * kv_cache_write copy their integer tables to the host after the work
 * already queued on `stream`, synchronise the stream, and return
 * ATTN_ERR_TABLE (launching nothing) when a check below fails.  The block
 * table is read only where the kernels would read it (ceil(kv_len /
 * block_size) entries a row), and only after every kv_len has been checked
 * against max_seqlen_k and the row stride.  Calls on a stream that is
 * being captured into a CUDA graph are not checked (no synchronisation is
 * possible there).  Without the variable no call reads its tables on the
 * host.
 *
 * attn_validate_tables -- the same checks on tables the caller holds in
 * HOST memory.  cu_seqlens_q may be NULL (decode: request r owns query row
 * r, and total_q must equal B); block_table holds B rows of bt_row_stride
 * entries.  ATTN_ERR_TABLE when
 *   cu_seqlens_q[0] != 0, cu_seqlens_q[B] != total_q, or a q_len is
 *   negative or above max_seqlen_q;
 *   a kv_len (seqused_k[r]) is negative or above max_seqlen_k;
 *   causal != 0 and kv_len < q_len (the new tokens' keys are part of kv_len);
 *   B > 1 and ceil(kv_len / block_size) > bt_row_stride;
 *   a block id among the first ceil(kv_len / block_size) of its row is
 *   outside [0, num_blocks).
 * ATTN_ERR_SHAPE for negative sizes, ATTN_ERR_NULL for a missing table.
 *
 * attn_validate_slots -- HOST slot_mapping of T tokens: ATTN_ERR_TABLE when
 * a slot is below -1 (padding) or at least num_blocks * block_size.
 *
 * attn_debug_validate_enabled -- 1 when the environment switch is on.
 */
attn_status attn_validate_tables(const int32_t *cu_seqlens_q, const int32_t *seqused_k,
                                 const int32_t *block_table, int64_t bt_row_stride, int B, int total_q,
                                 int max_seqlen_q, int max_seqlen_k, int block_size, int num_blocks, int causal);
attn_status attn_validate_slots(const int64_t *slot_mapping, int T, int block_size, int num_blocks);
int attn_debug_validate_enabled(void);

/* Human-readable name of a status code. */
const char *attn_status_string(attn_status s);

/*
 * attn_device_error_flag -- read (and with reset != 0, clear) the device
 * error word of the current device: bit 0 = a block id outside
 * [0, num_blocks) was met, bit 1 = a slot outside the cache was met, bit 2 =
 * a pipeline wait in the tensor-core kernel gave up after 2 s (an internal
 * error; that launch's output is invalid).
 * Returns -1 if the CUDA call failed.  Synchronises the device.
 */
int attn_device_error_flag(int reset);

/*
 * attn_selftest_wait_timeout -- failure-detection self-test of the bounded
 * waits (not an operation of the pages).  Launches one thread that waits,
 * through the same bounded wait as the tensor-core kernel's pipeline, on an
 * mbarrier phase that nothing completes.  After the wait limit (2 s) it
 * gives up and raises bit 2 (timeout) of the device error word, which
 * attn_device_error_flag() then reports; the context stays usable.
 * Asynchronous on `stream`.  ATTN_ERR_CUDA or ATTN_ERR_DEVICE as the other
 * entry points.
 */
attn_status attn_selftest_wait_timeout(attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
