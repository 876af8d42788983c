/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV-cache attention library.
 *
 * What it computes
 * ----------------
 * Scaled dot-product attention softmax(q K^T * scale + M) V for the decode
 * phase (one new query row per sequence) and for causal prefill chunks (many
 * query rows per sequence), over a PagedAttention KV cache: K and V live in
 * fixed-size physical blocks of 16 tokens that each sequence reaches through
 * its row of a block table, and new tokens' K/V are appended through a
 * slot mapping.  Query head h reads KV head floor(h / G), G = n_q / n_kv
 * (MHA: G = 1, GQA: 1 < G < n_q, MQA: n_kv = 1).
 *
 * Sources (page title, section):
 *  - "注意力演进与推理流程" (attention evolution and inference, jerryiiii.gitbook.io):
 *    section 1.1 (SDPA with causal mask M), section 3.1 (GQA group rule
 *    g = floor(h / G)), 变革 1 (PagedAttention: fixed blocks, e.g. 16 tokens,
 *    allocated on demand), 变革 3 (chunked prefill).
 *  - vLLM concepts deep dive, section 1 (yyzxw.github.io): decode attention
 *    Attention(q_t, K_<=t, V_<=t); attention kernels receive a block table and
 *    a slot mapping instead of contiguous K/V pointers.
 *  - "LLM 推理全过程的维度变化与核心公式" (research.frankk.site, LLM inference
 *    walkthrough): section "Decode 阶段维度流转" (write K/V at cache_len, then
 *    read the whole cache; decode needs no causal mask), section "KV Cache 的
 *    形状与增长" (paged blocks change only the layout), section "工程优化怎么嵌进
 *    公式" (Flash-Decoding: split cache_len, then a log-sum-exp reduction;
 *    chunked prefill leaves the formula unchanged).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All data pointers are DEVICE pointers owned by the caller; the library
 *    allocates nothing at run time and keeps no pointer after it returns.
 *    Its global state: a per-device cache of SM counts and kernel attributes,
 *    and one file-scope device array of PKV_STATIC_SCRATCH_BYTES (held by every
 *    GPU that loads the library) with its cached per-device address, used only
 *    by paged_attention_decode_static_scratch and shared by all its calls.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call only enqueues work on that stream and returns; it
 *    never synchronises.  Ordering between calls is the caller's: append the
 *    new tokens (kv_reshape_and_cache) before attending over them, on the
 *    same stream.
 *  - Layouts (all row-major, contiguous):
 *      k_cache, v_cache : bf16 [num_blocks][num_kv_heads][block_size][head_dim]
 *                         (one (block, head) tile of 16 x 128 bf16 is 4096
 *                         contiguous bytes; base 16-byte aligned)
 *      block_tables     : int32 [num_seqs][max_blocks_per_seq]; entries past
 *                         ceil(context_len / block_size) are never read
 *      context_lens     : int32 [num_seqs]; counts the tokens of this step
 *      q                : bf16 [rows][num_q_heads][head_dim]
 *      out              : out_dtype [rows][num_q_heads][head_dim]
 *  - Supported shapes: head_dim 128, block_size 16, bf16 K/V/q,
 *    num_q_heads % num_kv_heads == 0 with G <= 8 or G a multiple of 8.
 *  - Return value: PKV_OK or a negative PKV_ERR_* code; no exception crosses
 *    the ABI.  Argument errors are detected before anything is enqueued.
 *  - Data that only the device sees (context lengths, block ids) is checked
 *    by the kernels: a context length outside [1, max_blocks_per_seq *
 *    block_size] or a block id outside [0, num_blocks) never causes an
 *    out-of-bounds access; the offending block contributes nothing, a
 *    length < 1 yields zero output rows, and a PKV_STATUS_* bit is ORed into
 *    the 32-bit status word at byte 0 of the workspace.
 *    The word is sticky: clear it (e.g. cudaMemsetAsync) to reset.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element types. */
typedef enum pkv_dtype {
    PKV_DTYPE_BF16 = 0,     /* bfloat16 */
    PKV_DTYPE_FLOAT32 = 1,  /* IEEE binary32 */
    PKV_DTYPE_FP8_E4M3 = 2  /* 8-bit float: 1 sign, 4 exponent (bias 7), 3 mantissa bits, max 448 */
} pkv_dtype;

/* Description of the physical block pool shared by K and V. */
typedef struct pkv_cache_desc {
    int32_t num_blocks;    /* physical blocks in the pool (>= 1) */
    int32_t block_size;    /* tokens per block; must be 16 */
    int32_t num_kv_heads;  /* KV heads n_kv (>= 1) */
    int32_t head_dim;      /* per-head dimension; must be 128 */
    int32_t dtype;         /* pkv_dtype of K/V: PKV_DTYPE_BF16, or PKV_DTYPE_FP8_E4M3 for the
                              *_fp8 entry points and kv_copy_blocks */
} pkv_cache_desc;

/* Return codes. */
#define PKV_OK 0
#define PKV_ERR_INVALID_ARG (-1)         /* null pointer, bad size, misaligned pointer, n_q % n_kv != 0 */
#define PKV_ERR_UNSUPPORTED (-2)         /* head_dim, block_size, dtype or group size not supported */
#define PKV_ERR_WORKSPACE_TOO_SMALL (-3) /* workspace_bytes below the *_workspace_size() answer */
#define PKV_ERR_CUDA (-4)                /* a CUDA runtime call or launch failed */
#define PKV_ERR_OUT_OF_BLOCKS (-5)       /* block manager: not enough free blocks (nothing changed) */

/* Bits ORed into the device status word (workspace byte 0). */
#define PKV_STATUS_BAD_CONTEXT_LEN 0x1u /* context_len < 1 or > max_blocks_per_seq * block_size */
#define PKV_STATUS_BAD_BLOCK_ID 0x2u    /* a needed block_tables entry outside [0, num_blocks) */
#define PKV_STATUS_BAD_Q_LEN 0x4u       /* prefill: q_len < 0, > context_len or > max_q_len */
#define PKV_STATUS_TIMEOUT 0x8u         /* a bounded wait inside a kernel gave up (output invalid) */

/*
 * kv_reshape_and_cache -- append new tokens' K and V to the paged pool.
 *
 * For each token t < num_tokens and KV head h:
 *     slot = slot_mapping[t];  block = slot / block_size;  off = slot % block_size
 *     k_cache[block][h][off][:] = key[t][h][:];   v_cache[block][h][off][:] = value[t][h][:]
 * This is the write of the new token's K/V at position cache_len that precedes
 * the read in a decode step ("LLM 推理全过程的维度变化与核心公式", section
 * "Decode 阶段维度流转"), done through the slot mapping the vLLM concepts deep
 * dive (section 1) describes.  The copy is bit-exact.
 *
 *   key, value   : bf16 [num_tokens][num_kv_heads][head_dim], device, 16-B aligned
 *   k_cache, v_cache : the pool (layout above), written in place
 *   slot_mapping : int32 [num_tokens], device.  slot < 0 marks a padding
 *                  token and is skipped; slot >= num_blocks * block_size is
 *                  skipped too (nothing is written out of bounds).  Two
 *                  tokens with the same slot in one call race (undefined).
 *   num_tokens   : >= 0 (0 enqueues nothing)
 * Errors: PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED / PKV_ERR_CUDA.
 */
PKV_API int kv_reshape_and_cache(const void *key, const void *value, void *k_cache, void *v_cache,
                         const int32_t *slot_mapping, int32_t num_tokens,
                         const pkv_cache_desc *cache, void *stream);

/*
 * kv_reshape_and_cache_fp8 -- append new tokens' K and V to an FP8 (E4M3) pool.
 *
 * INT8 / FP8 KV caches quantise the cache per channel or per token, halving it
 * or more ("LLM 推理全过程的维度变化与核心公式", section "KV Cache 的形状与增长";
 * the error depends on the group size and the scaling: xinc.fun archive 233,
 * section 7).  Here: per token and KV head, one fp32 scale for its 128 values.
 * For each token t < num_tokens and KV head h, with x = key[t][h][:] (and the
 * same for value), slot = slot_mapping[t] (negative: skipped):
 *     a     = max(max_k |x_k|, 2^-100)
 *     code  = E4M3(x_k * (448 / a))   nearest even, saturating at +-448
 *     scale = a / 448
 *     k_cache[block][h][off][k] = code_k;  k_scale[block][h][off] = scale
 * Each step is one correctly rounded fp32 operation, so the codes are exactly
 * reproducible; x_k is recovered as E4M3 value(code_k) * scale.
 *
 *   key, value       : bf16 [num_tokens][num_kv_heads][head_dim], device, 16-B aligned
 *   k_cache, v_cache : uint8 E4M3 codes [num_blocks][num_kv_heads][16][128], device
 *   k_scale, v_scale : fp32 [num_blocks][num_kv_heads][16], device, 16-B aligned
 *   cache->dtype     : PKV_DTYPE_FP8_E4M3
 * Errors: as kv_reshape_and_cache.
 */
PKV_API int kv_reshape_and_cache_fp8(const void *key, const void *value, void *k_cache, void *v_cache, float *k_scale,
                                     float *v_scale, const int32_t *slot_mapping, int32_t num_tokens,
                                     const pkv_cache_desc *cache, void *stream);

/*
 * kv_copy_blocks -- copy whole physical blocks (the copy at a branch point).
 *
 * Sequences that share a prefix, or parallel candidates, reference the same
 * physical blocks until they branch; there the branch gets a new block
 * (xinc.fun archive 233, section 6).  The host block manager (pkv_bm_append)
 * reports such (source, destination) pairs; this call performs them:
 *     for i < num_pairs: block block_pairs[2i+1] := block block_pairs[2i]
 * in k_cache and v_cache (every head and slot), and for an FP8 cache also in
 * k_scale and v_scale (fp32 [num_blocks][num_kv_heads][block_size]).
 *
 *   block_pairs : int32 [num_pairs][2] = {source, destination}, DEVICE memory
 *   k_scale, v_scale : NULL for a bf16 cache; required when cache->dtype is
 *                      PKV_DTYPE_FP8_E4M3 (16-byte aligned)
 * The copies run concurrently: destinations must be distinct and must not be
 * sources of the same call.  A pair with an id outside [0, num_blocks) is
 * skipped.  Bit-exact.
 * Errors: PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED / PKV_ERR_CUDA.
 */
PKV_API int kv_copy_blocks(void *k_cache, void *v_cache, float *k_scale, float *v_scale, const int32_t *block_pairs,
                           int32_t num_pairs, const pkv_cache_desc *cache, void *stream);

/*
 * paged_attention_workspace_size -- bytes of device workspace that
 * paged_attention_decode needs for these sizes and this partition_size
 * (0 = automatic; the answer then covers every automatic choice).  Needs no
 * GPU.  Returns 0 for invalid arguments.
 */
PKV_API size_t paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                      int32_t partition_size, const pkv_cache_desc *cache);

/*
 * paged_attention_decode_partitions -- how many partitions per sequence the
 * decode entry points (paged_attention_decode, _append, _window, _fp8 and
 * _static_scratch) split a row's keys into for these sizes: 1 means no split
 * and no merge kernel; above 1 the log-sum-exp merge runs after the decode
 * kernel.  window = 0 for no sliding window.  With partition_size = 0 the
 * answer is the automatic choice for the current device (it reads the SM
 * count, so it needs a GPU: PKV_ERR_CUDA otherwise).  The automatic choice
 * uses 1024-token partitions; it does not split contexts of at most 2048
 * tokens whose (sequence, KV head) units already fill one wave of the GPU; for
 * a bf16 cache it never makes more than 32 partitions per sequence (the merge
 * folds a row's partitions in sequence); and with few units it shrinks the
 * partitions (to no less than 256 tokens) until the grid covers every SM
 * twice.  For an FP8 cache (half the bytes per CTA) contexts of at most 2048
 * tokens whose units fill every SM are not split, and contexts of 16K tokens
 * and more double the partition while at least 3 CTAs per SM remain.
 * Returns the count, or a negative PKV_ERR_* for invalid arguments.
 */
PKV_API int32_t paged_attention_decode_partitions(int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                                  int32_t partition_size, int32_t window,
                                                  const pkv_cache_desc *cache);

/*
 * paged_attention_decode -- decode-phase attention over the paged cache.
 *
 * For each sequence b (ctx = context_lens[b], which already counts the token
 * appended this step) and query head h with KV head g = floor(h / G):
 *     s_j    = scale * <q[b][h], K_b[j][g]>                     j = 0 .. ctx-1
 *     out[b][h] = sum_j softmax(s)_j * V_b[j][g]
 * where K_b[j] is row j % block_size of block block_tables[b][j / block_size]
 * ("LLM 推理全过程的维度变化与核心公式", section "Decode 阶段维度流转": scores
 * [B, n_q, 1, cache_len], GQA broadcast, no causal mask).
 *
 * Long contexts are split into partitions of `partition_size` tokens that are
 * processed in parallel and then combined by a log-sum-exp merge
 * (Flash-Decoding; same page, section "工程优化怎么嵌进公式").  The result
 * does not depend on the partition size beyond float rounding.
 *
 *   out            : out_dtype [num_seqs][num_q_heads][head_dim], device
 *   out_dtype      : PKV_DTYPE_FLOAT32 or PKV_DTYPE_BF16 (round to nearest even)
 *   q              : bf16 [num_seqs][num_q_heads][head_dim], device
 *   block_tables   : int32 [num_seqs][max_blocks_per_seq], device
 *   context_lens   : int32 [num_seqs], device
 *   num_seqs       : 1 .. 65535;  num_q_heads: multiple of cache->num_kv_heads
 *   scale          : softmax scale (usually 1/sqrt(head_dim))
 *   partition_size : tokens per partition, a positive multiple of 16, or 0
 *                    for an automatic choice sized to the GPU's SM count
 *   workspace      : device scratch, 256-B aligned, of at least
 *                    paged_attention_workspace_size(num_seqs, num_q_heads,
 *                    max_blocks_per_seq, partition_size, cache) bytes; holds
 *                    the status word (byte 0) and the per-partition partials
 *                    (written before they are read, so only the status word
 *                    needs clearing; it is sticky).  The same workspace serves
 *                    later calls.  Calls that share a workspace must not
 *                    overlap in time (they race on it).
 * Enqueues the decode kernel and, when a context is split into partitions,
 * the log-sum-exp merge kernel (both with programmatic dependent launch).
 * Errors: PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED /
 *         PKV_ERR_WORKSPACE_TOO_SMALL / PKV_ERR_CUDA.
 */
PKV_API int paged_attention_decode(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                           const void *v_cache, const int32_t *block_tables,
                           const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                           int32_t max_blocks_per_seq, float scale, int32_t partition_size,
                           const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes,
                           void *stream);

/*
 * Largest workspace that paged_attention_decode_static_scratch can stand in
 * for: 16 MiB of device memory, held by every GPU that loads this library for
 * as long as the process lives.
 */
#define PKV_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * paged_attention_decode_append -- one decode step in one launch: appends each
 * sequence's new K/V row and attends over the cache including it.
 *
 * Same result as kv_reshape_and_cache() with slot_mapping[b] = the slot of
 * position ctx_b - 1 (row (ctx_b - 1) % 16 of block
 * block_tables[b][(ctx_b - 1) / 16]) followed by paged_attention_decode()
 * (sections as for those two calls: "LLM 推理全过程的维度变化与核心公式", "Decode
 * 阶段维度流转" -- the step's K/V is appended to the cache, then the single query
 * row attends over all of it).  The CTAs that read a sequence's last block put
 * the new row into their shared-memory copy of it, and one CTA per KV head
 * writes it to the pool, so no separate append kernel runs and no CTA reads the
 * slot from memory.  The pool afterwards equals the two-call result bit for bit.
 *
 *   key, value : bf16 [num_seqs][num_kv_heads][head_dim], device, 16-B aligned:
 *                the row of position ctx_b - 1 of each sequence
 *   k_cache, v_cache : the bf16 pool (written at those slots)
 *   other arguments and the workspace: as paged_attention_decode (no window,
 *   bf16 cache only).
 * A sequence with an out-of-range context length or an invalid id in its last
 * block gets no row written (the status word flags it, as for the decode).
 * Errors: as paged_attention_decode; PKV_ERR_INVALID_ARG for a null or
 * misaligned key / value.
 */
PKV_API int paged_attention_decode_append(void *out, int32_t out_dtype, const void *q, const void *key,
                                          const void *value, void *k_cache, void *v_cache,
                                          const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                                          int32_t num_q_heads, int32_t max_blocks_per_seq, float scale,
                                          int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * paged_attention_decode_static_scratch -- paged_attention_decode without a
 * caller-provided workspace; it allocates nothing.  (The pages have no
 * counterpart: this is a deployment convenience, not part of the method.)
 *
 * For callers that cannot allocate device memory at the point of the call:
 * code running under a framework or allocator that owns all device memory
 * (where a raw cudaMalloc would bypass its pool or its accounting), real-time
 * or latency-critical loops where cudaMalloc/cudaFree would synchronise the
 * device and stall, and callers such as plugins or other libraries that are
 * handed only the input and output buffers.
 *
 * The split-KV scratch (status word and per-partition partials) lives in one
 * file-scope device array of PKV_STATIC_SCRATCH_BYTES
 * bytes instead of a workspace argument.  Everything else -- arguments,
 * layouts, result and error codes -- is exactly paged_attention_decode's.
 *
 *   status : device pointer to one uint32 that receives this call's
 *            PKV_STATUS_* bits (copied out of the scratch after the kernels),
 *            or NULL to discard them.
 * Limits and sharing:
 *  - Sizes whose paged_attention_workspace_size(num_seqs, num_q_heads,
 *    max_blocks_per_seq, partition_size, cache) exceeds
 *    PKV_STATIC_SCRATCH_BYTES are rejected with PKV_ERR_WORKSPACE_TOO_SMALL
 *    before anything is enqueued (use a larger partition_size, fewer
 *    sequences per call, or paged_attention_decode with a workspace).
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and caches it once the
 *    lookup succeeds (a failed lookup is retried by the next call); make
 *    that first call outside any stream capture.
 *  - Every call on a device shares the one array, which keeps the last
 *    call's contents: each call clears the 256-byte status word (an
 *    asynchronous memset on `stream`) before its kernels run; the partials
 *    are written before they are read.  Calls
 *    whose execution overlaps on the GPU (different streams without ordering
 *    between them, or different host threads) race on the array and give
 *    undefined results; serialise them.
 * Errors: as paged_attention_decode; PKV_ERR_CUDA if the array's address
 * cannot be obtained.
 */
PKV_API int paged_attention_decode_static_scratch(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                                                  const void *v_cache, const int32_t *block_tables,
                                                  const int32_t *context_lens, int32_t num_seqs,
                                                  int32_t num_q_heads, int32_t max_blocks_per_seq, float scale,
                                                  int32_t partition_size, const pkv_cache_desc *cache,
                                                  uint32_t *status, void *stream);

/*
 * paged_attention_decode_window -- decode attention under a sliding window.
 *
 * As paged_attention_decode, except that sequence b's row sees only its newest
 * `window` keys, j >= max(0, ctx_b - window): Sliding Window Attention keeps
 * only the most recent W tokens' K and V ("LLM 推理全过程的维度变化与核心公式",
 * section "KV Cache 的形状与增长").  Blocks wholly before the window are never
 * read (their table entries may be stale or freed ids); the work and bytes per
 * row are bounded by the window, not by the context.  window >= ctx gives
 * exactly paged_attention_decode's result.
 *   window : >= 1 (PKV_ERR_INVALID_ARG otherwise)
 * The workspace that paged_attention_workspace_size() gives for the same
 * arguments is always enough (a window needs at most that).
 */
PKV_API int paged_attention_decode_window(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                                          const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_blocks_per_seq, float scale, int32_t window,
                                          int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * paged_attention_decode_fp8 -- decode attention over an FP8 (E4M3) pool.
 *
 * As paged_attention_decode_window (window 0 = no window), with K_j and V_j the
 * dequantised rows code * scale written by kv_reshape_and_cache_fp8:
 *     s_j = scale * <q, K_j>,  out = sum_j softmax(s)_j V_j
 * Every K/V byte read per token and head is halved.  The dot products run on
 * fp16 tensor-core MMAs: E4M3 values are exact fp16 numbers, q is scaled by a
 * power of two per CTA into the fp16 range (exact), the K scale multiplies the
 * scores and the V scale is folded into the softmax weights (kept to about
 * 2^-22 relative as an fp16 head and remainder).
 *   k_cache, v_cache : uint8 E4M3 codes, cache->dtype PKV_DTYPE_FP8_E4M3
 *   k_scale, v_scale : fp32 [num_blocks][num_kv_heads][16], device, 16-B aligned
 *   window           : 0, or >= 1 as in paged_attention_decode_window
 * Workspace: paged_attention_workspace_size() with this cache descriptor.
 * Errors: as paged_attention_decode.
 */
PKV_API int paged_attention_decode_fp8(void *out, int32_t out_dtype, const void *q, const void *k_cache,
                                       const void *v_cache, const float *k_scale, const float *v_scale,
                                       const int32_t *block_tables, const int32_t *context_lens, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t max_blocks_per_seq, float scale, int32_t window,
                                       int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                                       size_t workspace_bytes, void *stream);

/*
 * paged_attention_prefill_workspace_size -- the least workspace that
 * paged_attention_prefill_chunk accepts: the status word (256 bytes).  With
 * it the kernel runs one CTA per (KV head, sequence, pair of 128-row tiles).
 * Needs no GPU.
 */
PKV_API size_t paged_attention_prefill_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                              const pkv_cache_desc *cache);

/*
 * paged_attention_prefill_chunk_workspace_size -- the workspace with which
 * paged_attention_prefill_chunk (and its _window / _fp8 forms) may split the
 * keys (split-KV) for these sizes on the current device: when its CTAs would
 * not fill the GPU (few sequences, short chunks, long contexts), each pair of
 * row tiles walks 2..16 key ranges in separate CTAs whose partials (m, l, O)
 * a log-sum-exp merge folds ("LLM 推理全过程的维度变化与核心公式", section "工程
 * 优化怎么嵌进公式", Flash-Decoding, applied to a chunk's rows).  The result does
 * not depend on the split beyond float rounding.  Layout [status 256 B | m | l |
 * O], fp32 partials of total_q_rows x num_q_heads rows per split; 256 bytes
 * (no split) when the CTAs already fill the GPU.  Reads the current device's
 * SM count (152 assumed without a GPU).  Returns 0 for invalid arguments.
 */
PKV_API size_t paged_attention_prefill_chunk_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                            int32_t total_q_rows, int32_t max_q_len,
                                                            int32_t max_blocks_per_seq, const pkv_cache_desc *cache);

/*
 * paged_attention_prefill_chunk -- causal attention of a chunk of new query
 * rows per sequence over that sequence's paged cache.
 *
 * Sequence b owns query rows cu_q_lens[b] .. cu_q_lens[b+1]-1 (q_len rows);
 * its context length ctx = context_lens[b] counts those q_len tokens, whose
 * K/V must already be in the cache.  Row i (0-based within the chunk) sits at
 * absolute position c + i with c = ctx - q_len and sees keys j <= c + i:
 * the causal mask M_ij = 0 for j <= i, -inf otherwise ("注意力演进与推理流程",
 * section 1.1) shifted by the cached prefix, which is what chunked prefill
 * computes (same page, 变革 3; walkthrough page, Chunked Prefill: "formula
 * unchanged").  With q_len = 1 a row is a decode row.
 *
 *   out        : out_dtype [cu_q_lens[num_seqs]][num_q_heads][head_dim], device,
 *                16-B aligned
 *   q          : bf16 [cu_q_lens[num_seqs]][num_q_heads][head_dim], device,
 *                16-B aligned
 *   cu_q_lens  : int32 [num_seqs + 1], device, non-decreasing, cu_q_lens[0] = 0
 *   max_q_len  : host upper bound of every q_len (sizes the launch grid)
 *   total_q_rows : host value of cu_q_lens[num_seqs] (bounds the q/out tensors)
 *   workspace  : device, 256-B aligned, >= paged_attention_prefill_workspace_size()
 *                bytes (the status word); with at least
 *                paged_attention_prefill_chunk_workspace_size() bytes for the
 *                same sizes the call may split the keys (and then launches the
 *                merge kernel after the prefill kernel)
 * Uses the 5th-generation tensor cores (tcgen05, accumulators in tensor memory).
 * Errors: PKV_ERR_INVALID_ARG (null or misaligned pointer, bad size) /
 *         PKV_ERR_UNSUPPORTED (group size not in {1,2,4,8,16}, more than 65535
 *         row tiles x group, or num_blocks x num_kv_heads above INT32_MAX) /
 *         PKV_ERR_WORKSPACE_TOO_SMALL / PKV_ERR_CUDA.
 */
PKV_API int paged_attention_prefill_chunk(void *out, int32_t out_dtype, const void *q, const int32_t *cu_q_lens,
                                  int32_t max_q_len, int32_t total_q_rows, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                  int32_t max_blocks_per_seq, float scale, const pkv_cache_desc *cache,
                                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_attention_prefill_chunk_window -- paged_attention_prefill_chunk with a
 * sliding window of `window` >= 1 tokens ("LLM 推理全过程的维度变化与核心公式",
 * section "KV Cache 的形状与增长", Sliding Window Attention: only the most
 * recent W tokens' K and V are kept): row i at position pos = c + i sees keys
 * pos - window < j <= pos.  Key tiles wholly before the earliest visible key
 * of a CTA's rows are never fetched, and block_tables entries of blocks that
 * lie wholly before it are never read (they may be stale); every other entry
 * is checked as in paged_attention_prefill_chunk.  A window at least as long
 * as the context gives exactly the unwindowed result.
 * Errors: as paged_attention_prefill_chunk; PKV_ERR_INVALID_ARG for window < 1.
 */
PKV_API int paged_attention_prefill_chunk_window(void *out, int32_t out_dtype, const void *q,
                                         const int32_t *cu_q_lens, int32_t max_q_len, int32_t total_q_rows,
                                         const void *k_cache, const void *v_cache, const int32_t *block_tables,
                                         const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                         int32_t max_blocks_per_seq, float scale, int32_t window,
                                         const pkv_cache_desc *cache, void *workspace, size_t workspace_bytes,
                                         void *stream);

/*
 * paged_attention_prefill_chunk_fp8 -- paged_attention_prefill_chunk over an FP8
 * (E4M3) cache (cache->dtype PKV_DTYPE_FP8_E4M3; codes and per-slot scales as
 * written by kv_reshape_and_cache_fp8; attention over code * scale as in
 * paged_attention_decode_fp8), with an optional sliding window (window = 0:
 * none; else as paged_attention_prefill_chunk_window).  The codes are fetched
 * by TMA and expanded to bf16 in shared memory (exact: every E4M3 value is a
 * bf16 value); the scales are applied in fp32, the K scale to the scores and
 * the V scale to the probabilities before P V.  Workspace:
 * paged_attention_prefill_workspace_size() with the FP8 cache descriptor.
 *   k_scale, v_scale : float [num_blocks][num_kv_heads][16], device, 16-B aligned
 * Errors: as paged_attention_prefill_chunk; PKV_ERR_INVALID_ARG for a missing or
 * misaligned scale array or window < 0.
 */
PKV_API int paged_attention_prefill_chunk_fp8(void *out, int32_t out_dtype, const void *q, const int32_t *cu_q_lens,
                                              int32_t max_q_len, int32_t total_q_rows, const void *k_cache,
                                              const void *v_cache, const float *k_scale, const float *v_scale,
                                              const int32_t *block_tables, const int32_t *context_lens,
                                              int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq,
                                              float scale, int32_t window, const pkv_cache_desc *cache,
                                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_attention_verify -- attention of k draft positions per sequence
 * (speculative decoding's verification step).
 *
 * A draft model proposes k tokens and the target model checks all k positions
 * in one pass, turning k decode steps into one k-row computation
 * ("LLM 推理全过程的维度变化与核心公式", section "工程优化怎么嵌进公式",
 * Speculative Decoding; xinc.fun archive 233, section 7).  The k tokens' K/V
 * are appended first, so ctx_b counts them; row i (0 <= i < k) of sequence b
 * sits at position ctx_b - k + i and sees keys j <= ctx_b - k + i (the causal
 * rule among the draft tokens; row k - 1 is an ordinary decode row).  The
 * acceptance rule itself (sampling) is not part of this library.
 *
 *   q, out    : [num_seqs * q_per_seq][num_q_heads][head_dim]; sequence b owns
 *               rows b * q_per_seq .. b * q_per_seq + q_per_seq - 1
 *   q_per_seq : k, 1 .. 16
 * Runs on the decode kernel, where the G heads x k positions of a KV head are
 * the MMA columns of ceil(G * k / 16) CTAs of up to 16 columns (one or two
 * 8-column tiles), each reading the K/V once; or on the tcgen05 prefill kernel
 * (then q and out must be 16-B aligned), which reads them once per row tile and
 * splits the keys when its CTAs cannot fill the GPU, when G is in {1,2,4,8,16}
 * and G * k >= 32 -- the route measured faster (paged_attention_verify_on
 * picks one explicitly).
 * num_seqs * k must not exceed 65535 (PKV_ERR_UNSUPPORTED).  A sequence with
 * ctx < k sets PKV_STATUS_BAD_Q_LEN and gets zero rows.
 * Workspace: paged_attention_verify_workspace_size() bytes (sized for the route
 * taken with the current device), zero-filled once.
 * Errors: as paged_attention_decode; PKV_ERR_INVALID_ARG for q_per_seq outside 1..16.
 */
PKV_API size_t paged_attention_verify_workspace_size(int32_t num_seqs, int32_t q_per_seq, int32_t num_q_heads,
                                                     int32_t max_blocks_per_seq, int32_t partition_size,
                                                     const pkv_cache_desc *cache);
/*
 * The kernel a verify call runs on: PKV_VERIFY_AUTO lets the measured rule
 * above choose; the other two force one (the prefill kernel only for G in
 * {1, 2, 4, 8, 16}).  The result does not depend on the kernel beyond float
 * rounding.
 */
#define PKV_VERIFY_AUTO (-1)
#define PKV_VERIFY_DECODE_KERNEL 0
#define PKV_VERIFY_PREFILL_KERNEL 1

/*
 * paged_attention_verify_workspace_size_on / paged_attention_verify_on --
 * paged_attention_verify_workspace_size and paged_attention_verify (with the
 * sliding window and the FP8 cache of _window / _fp8: window 0 for none,
 * k_scale and v_scale NULL for a bf16 cache) on the kernel `kernel` chooses.
 * Workspace: paged_attention_verify_workspace_size_on() for the same kernel.
 * Errors: as paged_attention_verify; PKV_ERR_UNSUPPORTED for the prefill
 * kernel with a group size it cannot pack; the size query returns 0.
 */
PKV_API size_t paged_attention_verify_workspace_size_on(int32_t kernel, int32_t num_seqs, int32_t q_per_seq,
                                                        int32_t num_q_heads, int32_t max_blocks_per_seq,
                                                        int32_t partition_size, const pkv_cache_desc *cache);
PKV_API int paged_attention_verify_on(int32_t kernel, void *out, int32_t out_dtype, const void *q, int32_t q_per_seq,
                                      const void *k_cache, const void *v_cache, const float *k_scale,
                                      const float *v_scale, const int32_t *block_tables,
                                      const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                      int32_t max_blocks_per_seq, float scale, int32_t window,
                                      int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                                      size_t workspace_bytes, void *stream);

/*
 * paged_attention_verify_on_prefill -- the kernel paged_attention_verify (and
 * _window / _fp8, per cache->dtype) takes for these sizes on the current
 * device: 1 the tcgen05 prefill kernel, 0 the decode kernel; a negative
 * PKV_ERR_* for invalid arguments.  Needs no GPU.
 */
PKV_API int paged_attention_verify_on_prefill(int32_t num_seqs, int32_t q_per_seq, int32_t num_q_heads,
                                              const pkv_cache_desc *cache);
PKV_API int paged_attention_verify(void *out, int32_t out_dtype, const void *q, int32_t q_per_seq, const void *k_cache,
                                   const void *v_cache, const int32_t *block_tables, const int32_t *context_lens,
                                   int32_t num_seqs, int32_t num_q_heads, int32_t max_blocks_per_seq, float scale,
                                   int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * paged_attention_verify_window -- paged_attention_verify with a sliding window
 * of `window` >= 1 tokens (same page and section as the decode's window): row i
 * of a sequence, at position pos = ctx - k + i, sees keys pos - window < j <=
 * pos.  Blocks wholly before the first row's window are not fetched and their
 * table entries are not read.  Same paths, workspace and errors as
 * paged_attention_verify; PKV_ERR_INVALID_ARG for window < 1.
 */
PKV_API int paged_attention_verify_window(void *out, int32_t out_dtype, const void *q, int32_t q_per_seq,
                                          const void *k_cache, const void *v_cache, const int32_t *block_tables,
                                          const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_blocks_per_seq, float scale, int32_t partition_size,
                                          int32_t window, const pkv_cache_desc *cache, void *workspace,
                                          size_t workspace_bytes, void *stream);

/*
 * paged_attention_verify_fp8 -- paged_attention_verify over an FP8 (E4M3) cache
 * (cache->dtype PKV_DTYPE_FP8_E4M3; codes and scales as written by
 * kv_reshape_and_cache_fp8, attention over code * scale as in
 * paged_attention_decode_fp8), with an optional sliding window (window = 0:
 * none).  On the decode kernel, one 8-column MMA tile per CTA: the G * k
 * (position, head) columns of a KV head are shared out over ceil(G * k / 8)
 * CTAs, each reading the K/V codes once; or, when G is in {1,2,4,8,16} and
 * G * k >= 32, on the FP8 prefill kernel (paged_attention_prefill_chunk_fp8
 * with k rows per sequence, split-KV for few units; q and out then 16-B
 * aligned), which reads the codes once per row tile.  Workspace:
 * paged_attention_verify_workspace_size() with the FP8 cache descriptor.
 * Errors: as paged_attention_verify; PKV_ERR_INVALID_ARG for a missing or
 * misaligned scale array.
 */
PKV_API int paged_attention_verify_fp8(void *out, int32_t out_dtype, const void *q, int32_t q_per_seq,
                                       const void *k_cache, const void *v_cache, const float *k_scale,
                                       const float *v_scale, const int32_t *block_tables,
                                       const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                       int32_t max_blocks_per_seq, float scale, int32_t window,
                                       int32_t partition_size, const pkv_cache_desc *cache, void *workspace,
                                       size_t workspace_bytes, void *stream);

/*
 * ---- Host block manager ---------------------------------------------------------
 * Hands out the pool's physical blocks to sequences and emits the block tables
 * and slot mappings the kernels above consume.  Sources: "注意力演进与推理流程",
 * 变革 1 (the cache is cut into fixed-size blocks of e.g. 16 tokens and a block
 * is allocated on demand as a sequence grows) and 变革 3 (prefix caching: a
 * repeated prefix hits cached KV and skips its prefill); xinc.fun archive 233,
 * section 6 (sequences sharing a prefix, or parallel candidates, reference the
 * same physical blocks until they branch, where a new block is allocated).
 *
 * Model: every block has a reference count (sequences whose table holds it).
 * A sequence is a list of blocks plus a length in tokens.  Appending never
 * writes into a block that another sequence also references: if a sequence's
 * partially filled last block is shared, the append first moves the sequence
 * to a fresh block and reports a (source, destination) pair that the caller
 * must copy on the device (kv_copy_blocks) before the tokens are written.
 * Full blocks can be published under a hash of all token ids up to their end;
 * a new sequence whose prompt starts with published blocks takes them over
 * (reference +1).  A block whose count drops to 0 becomes free; a published
 * free block stays findable until the allocator reuses it (unpublished free
 * blocks are reused first, published ones oldest first).
 *
 * Host memory only; needs no GPU.  Not thread-safe: one thread owns a manager.
 * Sequence ids are the caller's 64-bit keys.  Every call either succeeds or
 * returns an error with the manager unchanged.
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A manager for blocks 0 .. num_blocks-1 (all free).  *out receives it. */
PKV_API int pkv_bm_create(int32_t num_blocks, pkv_block_manager **out);
PKV_API void pkv_bm_destroy(pkv_block_manager *bm);
/* Free blocks (including published ones that no sequence holds). */
PKV_API int32_t pkv_bm_num_free(const pkv_block_manager *bm);
/* Reference count of one block (0 when free). */
PKV_API int pkv_bm_ref_count(const pkv_block_manager *bm, int32_t block, int32_t *count);

/* A new, empty sequence.  PKV_ERR_INVALID_ARG if the id is taken. */
PKV_API int pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id);
/* child_id starts as a copy of parent_id's table and length, sharing every block. */
PKV_API int pkv_bm_fork(pkv_block_manager *bm, int64_t parent_id, int64_t child_id);
/*
 * Reserve slots for num_tokens new tokens at positions length .. length+num_tokens-1:
 * slot_mapping[t] = table[p / 16] * 16 + p % 16 (host array of num_tokens).
 * New blocks are allocated as positions cross a block boundary.  copy_pair
 * (host int32[2]) receives {source, destination} and *num_copies is 1 when
 * the shared last block had to be replaced first (0 otherwise).
 * PKV_ERR_OUT_OF_BLOCKS if the free blocks do not suffice.
 */
PKV_API int pkv_bm_append(pkv_block_manager *bm, int64_t seq_id, int32_t num_tokens, int32_t *slot_mapping,
                          int32_t *copy_pair, int32_t *num_copies);
/*
 * One call for a batch (e.g. one decode step): num_tokens[i] new tokens for
 * seq_ids[i] (num_tokens NULL: one each), in order.  slot_mapping (host, sum of
 * num_tokens) receives the slots sequence after sequence; copy_pairs (host,
 * room for num_seqs pairs) receives the {source, destination} pairs to copy
 * first, *num_copies of them.  All or nothing: PKV_ERR_OUT_OF_BLOCKS (or an
 * invalid or repeated id) changes nothing.
 */
PKV_API int pkv_bm_append_batch(pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs,
                                const int32_t *num_tokens, int32_t *slot_mapping, int32_t *copy_pairs,
                                int32_t *num_copies);
/* Drop a sequence: every block's count decreases; blocks reaching 0 become free. */
PKV_API int pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);
PKV_API int pkv_bm_sequence_length(const pkv_block_manager *bm, int64_t seq_id, int64_t *length);
/*
 * Emit the block-table rows and context lengths of num_seqs sequences (host
 * arrays): block_tables [num_seqs][max_blocks_per_seq], entries past a
 * sequence's blocks set to pad_block.  PKV_ERR_INVALID_ARG if a sequence
 * needs more than max_blocks_per_seq blocks (nothing written).
 */
PKV_API int pkv_bm_block_tables(const pkv_block_manager *bm, const int64_t *seq_ids, int32_t num_seqs,
                                int32_t max_blocks_per_seq, int32_t pad_block, int32_t *block_tables,
                                int32_t *context_lens);
/*
 * Prefix caching.  pkv_bm_publish: tokens[0 .. num_tokens) are the token ids
 * at positions 0.. of seq_id (num_tokens <= its length); every full block
 * among them is published under a hash of tokens[0 .. end of block) unless
 * that prefix is already published.  pkv_bm_add_sequence_cached: a new
 * sequence whose prompt is tokens[0 .. num_tokens); it takes over the
 * longest run of published leading blocks, leaving at least one prompt token
 * to compute, and *num_cached_tokens = 16 x blocks taken (its length).
 * Matches compare the stored token ids, so a hash collision never shares a
 * block.
 */
PKV_API int pkv_bm_publish(pkv_block_manager *bm, int64_t seq_id, const int32_t *tokens, int32_t num_tokens);
PKV_API int pkv_bm_add_sequence_cached(pkv_block_manager *bm, int64_t seq_id, const int32_t *tokens,
                                       int32_t num_tokens, int32_t *num_cached_tokens);

/* Human-readable name of a return code (static string, never NULL). */
PKV_API const char *pagedkv_status_string(int status);

/* Library version: major * 10000 + minor * 100 + patch. */
PKV_API int pagedkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
