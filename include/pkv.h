/*
 * pkv — decode-phase attention over a paged KV cache, for NVIDIA GB300 (sm_103a).
 *
 * Sources, cited below by short name:
 *   [inference]  LLM-101-CN, "推理优化" (engineering/inference.html)
 *   [essay]      gsyq.cn essay on the three dimensions of LLM inference
 *   [vllm-06]    "Deep dive into vLLM 06: GPU execution, kernels and graphs"
 *   [chapter12]  tutorial chapter "12-推理优化" (docs.yz520gzy.top)
 *
 * Conventions shared by every call:
 *   - All tensors are dense, row-major (C order), in device memory owned by the
 *     caller.  The library allocates nothing on the device, keeps no per-call
 *     state, and every call is asynchronous on `stream` (a cudaStream_t; NULL
 *     is the legacy default stream).  Only pkv_check_error synchronises.
 *   - Device pointers must be 16-byte aligned.
 *   - 16-bit element types: PKV_FP16 (IEEE binary16) or PKV_BF16 (bfloat16).
 *   - Cache layout, "organised by page" ([inference] "PagedAttention 内核实现"):
 *       k_cache, v_cache: [num_blocks][block_size][num_kv_heads][head_dim]
 *     or, with PKV_LAYOUT_HND OR-ed into the dtype argument of a call, head
 *     major ([chapter12] PagedKVCache, one [heads][page_size][head_dim] slab
 *     per page):
 *       k_cache, v_cache: [num_blocks][num_kv_heads][block_size][head_dim]
 *     where each (page, head) is one contiguous block_size x head_dim tile.
 *   - Argument errors are found on the host before any launch: the call
 *     returns a status and launches nothing.
 *   - Bad indices found on the device (a block id outside [0, num_blocks), a
 *     slot beyond the pool, a context longer than the block table or than
 *     max_context_len) never fault: the offending token is skipped and a bit
 *     is OR-ed into the optional device word *err_flag (PKV_EFLAG_*), which
 *     the caller zero-initialises and reads back with pkv_check_error.
 *   - Supported sizes: head_dim in {64, 128}; block_size in {16, 32, 64, 128};
 *     num_q_heads a multiple of num_kv_heads with at most 16 query heads per
 *     KV head.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,    /* null pointer, bad size, misaligned pointer */
    PKV_ERR_UNSUPPORTED = 2,    /* valid but not implemented (head_dim, block_size, group) */
    PKV_ERR_WORKSPACE = 3,      /* workspace missing or smaller than required */
    PKV_ERR_CUDA = 4,           /* a CUDA runtime call failed (launch, query, copy) */
    PKV_ERR_DEVICE_INDEX = 5,   /* pkv_check_error: a kernel skipped an out-of-range index */
    PKV_ERR_DEVICE_TIMEOUT = 6  /* pkv_check_error: a bounded in-kernel wait gave up */
} pkv_status;

typedef enum { PKV_FP16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* OR-ed into the dtype argument of a call that reads or writes the cache:
   the caches are head major, [num_blocks][num_kv_heads][block_size][head_dim]. */
#define PKV_LAYOUT_HND 0x100

/* Bits OR-ed into *err_flag by the kernels. */
#define PKV_EFLAG_BLOCK_ID      0x1  /* block id outside [0, num_blocks) */
#define PKV_EFLAG_SLOT          0x2  /* slot >= num_blocks * block_size */
#define PKV_EFLAG_CONTEXT_LEN   0x4  /* context_len > max_blocks_per_seq * block_size,
                                        > max_context_len, or negative */
#define PKV_EFLAG_TIMEOUT       0x8  /* a bounded wait inside a kernel expired */
#define PKV_EFLAG_GROUP         0x10 /* a shared-prefix group was malformed (its members were
                                        decoded without the shared prefix) */

#define PKV_MAX_SPLITS 1024           /* upper bound on split-K partitions per sequence */

/*
 * Append (scatter) each step's new K/V token into its slot.
 *
 * For every i < num_tokens with s = slot_mapping[i] >= 0:
 *     k_cache[s / block_size][s % block_size][:][:] = k_new[i][:][:]   (same for V)
 * The block/offset split of a slot follows the token-to-page addressing of
 * [essay] §三.2 (get_kv_cache) and [chapter12] PagedKVCache.update; writing
 * the new token at the current page and offset follows [inference]
 * KVCachePool.write_tokens.  A negative slot is padding and is skipped.  The
 * copy is bit-exact.
 *
 *   k_new, v_new   [num_tokens][num_kv_heads][head_dim] (read)
 *   k_cache, v_cache                                    (written at the slots only)
 *   slot_mapping   int64 [num_tokens]; slots must be distinct within one call
 *   err_flag       nullable; PKV_EFLAG_SLOT if a slot lies beyond the pool
 */
pkv_status pkv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                      const int64_t* slot_mapping, int num_tokens, int num_blocks,
                      int block_size, int num_kv_heads, int head_dim, pkv_dtype dtype,
                      int32_t* err_flag, void* stream);

/*
 * Bytes of device workspace pkv_decode_attention (and pkv_decode_attention_fp8)
 * needs for these arguments on the current device (the split-K plan depends on
 * the device's SM count; the automatic plan picks, among partitions of 256 to
 * 2048 tokens, the count with the least estimated time: waves of resident CTAs,
 * rounded up, times the partition's tokens plus a fixed per-CTA start; the
 * E4M3 kernel, with more resident CTAs per SM, may pick another count, and
 * this size covers both).  Returns 0 when no workspace is needed and SIZE_MAX
 * when the arguments are invalid or the device cannot be queried.
 */
size_t pkv_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int max_context_len, int num_splits);

/*
 * The number of KV partitions per sequence (split-K) pkv_decode_attention
 * uses for these arguments on the current device (16-bit caches): >= 1, or -1
 * when the arguments are invalid or the device cannot be queried.  num_splits
 * as in pkv_decode_attention (0 = automatic).
 */
int pkv_decode_num_splits(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int max_context_len, int num_splits);

/* The same for pkv_decode_attention_fp8 (E4M3 caches), whose kernel holds more
 * CTAs per SM, so its automatic plan may pick another count. */
int pkv_decode_num_splits_fp8(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_context_len, int num_splits);

/*
 * Decode attention: one query token per sequence against its paged context.
 *
 * For sequence b, query head h, KV head g = h / (num_q_heads / num_kv_heads)
 * (contiguous GQA groups, [essay] §三.6) and n = context_lens[b]:
 *     K_t = k_cache[block_tables[b][t / block_size]][t % block_size][g][:]   t < n
 *     s_t = scale * <q[b][h], K_t>            (scale = 1/sqrt(head_dim) normally,
 *                                              [inference] chunked prefill, NPUAttention)
 *     out[b][h] = sum_t softmax(s)_t V_t      ([chapter12] Attention(Q_t, K_1:t, V_1:t))
 * computed in fp32 with an online softmax ([vllm-06] FlashAttention, online
 * softmax) and, for long contexts, split over the KV length into partitions
 * merged by log-sum-exp ([vllm-06] Flash-Decoding; [inference] combine_result).
 * Tokens at positions >= n are never read.  n == 0 gives a zero row.
 *
 *   out            [num_seqs][num_q_heads][head_dim] (written), dtype
 *   q              [num_seqs][num_q_heads][head_dim] (read), dtype
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]; entries past the
 *                  context are never read
 *   context_lens   int32 [num_seqs], in device memory
 *   max_context_len  host-side upper bound of context_lens, used to plan the
 *                  split; a longer context is truncated and flagged
 *   num_splits     0 = automatic, else the requested number of KV partitions
 *                  per sequence (1 .. PKV_MAX_SPLITS; fewer are used when the
 *                  context has fewer pages)
 *   workspace      device scratch of at least pkv_decode_workspace_size(...)
 *                  bytes (may be NULL when that size is 0); its contents on
 *                  entry do not matter and are clobbered
 *   err_flag       nullable; PKV_EFLAG_BLOCK_ID / PKV_EFLAG_CONTEXT_LEN /
 *                  PKV_EFLAG_TIMEOUT
 */
pkv_status pkv_decode_attention(void* out, const void* q, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* context_lens,
                                int max_context_len, int num_seqs, int num_blocks,
                                int block_size, int num_q_heads, int num_kv_heads, int head_dim,
                                float scale, int num_splits, void* workspace,
                                size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag,
                                void* stream);

/*
 * FP8 (E4M3) KV cache ([vllm-06] 3.3 FP8 inference: E4M3 for inference, the
 * value range held by a scale; 2.2 kernel fusion: the KV-cache write fused
 * with quantisation).  The caches hold E4M3 codes, one byte per element, in
 * either layout; one fp32 scale for K and one for V (finite, > 0): a code c
 * stands for the value c * k_scale (c * v_scale).  E4M3: 1 sign bit, 4
 * exponent bits (bias 7), 3 fraction bits, no infinities, S.1111.111 = NaN,
 * largest finite value 448.
 *
 * pkv_append_fp8: pkv_append with quantisation: element x of a new K row is
 *   stored as E4M3(x / k_scale), the quotient rounded to fp32 and then to the
 *   nearest E4M3 value (ties to even), saturating at +-448; likewise V.
 *   k_new, v_new are 16-bit values of dtype (which may carry PKV_LAYOUT_HND);
 *   the caches must be 8-byte aligned; head_dim a multiple of 8.
 * pkv_decode_attention_fp8: pkv_decode_attention over E4M3 caches; q and out
 *   are dtype; head_dim 128 only; workspace as pkv_decode_workspace_size.
 *   Each code is converted exactly (every E4M3 value is an fp16 and a bf16
 *   value); k_scale enters the scores, v_scale the output.
 */
pkv_status pkv_append_fp8(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, int num_blocks,
                          int block_size, int num_kv_heads, int head_dim, float k_scale,
                          float v_scale, pkv_dtype dtype, int32_t* err_flag, void* stream);

pkv_status pkv_decode_attention_fp8(void* out, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* context_lens,
                                    int max_context_len, int num_seqs, int num_blocks,
                                    int block_size, int num_q_heads, int num_kv_heads,
                                    int head_dim, float scale, float k_scale, float v_scale,
                                    int num_splits, void* workspace, size_t workspace_bytes,
                                    pkv_dtype dtype, int32_t* err_flag, void* stream);

/*
 * One decode step in one launch: the append of one new token per sequence
 * followed by decode attention, with the append done by the decode kernel
 * itself (the pages list KV-cache writes among the ops worth fusing into
 * their neighbours: [vllm-06] kernel fusion).  The result, and the cache after
 * the call, are those of pkv_append with slot_mapping[b] = the slot of
 * position context_lens[b] - 1 of sequence b (block
 * block_tables[b][(n-1) / block_size], offset (n-1) % block_size), followed by
 * pkv_decode_attention.
 *
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim], dtype: sequence b's new
 *                 token, written at position context_lens[b] - 1
 *   k_cache, v_cache  written at those slots; the slots must not be shared
 *                 with another sequence (a page being appended to is private)
 *   other arguments as for pkv_decode_attention
 * A sequence with a bad last block id, or a context_len that is negative or
 * too long, is flagged and its new token is not written.
 */
pkv_status pkv_append_decode_attention(void* out, const void* q, const void* k_new,
                                       const void* v_new, void* k_cache, void* v_cache,
                                       const int32_t* block_tables, int max_blocks_per_seq,
                                       const int32_t* context_lens, int max_context_len,
                                       int num_seqs, int num_blocks, int block_size,
                                       int num_q_heads, int num_kv_heads, int head_dim,
                                       float scale, int num_splits, void* workspace,
                                       size_t workspace_bytes, pkv_dtype dtype,
                                       int32_t* err_flag, void* stream);

/*
 * The same one-launch step over E4M3 caches ([vllm-06] 3.3 FP8 inference;
 * 2.2, the KV-cache write fused with quantisation): the result, and the cache
 * after the call, are those of pkv_append_fp8 with slot_mapping[b] = the slot
 * of position context_lens[b] - 1 of sequence b, followed by
 * pkv_decode_attention_fp8.  The new rows are quantised exactly as
 * pkv_append_fp8 does (the same codes, bit for bit).
 *
 *   k_new, v_new  [num_seqs][num_kv_heads][head_dim], dtype (fp16 or bf16)
 *   k_cache, v_cache  uint8 E4M3 codes, written at those slots (private pages)
 *   k_scale, v_scale, other arguments as for pkv_decode_attention_fp8
 */
pkv_status pkv_append_decode_attention_fp8(void* out, const void* q, const void* k_new,
                                           const void* v_new, void* k_cache, void* v_cache,
                                           const int32_t* block_tables, int max_blocks_per_seq,
                                           const int32_t* context_lens, int max_context_len,
                                           int num_seqs, int num_blocks, int block_size,
                                           int num_q_heads, int num_kv_heads, int head_dim,
                                           float scale, float k_scale, float v_scale,
                                           int num_splits, void* workspace,
                                           size_t workspace_bytes, pkv_dtype dtype,
                                           int32_t* err_flag, void* stream);

/*
 * Decode attention for callers that cannot allocate device memory.
 *
 * The paper has no counterpart to this call; it exists for integration.  Some
 * callers have no way to provide the workspace pkv_decode_attention needs:
 * plain-C hosts with no device allocator of their own, plug-ins living inside
 * another runtime whose memory pool they must not bypass, and latency-bound
 * decode loops that cannot afford cudaMalloc / cudaFree (both may synchronise
 * the whole device).  This entry point takes the same arguments minus the
 * workspace and computes the same result with the same kernels, using instead
 * a fixed scratch array of PKV_NOALLOC_SCRATCH_BYTES that lives in the
 * library's own device memory.  It calls no allocating routine.
 *
 *   - The array is reserved on every GPU that loads the library and stays
 *     reserved until the process exits.
 *   - The array's device address belongs to one CUDA context.  The first
 *     call in each context (for most programs the device's primary context,
 *     so once per device) looks the address up with that context current and
 *     remembers it under the context's id; make that first call before any
 *     stream capture.  A context destroyed and replaced (cudaDeviceReset)
 *     gets a new id, so its successor looks the address up again.
 *   - All calls share the one array, which keeps the previous call's contents.
 *     The kernels overwrite every scratch entry they read, so nothing has to be
 *     cleared, but calls that may run at the same time on the GPU (for
 *     example on two streams without ordering between them) race on it and
 *     corrupt each other's results.  Order them on one stream.
 *   - Returns PKV_ERR_WORKSPACE, launching nothing, when the split plan for
 *     these arguments (the plan pkv_decode_attention makes for a 16-bit
 *     cache) needs more than PKV_NOALLOC_SCRATCH_BYTES; pass a smaller
 *     num_splits, or use pkv_decode_attention.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (8u << 20)

pkv_status pkv_decode_attention_noalloc(void* out, const void* q, const void* k_cache,
                                        const void* v_cache, const int32_t* block_tables,
                                        int max_blocks_per_seq, const int32_t* context_lens,
                                        int max_context_len, int num_seqs, int num_blocks,
                                        int block_size, int num_q_heads, int num_kv_heads,
                                        int head_dim, float scale, int num_splits,
                                        pkv_dtype dtype, int32_t* err_flag, void* stream);

/*
 * Decode attention with shared prompt prefixes.
 *
 * Same result as pkv_decode_attention, for batches whose sequences share
 * physical prefix blocks (Copy-on-Write sharing of a common prefix,
 * [inference] "PagedAttention", Copy-on-Write; prefix trees, [chapter12]
 * RadixAttention): sequences group_start[p] .. group_start[p+1]-1 form group
 * p, and the first group_prefix_len[p] tokens of each member are the same
 * blocks, listed in the block table of the group's first member.  Each group's
 * prefix K/V is read once for all members' queries (the members' query rows
 * stand in for a GQA group's heads on the tensor cores); the suffixes are
 * decoded per sequence; the partials are merged by log-sum-exp.
 *
 *   group_start       int32 [num_groups + 1], device: 0 = group_start[0] <= ...
 *                     <= group_start[num_groups] = num_seqs (a sequence that
 *                     shares nothing is a group of one with prefix 0)
 *   group_prefix_len  int32 [num_groups], device: a multiple of block_size,
 *                     at most max_prefix_len and each member's context
 *                     (members with a shorter context are masked correctly)
 *   max_group_size, max_prefix_len  host-side bounds used to plan
 *   workspace         at least pkv_prefix_shared_workspace_size(...) bytes;
 *                     contents on entry do not matter
 *   err_flag          nullable; also PKV_EFLAG_GROUP for a malformed group, whose
 *                     members are then decoded without the shared prefix
 *                     (still the correct result)
 * The precondition that members' tables hold the group's prefix blocks is not
 * checked: the prefix is read from the first member's table.
 *
 * Streams: the call queues a plan on `stream`, then runs the prefix kernel on a
 * second stream of the library's own (one per CUDA context, made on the
 * context's first such call, highest priority), forked from `stream` after the
 * plan by an event and joined back before the call returns, so that the
 * prefix and the suffix decode run at the same time.  Work queued on `stream`
 * before the call is complete before either starts, and work queued after it
 * sees the whole result, as with a single-stream call; the fork and join are
 * ordinary event records and waits, so the call can be captured in a CUDA
 * graph (make the first call in each context outside the capture, since it
 * creates the stream and its events).  Calls from several host threads are
 * serialised on the host around the fork and join.  When the side stream cannot
 * be had (no current context id, more than 64 contexts), the prefix kernel runs
 * on `stream` between the plan and the decode.  There is no separate merge
 * launch: the CTA that writes the last partial of a (sequence, KV head) merges
 * it, counting down a per-unit count that the plan sets in the workspace.
 */
size_t pkv_prefix_shared_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_context_len,
                                        int num_groups, int max_group_size, int max_prefix_len);

pkv_status pkv_decode_attention_prefix_shared(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int num_blocks, int block_size, int num_q_heads,
    int num_kv_heads, int head_dim, float scale, int num_groups, const int32_t* group_start,
    const int32_t* group_prefix_len, int max_group_size, int max_prefix_len, void* workspace,
    size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag, void* stream);

/*
 * Multi-query attention over the paged cache: q_len new query tokens per
 * sequence, causal within the chunk.  This is the attention of a chunked-prefill
 * chunk ([inference] "Chunked Prefill": the chunk's queries against the cached
 * KV and the chunk's own KV) and of speculative verification, where the large
 * model scores K drafted tokens plus one in a single pass ([inference]
 * "投机采样 (Speculative Decoding)").  The chunk's K/V are appended first
 * (pkv_append with q_len slots per sequence), so context_lens[b] counts them,
 * and query token i of sequence b attends to positions 0 .. n_b - q_len + i
 * (each query sees the keys up to its own position: [chapter12]
 * Attention(Q_t, K_1:t, V_1:t)).
 *
 *   q, out        [num_seqs][q_len][num_q_heads][head_dim], dtype
 *   context_lens  int32 [num_seqs], device: tokens in the cache per sequence,
 *                 at least q_len (a shorter one is flagged PKV_EFLAG_CONTEXT_LEN;
 *                 rows whose limit is not positive get a zero output)
 *   other arguments as for pkv_decode_attention; workspace of at least
 *   pkv_multi_query_workspace_size(...) bytes (contents on entry do not matter)
 * Limits: num_seqs * num_kv_heads and num_seqs * q_len at most 65535.
 * The (query token, query head) rows of one KV head form a dense matrix that
 * meets every context token.  With at most pkv_max_group_size() rows per
 * (sequence, KV head) (q_len * num_q_heads / num_kv_heads: verifying a few
 * drafted tokens, or a small GQA group) the decode kernel serves them as it
 * serves the heads of a GQA group, streaming the context once at the HBM
 * rate, with per-row causal limits on the last positions; up to twice as many
 * rows take two adjacent CTAs that read the context together (the second
 * copy mostly from L2).  With more rows the products run on the tensor cores
 * (tcgen05, 128 rows per CTA, accumulators in tensor memory).  Either way the
 * context is split into partitions whose partials are merged by log-sum-exp
 * as in pkv_merge.
 */
size_t pkv_multi_query_workspace_size(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int max_context_len);

/*
 * The kernel a pkv_multi_query_attention call with these arguments runs on
 * the current device: 1 for the decode kernel, 0 for the tensor-core kernel,
 * -1 when the arguments are invalid or the device cannot be queried.  When
 * num_partitions is not null it receives the context partitions (partial
 * slots per row are the same, or twice as many on the tensor-core kernel with
 * at most 64 rows per (sequence, KV head)).
 */
int pkv_multi_query_plan(int num_seqs, int q_len, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int max_context_len, int* num_partitions);

pkv_status pkv_multi_query_attention(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int num_seqs, int q_len, int num_blocks, int block_size,
    int num_q_heads, int num_kv_heads, int head_dim, float scale, void* workspace,
    size_t workspace_bytes, pkv_dtype dtype, int32_t* err_flag, void* stream);

/*
 * Log-sum-exp merge of split-K partials ([inference] combine_result and the
 * exactness remark after it; [vllm-06] Flash-Decoding merges with the same
 * m / l rescale rule).  Each partial is stored normalised with its
 * log-sum-exp lse_p = M_p + ln L_p; since exp(M_p - M*) L_p = exp(lse_p - M*),
 *     lse* = max_p lse_p,  w_p = exp(lse_p - lse*),  out = sum_p w_p O_p / sum_p w_p
 * is the pages' combine.  lse_p = -inf marks an empty partition (weight 0);
 * a row whose partitions are all empty becomes 0.
 *
 *   out          [num_seqs][num_q_heads][head_dim] (written), dtype
 *   partial_o    float32 [num_seqs][num_q_heads][num_splits][head_dim]
 *   partial_lse  float32 [num_seqs][num_q_heads][num_splits], natural log
 *   head_dim must be a multiple of 4, at most 512 (PKV_ERR_UNSUPPORTED otherwise).
 */
pkv_status pkv_merge(void* out, const float* partial_o, const float* partial_lse, int num_seqs,
                     int num_q_heads, int num_splits, int head_dim, pkv_dtype dtype,
                     void* stream);

/*
 * Block-table gather: copies each sequence's cached K and V rows, in token
 * order, into contiguous buffers ([essay] §三.2 get_kv_cache;
 * [chapter12] PagedKVCache.get):
 *     k_out[b][t][:][:] = k_cache[block_tables[b][t / block_size]][t % block_size][:][:]
 * for t < min(context_lens[b], max_context_len); rows t >= that are left
 * untouched.  Bit-exact.
 *
 *   k_out, v_out   [num_seqs][max_context_len][num_kv_heads][head_dim] (written)
 *   err_flag       nullable; PKV_EFLAG_BLOCK_ID / PKV_EFLAG_CONTEXT_LEN
 */
pkv_status pkv_gather(void* k_out, void* v_out, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int max_context_len, int num_seqs,
                      int num_blocks, int block_size, int num_kv_heads, int head_dim,
                      pkv_dtype dtype, int32_t* err_flag, void* stream);

/*
 * Synchronises `stream`, then reads the device error word.  Returns PKV_OK
 * when it is 0, PKV_ERR_DEVICE_TIMEOUT when PKV_EFLAG_TIMEOUT is set,
 * PKV_ERR_DEVICE_INDEX for any other bit, PKV_ERR_CUDA if the copy fails.
 * When flags_out is not NULL it receives the word.  The word is not cleared.
 */
pkv_status pkv_check_error(const int32_t* err_flag, void* stream, int32_t* flags_out);

/*
 * Self-test of the kernels' failure path (the pages have no counterpart):
 * launches one warp that waits, with the same bounded-wait routine the decode
 * kernel uses, on an mbarrier phase that nothing completes.  After limit_ns
 * nanoseconds (1 .. 1e9) the wait gives up and PKV_EFLAG_TIMEOUT is OR-ed into
 * *err_flag, so pkv_check_error then returns PKV_ERR_DEVICE_TIMEOUT and the
 * context stays usable.  Asynchronous on `stream`.
 */
pkv_status pkv_selftest_wait_timeout(int32_t* err_flag, unsigned long long limit_ns,
                                     void* stream);

/* A static, human-readable name for a status. */
const char* pkv_status_string(pkv_status status);

/* Number of query heads one CTA of the decode kernel serves at most. */
int pkv_max_group_size(void);

/*
 * 1 when the library was compiled with -DPKV_DEBUG, else 0.  A debug build
 * fills every shared-memory ring slot of the decode and tensor-core kernels
 * with NaN bytes at the start and again whenever its stage is released, so a
 * read of a slot whose copy has not landed (or of a stage already released)
 * shows up as NaN in the output.  Slower; for testing only.
 */
int pkv_debug_build(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
