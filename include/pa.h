/*
 * pa.h -- C ABI of the paged decode-attention library (libpa.so), sm_103a.
 *
 * The library implements the decode-time hot path of PagedAttention as the
 * four source pages describe it:
 *   - "Optimizing Llama 3.1 405B Inference with vLLM PagedAttention",
 *     "Why Standard Attention Fails at Scale": the KV cache is split into
 *     fixed-size pages (16 tokens by default) mapped from logical blocks;
 *     "PagedAttention Mechanics": a page table per sequence, a new token is
 *     appended into the sequence's last page (a fresh page only when needed),
 *     and sequences may point at the same physical pages (shared prefixes).
 *   - "vLLM PagedAttention: Memory Optimization & High-Throughput LLM
 *     Inference Tuning", section 2: the attention kernel fetches the K/V
 *     vectors by walking the block table; only a request's last block is
 *     partially filled.  Section 1: the new token attends to every cached one.
 *   - "Optimizing vLLM Throughput with PagedAttention and Continuous Batching
 *     for Llama 3": grouped-query attention, several query heads per KV head.
 *   - "vLLM PagedAttention Optimization: Complete Step-by-Step Tuning Guide",
 *     Step 3: an FP8 KV cache halves the bytes read; the format is E4M3
 *     ("Optimizing Llama 3.1 405B Inference with vLLM PagedAttention",
 *     section "Quantization Without Quality Loss").
 *
 * Conventions for every entry point
 *   - All pointers are DEVICE pointers of the current CUDA device unless a
 *     comment says otherwise; the caller owns every buffer.  The library
 *     allocates no device memory, never synchronises the stream it is given,
 *     and enqueues its kernels on `stream` (0 = the legacy default stream).
 *   - Tensors are dense, row-major, in the shapes given below:
 *       q            bf16  [num_seqs][num_q_heads][head_dim]
 *       k_cache/v_cache    [num_blocks][num_kv_heads][block_size][head_dim]
 *                          of bf16 (PA_KV_BF16) or E4M3 bytes (PA_KV_FP8_E4M3)
 *       block_tables int32 [num_seqs][max_blocks_per_seq]; entry j of row s is
 *                          the physical block holding logical tokens
 *                          [j*block_size, (j+1)*block_size) of sequence s
 *       context_lens int32 [num_seqs]; includes the token appended this step
 *       out          bf16  [num_seqs][num_q_heads][head_dim]
 *   - Query head hq attends with KV head hq / (num_q_heads / num_kv_heads).
 *   - Logical token t of sequence s is slot block_tables[s][t / block_size] *
 *     block_size + t % block_size; slot x is row x % block_size of block
 *     x / block_size.
 *   - Supported: head_dim 64 or 128; block_size 16 or 32; group size
 *     num_q_heads / num_kv_heads from 1 to 16; partition_size 0 or a
 *     positive multiple of block_size.  Other values return
 *     PA_ERR_UNSUPPORTED before anything is launched.
 *   - Host-side checks (null or misaligned pointers, negative sizes, shapes
 *     out of range) return an error before anything is launched.  Pointers
 *     must be 16-byte aligned.  A failed CUDA call returns PA_ERR_CUDA; the
 *     message is available from pa_last_error().
 *   - Checks that need the device data (a block id outside [0, num_blocks),
 *     a context longer than the table, a slot outside the pool) are made in
 *     the kernels, which skip the offending item and set a bit in the
 *     library's device error word; read it with pa_device_errors().
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null / misaligned pointer, negative or inconsistent size */
    PA_ERR_UNSUPPORTED = 2, /* well-formed but not built: head_dim, block_size, group, dtype */
    PA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than pa_decode_workspace_size */
    PA_ERR_CUDA = 4         /* a CUDA call failed; see pa_last_error() */
} pa_status;

typedef enum pa_kv_dtype {
    PA_KV_BF16 = 0,      /* cache holds bf16 */
    PA_KV_FP8_E4M3 = 1   /* cache holds OCP E4M3 bytes; value = e4m3(byte) * kv_scale */
} pa_kv_dtype;

/* Bits of the device error word (pa_device_errors). */
#define PA_DEVERR_BAD_BLOCK   0x1u /* a block-table entry outside [0, num_blocks): page read as zeros */
#define PA_DEVERR_BAD_CONTEXT 0x2u /* context_lens[s] > max_blocks_per_seq * block_size: clamped */
#define PA_DEVERR_TIMEOUT     0x4u /* a wait for a page copy exceeded its time limit; output invalid */
#define PA_DEVERR_BAD_SLOT    0x8u /* slot_mapping entry >= num_blocks * block_size: token skipped */
#define PA_DEVERR_OUT_OF_BLOCKS 0x10u /* pa_block_alloc: free stack too short; nothing changed */

/*
 * pa_slot_mapping -- slot of each sequence's newest token.
 * Source: "Optimizing Llama 3.1 405B Inference with vLLM PagedAttention",
 * section "PagedAttention Mechanics": the arriving token is appended at the
 * end of the sequence's logical blocks.
 *   slot_mapping[s] = block_tables[s][(n-1) / block_size] * block_size
 *                     + (n-1) % block_size,   n = context_lens[s] > 0
 *   slot_mapping[s] = -1                      n <= 0
 * The host allocator must already have put a block in the table for
 * position n-1 (a new block is taken only when a token starts one).
 * block_tables, context_lens: inputs as above.  slot_mapping: int32
 * [num_seqs] output.  One kernel.
 */
pa_status pa_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int num_seqs, int block_size,
                          int32_t *slot_mapping, cudaStream_t stream);

/*
 * pa_cache_append -- write each new token's K and V into its cache slot.
 * Source: "Optimizing Llama 3.1 405B Inference with vLLM PagedAttention",
 * section "PagedAttention Mechanics" (append on token arrival); Step 3 of
 * "vLLM PagedAttention Optimization: Complete Step-by-Step Tuning Guide"
 * (FP8 KV cache).
 *   k, v          bf16 [num_tokens][num_kv_heads][head_dim] (inputs)
 *   slot_mapping  int32 [num_tokens]; a negative slot skips the token
 *   k_cache, v_cache  written in place at row slot % block_size of block
 *                 slot / block_size, for every KV head
 *   kv_dtype      PA_KV_BF16: the bf16 bits are copied.
 *                 PA_KV_FP8_E4M3: each element is stored as
 *                 e4m3_rn_satfinite((float)x / scale) (IEEE fp32 division,
 *                 round to nearest even, saturating to +-448).
 *   scale         > 0 and finite for FP8; ignored for bf16.
 * Distinct tokens must have distinct slots.  One kernel.
 */
pa_status pa_cache_append(const void *k, const void *v, const int32_t *slot_mapping,
                          int num_tokens, void *k_cache, void *v_cache, int num_blocks,
                          int num_kv_heads, int head_dim, int block_size,
                          pa_kv_dtype kv_dtype, float scale, cudaStream_t stream);

/*
 * Number of context partitions the workspace is laid out for:
 * ceil(max_blocks_per_seq * block_size / partition_size); 1 when
 * partition_size == 0.
 */
int pa_decode_max_partitions(int max_blocks_per_seq, int block_size, int partition_size);

/*
 * Bytes of workspace pa_decode / pa_decode_partitions need (0 when
 * partition_size == 0).  Layout, with P = pa_decode_max_partitions(...):
 *   float o[num_seqs][num_q_heads][P][head_dim]  partition output, normalised
 *                                                (sum_t p_t V[t] / sum_t p_t)
 *   float m[num_seqs][num_q_heads][P]            partition max of
 *                                                softmax_scale * q.K[t]
 *   float l[num_seqs][num_q_heads][P]            sum_t exp(score_t - m)
 * Only partitions p < ceil(context_lens[s] / partition_size) are written.
 */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                int max_blocks_per_seq, int block_size, int partition_size);

/*
 * pa_decode_partitions -- single-query paged attention, per context partition.
 * Source: section 2 of "vLLM PagedAttention: Memory Optimization ..." (the
 * kernel walks the block table), the GQA passage of the Llama 3 page, and
 * the FP8 KV passage of the tuning guide; the split over long contexts with
 * a log-sum-exp merge is this library's design for 128K contexts (the pages
 * only motivate them: 128000-token max_model_len, ~40 GB per sequence).
 * For every sequence s, KV head h and partition p < ceil(n_s / partition_size)
 * (n_s = context_lens[s]), and every query head hq of h's group, computes
 * over logical tokens t in [p*partition_size, min((p+1)*partition_size, n_s)):
 *   score_t = softmax_scale * kscale * (q[s][hq] . K[t]),
 *   m = max_t score_t, l = sum_t exp(score_t - m),
 *   o = sum_t exp(score_t - m) * vscale * V[t] / l
 * and stores (o, m, l) into the workspace (layout above).  kscale = vscale =
 * kv_scale for FP8, 1 for bf16.  partition_size must be > 0.
 * One kernel.  For the FP8 cache the query is rounded to fp16 for the tensor
 * core product (exact for bf16 values of magnitude in [2^-14, 65504]).
 */
pa_status pa_decode_partitions(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int num_blocks, int block_size,
                               pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                               int partition_size, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * pa_decode_reduce -- log-sum-exp merge of the partitions into the output.
 * Source: the pages motivate contexts of 128K tokens ("vLLM PagedAttention
 * Optimization: Complete Step-by-Step Tuning Guide", Step 1: ~40 GB of KV
 * per 128k-token sequence; "Optimizing Llama 3.1 405B Inference with vLLM
 * PagedAttention", "Why Standard Attention Fails at Scale") but give no
 * split; cutting a long context into partitions and merging them by the
 * log-sum-exp identity is this library's design for such contexts, and the
 * merge reproduces exactly the softmax over the whole context that section 2
 * of "vLLM PagedAttention: Memory Optimization & High-Throughput LLM
 * Inference Tuning" computes through the block table.
 * For each (s, hq) with n = ceil(context_lens[s] / partition_size) > 0:
 *   M = max_p m_p,  w_p = l_p * exp(m_p - M),
 *   out[s][hq] = bf16_rn( sum_p w_p o_p / sum_p w_p )
 * and zeros when n = 0.  workspace as written by pa_decode_partitions (or
 * by the caller in the documented layout) for the same max_blocks_per_seq,
 * block_size and partition_size.  One kernel.
 */
pa_status pa_decode_reduce(const void *workspace, size_t workspace_bytes,
                           const int32_t *context_lens, int num_seqs, int num_q_heads,
                           int head_dim, int max_blocks_per_seq, int block_size,
                           int partition_size, void *out, cudaStream_t stream);

/*
 * pa_decode -- single-query paged decode attention, bf16 output.
 * Source: "vLLM PagedAttention: Memory Optimization & High-Throughput LLM
 * Inference Tuning", section 2 (the kernel gathers each token's K and V by
 * walking the sequence's block table; only the last block is partly
 * filled) and section 1 (the new token attends to every cached token);
 * grouped-query heads as in "Optimizing vLLM Throughput with PagedAttention
 * and Continuous Batching for Llama 3"; the E4M3 cache of Step 3 of the
 * tuning guide.  The optional split (partition_size > 0) is this library's
 * design for long contexts, merged as pa_decode_reduce states.
 *   out[s][hq] = bf16_rn( softmax_t(softmax_scale * kscale * q[s][hq] . K[t])
 *                         . vscale * V )  over the n_s cached tokens of KV head
 *                hq / group; zeros when n_s = 0.
 * partition_size == 0: one pass per (sequence, KV head); workspace unused
 * (may be NULL).  partition_size > 0: pa_decode_partitions followed by
 * pa_decode_reduce on the same stream (two kernels).
 */
pa_status pa_decode(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int num_blocks, int block_size,
                    pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                    int partition_size, void *workspace, size_t workspace_bytes,
                    void *out, cudaStream_t stream);

/*
 * pa_decode_step -- one whole decode step of one layer in one launch (two
 * when split): slot mapping, append and attention fused.
 * For every sequence s with n = context_lens[s] > 0, the new token's rows
 * k_new[s], v_new[s] (bf16 [num_seqs][num_kv_heads][head_dim]) are written
 * into slot block_tables[s][(n-1)/block_size]*block_size + (n-1)%block_size
 * exactly as pa_cache_append writes them (FP8: with scale kv_scale), and then
 * out is computed exactly as pa_decode computes it over the n tokens,
 * including the new one ("PagedAttention Mechanics": append, then attend).
 * slot_mapping (optional, int32 [num_seqs], may be NULL) receives the slots
 * (-1 for empty sequences).  The appended token's block must not be shared
 * with another sequence.  Workspace as for pa_decode.  The append is done by
 * the attention kernel's CTA that owns the token's partition, before it
 * reads that page.
 */
pa_status pa_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int num_blocks, int block_size,
                         pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                         int partition_size, void *workspace, size_t workspace_bytes,
                         int32_t *slot_mapping, void *out, cudaStream_t stream);

/*
 * pa_cache_append_scaled / pa_decode_step_scaled -- the E4M3 cache with its
 * own scale per KV head for K and for V.
 * The tuning guide's FP8 KV passage (Step 3) fixes no scale granularity;
 * these entry points take the per-head reading: K elements of KV head h
 * are stored as e4m3_rn_satfinite((float)x / k_scales[h]) and read back as
 * e4m3(b) * k_scales[h]; V likewise with v_scales[h].  k_scales and
 * v_scales are DEVICE float arrays [num_kv_heads] of positive finite values
 * (not checked); equal entries give the one-scale behaviour of
 * pa_cache_append / pa_decode_step.  The cache dtype is E4M3.
 * pa_decode_step_scaled: as pa_decode_step; k_new and v_new may both be NULL
 * for attention without an append (slot_mapping is then not written).
 */
pa_status pa_cache_append_scaled(const void *k, const void *v, const int32_t *slot_mapping,
                                 int num_tokens, void *k_cache, void *v_cache, int num_blocks,
                                 int num_kv_heads, int head_dim, int block_size,
                                 const float *k_scales, const float *v_scales,
                                 cudaStream_t stream);
pa_status pa_decode_step_scaled(const void *q, const void *k_new, const void *v_new,
                                void *k_cache, void *v_cache, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                int block_size, const float *k_scales, const float *v_scales,
                                float softmax_scale, int partition_size, void *workspace,
                                size_t workspace_bytes, int32_t *slot_mapping, void *out,
                                cudaStream_t stream);

/*
 * pa_block_alloc -- device-side block allocation for the newest tokens, with
 * copy-on-write of shared blocks.
 * Source: a new block is taken only when a token starts one ("Optimizing
 * Llama 3.1 405B Inference with vLLM PagedAttention", section
 * "PagedAttention Mechanics"), and requests may share blocks ("vLLM
 * PagedAttention: Memory Optimization & High-Throughput LLM Inference
 * Tuning", section 2).  Reading for writes into a shared block (the pages
 * are silent): the writer first gets a private copy.
 *   context_lens int32 [num_seqs] (device, in/out): the length including the
 *                token being appended; with advance != 0 every entry > 0 is
 *                first increased by one (one new token per active sequence)
 *                and written back.
 *   For each sequence with n > 0, pos = n - 1, j = pos / block_size:
 *     pos % block_size == 0: block_tables[s][j] = a fresh block;
 *     else if refcounts[block_tables[s][j]] > 1 (counted before the call):
 *       block_tables[s][j] = a fresh block holding a copy of rows
 *       [0, pos % block_size) of the old block (every KV head, K and V), and
 *       the old block loses one reference;
 *     else nothing (the sole owner appends in place).
 *   free_blocks int32 [num_blocks] (device, in/out): a stack whose first
 *                *free_count entries are the free blocks; fresh blocks come
 *                off its top in sequence order (refcount set to 1); blocks
 *                whose count reaches 0 are pushed back afterwards in the
 *                order of the last sequence that copied out of them.
 *   free_count   int32 scalar (device, in/out).
 *   refcounts    int32 [num_blocks] (device, in/out): references per block.
 *   cow_src      int32 [num_seqs] (device, out): block copied from, or -1.
 * If the stack holds fewer blocks than needed nothing changes and the device
 * error word gets PA_DEVERR_OUT_OF_BLOCKS.  Deterministic (one CTA decides
 * in sequence order).  num_seqs <= 16384.  Two kernels (decide, copy).
 */
pa_status pa_block_alloc(int32_t *block_tables, int max_blocks_per_seq, int32_t *context_lens,
                         int num_seqs, int block_size, int advance, int32_t *free_blocks,
                         int32_t *free_count, int32_t *refcounts, int num_blocks, void *k_cache,
                         void *v_cache, int num_kv_heads, int head_dim, pa_kv_dtype kv_dtype,
                         int32_t *cow_src, cudaStream_t stream);

/*
 * pa_block_alloc_chunk -- the same for a chunk of new tokens per sequence
 * (chunked prefill).  Same source and readings as pa_block_alloc.
 *   query_start  int32 [num_seqs + 1] (device): sequence s brings
 *                c = query_start[s+1] - query_start[s] tokens at the end of
 *                its context; context_lens[s] (device, read only) counts
 *                them, so old = context_lens[s] - c tokens are cached.
 *   For each sequence with c > 0:
 *     if old % block_size != 0 and refcounts[block_tables[s][old / B]] > 1
 *       (counted before the call): that entry = a fresh block holding a
 *       copy of rows [0, old % block_size) of the old block (every KV head,
 *       K and V), and the old block loses one reference;
 *     every logical block from (old % B ? old / B + 1 : old / B) to
 *       (context_lens[s] - 1) / B gets a fresh block.
 *   Fresh blocks come off the top of the stack in sequence order, a
 *   sequence's copy first and then its new blocks in logical order; freed
 *   blocks go back as in pa_block_alloc.  A sequence with c > context_lens[s]
 *   or a last block past max_blocks_per_seq is left alone and
 *   PA_DEVERR_BAD_CONTEXT is set.  If the stack holds fewer blocks than
 *   needed nothing changes and PA_DEVERR_OUT_OF_BLOCKS is set.
 *   num_seqs <= 16384.  Two kernels (decide, copy).
 */
pa_status pa_block_alloc_chunk(int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, const int32_t *query_start,
                               int num_seqs, int block_size, int32_t *free_blocks,
                               int32_t *free_count, int32_t *refcounts, int num_blocks,
                               void *k_cache, void *v_cache, int num_kv_heads, int head_dim,
                               pa_kv_dtype kv_dtype, int32_t *cow_src, cudaStream_t stream);

/*
 * pa_decode_step_fp8_qk -- pa_decode_step_scaled with the scores taken as an
 * E4M3 x E4M3 tensor-core product (the first ranked variant of the FP8 KV
 * cache; the tuning guide's Step 3 quantises only the cache, so this is an
 * opt-in change to what is computed).  Every query element is first rounded
 * exactly as the cache's values are: q8 = e4m3_rn_satfinite((float)q / q_scale),
 * and the scores are softmax_scale * q_scale * k_scales[h] * sum_d
 * e4m3(q8[d]) * e4m3(k[t][d]); the softmax, PV and output are as in
 * pa_decode_step_scaled.  q_scale: a HOST float, positive and finite
 * (PA_ERR_INVALID_ARG otherwise); queries with |q| / q_scale above 448
 * saturate.  Other arguments and layouts as pa_decode_step_scaled.
 */
pa_status pa_decode_step_fp8_qk(const void *q, const void *k_new, const void *v_new,
                                void *k_cache, void *v_cache, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                int block_size, const float *k_scales, const float *v_scales,
                                float q_scale, float softmax_scale, int partition_size,
                                void *workspace, size_t workspace_bytes, int32_t *slot_mapping,
                                void *out, cudaStream_t stream);

/*
 * pa_chunk_slot_mapping / pa_prefill -- chunked prefill over the paged cache.
 * Chunked prefill is named in the "Production Checklist" of "Optimizing
 * Llama 3.1 405B Inference with vLLM PagedAttention" and in Step 2 of "vLLM
 * PagedAttention Optimization: Complete Step-by-Step Tuning Guide"; the
 * attention walks the block table as the decode does ("vLLM PagedAttention:
 * Memory Optimization & High-Throughput LLM Inference Tuning", section 2).
 * Sequence s brings C_s = query_start[s+1] - query_start[s] new tokens at the
 * END of its context: context_lens[s] >= C_s counts them, and chunk row i
 * (query_start[s] <= i < query_start[s+1]) is logical position
 * p_i = context_lens[s] - C_s + (i - query_start[s]).
 *   query_start  int32 [num_seqs + 1] (device), query_start[0] = 0.
 * pa_chunk_slot_mapping: slot_mapping[i] = slot of position p_i (int32
 *   [query_start[num_seqs]] output), for pa_cache_append of the chunk's K/V.
 * pa_prefill: for every chunk row i and query head hq,
 *   out[i][hq] = bf16_rn( softmax_{t <= p_i}(softmax_scale * q[i][hq] . K[t])
 *                         . V ),  K/V of KV head hq / group, t over the
 *   sequence's logical tokens 0..p_i through the block table (the chunk's
 *   own K/V must already be in the cache).
 *   q, out bf16 [num_tokens][num_q_heads][head_dim], num_tokens =
 *   query_start[num_seqs] (the host's count of chunk rows).
 *   max_query_len >= every C_s (host-side bound used for the grid).
 *   Supported: group 1, 2, 4, 8 or 16, block 16/32, softmax_scale > 0, and
 *   a bf16 cache at head_dim 64/128 or an E4M3 cache (x / kv_scale, one
 *   scale for K and V, kv_scale > 0) at head_dim 128 (PA_ERR_UNSUPPORTED
 *   otherwise; the E4M3 cache is the one "Step 3 (FP8 KV cache)" of the
 *   tuning guide names).  One kernel on the tcgen05 tensor cores
 *   (accumulators in tensor memory); with an E4M3 cache the pages are
 *   widened exactly to fp16 in shared memory and the products run in
 *   fp16 (the query rounded to fp16, exact for bf16 values in its range).
 *   kv_scale is unused for a bf16 cache.
 * pa_prefill_scaled: the same over an E4M3 cache with a K and a V scale per
 *   KV head (k_scales, v_scales: float32 [num_kv_heads], device), the cache
 *   holding x / scale[h] as pa_cache_append_scaled writes it ("Step 3 (FP8
 *   KV cache)" of the tuning guide; per-head scales are a reading, as for
 *   pa_decode_step_scaled).  head_dim 128; null scale arrays are rejected.
 * pa_prefill_mma: the same computation always with the warp-level MMA
 *   kernel (kept as the comparison point for the tensor-memory kernel);
 *   bf16 caches only.
 */
pa_status pa_chunk_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, const int32_t *query_start,
                                int num_seqs, int block_size, int32_t *slot_mapping,
                                cudaStream_t stream);
pa_status pa_prefill(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                     int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                     int head_dim, int num_blocks, int block_size, pa_kv_dtype kv_dtype,
                     float kv_scale, float softmax_scale, void *out, cudaStream_t stream);
pa_status pa_prefill_scaled(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                            int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int num_blocks, int block_size, const float *k_scales,
                            const float *v_scales, float softmax_scale, void *out, cudaStream_t stream);
pa_status pa_prefill_mma(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                         int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                         int head_dim, int num_blocks, int block_size, pa_kv_dtype kv_dtype,
                         float kv_scale, float softmax_scale, void *out, cudaStream_t stream);

/*
 * pa_decode_static_workspace -- pa_decode with partition_size > 0, without
 * the caller's workspace.
 * The source pages have no counterpart to this entry point.  It exists for
 * callers that cannot allocate device memory at the time they run attention
 * (device memory owned by another framework's pool, hosts that forbid
 * allocation after start-up, paths where the device-wide synchronisation of
 * cudaMalloc/cudaFree is not acceptable).  The split path's scratch lives in
 * a fixed array of PA_STATIC_WORKSPACE_BYTES inside the library, which every
 * GPU holds from the moment the library's module is loaded on it until the
 * process exits.  The call allocates nothing.
 *   Arguments, layouts and results: as pa_decode; partition_size must be
 *   > 0.  A call whose scratch (pa_decode_workspace_size) would exceed
 *   PA_STATIC_WORKSPACE_BYTES returns PA_ERR_WORKSPACE before launching.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current, and looks it up again
 *   when the device's context has been re-created (after cudaDeviceReset);
 *   make that first call before capturing any stream.
 *   All calls share the one array and nothing in it needs to start at zero;
 *   calls that can overlap on the GPU (other streams, other host threads)
 *   race on it and must be serialised by the caller.  Two kernels.
 */
#define PA_STATIC_WORKSPACE_BYTES (32u << 20)
pa_status pa_decode_static_workspace(const void *q, const void *k_cache, const void *v_cache,
                                     const int32_t *block_tables, int max_blocks_per_seq,
                                     const int32_t *context_lens, int num_seqs, int num_q_heads,
                                     int num_kv_heads, int head_dim, int num_blocks,
                                     int block_size, pa_kv_dtype kv_dtype, float kv_scale,
                                     float softmax_scale, int partition_size, void *out,
                                     cudaStream_t stream);

/*
 * pa_device_errors -- read (and with clear != 0, reset) the device error
 * word of the current device into *flags (PA_DEVERR_* bits).  This call
 * synchronises the device.  flags is a HOST pointer.
 */
pa_status pa_device_errors(unsigned int *flags, int clear);

/*
 * pa_test_set_wait -- TEST HOOK for the kernels' bounded waits; not for
 * production use.  The pages have no counterpart: every wait of the decode
 * kernel and of the tensor-memory prefill kernel gives up after a time
 * limit, sets PA_DEVERR_TIMEOUT, waits for the copies still in flight and
 * finishes (the decode with zeros for the affected rows, the prefill with
 * an invalid output), so a copy that never lands cannot hang the GPU.
 * This call sets that limit for kernels launched afterwards (limit_ns = 0
 * restores the default of 2 s; above 60 s is refused).  With
 * stall_first_wait != 0 the first wait (each warp's in a pa_decode*
 * kernel, the MMA threads' in pa_prefill's tensor-memory kernel) is made on
 * a barrier that nothing completes, so it runs out after limit_ns: tests use
 * this to drive the give-up path without a real fault.  The drain of the
 * copies already issued always keeps the 2 s limit.  Process-wide; read at
 * launch time on the host, so set it while none of the library's calls is
 * being made.
 */
pa_status pa_test_set_wait(uint64_t limit_ns, int stall_first_wait);

/* Static description of a status code (never NULL). */
const char *pa_status_string(pa_status status);

/* Message describing the most recent failure on the calling host thread
 * (which argument was rejected, or the CUDA error); "" if none. */
const char *pa_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H */
