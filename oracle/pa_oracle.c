/*
 * Reference oracle for paged decode attention and the KV-cache append step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously-correct
 * statement of what the GPU path computes.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline leg may load it.  It shares no code,
 * header, table or constant generator with the CUDA library, and it never
 * reads a value produced by that library.
 *
 * Sources (four web pages on vLLM PagedAttention):
 *   - "Optimizing Llama 3.1 405B Inference with vLLM PagedAttention",
 *     sections "Why Standard Attention Fails at Scale" (fixed-size pages of
 *     16 tokens, logical blocks mapped to physical pages) and "PagedAttention
 *     Mechanics" (a page table per sequence; appending a token writes into the
 *     sequence's last page, a fresh page only when needed; shared prefix pages).
 *   - "vLLM PagedAttention: Memory Optimization & High-Throughput LLM Inference
 *     Tuning", section 2 (the kernel fetches K/V by walking the block table;
 *     only the last block of a request is partially filled; shared prompt
 *     blocks) and section 1 (each new token attends to all cached tokens).
 *   - "Optimizing vLLM Throughput with PagedAttention and Continuous Batching
 *     for Llama 3" (grouped-query attention: several query heads share one KV
 *     head).
 *   - "vLLM PagedAttention Optimization: Complete Step-by-Step Tuning Guide",
 *     Step 1 (KV bytes per token formula) and Step 3 (FP8 KV cache); the
 *     E4M3 format is named in "Optimizing Llama 3.1 405B Inference with vLLM
 *     PagedAttention", section "Quantization Without Quality Loss".
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - cache layout [num_blocks][num_kv_heads][block_size][head_dim];
 *   - logical token t of a sequence lives in block_tables[s][t / B] at
 *     offset t % B;
 *   - query head hq reads KV head hq / G with G = Hq / Hkv;
 *   - the new token is appended before attention, so context_lens includes it;
 *   - a negative slot means "skip"; a zero-length context yields zeros;
 *   - FP8 uses one per-tensor scale: stored = e4m3(x / scale) rounded to
 *     nearest-even with saturation to +-448; read back as e4m3(b) * scale.
 *
 * Arithmetic is fp64 except the fp8 encode, which divides in fp32 as the
 * quantisation step is defined on fp32 values.  No blocking, no fusion, no
 * reordering: one (sequence, query head) at a time, tokens in logical order.
 * The outer loop over (sequence, query head) may run on several host threads
 * (OpenMP); every output is written by exactly one thread.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* number formats                                                             */
/* ------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32: widen and convert. */
double pa_oracle_bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 flavour: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * (m/8 * 2^-6); S.1111.111 is NaN; there is no infinity, so the largest
 * finite magnitude is 1.75 * 2^8 = 448. */
double pa_oracle_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 15;
    int mant = code & 7;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant / 8.0, 1 - 7);
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

/* Encode a binary32 value as E4M3: round to the nearest representable value,
 * ties to the code whose mantissa LSB is zero; magnitudes beyond the largest
 * finite value saturate to +-448 (no NaN or infinity is produced from a
 * finite or infinite input); NaN maps to the NaN code 0x7F.  Done by plain
 * search over the 127 non-negative finite codes. */
uint8_t pa_oracle_e4m3_from_float(float x)
{
    if (isnan(x))
        return 0x7F;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double v = pa_oracle_e4m3_to_double((uint8_t)c);
        double err = fabs(v - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(best | (neg << 7));
}

/* ------------------------------------------------------------------------ */
/* KV bytes per token (Step 1 of the tuning guide)                            */
/* ------------------------------------------------------------------------ */

/* 2 (K and V) * layers * KV heads * head_dim * bytes per element. */
int64_t pa_oracle_kv_bytes_per_token(int64_t num_layers, int64_t num_kv_heads,
                                     int64_t head_dim, int64_t bytes_per_elem)
{
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem;
}

/* ------------------------------------------------------------------------ */
/* slot of the newest token                                                  */
/* ------------------------------------------------------------------------ */

/* The token that just arrived sits at logical position ctx - 1; its slot is
 * the physical block holding that position times B plus the offset in it.
 * An empty sequence has no newest token: slot -1. */
void pa_oracle_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs,
                            int block_size, int32_t *slot_mapping)
{
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        if (ctx <= 0) {
            slot_mapping[s] = -1;
            continue;
        }
        int pos = ctx - 1;
        int32_t block = block_tables[(int64_t)s * max_blocks_per_seq + pos / block_size];
        slot_mapping[s] = block * block_size + pos % block_size;
    }
}

/* ------------------------------------------------------------------------ */
/* append                                                                    */
/* ------------------------------------------------------------------------ */

/* Scatter token i's K and V rows (bf16 [T][Hkv][D]) into the cache slot
 * slot_mapping[i].  kv_dtype 0: copy the bf16 bits.  kv_dtype 1: store
 * e4m3(float(x) / scale).  Negative slots are skipped. */
void pa_oracle_cache_append(const uint16_t *k, const uint16_t *v,
                            const int32_t *slot_mapping, int num_tokens,
                            void *k_cache, void *v_cache, int num_kv_heads,
                            int head_dim, int block_size, int kv_dtype, float scale)
{
    for (int i = 0; i < num_tokens; ++i) {
        int32_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim + d;
                int64_t dst = ((block * num_kv_heads + h) * block_size + off) * head_dim + d;
                if (kv_dtype == 0) {
                    ((uint16_t *)k_cache)[dst] = k[src];
                    ((uint16_t *)v_cache)[dst] = v[src];
                } else {
                    float kf = (float)pa_oracle_bf16_to_double(k[src]);
                    float vf = (float)pa_oracle_bf16_to_double(v[src]);
                    ((uint8_t *)k_cache)[dst] = pa_oracle_e4m3_from_float(kf / scale);
                    ((uint8_t *)v_cache)[dst] = pa_oracle_e4m3_from_float(vf / scale);
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* attention                                                                 */
/* ------------------------------------------------------------------------ */

/* Read back one cached element as a real number. */
static double cache_value(const void *cache, int64_t index, int kv_dtype, double kv_scale)
{
    if (kv_dtype == 0)
        return pa_oracle_bf16_to_double(((const uint16_t *)cache)[index]);
    return pa_oracle_e4m3_to_double(((const uint8_t *)cache)[index]) * kv_scale;
}

/* Element index of (logical token t, KV head h, dim d) of sequence s. */
static int64_t token_index(const int32_t *block_tables, int max_blocks_per_seq,
                           int s, int t, int h, int d, int num_kv_heads,
                           int head_dim, int block_size)
{
    int64_t block = block_tables[(int64_t)s * max_blocks_per_seq + t / block_size];
    int64_t off = t % block_size;
    return ((block * num_kv_heads + h) * block_size + off) * head_dim + d;
}

/* Attention of one query head over logical tokens [t_begin, t_end) of one
 * sequence.  Writes o[d] = sum_t p_t V[t][d] with p = softmax over the range
 * of x_t = softmax_scale * q . K[t], and returns the range's max m = max_t x_t
 * and l = sum_t exp(x_t - m) through *m_out and *l_out.  An empty range gives
 * o = 0, m = -inf, l = 0. */
static void attend_range(const uint16_t *q_row, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq, int s, int kvh,
                         int t_begin, int t_end, int num_kv_heads, int head_dim, int block_size,
                         double softmax_scale, int kv_dtype, double k_scale, double v_scale,
                         double *x, double *o, double *m_out, double *l_out)
{
    int n = t_end - t_begin;
    for (int d = 0; d < head_dim; ++d)
        o[d] = 0.0;
    if (n <= 0) {
        *m_out = -INFINITY;
        *l_out = 0.0;
        return;
    }
    /* scores */
    for (int i = 0; i < n; ++i) {
        int t = t_begin + i;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) {
            int64_t idx = token_index(block_tables, max_blocks_per_seq, s, t, kvh, d,
                                      num_kv_heads, head_dim, block_size);
            dot += pa_oracle_bf16_to_double(q_row[d]) * cache_value(k_cache, idx, kv_dtype, k_scale);
        }
        x[i] = softmax_scale * dot;
    }
    /* softmax (max-subtracted for range safety; mathematically the same) */
    double m = x[0];
    for (int i = 1; i < n; ++i)
        if (x[i] > m)
            m = x[i];
    double l = 0.0;
    for (int i = 0; i < n; ++i) {
        x[i] = exp(x[i] - m);
        l += x[i];
    }
    /* weighted sum of values */
    for (int i = 0; i < n; ++i) {
        int t = t_begin + i;
        double p = x[i] / l;
        for (int d = 0; d < head_dim; ++d) {
            int64_t idx = token_index(block_tables, max_blocks_per_seq, s, t, kvh, d,
                                      num_kv_heads, head_dim, block_size);
            o[d] += p * cache_value(v_cache, idx, kv_dtype, v_scale);
        }
    }
    *m_out = m;
    *l_out = l;
}

/* Single-query decode attention through the block table.
 *   q            bf16 [S][Hq][D]
 *   caches       [num_blocks][Hkv][B][D] of kv_dtype (0 bf16, 1 e4m3)
 *   block_tables int32 [S][max_blocks_per_seq]
 *   context_lens int32 [S]
 *   out          fp64 [S][Hq][D]
 * out[s][hq] = softmax(softmax_scale * q[s][hq] . K_s^T) V_s with K_s, V_s the
 * first context_lens[s] logical tokens of KV head hq / (Hq / Hkv). */
void pa_oracle_decode(const uint16_t *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size,
                      double softmax_scale, int kv_dtype, double kv_scale, double *out)
{
    int group = num_q_heads / num_kv_heads;
    int max_ctx = 0;
    for (int s = 0; s < num_seqs; ++s)
        if (context_lens[s] > max_ctx)
            max_ctx = context_lens[s];
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)(max_ctx > 0 ? max_ctx : 1));
#pragma omp for collapse(2) schedule(dynamic)
        for (int s = 0; s < num_seqs; ++s) {
            for (int hq = 0; hq < num_q_heads; ++hq) {
                int kvh = hq / group;
                double m, l;
                attend_range(q + ((int64_t)s * num_q_heads + hq) * head_dim, k_cache, v_cache,
                             block_tables, max_blocks_per_seq, s, kvh, 0, context_lens[s],
                             num_kv_heads, head_dim, block_size, softmax_scale, kv_dtype,
                             kv_scale, kv_scale, x, out + ((int64_t)s * num_q_heads + hq) * head_dim,
                             &m, &l);
            }
        }
        free(x);
    }
}

/* Decode attention for a subset of (sequence, query head) pairs, used to
 * check sampled outputs of large workloads one by one.  pairs is int32
 * [n_pairs][2] of (s, hq); out is fp64 [n_pairs][D]. */
void pa_oracle_decode_pairs(const uint16_t *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size,
                            double softmax_scale, int kv_dtype, double kv_scale,
                            const int32_t *pairs, int n_pairs, double *out)
{
    int group = num_q_heads / num_kv_heads;
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < n_pairs; ++i) {
        int s = pairs[2 * i], hq = pairs[2 * i + 1];
        int n = context_lens[s];
        double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        double m, l;
        attend_range(q + ((int64_t)s * num_q_heads + hq) * head_dim, k_cache, v_cache,
                     block_tables, max_blocks_per_seq, s, hq / group, 0, n, num_kv_heads,
                     head_dim, block_size, softmax_scale, kv_dtype, kv_scale, kv_scale, x,
                     out + (int64_t)i * head_dim, &m, &l);
        free(x);
    }
}

/* Attention restricted to context partition p = [p * P, min((p + 1) * P, ctx))
 * of every (sequence, query head): o fp64 [S][Hq][max_partitions][D],
 * m and l fp64 [S][Hq][max_partitions].  Partitions at or past the end of a
 * sequence get o = 0, m = -inf, l = 0. */
void pa_oracle_decode_partitions(const uint16_t *q, const void *k_cache, const void *v_cache,
                                 const int32_t *block_tables, int max_blocks_per_seq,
                                 const int32_t *context_lens, int num_seqs, int num_q_heads,
                                 int num_kv_heads, int head_dim, int block_size,
                                 double softmax_scale, int kv_dtype, double kv_scale,
                                 int partition_size, int max_partitions,
                                 double *o, double *m, double *l)
{
    int group = num_q_heads / num_kv_heads;
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)partition_size);
#pragma omp for collapse(2) schedule(dynamic)
        for (int s = 0; s < num_seqs; ++s) {
            for (int hq = 0; hq < num_q_heads; ++hq) {
                for (int p = 0; p < max_partitions; ++p) {
                    int64_t row = ((int64_t)s * num_q_heads + hq) * max_partitions + p;
                    int t0 = p * partition_size;
                    int t1 = t0 + partition_size;
                    if (t1 > context_lens[s])
                        t1 = context_lens[s];
                    attend_range(q + ((int64_t)s * num_q_heads + hq) * head_dim, k_cache,
                                 v_cache, block_tables, max_blocks_per_seq, s, hq / group, t0,
                                 t1, num_kv_heads, head_dim, block_size, softmax_scale,
                                 kv_dtype, kv_scale, kv_scale, x, o + row * head_dim, &m[row],
                                 &l[row]);
                }
            }
        }
        free(x);
    }
}

/* Log-sum-exp merge of partition results.  For each (s, hq) with
 * n = ceil(ctx / P) partitions: M = max_p m_p, w_p = l_p exp(m_p - M),
 * out = sum_p w_p o_p / sum_p w_p.  n = 0 gives zeros.  Inputs are the
 * partial arrays laid out as in pa_oracle_decode_partitions (fp32 here, as
 * a caller stores them); out is fp64 [S][Hq][D]. */
void pa_oracle_merge_partitions(const float *o, const float *m, const float *l,
                                const int32_t *context_lens, int num_seqs, int num_q_heads,
                                int head_dim, int partition_size, int max_partitions,
                                double *out)
{
    for (int s = 0; s < num_seqs; ++s) {
        int ctx = context_lens[s];
        int n = ctx > 0 ? (ctx + partition_size - 1) / partition_size : 0;
        for (int hq = 0; hq < num_q_heads; ++hq) {
            int64_t base = ((int64_t)s * num_q_heads + hq) * max_partitions;
            double *dst = out + ((int64_t)s * num_q_heads + hq) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                dst[d] = 0.0;
            if (n == 0)
                continue;
            double big = -INFINITY;
            for (int p = 0; p < n; ++p)
                if ((double)m[base + p] > big)
                    big = (double)m[base + p];
            double total = 0.0;
            for (int p = 0; p < n; ++p)
                total += (double)l[base + p] * exp((double)m[base + p] - big);
            for (int p = 0; p < n; ++p) {
                double w = (double)l[base + p] * exp((double)m[base + p] - big) / total;
                for (int d = 0; d < head_dim; ++d)
                    dst[d] += w * (double)o[(base + p) * head_dim + d];
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* E4M3 cache with a scale per KV head for K and for V                        */
/* ------------------------------------------------------------------------ */

/* The tuning guide's FP8 KV passage (Step 3) fixes no scale granularity.
 * This variant gives every KV head h its own scales: K elements of head h
 * are stored as e4m3(float(x) / k_scales[h]) and read back as
 * e4m3(b) * k_scales[h]; V likewise with v_scales[h].  One scale for the
 * whole cache is the case where every entry is equal. */
void pa_oracle_cache_append_scaled(const uint16_t *k, const uint16_t *v,
                                   const int32_t *slot_mapping, int num_tokens,
                                   uint8_t *k_cache, uint8_t *v_cache, int num_kv_heads,
                                   int head_dim, int block_size, const float *k_scales,
                                   const float *v_scales)
{
    for (int i = 0; i < num_tokens; ++i) {
        int32_t slot = slot_mapping[i];
        if (slot < 0)
            continue;
        int64_t block = slot / block_size;
        int64_t off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            for (int d = 0; d < head_dim; ++d) {
                int64_t src = ((int64_t)i * num_kv_heads + h) * head_dim + d;
                int64_t dst = ((block * num_kv_heads + h) * block_size + off) * head_dim + d;
                float kf = (float)pa_oracle_bf16_to_double(k[src]);
                float vf = (float)pa_oracle_bf16_to_double(v[src]);
                k_cache[dst] = pa_oracle_e4m3_from_float(kf / k_scales[h]);
                v_cache[dst] = pa_oracle_e4m3_from_float(vf / v_scales[h]);
            }
        }
    }
}

/* Decode attention over an E4M3 cache with per-head K and V scales, for the
 * listed (sequence, query head) pairs (all pairs when pairs is NULL, in
 * [S][Hq] order).  out is fp64 [n][D]. */
void pa_oracle_decode_scaled(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, int num_seqs, int num_q_heads,
                             int num_kv_heads, int head_dim, int block_size,
                             double softmax_scale, const float *k_scales, const float *v_scales,
                             const int32_t *pairs, int n_pairs, double *out)
{
    int group = num_q_heads / num_kv_heads;
    int n = pairs ? n_pairs : num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < n; ++i) {
        int s = pairs ? pairs[2 * i] : i / num_q_heads;
        int hq = pairs ? pairs[2 * i + 1] : i % num_q_heads;
        int kvh = hq / group;
        int len = context_lens[s];
        double *x = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
        double m, l;
        attend_range(q + ((int64_t)s * num_q_heads + hq) * head_dim, k_cache, v_cache,
                     block_tables, max_blocks_per_seq, s, kvh, 0, len, num_kv_heads, head_dim,
                     block_size, softmax_scale, 1, (double)k_scales[kvh], (double)v_scales[kvh],
                     x, out + (int64_t)i * head_dim, &m, &l);
        free(x);
    }
}

/* Decode attention whose scores take the query rounded to E4M3 the way the
 * cache's values are (the first ranked variant of the FP8 KV cache, beyond
 * the tuning guide's Step 3, which quantises only the cache): every query
 * element becomes e4m3(float(q) / q_scale) and is read back as
 * e4m3(code) * q_scale.  An E4M3 value is exact in bf16, so the rounded row
 * is passed on as bf16 bits of e4m3(code) with q_scale folded into the
 * softmax scale.  Cache scales per KV head as pa_oracle_decode_scaled. */
void pa_oracle_decode_fp8_qk(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                             const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, int num_seqs, int num_q_heads,
                             int num_kv_heads, int head_dim, int block_size,
                             double softmax_scale, float q_scale, const float *k_scales,
                             const float *v_scales, const int32_t *pairs, int n_pairs,
                             double *out)
{
    int group = num_q_heads / num_kv_heads;
    int n = pairs ? n_pairs : num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < n; ++i) {
        int s = pairs ? pairs[2 * i] : i / num_q_heads;
        int hq = pairs ? pairs[2 * i + 1] : i % num_q_heads;
        int kvh = hq / group;
        int len = context_lens[s];
        const uint16_t *q_row = q + ((int64_t)s * num_q_heads + hq) * head_dim;
        uint16_t *q8 = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)head_dim);
        for (int d = 0; d < head_dim; ++d) {
            float x = (float)pa_oracle_bf16_to_double(q_row[d]);
            float r = (float)pa_oracle_e4m3_to_double(pa_oracle_e4m3_from_float(x / q_scale));
            uint32_t bits;
            memcpy(&bits, &r, sizeof bits);
            q8[d] = (uint16_t)(bits >> 16); /* exact: an E4M3 value has 3 fraction bits */
        }
        double *x = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
        double m, l;
        attend_range(q8, k_cache, v_cache, block_tables, max_blocks_per_seq, s, kvh, 0, len,
                     num_kv_heads, head_dim, block_size, softmax_scale * (double)q_scale, 1,
                     (double)k_scales[kvh], (double)v_scales[kvh], x, out + (int64_t)i * head_dim,
                     &m, &l);
        free(x);
        free(q8);
    }
}

/* ------------------------------------------------------------------------ */
/* chunked prefill: many new tokens per sequence                             */
/* ------------------------------------------------------------------------ */

/* Slots of a chunk of new tokens.  Sequence s brings the
 * C = query_start[s+1] - query_start[s] tokens at the end of its context
 * (context_lens[s] counts them): row i of the chunk is logical position
 * context_lens[s] - C + (i - query_start[s]); its slot is found through the
 * block table as for a single token ("PagedAttention Mechanics"). */
void pa_oracle_chunk_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *context_lens, const int32_t *query_start,
                                  int num_seqs, int block_size, int32_t *slot_mapping)
{
    for (int s = 0; s < num_seqs; ++s) {
        int c = query_start[s + 1] - query_start[s];
        for (int i = query_start[s]; i < query_start[s + 1]; ++i) {
            int pos = context_lens[s] - c + (i - query_start[s]);
            int32_t block = block_tables[(int64_t)s * max_blocks_per_seq + pos / block_size];
            slot_mapping[i] = block * block_size + pos % block_size;
        }
    }
}

/* Chunked prefill attention: each new token attends to every token at or
 * before its own position -- the cached prefix and the chunk's earlier
 * tokens -- read through the block table (the chunk's own K/V are already
 * in the cache).  q and out are [Tq][Hq][D] with the rows of sequence s at
 * [query_start[s], query_start[s+1]); out is fp64. */
void pa_oracle_prefill(const uint16_t *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       double softmax_scale, int kv_dtype, double kv_scale, double *out)
{
    int group = num_q_heads / num_kv_heads;
    int total = query_start[num_seqs];
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < total; ++i) {
        int s = 0;
        while (query_start[s + 1] <= i)
            ++s;
        int c = query_start[s + 1] - query_start[s];
        int pos = context_lens[s] - c + (i - query_start[s]);
        double *x = (double *)malloc(sizeof(double) * (size_t)(context_lens[s] > 0 ? context_lens[s] : 1));
        for (int hq = 0; hq < num_q_heads; ++hq) {
            double m, l;
            attend_range(q + ((int64_t)i * num_q_heads + hq) * head_dim, k_cache, v_cache,
                         block_tables, max_blocks_per_seq, s, hq / group, 0, pos + 1,
                         num_kv_heads, head_dim, block_size, softmax_scale, kv_dtype, kv_scale,
                         kv_scale, x, out + ((int64_t)i * num_q_heads + hq) * head_dim, &m, &l);
        }
        free(x);
    }
}

/* Chunked prefill over an E4M3 cache with a K scale and a V scale per KV
 * head (k_scales[h], v_scales[h]), as pa_oracle_decode_scaled reads it;
 * otherwise as pa_oracle_prefill. */
void pa_oracle_prefill_scaled(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                              double softmax_scale, const float *k_scales, const float *v_scales,
                              double *out)
{
    int group = num_q_heads / num_kv_heads;
    int total = query_start[num_seqs];
#pragma omp parallel for schedule(dynamic)
    for (int i = 0; i < total; ++i) {
        int s = 0;
        while (query_start[s + 1] <= i)
            ++s;
        int c = query_start[s + 1] - query_start[s];
        int pos = context_lens[s] - c + (i - query_start[s]);
        double *x = (double *)malloc(sizeof(double) * (size_t)(context_lens[s] > 0 ? context_lens[s] : 1));
        for (int hq = 0; hq < num_q_heads; ++hq) {
            int kvh = hq / group;
            double m, l;
            attend_range(q + ((int64_t)i * num_q_heads + hq) * head_dim, k_cache, v_cache,
                         block_tables, max_blocks_per_seq, s, kvh, 0, pos + 1, num_kv_heads, head_dim,
                         block_size, softmax_scale, 1, (double)k_scales[kvh], (double)v_scales[kvh], x,
                         out + ((int64_t)i * num_q_heads + hq) * head_dim, &m, &l);
        }
        free(x);
    }
}

/* ------------------------------------------------------------------------ */
/* block allocation for the newest tokens, with copy-on-write                */
/* ------------------------------------------------------------------------ */

/* A token that arrives is added at the end of its sequence, and a new
 * physical block is taken only when the token starts one ("Optimizing Llama
 * 3.1 405B Inference with vLLM PagedAttention", section "PagedAttention
 * Mechanics"); sequences may share the physical blocks of a common prompt
 * ("vLLM PagedAttention: Memory Optimization & High-Throughput LLM Inference
 * Tuning", section 2).  Reading for a shared block that
 * is about to be written (the pages are silent): the writer first gets its
 * own copy (copy-on-write).
 *
 * For every sequence s with n = context_lens[s] > 0 (n counts the token
 * being appended, at position pos = n - 1, logical block j = pos / B):
 *   - pos % B == 0: the token opens block j: it gets a fresh block;
 *   - otherwise, if the block table[s][j] is referenced by more than one
 *     sequence (refcounts[block] > 1, counted before this call): it gets a
 *     fresh block, the rows [0, pos % B) of every KV head of K and V are
 *     copied into it, and the old block loses one reference;
 *   - otherwise nothing changes (the sole owner appends in place).
 * Fresh blocks are taken from the top of the free stack
 * free_blocks[0 .. *free_count) in sequence order (the first sequence that
 * needs one takes free_blocks[*free_count - 1]); each gets refcount 1.
 * Blocks whose count drops to zero are pushed back afterwards, in the order
 * of the last sequence (by index) that copied out of them.  If the stack
 * holds fewer blocks than needed, nothing changes and the call returns 1
 * (else 0).  cow_src[s] receives the block copied from, or -1.
 * Caches are bf16 (elem_bytes 2) or E4M3 (1); layout as elsewhere. */
int pa_oracle_block_alloc(int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int num_seqs, int block_size,
                          int32_t *free_blocks, int32_t *free_count, int32_t *refcounts,
                          int num_blocks, uint8_t *k_cache, uint8_t *v_cache, int num_kv_heads,
                          int head_dim, int elem_bytes, int32_t *cow_src)
{
    int need = 0;
    int *action = (int *)malloc(sizeof(int) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    /* decide, from the state before the call */
    for (int s = 0; s < num_seqs; ++s) {
        int n = context_lens[s];
        action[s] = 0; /* 0 none, 1 fresh, 2 copy */
        cow_src[s] = -1;
        if (n <= 0)
            continue;
        int pos = n - 1;
        int j = pos / block_size;
        if (j >= max_blocks_per_seq)
            continue;
        if (pos % block_size == 0) {
            action[s] = 1;
        } else {
            int32_t cur = block_tables[(int64_t)s * max_blocks_per_seq + j];
            if (cur < 0 || cur >= num_blocks)
                continue;
            if (refcounts[cur] > 1)
                action[s] = 2;
        }
        if (action[s])
            ++need;
    }
    if (need > *free_count) {
        free(action);
        return 1;
    }
    int top = *free_count;
    int taken = 0;
    int32_t *freed = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    int nfreed = 0;
    int64_t row_bytes = (int64_t)head_dim * elem_bytes;
    for (int s = 0; s < num_seqs; ++s) {
        if (!action[s])
            continue;
        int pos = context_lens[s] - 1;
        int j = pos / block_size;
        int64_t entry = (int64_t)s * max_blocks_per_seq + j;
        int32_t fresh = free_blocks[top - 1 - taken];
        ++taken;
        if (action[s] == 2) {
            int32_t old = block_tables[entry];
            int rows = pos % block_size;
            for (int h = 0; h < num_kv_heads; ++h) {
                int64_t src = (((int64_t)old * num_kv_heads + h) * block_size) * row_bytes;
                int64_t dst = (((int64_t)fresh * num_kv_heads + h) * block_size) * row_bytes;
                memcpy(k_cache + dst, k_cache + src, (size_t)(rows * row_bytes));
                memcpy(v_cache + dst, v_cache + src, (size_t)(rows * row_bytes));
            }
            refcounts[old] -= 1;
            cow_src[s] = old;
        }
        block_tables[entry] = fresh;
        refcounts[fresh] = 1;
    }
    /* push blocks left without references, in order of their last copier */
    for (int s = 0; s < num_seqs; ++s) {
        if (action[s] != 2 || refcounts[cow_src[s]] != 0)
            continue;
        int last = 1;
        for (int t = s + 1; t < num_seqs; ++t)
            if (action[t] == 2 && cow_src[t] == cow_src[s])
                last = 0;
        if (last)
            freed[nfreed++] = cow_src[s];
    }
    *free_count = top - taken;
    for (int i = 0; i < nfreed; ++i)
        free_blocks[(*free_count)++] = freed[i];
    free(freed);
    free(action);
    return 0;
}

/* The same for a chunk of new tokens per sequence (chunked prefill): sequence
 * s with c = query_start[s+1] - query_start[s] > 0 new tokens and
 * n = context_lens[s] (which counts them) holds old = n - c tokens already.
 *   - if old % B != 0 and the block holding them, j0 = old / B, is
 *     referenced by more than one sequence (counted before the call): it
 *     gets a fresh block holding a copy of rows [0, old % B) (every KV head,
 *     K and V), and the old block loses one reference;
 *   - every logical block the chunk reaches beyond that, from
 *     (old % B == 0 ? old / B : old / B + 1) to (n - 1) / B, gets a fresh
 *     block.
 * Fresh blocks come off the top of the stack in sequence order, a
 * sequence's copy first and then its new blocks in logical order; each gets
 * refcount 1.  Sequences with c <= 0, with c > n or whose last block lies
 * past max_blocks_per_seq are left alone.  Freed blocks go back as in
 * pa_oracle_block_alloc.  If the stack holds fewer blocks than needed
 * nothing changes and the call returns 1 (else 0). */
int pa_oracle_block_alloc_chunk(int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, const int32_t *query_start,
                                int num_seqs, int block_size, int32_t *free_blocks,
                                int32_t *free_count, int32_t *refcounts, int num_blocks,
                                uint8_t *k_cache, uint8_t *v_cache, int num_kv_heads, int head_dim,
                                int elem_bytes, int32_t *cow_src)
{
    int need = 0;
    int *copy = (int *)malloc(sizeof(int) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    int *first = (int *)malloc(sizeof(int) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    int *last = (int *)malloc(sizeof(int) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    /* decide, from the state before the call */
    for (int s = 0; s < num_seqs; ++s) {
        int c = query_start[s + 1] - query_start[s];
        int n = context_lens[s];
        int old = n - c;
        copy[s] = 0;
        first[s] = 0;
        last[s] = -1; /* no new blocks */
        cow_src[s] = -1;
        if (c <= 0 || old < 0 || (n - 1) / block_size >= max_blocks_per_seq)
            continue;
        if (old % block_size != 0) {
            int32_t cur = block_tables[(int64_t)s * max_blocks_per_seq + old / block_size];
            if (cur >= 0 && cur < num_blocks && refcounts[cur] > 1)
                copy[s] = 1;
            first[s] = old / block_size + 1;
        } else {
            first[s] = old / block_size;
        }
        last[s] = (n - 1) / block_size;
        need += copy[s] + (last[s] - first[s] + 1);
    }
    if (need > *free_count) {
        free(copy);
        free(first);
        free(last);
        return 1;
    }
    int top = *free_count;
    int taken = 0;
    int32_t *freed = (int32_t *)malloc(sizeof(int32_t) * (size_t)(num_seqs > 0 ? num_seqs : 1));
    int nfreed = 0;
    int64_t row_bytes = (int64_t)head_dim * elem_bytes;
    for (int s = 0; s < num_seqs; ++s) {
        int64_t row0 = (int64_t)s * max_blocks_per_seq;
        if (copy[s]) {
            int old = context_lens[s] - (query_start[s + 1] - query_start[s]);
            int64_t entry = row0 + old / block_size;
            int32_t src_block = block_tables[entry];
            int32_t fresh = free_blocks[top - 1 - taken];
            ++taken;
            int rows = old % block_size;
            for (int h = 0; h < num_kv_heads; ++h) {
                int64_t src = (((int64_t)src_block * num_kv_heads + h) * block_size) * row_bytes;
                int64_t dst = (((int64_t)fresh * num_kv_heads + h) * block_size) * row_bytes;
                memcpy(k_cache + dst, k_cache + src, (size_t)(rows * row_bytes));
                memcpy(v_cache + dst, v_cache + src, (size_t)(rows * row_bytes));
            }
            refcounts[src_block] -= 1;
            cow_src[s] = src_block;
            block_tables[entry] = fresh;
            refcounts[fresh] = 1;
        }
        for (int j = first[s]; j <= last[s]; ++j) {
            int32_t fresh = free_blocks[top - 1 - taken];
            ++taken;
            block_tables[row0 + j] = fresh;
            refcounts[fresh] = 1;
        }
    }
    /* push blocks left without references, in order of their last copier */
    for (int s = 0; s < num_seqs; ++s) {
        if (!copy[s] || refcounts[cow_src[s]] != 0)
            continue;
        int is_last = 1;
        for (int t = s + 1; t < num_seqs; ++t)
            if (copy[t] && cow_src[t] == cow_src[s])
                is_last = 0;
        if (is_last)
            freed[nfreed++] = cow_src[s];
    }
    *free_count = top - taken;
    for (int i = 0; i < nfreed; ++i)
        free_blocks[(*free_count)++] = freed[i];
    free(freed);
    free(copy);
    free(first);
    free(last);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* threads                                                                   */
/* ------------------------------------------------------------------------ */

void pa_oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int pa_oracle_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
