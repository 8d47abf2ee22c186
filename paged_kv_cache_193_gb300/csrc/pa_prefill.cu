// Chunked prefill over the paged cache, for sm_103a.
//
// A chunk of C new tokens ends its sequence's context; each of them attends
// to every token at or before its own position (the cached prefix and the
// chunk's earlier tokens), all read through the sequence's block table
// ("vLLM PagedAttention: Memory Optimization & High-Throughput LLM
// Inference Tuning", section 2).  Chunked prefill itself is named in the
// "Production Checklist" of "Optimizing Llama 3.1 405B Inference with vLLM
// PagedAttention" and in Step 2 of "vLLM PagedAttention Optimization:
// Complete Step-by-Step Tuning Guide".
//
// One CTA per (query tile, KV head, sequence).  A query tile is 64 rows of
// (chunk token, query head of the KV head's group), 16 per consumer warp, so
// every K/V page brought on chip serves the whole group.  A producer warp
// streams the tile's pages (keys up to the tile's last position) with 2-D
// TMA tile loads into a ring of stages shared by the four consumer warps
// (full barrier: the copy landed; empty barrier: all four warps are done).
// Each consumer warp computes S = Q K^T (m16n8k16 MMA, query rows as M, keys
// as N), applies the causal mask, keeps a running max / sum per row, and
// accumulates O += P V with P reused from the S registers.
#include <math.h>

#include <atomic>

#include "pa_prefill.cuh"

namespace pa {

struct PrefillArgs {
    const __nv_bfloat16 *q;      // [total chunk tokens][Hq][D]
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start;  // [S + 1]
    int max_blocks;
    int num_blocks;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int tile_tokens;             // chunk tokens per CTA (64 rows / group)
    float score_scale;           // softmax_scale * log2(e)
    __nv_bfloat16 *out;          // [total chunk tokens][Hq][D]
    unsigned int *err;
};

constexpr int kPrefillWarps = 4;  // consumer warps, 16 query rows each
constexpr int kPrefillRows = kPrefillWarps * 16;
constexpr int kPrefillRingBytes = 64 * 1024;
constexpr uint64_t kPrefillWaitNs = 2000000000ull;

template <int D, int BS>
struct PrefillCfg {
    static constexpr int ROWB = D * 2;
    static constexpr int SLAB = ROWB >= 128 ? 128 : ROWB;
    static constexpr int NSLAB = ROWB / SLAB;
    static constexpr int PAGE = BS * ROWB;
    static constexpr int STAGE = 2 * PAGE;
    static constexpr int NS = kPrefillRingBytes / STAGE >= 2 ? kPrefillRingBytes / STAGE : 2;
    static constexpr int SMEM = NS * STAGE + 1024;
    static constexpr int KSTEPS = D / 16;
    static constexpr int NTK = BS / 8;   // 8-key n-tiles per page
    static constexpr int DT = D / 8;     // 8-dim n-tiles of the output
};

__device__ __forceinline__ uint32_t keep_halves(uint32_t v, bool lo, bool hi) {
    return (lo ? (v & 0xFFFFu) : 0u) | (hi ? (v & 0xFFFF0000u) : 0u);
}

template <int D, int BS>
__global__ void __launch_bounds__((kPrefillWarps + 1) * 32, 2)
    prefill_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const PrefillArgs a) {
    using C = PrefillCfg<D, BS>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[C::NS];
    __shared__ __align__(8) uint64_t empty[C::NS];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;

    const int tile = gridDim.x - 1 - blockIdx.x;  // later (longer) tiles start first
    const int h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q0 = a.query_start[s];
    const int chunk = a.query_start[s + 1] - q0;
    const int ctx = a.context_lens[s];
    const int tok_begin = tile * a.tile_tokens;
    if (tok_begin >= chunk) return;
    if (ctx > a.max_blocks * BS || ctx < chunk) {
        if (tid == 0) set_device_error(a.err, PA_DEVERR_BAD_CONTEXT);
        return;
    }
    const int tok_end = min(tok_begin + a.tile_tokens, chunk);
    const int first_pos = ctx - chunk;            // position of chunk token 0
    const int kend = first_pos + tok_end;         // keys [0, kend) reach the tile's last token
    const int npages = (kend + BS - 1) / BS;

    if (tid == 0) {
        for (int i = 0; i < C::NS; ++i) {
            mbar_init(smem_addr(&full[i]), 1);
            mbar_init(smem_addr(&empty[i]), kPrefillWarps);
        }
        fence_barrier_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();

    if (warp == kPrefillWarps) {
        // ---- producer: pages 0 .. npages-1, table entries 32 at a time ----
        const int32_t *bt = a.block_tables + static_cast<int64_t>(s) * a.max_blocks;
        const uint64_t policy = l2_evict_first_policy();
        const int rows_total = a.num_blocks * a.num_kv_heads * BS;
        bool ok = true;
        for (int j0 = 0; j0 < npages && ok; j0 += 32) {
            const int ent = j0 + lane < npages ? __ldg(bt + j0 + lane) : -1;
            const int cnt = min(32, npages - j0);
            for (int jj = 0; jj < cnt; ++jj) {
                const int blk = __shfl_sync(0xffffffffu, ent, jj);
                if (lane == 0 && ok) {
                    const int j = j0 + jj, st = j % C::NS, use = j / C::NS;
                    if (!mbar_wait_bounded(smem_addr(&empty[st]), (use & 1) ^ 1, kPrefillWaitNs)) {
                        set_device_error(a.err, PA_DEVERR_TIMEOUT);
                        ok = false;
                    } else {
                        int y;
                        if (blk < 0 || blk >= a.num_blocks) {
                            set_device_error(a.err, PA_DEVERR_BAD_BLOCK);
                            y = rows_total;  // wholly outside the tensor: zeros
                        } else {
                            y = (blk * a.num_kv_heads + h) * BS;
                        }
                        const uint32_t bar = smem_addr(&full[st]);
                        const uint32_t kdst = ring + st * C::STAGE, vdst = kdst + C::PAGE;
                        mbar_arrive_expect_tx(bar, C::STAGE);
#pragma unroll
                        for (int sl = 0; sl < C::NSLAB; ++sl) {
                            tma_load_2d(kdst + sl * (BS * C::SLAB), &tmK, sl * (C::SLAB / 2), y, bar, policy);
                            tma_load_2d(vdst + sl * (BS * C::SLAB), &tmV, sl * (C::SLAB / 2), y, bar, policy);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        }
        return;
    }

    // ---- consumers: rows r0 = warp*16 + lane/4 and r1 = r0 + 8 ----------------
    const int r = lane >> 2, c = lane & 3;
    const int rows_valid = (tok_end - tok_begin) * a.group;
    int pos[2];            // query position of each row (-1: padding row)
    const __nv_bfloat16 *qrow[2];
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        const int row = warp * 16 + r + hi * 8;
        const int t = row / a.group, g = row % a.group;
        const bool live = row < rows_valid;
        pos[hi] = live ? first_pos + tok_begin + t : -1;
        qrow[hi] = live ? a.q + ((static_cast<int64_t>(q0) + tok_begin + t) * a.num_q_heads +
                                 h * a.group + g) * D
                        : nullptr;
    }
    uint32_t qa[C::KSTEPS][4];
#pragma unroll
    for (int kk = 0; kk < C::KSTEPS; ++kk) {
        const int d0 = kk * 16 + 2 * c;
        qa[kk][0] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[0] + d0)) : 0u;
        qa[kk][1] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[1] + d0)) : 0u;
        qa[kk][2] = qrow[0] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[0] + d0 + 8)) : 0u;
        qa[kk][3] = qrow[1] ? __ldg(reinterpret_cast<const uint32_t *>(qrow[1] + d0 + 8)) : 0u;
    }
    float o[C::DT][4];
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[dt][e] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    // last key any row of this warp needs: later pages are masked out for all
    // of its rows, so the warp only waits for them and hands them back
    const int warp_last = __reduce_max_sync(0xffffffffu, max(pos[0], pos[1]));

    for (int j = 0; j < npages; ++j) {
        const int st = j % C::NS, use = j / C::NS;
        if (!mbar_wait_bounded(smem_addr(&full[st]), use & 1, kPrefillWaitNs)) {
            // a copy never arrived: flag it, wait (bounded) for the copies
            // that may still be in flight, and finish with what we have
            if (lane == 0) set_device_error(a.err, PA_DEVERR_TIMEOUT);
            for (int jj = j + 1; jj < min(npages, j + C::NS); ++jj)
                mbar_wait_bounded(smem_addr(&full[jj % C::NS]), (jj / C::NS) & 1, kPrefillWaitNs);
            break;
        }
        const int tok0 = j * BS;
        if (tok0 <= warp_last) {
            const uint32_t kbase = ring + st * C::STAGE, vbase = kbase + C::PAGE;
            const int valid = min(BS, kend - tok0);
            float sc[C::NTK][4];
#pragma unroll
            for (int nt = 0; nt < C::NTK; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[nt][e] = 0.f;
            // S = Q K^T over 16-key groups
#pragma unroll
            for (int kg = 0; kg < BS / 16; ++kg) {
                const int mi = lane >> 3;
                const int key = kg * 16 + (mi >> 1) * 8 + (lane & 7);
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(swz_addr<C::SLAB, BS>(kbase, key, (kk * 16 + (mi & 1) * 8) * 2), b0, b1, b2, b3);
                    mma16816<false>(sc[2 * kg], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
                    mma16816<false>(sc[2 * kg + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
                }
            }
            // causal mask, scale, online softmax (2 rows per thread)
#pragma unroll
            for (int hi = 0; hi < 2; ++hi) {
                float mx = -INFINITY;
#pragma unroll
                for (int nt = 0; nt < C::NTK; ++nt)
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int key = tok0 + nt * 8 + 2 * c + jj;
                        float x = sc[nt][hi * 2 + jj] * a.score_scale;
                        x = key <= pos[hi] ? x : -INFINITY;
                        sc[nt][hi * 2 + jj] = x;
                        mx = fmaxf(mx, x);
                    }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
                const float m_new = fmaxf(m_run[hi], mx);
                const float m_use = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = fast_exp2(m_run[hi] - m_use);
                m_run[hi] = m_new;
                float sum = 0.f;
#pragma unroll
                for (int nt = 0; nt < C::NTK; ++nt)
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const float p = fast_exp2(sc[nt][hi * 2 + jj] - m_use);
                        sc[nt][hi * 2 + jj] = p;
                        sum += p;
                    }
                l_run[hi] = l_run[hi] * alpha + sum;
#pragma unroll
                for (int dt = 0; dt < C::DT; ++dt) {
                    o[dt][hi * 2] *= alpha;
                    o[dt][hi * 2 + 1] *= alpha;
                }
            }
            // O += P V over 16-key groups; P reused from the S registers
#pragma unroll
            for (int kg = 0; kg < BS / 16; ++kg) {
                const uint32_t pa0 = pack2<false>(sc[2 * kg][0], sc[2 * kg][1]);
                const uint32_t pa1 = pack2<false>(sc[2 * kg][2], sc[2 * kg][3]);
                const uint32_t pa2 = pack2<false>(sc[2 * kg + 1][0], sc[2 * kg + 1][1]);
                const uint32_t pa3 = pack2<false>(sc[2 * kg + 1][2], sc[2 * kg + 1][3]);
                const int mi = lane >> 3;
                const int key = kg * 16 + (mi & 1) * 8 + (lane & 7);
                // keys at or past `valid` hold whatever the pool held: drop them
                const int kb = kg * 16 + 2 * c;
                const bool partial = valid < BS;
#pragma unroll
                for (int dp = 0; dp < C::DT / 2; ++dp) {
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_trans(swz_addr<C::SLAB, BS>(vbase, key, (dp * 16 + (mi >> 1) * 8) * 2), b0, b1, b2, b3);
                    if (partial) {
                        b0 = keep_halves(b0, kb < valid, kb + 1 < valid);
                        b1 = keep_halves(b1, kb + 8 < valid, kb + 9 < valid);
                        b2 = keep_halves(b2, kb < valid, kb + 1 < valid);
                        b3 = keep_halves(b3, kb + 8 < valid, kb + 9 < valid);
                    }
                    mma16816<false>(o[2 * dp], pa0, pa1, pa2, pa3, b0, b1);
                    mma16816<false>(o[2 * dp + 1], pa0, pa1, pa2, pa3, b2, b3);
                }
            }
        }
        __syncwarp();
        if (lane == 0) asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty[st])) : "memory");
    }

    // ---- epilogue: O / l per row -------------------------------------------------
#pragma unroll
    for (int hi = 0; hi < 2; ++hi) {
        float l = l_run[hi];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        const float inv = l > 0.f ? 1.f / l : 0.f;
        if (pos[hi] < 0) continue;
        const int row = warp * 16 + r + hi * 8;
        const int t = row / a.group, g = row % a.group;
        __nv_bfloat16 *dst = a.out + ((static_cast<int64_t>(q0) + tok_begin + t) * a.num_q_heads +
                                      h * a.group + g) * D;
#pragma unroll
        for (int dt = 0; dt < C::DT; ++dt)
            *reinterpret_cast<__nv_bfloat162 *>(dst + dt * 8 + 2 * c) =
                __floats2bfloat162_rn(o[dt][hi * 2] * inv, o[dt][hi * 2 + 1] * inv);
    }
}

// Slots of every chunk token: one CTA per sequence.
__global__ void chunk_slot_kernel(const int32_t *__restrict__ block_tables, int max_blocks,
                                  const int32_t *__restrict__ context_lens,
                                  const int32_t *__restrict__ query_start, int block_size,
                                  int32_t *__restrict__ slot_mapping, unsigned int *err) {
    const int s = blockIdx.x;
    const int q0 = query_start[s], q1 = query_start[s + 1];
    const int ctx = context_lens[s];
    for (int i = q0 + threadIdx.x; i < q1; i += blockDim.x) {
        const int pos = ctx - (q1 - q0) + (i - q0);
        if (pos < 0 || pos / block_size >= max_blocks) {
            set_device_error(err, PA_DEVERR_BAD_CONTEXT);
            slot_mapping[i] = -1;
            continue;
        }
        const int32_t blk = block_tables[static_cast<int64_t>(s) * max_blocks + pos / block_size];
        slot_mapping[i] = blk * block_size + pos % block_size;
    }
}

template <int D, int BS>
static pa_status launch_prefill(const CUtensorMap &tk, const CUtensorMap &tv, const PrefillArgs &a,
                                dim3 grid, cudaStream_t stream) {
    using C = PrefillCfg<D, BS>;
    auto kern = prefill_kernel<D, BS>;
    static std::atomic<uint64_t> raised{0};
    int dev = 0;
    pa_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != PA_OK) return st;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(raised.load(std::memory_order_acquire) & bit)) {
        st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM),
                        "cudaFuncSetAttribute(prefill)");
        if (st != PA_OK) return st;
        raised.fetch_or(bit, std::memory_order_release);
    }
    kern<<<grid, (kPrefillWarps + 1) * 32, C::SMEM, stream>>>(tk, tv, a);
    return cuda_check(cudaGetLastError(), "prefill launch");
}

pa_status launch_prefill_tc(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                            int total_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int num_blocks, int block_size, bool fp8, float kv_scale,
                            const float *k_scales, const float *v_scales, float softmax_scale, void *out,
                            unsigned int *err, cudaStream_t stream);
static pa_status prefill_impl(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, const int32_t *query_start,
                              int num_seqs, int num_tokens, int max_query_len, int num_q_heads,
                              int num_kv_heads, int head_dim, int num_blocks, int block_size,
                              pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                              void *out, cudaStream_t stream, bool tensor_memory,
                              const float *k_scales = nullptr, const float *v_scales = nullptr);

}  // namespace pa

using namespace pa;

extern "C" {

pa_status pa_chunk_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                                const int32_t *context_lens, const int32_t *query_start,
                                int num_seqs, int block_size, int32_t *slot_mapping,
                                cudaStream_t stream) {
    clear_error();
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad size (num_seqs=%d, max_blocks_per_seq=%d, block_size=%d)",
                    num_seqs, max_blocks_per_seq, block_size);
    if (num_seqs == 0) return PA_OK;
    if (num_seqs > 0x7fffffff / 2) return fail(PA_ERR_UNSUPPORTED, "too many sequences");
    if (!block_tables || !context_lens || !query_start || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    unsigned int *err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    chunk_slot_kernel<<<num_seqs, 128, 0, stream>>>(block_tables, max_blocks_per_seq, context_lens,
                                                    query_start, block_size, slot_mapping, err);
    return cuda_check(cudaGetLastError(), "chunk slot launch");
}

pa_status pa_prefill(const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                     int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                     int head_dim, int num_blocks, int block_size, pa_kv_dtype kv_dtype,
                     float kv_scale, float softmax_scale, void *out, cudaStream_t stream) {
    return prefill_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        query_start, num_seqs, num_tokens, max_query_len, num_q_heads,
                        num_kv_heads, head_dim, num_blocks, block_size, kv_dtype, kv_scale,
                        softmax_scale, out, stream, true);
}

pa_status pa_prefill_mma(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                         int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                         int head_dim, int num_blocks, int block_size, pa_kv_dtype kv_dtype,
                         float kv_scale, float softmax_scale, void *out, cudaStream_t stream) {
    return prefill_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        query_start, num_seqs, num_tokens, max_query_len, num_q_heads,
                        num_kv_heads, head_dim, num_blocks, block_size, kv_dtype, kv_scale,
                        softmax_scale, out, stream, false);
}

pa_status pa_prefill_scaled(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                            int num_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int num_blocks, int block_size, const float *k_scales,
                            const float *v_scales, float softmax_scale, void *out, cudaStream_t stream) {
    if (!k_scales || !v_scales) {
        clear_error();
        return fail(PA_ERR_INVALID_ARG, "null scale array");
    }
    return prefill_impl(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        query_start, num_seqs, num_tokens, max_query_len, num_q_heads,
                        num_kv_heads, head_dim, num_blocks, block_size, PA_KV_FP8_E4M3, 1.f,
                        softmax_scale, out, stream, true, k_scales, v_scales);
}

}  // extern "C"

namespace pa {

static pa_status prefill_impl(const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, int max_blocks_per_seq,
                              const int32_t *context_lens, const int32_t *query_start,
                              int num_seqs, int num_tokens, int max_query_len, int num_q_heads,
                              int num_kv_heads, int head_dim, int num_blocks, int block_size,
                              pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                              void *out, cudaStream_t stream, bool tensor_memory,
                              const float *k_scales, const float *v_scales) {
    clear_error();
    if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || num_q_heads <= 0 ||
        num_kv_heads <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad size");
    if (num_q_heads % num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    num_q_heads, num_kv_heads);
    const int group = num_q_heads / num_kv_heads;
    if (group > 16 || (group & (group - 1)) != 0)
        return fail(PA_ERR_UNSUPPORTED, "query group of %d heads (prefill supports 1, 2, 4, 8, 16)", group);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (block_size != 16 && block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: 16, 32)", block_size);
    const bool fp8 = kv_dtype == PA_KV_FP8_E4M3;
    if (kv_dtype != PA_KV_BF16 && !fp8) return fail(PA_ERR_INVALID_ARG, "unknown kv_dtype %d", static_cast<int>(kv_dtype));
    if (fp8 && !(tensor_memory && head_dim == 128))
        return fail(PA_ERR_UNSUPPORTED, "E4M3 caches: pa_prefill at head_dim 128 only");
    if (fp8 && !k_scales && !(kv_scale > 0.f && isfinite(kv_scale)))
        return fail(PA_ERR_INVALID_ARG, "kv_scale must be positive and finite for an E4M3 cache");
    if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size > 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "pool exceeds 2^31 rows");
    if (num_seqs > 65535 || num_kv_heads > 65535) return fail(PA_ERR_UNSUPPORTED, "grid too large");
    if (!isfinite(softmax_scale)) return fail(PA_ERR_INVALID_ARG, "softmax_scale is not finite");
    // The prefill kernels take each row's maximum over the raw scores and
    // scale it afterwards, which keeps the order only for a positive scale.
    if (!(softmax_scale > 0.f))
        return fail(PA_ERR_UNSUPPORTED, "prefill needs softmax_scale > 0 (got %g)",
                    static_cast<double>(softmax_scale));
    if (num_seqs == 0 || max_query_len == 0 || num_tokens == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start || !out)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return fail(PA_ERR_INVALID_ARG, "q, caches and out must be 16-byte aligned");
    unsigned int *err0 = device_error_word();
    if (!err0) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    if (tensor_memory)
        return launch_prefill_tc(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                 context_lens, query_start, num_seqs, num_tokens, max_query_len,
                                 num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, fp8,
                                 kv_scale, k_scales, v_scales, softmax_scale, out, err0, stream);
    const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
    CUtensorMap tk, tv;
    pa_status st = make_map(&tk, k_cache, false, head_dim, rows, block_size);
    if (st != PA_OK) return st;
    st = make_map(&tv, v_cache, false, head_dim, rows, block_size);
    if (st != PA_OK) return st;
    unsigned int *err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    PrefillArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    a.tile_tokens = kPrefillRows / group;
    a.score_scale = softmax_scale * 1.4426950408889634f;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    dim3 grid((max_query_len + a.tile_tokens - 1) / a.tile_tokens, num_kv_heads, num_seqs);
    if (head_dim == 128)
        return block_size == 16 ? launch_prefill<128, 16>(tk, tv, a, grid, stream)
                                : launch_prefill<128, 32>(tk, tv, a, grid, stream);
    return block_size == 16 ? launch_prefill<64, 16>(tk, tv, a, grid, stream)
                            : launch_prefill<64, 32>(tk, tv, a, grid, stream);
}

}  // namespace pa
