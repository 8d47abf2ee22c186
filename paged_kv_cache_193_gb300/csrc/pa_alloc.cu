// Device-side block allocation for the newest tokens, with copy-on-write.
//
// A token that arrives is added at the end of its sequence, and a new
// physical block is taken only when the token starts one ("Optimizing Llama
// 3.1 405B Inference with vLLM PagedAttention", section "PagedAttention
// Mechanics");
// sequences may share the blocks of a common prompt ("vLLM PagedAttention:
// Memory Optimization & High-Throughput LLM Inference Tuning", section 2).  A
// token written into a block that other sequences also reference first gets a
// private copy of the block's rows.
//
// One CTA of 1024 threads makes every decision with block-wide scans in
// sequence order, so the result is deterministic: fresh blocks come off the
// top of the free stack in sequence order, and blocks left without
// references are pushed back in the order of the last sequence that copied
// out of them.  A second kernel copies the rows, one CTA per (sequence, KV
// head).
#include "pa_device.cuh"

namespace pa {

constexpr int kAllocThreads = 1024;
constexpr int kAllocChunks = 16;  // sequences per thread: up to 16384 sequences
constexpr int kMaxAllocSeqs = kAllocThreads * kAllocChunks;

// Exclusive prefix sum over the CTA of one int per thread; returns this
// thread's offset and leaves the CTA total in *total for every thread.
__device__ __forceinline__ int cta_exclusive_scan(int v, int *total) {
    __shared__ int warp_off[kAllocThreads / 32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_off[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const int w = warp_off[lane];
        int y = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int z = __shfl_up_sync(0xffffffffu, y, o);
            if (lane >= o) y += z;
        }
        warp_off[lane] = y - w;
        if (lane == 31) *total = y;
    }
    __syncthreads();
    const int res = warp_off[warp] + x - v;
    __syncthreads();
    return res;
}

// Per-sequence decision kept in cow_src while the kernel runs:
// >= 0 copy-on-write from that block, kFresh a fresh block, kNone nothing.
constexpr int kNone = -1;
constexpr int kFresh = -2;

__global__ void __launch_bounds__(kAllocThreads)
    block_alloc_kernel(int32_t *__restrict__ block_tables, int max_blocks,
                       int32_t *__restrict__ context_lens, int num_seqs, int block_size,
                       int advance, int32_t *__restrict__ free_blocks,
                       int32_t *__restrict__ free_count, int32_t *__restrict__ refcounts,
                       int num_blocks, int32_t *__restrict__ cow_src, unsigned int *err) {
    __shared__ int total_s;
    __shared__ unsigned int zero_bits[kMaxAllocSeqs / 32];    // copied-from block reached 0
    __shared__ unsigned int pusher_bits[kMaxAllocSeqs / 32];  // ... and this sequence pushes it
    const int tid = threadIdx.x;
    const int top = *free_count;
    // context length of sequence s including the token appended now
    auto ctx_of = [&](int s) {
        const int n = context_lens[s];
        return (advance && n > 0) ? n + 1 : n;
    };
    auto bit_get = [](const unsigned int *bits, int s) { return (bits[s >> 5] >> (s & 31)) & 1u; };

    for (int i = tid; i < kMaxAllocSeqs / 32; i += kAllocThreads) zero_bits[i] = pusher_bits[i] = 0;

    // 1. decide every sequence's action from the state before the call
    int need = 0;
    for (int s = tid; s < num_seqs; s += kAllocThreads) {
        int act = kNone;
        const int n = ctx_of(s);
        if (n > 0) {
            const int pos = n - 1, j = pos / block_size;
            if (j >= max_blocks) {
                set_device_error(err, PA_DEVERR_BAD_CONTEXT);
            } else if (pos % block_size == 0) {
                act = kFresh;
            } else {
                const int b = block_tables[static_cast<int64_t>(s) * max_blocks + j];
                if (b < 0 || b >= num_blocks)
                    set_device_error(err, PA_DEVERR_BAD_BLOCK);
                else if (refcounts[b] > 1)
                    act = b;
            }
        }
        cow_src[s] = act;
        need += act != kNone;
    }
    cta_exclusive_scan(need, &total_s);
    const int total = total_s;
    if (total > top) {  // not enough free blocks: change nothing
        if (tid == 0) set_device_error(err, PA_DEVERR_OUT_OF_BLOCKS);
        for (int s = tid; s < num_seqs; s += kAllocThreads) cow_src[s] = kNone;
        return;
    }

    // 2. hand out fresh blocks in sequence order; drop the copied-from refs
    int taken = 0;
    for (int base = 0; base < num_seqs; base += kAllocThreads) {  // uniform trip count
        const int s = base + tid;
        const int act = s < num_seqs ? cow_src[s] : kNone;
        const int rank = cta_exclusive_scan(act != kNone, &total_s);
        if (act != kNone) {
            const int fresh = free_blocks[top - 1 - (taken + rank)];
            const int pos = ctx_of(s) - 1;
            block_tables[static_cast<int64_t>(s) * max_blocks + pos / block_size] = fresh;
            refcounts[fresh] = 1;
            if (act >= 0) atomicSub(&refcounts[act], 1);
        }
        taken += total_s;
        __syncthreads();
    }

    // 3. blocks whose count reached zero go back on the stack in the order of
    //    their last copier: each copier of such a block bids -(index + 1)
    //    into the (zero) count with atomicMin; the largest index wins.
    for (int s = tid; s < num_seqs; s += kAllocThreads) {
        const int act = cow_src[s];
        if (act >= 0 && refcounts[act] == 0) atomicOr(&zero_bits[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    for (int s = tid; s < num_seqs; s += kAllocThreads)
        if (bit_get(zero_bits, s)) atomicMin(&refcounts[cow_src[s]], -(s + 1));
    __syncthreads();
    for (int s = tid; s < num_seqs; s += kAllocThreads)
        if (bit_get(zero_bits, s) && refcounts[cow_src[s]] == -(s + 1))
            atomicOr(&pusher_bits[s >> 5], 1u << (s & 31));
    __syncthreads();
    const int base_top = top - total;
    int pushed = 0;
    for (int base = 0; base < num_seqs; base += kAllocThreads) {
        const int s = base + tid;
        const int p = s < num_seqs ? static_cast<int>(bit_get(pusher_bits, s)) : 0;
        const int rank = cta_exclusive_scan(p, &total_s);
        if (p) {
            refcounts[cow_src[s]] = 0;
            free_blocks[base_top + pushed + rank] = cow_src[s];
        }
        pushed += total_s;
        __syncthreads();
    }
    for (int s = tid; s < num_seqs; s += kAllocThreads) {
        if (cow_src[s] == kFresh) cow_src[s] = kNone;
        if (advance) context_lens[s] = ctx_of(s);
    }
    if (tid == 0) *free_count = base_top + pushed;
}

// Copy rows [0, pos % B) of KV head blockIdx.y from the shared block to the
// sequence's new block, for K and V; pos is the first new token's position
// (n - 1, or n - c for a chunk of c tokens when query_start is given).
__global__ void cow_copy_kernel(const int32_t *__restrict__ block_tables, int max_blocks,
                                const int32_t *__restrict__ context_lens,
                                const int32_t *__restrict__ query_start,
                                const int32_t *__restrict__ cow_src, int block_size,
                                int num_kv_heads, int row_bytes, uint8_t *__restrict__ k_cache,
                                uint8_t *__restrict__ v_cache) {
    const int s = blockIdx.x, h = blockIdx.y;
    const int src = cow_src[s];
    if (src < 0) return;
    const int pos = context_lens[s] - (query_start ? query_start[s + 1] - query_start[s] : 1);
    const int dst = block_tables[static_cast<int64_t>(s) * max_blocks + pos / block_size];
    const int64_t head_bytes = static_cast<int64_t>(block_size) * row_bytes;
    const int64_t so = (static_cast<int64_t>(src) * num_kv_heads + h) * head_bytes;
    const int64_t dof = (static_cast<int64_t>(dst) * num_kv_heads + h) * head_bytes;
    const int vecs = (pos % block_size) * row_bytes / 16;
    for (int i = threadIdx.x; i < vecs; i += blockDim.x) {
        reinterpret_cast<uint4 *>(k_cache + dof)[i] = reinterpret_cast<const uint4 *>(k_cache + so)[i];
        reinterpret_cast<uint4 *>(v_cache + dof)[i] = reinterpret_cast<const uint4 *>(v_cache + so)[i];
    }
}

// The same for a chunk of c = query_start[s+1] - query_start[s] new tokens
// per sequence (context_lens counts them): a copy of a shared, partly filled
// last block, then a fresh block for every further block the chunk reaches;
// a sequence's fresh blocks come off the stack one after the other (its copy
// first, then its new blocks in logical order), the sequences in order.
__global__ void __launch_bounds__(kAllocThreads)
    block_alloc_chunk_kernel(int32_t *__restrict__ block_tables, int max_blocks,
                             const int32_t *__restrict__ context_lens,
                             const int32_t *__restrict__ query_start, int num_seqs, int block_size,
                             int32_t *__restrict__ free_blocks, int32_t *__restrict__ free_count,
                             int32_t *__restrict__ refcounts, int num_blocks,
                             int32_t *__restrict__ cow_src, unsigned int *err) {
    __shared__ int total_s;
    __shared__ unsigned int zero_bits[kMaxAllocSeqs / 32];    // copied-from block reached 0
    __shared__ unsigned int pusher_bits[kMaxAllocSeqs / 32];  // ... and this sequence pushes it
    const int tid = threadIdx.x;
    const int top = *free_count;
    auto bit_get = [](const unsigned int *bits, int s) { return (bits[s >> 5] >> (s & 31)) & 1u; };
    // sequence s's new blocks [first, last] (none if last < first), from the
    // state before the call; `report` flags bad inputs once
    auto span = [&](int s, bool report, int &first, int &last) {
        first = 0;
        last = -1;
        const int c = query_start[s + 1] - query_start[s];
        const int n = context_lens[s], old = n - c;
        if (c <= 0) return;
        if (old < 0 || (n - 1) / block_size >= max_blocks) {
            if (report) set_device_error(err, PA_DEVERR_BAD_CONTEXT);
            return;
        }
        first = old % block_size ? old / block_size + 1 : old / block_size;
        last = (n - 1) / block_size;
    };

    for (int i = tid; i < kMaxAllocSeqs / 32; i += kAllocThreads) zero_bits[i] = pusher_bits[i] = 0;

    // 1. decide every sequence's copy and count its blocks
    int need = 0;
    for (int s = tid; s < num_seqs; s += kAllocThreads) {
        int first, last;
        span(s, true, first, last);
        int act = kNone;
        if (last >= 0) {
            const int old = context_lens[s] - (query_start[s + 1] - query_start[s]);
            if (old % block_size) {
                const int b = block_tables[static_cast<int64_t>(s) * max_blocks + old / block_size];
                if (b < 0 || b >= num_blocks)
                    set_device_error(err, PA_DEVERR_BAD_BLOCK);
                else if (refcounts[b] > 1)
                    act = b;
            }
        }
        cow_src[s] = act;
        need += (act >= 0) + max(0, last - first + 1);
    }
    cta_exclusive_scan(need, &total_s);
    const int total = total_s;
    if (total > top) {  // not enough free blocks: change nothing
        if (tid == 0) set_device_error(err, PA_DEVERR_OUT_OF_BLOCKS);
        for (int s = tid; s < num_seqs; s += kAllocThreads) cow_src[s] = kNone;
        return;
    }

    // 2. hand out fresh blocks in sequence order; drop the copied-from refs
    int taken = 0;
    for (int base = 0; base < num_seqs; base += kAllocThreads) {  // uniform trip count
        const int s = base + tid;
        int first = 0, last = -1, act = kNone;
        if (s < num_seqs) {
            span(s, false, first, last);
            act = cow_src[s];
        }
        const int mine = (act >= 0) + max(0, last - first + 1);
        const int off = cta_exclusive_scan(mine, &total_s);
        if (mine > 0) {
            int32_t *row = block_tables + static_cast<int64_t>(s) * max_blocks;
            int k = taken + off;
            if (act >= 0) {
                const int old = context_lens[s] - (query_start[s + 1] - query_start[s]);
                const int fresh = free_blocks[top - 1 - k++];
                row[old / block_size] = fresh;
                refcounts[fresh] = 1;
                atomicSub(&refcounts[act], 1);
            }
            for (int j = first; j <= last; ++j) {
                const int fresh = free_blocks[top - 1 - k++];
                row[j] = fresh;
                refcounts[fresh] = 1;
            }
        }
        taken += total_s;
        __syncthreads();
    }

    // 3. blocks whose count reached zero go back on the stack in the order of
    //    their last copier (as in block_alloc_kernel)
    for (int s = tid; s < num_seqs; s += kAllocThreads) {
        const int act = cow_src[s];
        if (act >= 0 && refcounts[act] == 0) atomicOr(&zero_bits[s >> 5], 1u << (s & 31));
    }
    __syncthreads();
    for (int s = tid; s < num_seqs; s += kAllocThreads)
        if (bit_get(zero_bits, s)) atomicMin(&refcounts[cow_src[s]], -(s + 1));
    __syncthreads();
    for (int s = tid; s < num_seqs; s += kAllocThreads)
        if (bit_get(zero_bits, s) && refcounts[cow_src[s]] == -(s + 1))
            atomicOr(&pusher_bits[s >> 5], 1u << (s & 31));
    __syncthreads();
    const int base_top = top - total;
    int pushed = 0;
    for (int base = 0; base < num_seqs; base += kAllocThreads) {
        const int s = base + tid;
        const int p = s < num_seqs ? static_cast<int>(bit_get(pusher_bits, s)) : 0;
        const int rank = cta_exclusive_scan(p, &total_s);
        if (p) {
            refcounts[cow_src[s]] = 0;
            free_blocks[base_top + pushed + rank] = cow_src[s];
        }
        pushed += total_s;
        __syncthreads();
    }
    if (tid == 0) *free_count = base_top + pushed;
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_block_alloc(int32_t *block_tables, int max_blocks_per_seq,
                                    int32_t *context_lens, int num_seqs, int block_size,
                                    int advance, int32_t *free_blocks, int32_t *free_count,
                                    int32_t *refcounts, int num_blocks, void *k_cache,
                                    void *v_cache, int num_kv_heads, int head_dim,
                                    pa_kv_dtype kv_dtype, int32_t *cow_src, cudaStream_t stream) {
    clear_error();
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0 ||
        num_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad size (num_seqs=%d, max_blocks_per_seq=%d, "
                    "block_size=%d, num_blocks=%d, num_kv_heads=%d)", num_seqs,
                    max_blocks_per_seq, block_size, num_blocks, num_kv_heads);
    if (num_seqs > kMaxAllocSeqs)
        return fail(PA_ERR_UNSUPPORTED, "more than %d sequences", kMaxAllocSeqs);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (block_size != 16 && block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: 16, 32)", block_size);
    if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d", static_cast<int>(kv_dtype));
    if (num_seqs == 0) return PA_OK;
    if (!block_tables || !context_lens || !free_blocks || !free_count || !refcounts || !k_cache ||
        !v_cache || !cow_src)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "k_cache and v_cache must be 16-byte aligned");
    unsigned int *err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    block_alloc_kernel<<<1, kAllocThreads, 0, stream>>>(
        block_tables, max_blocks_per_seq, context_lens, num_seqs, block_size, advance, free_blocks,
        free_count, refcounts, num_blocks, cow_src, err);
    pa_status st = cuda_check(cudaGetLastError(), "block alloc launch");
    if (st != PA_OK) return st;
    const int row_bytes = head_dim * (kv_dtype == PA_KV_BF16 ? 2 : 1);
    cow_copy_kernel<<<dim3(num_seqs, num_kv_heads), 128, 0, stream>>>(
        block_tables, max_blocks_per_seq, context_lens, nullptr, cow_src, block_size, num_kv_heads,
        row_bytes, static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache));
    return cuda_check(cudaGetLastError(), "copy-on-write launch");
}

extern "C" pa_status pa_block_alloc_chunk(int32_t *block_tables, int max_blocks_per_seq,
                                          const int32_t *context_lens, const int32_t *query_start,
                                          int num_seqs, int block_size, int32_t *free_blocks,
                                          int32_t *free_count, int32_t *refcounts, int num_blocks,
                                          void *k_cache, void *v_cache, int num_kv_heads, int head_dim,
                                          pa_kv_dtype kv_dtype, int32_t *cow_src, cudaStream_t stream) {
    clear_error();
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || block_size <= 0 || num_blocks <= 0 ||
        num_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad size (num_seqs=%d, max_blocks_per_seq=%d, "
                    "block_size=%d, num_blocks=%d, num_kv_heads=%d)", num_seqs,
                    max_blocks_per_seq, block_size, num_blocks, num_kv_heads);
    if (num_seqs > kMaxAllocSeqs)
        return fail(PA_ERR_UNSUPPORTED, "more than %d sequences", kMaxAllocSeqs);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (block_size != 16 && block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: 16, 32)", block_size);
    if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d", static_cast<int>(kv_dtype));
    if (num_seqs == 0) return PA_OK;
    if (!block_tables || !context_lens || !query_start || !free_blocks || !free_count || !refcounts ||
        !k_cache || !v_cache || !cow_src)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "k_cache and v_cache must be 16-byte aligned");
    unsigned int *err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    block_alloc_chunk_kernel<<<1, kAllocThreads, 0, stream>>>(
        block_tables, max_blocks_per_seq, context_lens, query_start, num_seqs, block_size, free_blocks,
        free_count, refcounts, num_blocks, cow_src, err);
    pa_status st = cuda_check(cudaGetLastError(), "block alloc (chunk) launch");
    if (st != PA_OK) return st;
    const int row_bytes = head_dim * (kv_dtype == PA_KV_BF16 ? 2 : 1);
    cow_copy_kernel<<<dim3(num_seqs, num_kv_heads), 128, 0, stream>>>(
        block_tables, max_blocks_per_seq, context_lens, query_start, cow_src, block_size, num_kv_heads,
        row_bytes, static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache));
    return cuda_check(cudaGetLastError(), "copy-on-write launch");
}
