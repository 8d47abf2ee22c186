// Slot mapping, cache append and partition merge kernels, plus the library's
// shared host bookkeeping (status strings, last-error message, device error
// word).
//
// Slot mapping and append follow "Optimizing Llama 3.1 405B Inference with
// vLLM PagedAttention", section "PagedAttention Mechanics" (a new token is
// appended into the sequence's last page) and, for the FP8 cache, Step 3 of
// "vLLM PagedAttention Optimization: Complete Step-by-Step Tuning Guide".
// The merge is the log-sum-exp combination of softmax partitions used to
// split long contexts.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "pa_device.cuh"

namespace pa {

static thread_local char g_msg[512];

pa_status fail(pa_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return st;
}

void clear_error() { g_msg[0] = '\0'; }

pa_status cuda_check(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return PA_OK;
    return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// One word per device, set by kernels that meet bad device-side data.
__device__ unsigned int g_device_error;

unsigned int *device_error_word() {
    // cudaGetSymbolAddress resolves for the current device; cache per device.
    static unsigned int *cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
    if (dev < 64 && cache[dev]) return cache[dev];
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    if (dev < 64) cache[dev] = static_cast<unsigned int *>(p);
    return static_cast<unsigned int *>(p);
}

// Wait limit of the kernels and the test hook that makes the decode
// kernel's first waits run out (pa_test_set_wait).
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
static std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};
static std::atomic<int> g_stall_first_wait{0};

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int stall_first_wait() { return g_stall_first_wait.load(std::memory_order_relaxed); }

// ---------------------------------------------------------------------------
// slot mapping
// ---------------------------------------------------------------------------

__global__ void slot_mapping_kernel(const int32_t *__restrict__ block_tables, int max_blocks,
                                    const int32_t *__restrict__ context_lens, int num_seqs,
                                    int block_size, int32_t *__restrict__ slot_mapping,
                                    unsigned int *err) {
    int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= num_seqs) return;
    int n = context_lens[s];
    if (n <= 0) {
        slot_mapping[s] = -1;
        return;
    }
    int pos = n - 1;
    if (pos / block_size >= max_blocks) {
        set_device_error(err, PA_DEVERR_BAD_CONTEXT);
        slot_mapping[s] = -1;
        return;
    }
    int32_t block = block_tables[static_cast<int64_t>(s) * max_blocks + pos / block_size];
    slot_mapping[s] = block * block_size + pos % block_size;
}

// ---------------------------------------------------------------------------
// append: one thread moves 8 consecutive elements of one (token, head) row
// ---------------------------------------------------------------------------

template <bool FP8>
__global__ void append_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                              const int32_t *__restrict__ slot_mapping, int num_tokens,
                              uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache,
                              int64_t num_slots, int num_kv_heads, int head_dim, int block_size,
                              float scale, const float *__restrict__ k_scales,
                              const float *__restrict__ v_scales, unsigned int *err) {
    const int vec_per_row = head_dim / 8;
    int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * vec_per_row;
    if (idx >= total) return;
    int vec = static_cast<int>(idx % vec_per_row);
    int64_t row = idx / vec_per_row;  // token * num_kv_heads + head
    int head = static_cast<int>(row % num_kv_heads);
    int token = static_cast<int>(row / num_kv_heads);
    int32_t slot = slot_mapping[token];
    if (slot < 0) return;
    if (slot >= num_slots) {
        if (head == 0 && vec == 0) set_device_error(err, PA_DEVERR_BAD_SLOT);
        return;
    }
    int64_t block = slot / block_size;
    int64_t off = slot % block_size;
    int64_t dst = ((block * num_kv_heads + head) * block_size + off) * head_dim + vec * 8;
    uint4 kv = k[idx];
    uint4 vv = v[idx];
    if constexpr (!FP8) {
        *reinterpret_cast<uint4 *>(k_cache + dst * 2) = kv;
        *reinterpret_cast<uint4 *>(v_cache + dst * 2) = vv;
    } else {
        // one scale for the whole cache, or one per KV head for K and for V
        const float ks = k_scales ? k_scales[head] : scale;
        const float vs = v_scales ? v_scales[head] : scale;
        *reinterpret_cast<uint2 *>(k_cache + dst) = quantize8_e4m3(kv, ks);
        *reinterpret_cast<uint2 *>(v_cache + dst) = quantize8_e4m3(vv, vs);
    }
}

// ---------------------------------------------------------------------------
// partition merge: WPR warps per (sequence, query head)
// ---------------------------------------------------------------------------

// Merge launch shape (build-time): warps per row and partitions in flight
// per warp, for rows of 17-64 partitions (MID) and of more (WIDE).
#ifndef PA_REDUCE_MID_WPR
#define PA_REDUCE_MID_WPR 4
#endif
#ifndef PA_REDUCE_MID_U
#define PA_REDUCE_MID_U 4
#endif
#ifndef PA_REDUCE_WIDE_WPR
#define PA_REDUCE_WIDE_WPR 8
#endif
#ifndef PA_REDUCE_WIDE_U
#define PA_REDUCE_WIDE_U 8
#endif

// threads of a merge CTA: at least 128, and at least one row's WPR warps
template <int WPR>
constexpr int reduce_threads() { return WPR * 32 > 128 ? WPR * 32 : 128; }

// Wait until the grid this one depends on (programmatic dependent launch)
// has finished and its writes are visible; a no-op otherwise.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Cache-global loads as ordered asm statements: a chunk's loads are all
// issued before any of their values is used, so they are in flight
// together (left to itself the compiler interleaves each load with its use).
template <int VEC>
__device__ __forceinline__ void load_vec(float (&x)[VEC], const float *src) {
    if constexpr (VEC == 4) {
        asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(x[0]), "=f"(x[1]), "=f"(x[2]), "=f"(x[3])
                     : "l"(src));
    } else {
        asm volatile("ld.global.cg.v2.f32 {%0,%1}, [%2];" : "=f"(x[0]), "=f"(x[1]) : "l"(src));
    }
}

__device__ __forceinline__ float load_cg(const float *src) {
    float x;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(x) : "l"(src));
    return x;
}

// One pass over the partitions.  Each warp covers all D dims of its row
// (VEC per lane); each of the WPR warps of a row takes a contiguous range of
// partitions, U at a time with every load of the chunk in flight together,
// and keeps a running (max, sum, accumulator) rescaled when the max grows.
// The row's warps then combine their triples through shared memory.
template <int D, int WPR, int U>
__global__ void __launch_bounds__(reduce_threads<WPR>())
    reduce_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                  const float *__restrict__ ws_l, const int32_t *__restrict__ context_lens,
                  int num_rows, int num_q_heads, int partition_size, int max_partitions,
                  __nv_bfloat16 *__restrict__ out) {
    constexpr int VEC = D / 32;
    constexpr int ROWS = reduce_threads<WPR>() / 32 / WPR;
    __shared__ float part_o[WPR > 1 ? ROWS * WPR : 1][WPR > 1 ? D : 1];
    __shared__ float part_ml[WPR > 1 ? ROWS * WPR : 1][2];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int sub = warp % WPR;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * ROWS + warp / WPR;
    const bool live = row < num_rows;
    // the context lengths are inputs of the step, not results of the
    // attention kernel: read them before waiting for that kernel
    int n = 0;
    if (live) {
        const int ctx = context_lens[row / num_q_heads];
        n = ctx > 0 ? (ctx + partition_size - 1) / partition_size : 0;
        if (n > max_partitions) n = max_partitions;
    }
    grid_dependency_wait();
    float acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
    float mx = -INFINITY, tot = 0.f;
    const float *m = ws_m + row * max_partitions;
    const float *l = ws_l + row * max_partitions;
    const float *o = ws_o + row * max_partitions * D + lane * VEC;
    // warp sub takes the contiguous partitions [p_begin, p_end): every chunk
    // reads U consecutive partition rows, one contiguous run of memory
    const int per = (n + WPR - 1) / WPR;
    const int p_begin = sub * per, p_end = min(n, p_begin + per);
    for (int p0 = p_begin; p0 < p_end; p0 += U) {
        float mv[U], lv[U], ov[U][VEC];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int p = p0 + u;
            if (p < p_end) {
                mv[u] = load_cg(m + p);
                lv[u] = load_cg(l + p);
                load_vec<VEC>(ov[u], o + static_cast<int64_t>(p) * D);
            } else {
                mv[u] = -INFINITY;
                lv[u] = 0.f;
#pragma unroll
                for (int j = 0; j < VEC; ++j) ov[u][j] = 0.f;
            }
        }
        float cmax = mx;
#pragma unroll
        for (int u = 0; u < U; ++u) cmax = fmaxf(cmax, mv[u]);
        // a partition that holds tokens has l > 0 and a finite max; one
        // that gave up on a wait has l = 0 and weighs nothing
        const float keep = mx > -INFINITY ? __expf(mx - cmax) : 0.f;
        tot *= keep;
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[j] *= keep;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const float w = lv[u] > 0.f ? lv[u] * __expf(mv[u] - cmax) : 0.f;
            tot += w;
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc[j] += w * ov[u][j];
        }
        mx = cmax;
    }
    if constexpr (WPR > 1) {
#pragma unroll
        for (int j = 0; j < VEC; ++j) part_o[warp][lane * VEC + j] = acc[j];
        if (lane == 0) {
            part_ml[warp][0] = mx;
            part_ml[warp][1] = tot;
        }
        __syncthreads();
        if (sub != 0) return;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < WPR; ++w) M = fmaxf(M, part_ml[warp + w][0]);
        tot = 0.f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
#pragma unroll
        for (int w = 0; w < WPR; ++w) {
            const float tw = part_ml[warp + w][1];
            const float f = tw > 0.f ? __expf(part_ml[warp + w][0] - M) : 0.f;
            tot += f * tw;
#pragma unroll
            for (int j = 0; j < VEC; ++j) acc[j] += f * part_o[warp + w][lane * VEC + j];
        }
    }
    if (!live) return;
    const float inv = tot > 0.f ? 1.f / tot : 0.f;
    __nv_bfloat16 *dst = out + row * D + lane * VEC;
    if constexpr (VEC == 4) {
        __nv_bfloat162 a = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
        __nv_bfloat162 b = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t *>(&a);
        v.y = *reinterpret_cast<uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(dst) = v;
    } else {
        *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    }
}

// Shared by pa_decode (split path), pa_decode_step and pa_decode_reduce;
// arguments checked by the caller.  Launched as a programmatic dependent of
// the kernel before it on the stream, so its launch overlaps that kernel's
// tail; the kernel itself waits for the predecessor's results.
pa_status launch_reduce(const void *workspace, const int32_t *context_lens, int num_seqs,
                        int num_q_heads, int head_dim, int partition_size, int max_partitions,
                        void *out, cudaStream_t stream) {
    const float *ws_o = static_cast<const float *>(workspace);
    const int64_t rows = static_cast<int64_t>(num_seqs) * num_q_heads;
    const float *ws_m = ws_o + rows * max_partitions * head_dim;
    const float *ws_l = ws_m + rows * max_partitions;
    // one warp per row while partitions are few; more, each with several
    // partitions in flight, when there are many
    constexpr int kMidW = PA_REDUCE_MID_WPR, kMidU = PA_REDUCE_MID_U;
    constexpr int kWideW = PA_REDUCE_WIDE_WPR, kWideU = PA_REDUCE_WIDE_U;
    const int wpr = max_partitions > 64 ? kWideW : max_partitions > 16 ? kMidW : 1;
    const int threads = max_partitions > 64   ? reduce_threads<kWideW>()
                        : max_partitions > 16 ? reduce_threads<kMidW>()
                                              : reduce_threads<1>();
    const int rows_per_cta = threads / 32 / wpr;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>((rows + rows_per_cta - 1) / rows_per_cta));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int nrows = static_cast<int>(rows);
    __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(out);
    auto launch = [&](auto kern) {
        return cudaLaunchKernelEx(&cfg, kern, ws_o, ws_m, ws_l, context_lens, nrows, num_q_heads,
                                  partition_size, max_partitions, o);
    };
    cudaError_t e;
    if (head_dim == 128)
        e = max_partitions > 64   ? launch(reduce_kernel<128, kWideW, kWideU>)
            : max_partitions > 16 ? launch(reduce_kernel<128, kMidW, kMidU>)
                                  : launch(reduce_kernel<128, 1, 8>);
    else
        e = max_partitions > 64   ? launch(reduce_kernel<64, kWideW, kWideU>)
            : max_partitions > 16 ? launch(reduce_kernel<64, kMidW, kMidU>)
                                  : launch(reduce_kernel<64, 1, 8>);
    return cuda_check(e, "reduce launch");
}

}  // namespace pa

using namespace pa;

extern "C" {

const char *pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported configuration";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

const char *pa_last_error(void) { return g_msg; }

pa_status pa_test_set_wait(uint64_t limit_ns, int stall_first_wait) {
    clear_error();
    if (limit_ns > 60ull * 1000000000ull)
        return fail(PA_ERR_INVALID_ARG, "wait limit %llu ns is above 60 s",
                    static_cast<unsigned long long>(limit_ns));
    g_wait_limit_ns.store(limit_ns ? limit_ns : kDefaultWaitNs, std::memory_order_relaxed);
    g_stall_first_wait.store(stall_first_wait ? 1 : 0, std::memory_order_relaxed);
    return PA_OK;
}

pa_status pa_device_errors(unsigned int *flags, int clear) {
    clear_error();
    if (!flags) return fail(PA_ERR_INVALID_ARG, "flags is NULL");
    unsigned int *word = device_error_word();
    if (!word) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    pa_status st = cuda_check(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    if (st != PA_OK) return st;
    st = cuda_check(cudaMemcpy(flags, word, sizeof(unsigned int), cudaMemcpyDeviceToHost),
                    "read device error word");
    if (st != PA_OK || !clear) return st;
    return cuda_check(cudaMemset(word, 0, sizeof(unsigned int)), "clear device error word");
}

pa_status pa_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int num_seqs, int block_size,
                          int32_t *slot_mapping, cudaStream_t stream) {
    clear_error();
    if (num_seqs < 0 || max_blocks_per_seq < 0 || block_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "negative size (num_seqs=%d, max_blocks_per_seq=%d, block_size=%d)",
                    num_seqs, max_blocks_per_seq, block_size);
    if (num_seqs == 0) return PA_OK;
    if (!block_tables || !context_lens || !slot_mapping)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (max_blocks_per_seq == 0) return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq is 0");
    unsigned int *err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    int threads = 128;
    slot_mapping_kernel<<<(num_seqs + threads - 1) / threads, threads, 0, stream>>>(
        block_tables, max_blocks_per_seq, context_lens, num_seqs, block_size, slot_mapping, err);
    return cuda_check(cudaGetLastError(), "slot mapping launch");
}

static pa_status append_impl(const void *k, const void *v, const int32_t *slot_mapping,
                             int num_tokens, void *k_cache, void *v_cache, int num_blocks,
                             int num_kv_heads, int head_dim, int block_size, pa_kv_dtype kv_dtype,
                             float scale, const float *k_scales, const float *v_scales,
                             cudaStream_t stream) {
    if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad size (num_tokens=%d, num_blocks=%d, num_kv_heads=%d)",
                    num_tokens, num_blocks, num_kv_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (block_size != 16 && block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: 16, 32)", block_size);
    if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d", static_cast<int>(kv_dtype));
    if (kv_dtype == PA_KV_FP8_E4M3 && !k_scales && !(scale > 0.f && scale <= 3.4e38f))
        return fail(PA_ERR_INVALID_ARG, "fp8 scale must be positive and finite");
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "k, v, k_cache and v_cache must be 16-byte aligned");
    unsigned int *err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot resolve the device error word");
    int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim / 8);
    int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 0x7fffffff) return fail(PA_ERR_INVALID_ARG, "too many tokens");
    int64_t num_slots = static_cast<int64_t>(num_blocks) * block_size;
    if (kv_dtype == PA_KV_BF16)
        append_kernel<false><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
            static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), num_slots,
            num_kv_heads, head_dim, block_size, scale, nullptr, nullptr, err);
    else
        append_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
            static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), num_slots,
            num_kv_heads, head_dim, block_size, scale, k_scales, v_scales, err);
    return cuda_check(cudaGetLastError(), "append launch");
}

pa_status pa_cache_append(const void *k, const void *v, const int32_t *slot_mapping,
                          int num_tokens, void *k_cache, void *v_cache, int num_blocks,
                          int num_kv_heads, int head_dim, int block_size,
                          pa_kv_dtype kv_dtype, float scale, cudaStream_t stream) {
    clear_error();
    return append_impl(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, num_kv_heads,
                       head_dim, block_size, kv_dtype, scale, nullptr, nullptr, stream);
}

pa_status pa_cache_append_scaled(const void *k, const void *v, const int32_t *slot_mapping,
                                 int num_tokens, void *k_cache, void *v_cache, int num_blocks,
                                 int num_kv_heads, int head_dim, int block_size,
                                 const float *k_scales, const float *v_scales,
                                 cudaStream_t stream) {
    clear_error();
    if (!k_scales || !v_scales) return fail(PA_ERR_INVALID_ARG, "null scale array");
    return append_impl(k, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks, num_kv_heads,
                       head_dim, block_size, PA_KV_FP8_E4M3, 1.f, k_scales, v_scales, stream);
}

}  // extern "C"
