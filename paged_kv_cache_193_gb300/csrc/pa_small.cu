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
                              float scale, unsigned int *err) {
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
        const uint4 *src[2] = {&kv, &vv};
        uint8_t *cache[2] = {k_cache, v_cache};
#pragma unroll
        for (int which = 0; which < 2; ++which) {
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(src[which]);
            uint32_t words[2];
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                uint32_t packed = 0;
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    float2 f = __bfloat1622float2(h[w * 2 + j]);
                    float2 q = make_float2(__fdiv_rn(f.x, scale), __fdiv_rn(f.y, scale));
                    __nv_fp8x2_storage_t two = __nv_cvt_float2_to_fp8x2(q, __NV_SATFINITE, __NV_E4M3);
                    packed |= static_cast<uint32_t>(two) << (16 * j);
                }
                words[w] = packed;
            }
            *reinterpret_cast<uint2 *>(cache[which] + dst) = make_uint2(words[0], words[1]);
        }
    }
}

// ---------------------------------------------------------------------------
// partition merge: one CTA of 128 threads per (sequence, query head)
// ---------------------------------------------------------------------------

constexpr int kReduceThreads = 128;

template <int D>
__global__ void __launch_bounds__(kReduceThreads)
    reduce_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                  const float *__restrict__ ws_l, const int32_t *__restrict__ context_lens,
                  int num_q_heads, int partition_size, int max_partitions,
                  __nv_bfloat16 *__restrict__ out) {
    constexpr int VEC = D / 32;  // floats per lane across one warp
    constexpr int NWARP = kReduceThreads / 32;
    extern __shared__ float w_s[];  // [max_partitions] weights
    __shared__ float red[NWARP];
    __shared__ float acc_s[NWARP][D];

    const int hq = blockIdx.x, s = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = static_cast<int64_t>(s) * num_q_heads + hq;
    __nv_bfloat16 *dst = out + row * D;
    int n = context_lens[s];
    n = n > 0 ? (n + partition_size - 1) / partition_size : 0;
    if (n > max_partitions) n = max_partitions;
    if (n == 0) {
        for (int d = tid; d < D; d += kReduceThreads) dst[d] = __float2bfloat16_rn(0.f);
        return;
    }
    const float *m = ws_m + row * max_partitions;
    const float *l = ws_l + row * max_partitions;

    // M = max_p m_p
    float mx = -INFINITY;
    for (int p = tid; p < n; p += kReduceThreads) mx = fmaxf(mx, m[p]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int w = 1; w < NWARP; ++w) mx = fmaxf(mx, red[w]);
    __syncthreads();

    // w_p = l_p exp(m_p - M), W = sum_p w_p
    float sum = 0.f;
    for (int p = tid; p < n; p += kReduceThreads) {
        float w = l[p] * __expf(m[p] - mx);
        w_s[p] = w;
        sum += w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) red[warp] = sum;
    __syncthreads();
    float total = 0.f;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) total += red[w];

    // out = sum_p w_p o_p / W; warp w takes partitions p = w, w + 4, ...
    float acc[VEC];
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[j] = 0.f;
    const float *o = ws_o + row * max_partitions * D + lane * VEC;
    for (int p = warp; p < n; p += NWARP) {
        float w = w_s[p];
        const float *src = o + static_cast<int64_t>(p) * D;
        if constexpr (VEC == 4) {
            float4 x = *reinterpret_cast<const float4 *>(src);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
            acc[2] += w * x.z;
            acc[3] += w * x.w;
        } else {
            float2 x = *reinterpret_cast<const float2 *>(src);
            acc[0] += w * x.x;
            acc[1] += w * x.y;
        }
    }
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc_s[warp][lane * VEC + j] = acc[j];
    __syncthreads();
    float inv = 1.f / total;
    for (int d = tid; d < D; d += kReduceThreads) {
        float a = 0.f;
#pragma unroll
        for (int w = 0; w < NWARP; ++w) a += acc_s[w][d];
        dst[d] = __float2bfloat16_rn(a * inv);
    }
}

// Shared by pa_decode (split path) and pa_decode_reduce; arguments checked
// by the caller.
pa_status launch_reduce(const void *workspace, const int32_t *context_lens, int num_seqs,
                        int num_q_heads, int head_dim, int partition_size, int max_partitions,
                        void *out, cudaStream_t stream) {
    const float *ws_o = static_cast<const float *>(workspace);
    const int64_t rows = static_cast<int64_t>(num_seqs) * num_q_heads;
    const float *ws_m = ws_o + rows * max_partitions * head_dim;
    const float *ws_l = ws_m + rows * max_partitions;
    dim3 grid(num_q_heads, num_seqs);
    size_t smem = static_cast<size_t>(max_partitions) * sizeof(float);
    if (head_dim == 128) {
        if (smem > 48 * 1024) {
            pa_status st = cuda_check(cudaFuncSetAttribute(reduce_kernel<128>,
                                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           static_cast<int>(smem)),
                                      "cudaFuncSetAttribute(reduce)");
            if (st != PA_OK) return st;
        }
        reduce_kernel<128><<<grid, kReduceThreads, smem, stream>>>(
            ws_o, ws_m, ws_l, context_lens, num_q_heads, partition_size, max_partitions,
            static_cast<__nv_bfloat16 *>(out));
    } else {
        if (smem > 48 * 1024) {
            pa_status st = cuda_check(cudaFuncSetAttribute(reduce_kernel<64>,
                                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           static_cast<int>(smem)),
                                      "cudaFuncSetAttribute(reduce)");
            if (st != PA_OK) return st;
        }
        reduce_kernel<64><<<grid, kReduceThreads, smem, stream>>>(
            ws_o, ws_m, ws_l, context_lens, num_q_heads, partition_size, max_partitions,
            static_cast<__nv_bfloat16 *>(out));
    }
    return cuda_check(cudaGetLastError(), "reduce launch");
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

pa_status pa_cache_append(const void *k, const void *v, const int32_t *slot_mapping,
                          int num_tokens, void *k_cache, void *v_cache, int num_blocks,
                          int num_kv_heads, int head_dim, int block_size,
                          pa_kv_dtype kv_dtype, float scale, cudaStream_t stream) {
    clear_error();
    if (num_tokens < 0 || num_blocks < 0 || num_kv_heads <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad size (num_tokens=%d, num_blocks=%d, num_kv_heads=%d)",
                    num_tokens, num_blocks, num_kv_heads);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (block_size != 16 && block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: 16, 32)", block_size);
    if (kv_dtype != PA_KV_BF16 && kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d", static_cast<int>(kv_dtype));
    if (kv_dtype == PA_KV_FP8_E4M3 && !(scale > 0.f && scale <= 3.4e38f))
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
            num_kv_heads, head_dim, block_size, scale, err);
    else
        append_kernel<true><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            static_cast<const uint4 *>(k), static_cast<const uint4 *>(v), slot_mapping, num_tokens,
            static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), num_slots,
            num_kv_heads, head_dim, block_size, scale, err);
    return cuda_check(cudaGetLastError(), "append launch");
}

}  // extern "C"
