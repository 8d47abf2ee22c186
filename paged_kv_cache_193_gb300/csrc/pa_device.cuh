// Device-side building blocks for the paged-attention kernels (sm_103a):
// shared-memory mbarriers, TMA tile loads, warp-level tensor-core fragments,
// and the library's host-side bookkeeping (error messages, error word).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// ---------------------------------------------------------------------------
// host bookkeeping
// ---------------------------------------------------------------------------

// Record a formatted failure message for pa_last_error() and return `st`.
pa_status fail(pa_status st, const char *fmt, ...);
// Map a CUDA runtime error to PA_ERR_CUDA (recording the message) or PA_OK.
pa_status cuda_check(cudaError_t e, const char *what);
// Clear the thread's last-error message at the start of a call.
void clear_error();
// Device address of the library's error word on the current device.
unsigned int *device_error_word();
// Limit of a kernel's wait for a page copy (nanoseconds; 2 s unless a test
// set another), and whether the decode kernel's first waits are made to run
// out on purpose (test hook); both read when a kernel is launched.
uint64_t wait_limit_ns();
int stall_first_wait();
// Launch the partition merge (arguments already validated).
pa_status launch_reduce(const void *workspace, const int32_t *context_lens, int num_seqs,
                        int num_q_heads, int head_dim, int partition_size, int max_partitions,
                        void *out, cudaStream_t stream);

// Tensor map over a KV cache viewed as [num_blocks * num_kv_heads *
// block_size rows][head_dim]; one box is [block_size rows][min(row bytes,
// 128) bytes] with the hardware swizzle matching that width.
pa_status make_map(CUtensorMap *map, const void *cache, bool fp8, int head_dim, int64_t rows,
                   int block_size);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------------------
// device primitives (inline PTX)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's generic-proxy shared-memory accesses before later
// async-proxy (TMA) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's generic-proxy global writes before later async-proxy
// (TMA) reads of the same memory.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for phase `parity` of a barrier: spins on try_wait and gives
// up after `limit_ns` of wall time (checked every 1024 tries).  Returns false
// on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    uint64_t t0 = 0;
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 1023u) == 0) {
            uint64_t now = global_timer_ns();
            if (t0 == 0)
                t0 = now;
            else if (now - t0 > limit_ns)
                return false;
        }
    }
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// L2 policy for data read exactly once per step (the KV pages).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// Two 16 x 16 matrices of bytes, transposed: lanes 0-15 give the addresses
// of matrix 0's sixteen 16-byte rows, lanes 16-31 those of matrix 1.  Lane
// (g = lane / 4, c = lane % 4) receives in r0 bytes (rows 4c..4c+3, column
// g) of matrix 0, in r1 the same rows at column g + 8, and in r2, r3 the
// same of matrix 1 (lowest row in the lowest byte).
__device__ __forceinline__ void ldsm_x2_trans_b8(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                                 uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m16n16.x2.trans.shared.b8 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(addr), "r"(0u) : "memory");
}

// Transpose of an 8x8 b16 matrix held in the standard fragment layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// D += A * B, m16n8k16, fp32 accumulate, bf16 or fp16 operands.
template <bool F16>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (F16) {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// D += A * B, m16n8k32, both operands E4M3 (four per register, lowest k in
// the lowest byte), fp32 accumulate.
__device__ __forceinline__ void mma16832_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four E4M3 bytes b0..b3 of a word (b0 lowest) -> two fp16x2 registers:
// lo = {b0, b1}, hi = {b2, b3}, low half first.  Exact (every E4M3 value is
// an fp16 value).  The conversion reads the two 16-bit halves of the word
// directly, so no masking or shifting is needed.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (F16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    } else {
        __nv_bfloat162 b = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&b);
    }
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void set_device_error(unsigned int *err, unsigned int bits) {
    if (err) atomicOr(err, bits);
}

// Eight bf16 values -> eight E4M3 codes of x / scale: IEEE fp32 division,
// round to nearest even, saturating to +-448 (the append's FP8 encoding).
__device__ __forceinline__ uint2 quantize8_e4m3(const uint4 &bf16x8, float scale) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&bf16x8);
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
    return make_uint2(words[0], words[1]);
}

}  // namespace pa
