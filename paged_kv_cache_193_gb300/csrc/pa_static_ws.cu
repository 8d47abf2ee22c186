// Split-context decode that needs no allocation from its caller.
//
// Some callers cannot allocate device memory when they want to run attention:
// a process whose device memory is owned by another framework's pool, a host
// that forbids allocation once it has started serving, or code on a path where
// the device-wide synchronisation that cudaMalloc/cudaFree may cause would stall
// other streams.  For them, pa_decode_static_workspace keeps the split path's
// scratch (per-partition outputs, maxima and sums) in a fixed array that lives
// in this library's device image, so the call itself allocates nothing.
//
// Costs of that choice, which the header repeats: every GPU on which the
// library's module is loaded holds PA_STATIC_WORKSPACE_BYTES of device memory
// until the process exits; all calls share the one array, so calls that may
// overlap on the GPU (different streams, or different host threads) race and
// must be serialised by the caller.
#include <mutex>

#include "pa_device.cuh"

namespace pa {

pa_status decode_split_into(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int num_blocks, int block_size,
                            pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                            int partition_size, void *scratch, size_t capacity, void *out,
                            cudaStream_t stream);

// The scratch itself.  In host code this name is only a host-side handle of
// the symbol, not a device address; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) float g_static_scratch[PA_STATIC_WORKSPACE_BYTES / sizeof(float)];

// The driver's cuCtxGetCurrent, taken from the runtime so the library needs
// no link against libcuda.
static CUresult current_context(CUcontext *ctx) {
    using Fn = CUresult (*)(CUcontext *);
    static Fn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<Fn>(p);
    });
    return fn ? fn(ctx) : CUDA_ERROR_NOT_FOUND;
}

// Device address of g_static_scratch in the current device's context,
// looked up on the first call in that context.  The context handle is kept
// beside the address: after cudaDeviceReset (or any other teardown of the
// primary context) the module is loaded again at a possibly different
// address, and the changed handle triggers a fresh lookup.
static pa_status static_scratch_address(void **addr) {
    constexpr int kMaxDevices = 64;
    struct Entry {
        CUcontext ctx;
        void *ptr;
    };
    static Entry cache[kMaxDevices];
    static std::mutex lock;
    int dev = -1;
    pa_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != PA_OK) return st;
    if (dev < 0 || dev >= kMaxDevices)
        return fail(PA_ERR_UNSUPPORTED, "device ordinal %d is beyond the %d this entry point tracks",
                    dev, kMaxDevices);
    // Before the runtime's first real call on this thread no context may be
    // current yet (null handle); the symbol lookup creates and binds the
    // device's primary context, after which the handle is read again.
    CUcontext ctx = nullptr;
    if (current_context(&ctx) != CUDA_SUCCESS)
        return fail(PA_ERR_CUDA, "cannot read the current CUDA context");
    std::lock_guard<std::mutex> guard(lock);
    if (!ctx || cache[dev].ctx != ctx || !cache[dev].ptr) {
        void *p = nullptr;
        st = cuda_check(cudaGetSymbolAddress(&p, g_static_scratch),
                        "cudaGetSymbolAddress(static scratch)");
        if (st != PA_OK) return st;
        if (current_context(&ctx) != CUDA_SUCCESS || !ctx)
            return fail(PA_ERR_CUDA, "cannot read the current CUDA context");
        cache[dev] = Entry{ctx, p};
    }
    *addr = cache[dev].ptr;
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_static_workspace(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_tables,
    int max_blocks_per_seq, const int32_t *context_lens, int num_seqs, int num_q_heads,
    int num_kv_heads, int head_dim, int num_blocks, int block_size, pa_kv_dtype kv_dtype,
    float kv_scale, float softmax_scale, int partition_size, void *out, cudaStream_t stream) {
    clear_error();
    void *scratch = nullptr;
    pa_status st = static_scratch_address(&scratch);
    if (st != PA_OK) return st;
    // Nothing in the scratch has to start at zero: the merge reads only the
    // partitions that the attention kernel of the same call has just written.
    return decode_split_into(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                             num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                             kv_dtype, kv_scale, softmax_scale, partition_size, scratch,
                             PA_STATIC_WORKSPACE_BYTES, out, stream);
}
