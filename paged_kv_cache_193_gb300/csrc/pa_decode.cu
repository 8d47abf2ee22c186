// Paged decode attention for sm_103a.
//
// What it computes: for each sequence s and query head hq, softmax over the
// sequence's cached tokens of softmax_scale * q . K[t], applied to V, where
// K/V rows are found by walking the sequence's block table ("vLLM
// PagedAttention: Memory Optimization & High-Throughput LLM Inference
// Tuning", section 2) and hq reads KV head hq / group (grouped-query
// attention, "Optimizing vLLM Throughput with PagedAttention and Continuous
// Batching for Llama 3").  Long contexts are cut into partitions whose
// results are merged by log-sum-exp (reduce kernel in pa_small.cu).
//
// How (one CTA per (partition, KV head, sequence), NW warps):
//  * Each warp owns the partition's pages j = warp, warp + NW, ... and keeps
//    SPW of them in flight: lane 0 issues 2-D TMA tile loads of the K and V
//    page of this KV head (one [block_size x 128 B] box per 128-byte column
//    slab, hardware 128B/64B swizzle, L2 evict-first) completing on the
//    stage's mbarrier; when the warp has used a stage it refills it with its
//    page SPW further on.  Block-table entries are read 32 at a time by the
//    warp's lanes, one chunk ahead of use.
//  * The whole GQA group reuses each page: S^T = K Q^T is one m16n8k16
//    tensor-core product per 16 tokens x 16 head dims with the group (padded
//    to 8 or 16) as N, then a warp-shuffle online softmax over the tokens,
//    and O^T += V^T P^T with the head dim as M.  bf16 pages feed ldmatrix
//    directly (the swizzle makes it conflict-free); E4M3 pages are read with
//    plain shared loads and widened to fp16 in registers, with the head-dim
//    order permuted consistently on Q and K (and on the output) so every
//    thread reads whole 16-byte or 4-byte words.
//  * The warps' (max, sum, accumulator) triples are merged through shared
//    memory; the CTA writes bf16 output (unsplit) or the fp32 partition
//    result (o, m, l) to the workspace.
#include <cudaTypedefs.h>
#include <math.h>

#include <atomic>

#include "pa_device.cuh"

namespace pa {

struct DecodeArgs {
    const __nv_bfloat16 *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    int max_blocks;      // table row length
    int num_blocks;      // pool size
    int num_q_heads;
    int num_kv_heads;
    int group;           // query heads per KV head
    int partition_size;  // tokens per partition (the whole table when unsplit)
    int max_partitions;  // workspace stride
    float score_scale;   // softmax_scale * kscale * log2(e): scores in base-2 units
    float v_scale;       // vscale
    int split;           // 1: write (o, m, l) to the workspace; 0: write bf16 out
    __nv_bfloat16 *out;
    float *ws_o;
    float *ws_m;
    float *ws_l;
    unsigned int *err;
    // fused append (pa_decode_step): the CTA whose partition holds a
    // sequence's newest token first writes that token's K/V row of its KV
    // head into the cache; null k_new = no append
    const uint4 *k_new;  // bf16 [num_seqs][num_kv_heads][head_dim]
    const uint4 *v_new;
    uint8_t *k_cache_w;
    uint8_t *v_cache_w;
    int32_t *slot_out;   // optional: slot of each sequence's newest token
    float append_scale;  // E4M3 scale of the append (cache dtype FP8)
    // optional per-KV-head E4M3 scales (override the single scale above)
    const float *k_scales;
    const float *v_scales;
    float softmax_log2;  // softmax_scale * log2(e)
    float q_scale;       // E4M3 query scale of the E4M3 x E4M3 score product
    uint64_t wait_limit_ns;  // give up on a page copy after this long
    int stall_first_wait;    // test hook: each warp's first wait is on a barrier nothing completes
};

// Drain limit after a wait gave up: the copies still in flight into a
// warp's stages are always waited for with this (normal waits are
// microseconds), so no CTA leaves with a copy landing in its shared memory.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr float kLn2 = 0.693147180559945309f;

template <int D, int BS, bool FP8, int NT, int NW, int SPW>
struct Cfg {
    static constexpr int ELEM = FP8 ? 1 : 2;
    static constexpr int ROWB = D * ELEM;                     // bytes of one token row of one head
    static constexpr int SLAB = ROWB >= 128 ? 128 : ROWB;     // TMA box width in bytes = swizzle span
    static constexpr int NSLAB = ROWB / SLAB;
    static constexpr int PAGE = BS * ROWB;                    // one K (or V) page of one head
    // pages per iteration of a warp: two 16-token E4M3 pages (32 tokens per
    // pass amortise the per-pass work over twice the bytes), else one
    static constexpr int PPI = (FP8 && BS == 16) ? 2 : 1;
    static constexpr int STAGE = 2 * PPI * PAGE;              // PPI K pages, then PPI V pages
    static constexpr int NSTAGE = NW * SPW;
    static constexpr int RING = NSTAGE * STAGE;
    static constexpr int NP = 8 * NT;                         // group rows padded to the MMA N
    static constexpr int OSTR = D + 4;                        // epilogue row stride (floats)
    static constexpr int EPI = (NW * NP * OSTR + 4 * NW * NP + 2 * NP) * 4;
    static constexpr int SMEM = (RING > EPI ? RING : EPI) + 1024;  // + 1 KB for base alignment
    static constexpr int MT = BS / 16;                        // 16-token m-tiles per page
    static constexpr int MI = PPI * MT;                       // m-tiles per iteration
    static constexpr int KSTEPS = D / 16;
    static constexpr int DT = D / 16;                         // 16-dim tiles of the output
    static constexpr int CPT = D / 64;                        // fp8: 16-byte chunks per thread and row
    static_assert(SLAB == 128 || SLAB == 64, "swizzle span");
    static_assert((BS * SLAB) % 1024 == 0 || SLAB == 64, "slab alignment");
};

// Shared-memory address of byte `b` of token row `t` in a page tile laid
// down by the TMA with the swizzle that matches the slab width: 16-byte
// chunk c of a 128-byte row lands at c ^ (t & 7); of a 64-byte row at
// c ^ ((t >> 1) & 3).
template <class C, int BS>
__device__ __forceinline__ uint32_t swz(uint32_t base, int t, int b) {
    const int slab = b / C::SLAB;
    const int within = b % C::SLAB;
    const int chunk = within >> 4;
    const int phys = C::SLAB == 128 ? (chunk ^ (t & 7)) : (chunk ^ ((t >> 1) & 3));
    return base + slab * (BS * C::SLAB) + t * C::SLAB + (phys << 4) + (within & 15);
}

// FQ (E4M3 cache only): the query is rounded to E4M3 (x / q_scale) and the
// scores are an E4M3 x E4M3 tensor-core product over the cache bytes as
// they lie in shared memory.
// Groups above 8 with a bf16 cache of 16-token pages are held to three CTAs
// per SM (at most 168 registers, a 64 KB ring): their CTAs are short when the
// context is split, and a third CTA per SM hides more of each one's start.
template <int D, int BS, bool FP8, int NT, int NW, int SPW, bool FQ = false>
__global__ void __launch_bounds__(NW * 32, (NT == 2 && BS == 16 && !FP8) ? 3 : (NW >= 8 ? 1 : 8 / NW))
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeArgs a) {
    static_assert(!FQ || FP8, "the E4M3 score product needs the E4M3 cache");
    using C = Cfg<D, BS, FP8, NT, NW, SPW>;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t bars[C::NSTAGE];
    __shared__ __align__(8) uint64_t stall_bar;  // never completed (wait-limit test hook)

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t ring = (raw + 1023u) & ~1023u;
    float *epi = reinterpret_cast<float *>(smem_raw + (ring - raw));

    const int part = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r = lane >> 2, c = lane & 3;

    // scales of this KV head: one for the whole cache, or K and V per head
    float score_scale = a.score_scale, v_scale = a.v_scale;
    float append_k_scale = a.append_scale, append_v_scale = a.append_scale;
    if (a.k_scales) {
        append_k_scale = __ldg(a.k_scales + h);
        append_v_scale = __ldg(a.v_scales + h);
        score_scale = a.softmax_log2 * append_k_scale;
        v_scale = append_v_scale;
    }
    if constexpr (FQ) score_scale *= a.q_scale;

    // let a dependent merge kernel launch now; it waits for our results
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // Block-table entries and the query do not depend on the context length:
    // load them first so their latency overlaps the context-length load.
    const int t_begin = part * a.partition_size;
    const int page0 = t_begin / BS;
    const int lim = min(a.max_blocks - page0, a.partition_size / BS) - warp;  // table entries left
    const int32_t *bt = a.block_tables + static_cast<int64_t>(s) * a.max_blocks + page0 + warp;
    int ent_cur = lane * NW < lim ? __ldg(bt + lane * NW) : -1;
    int ent_next = (32 + lane) * NW < lim ? __ldg(bt + (32 + lane) * NW) : -1;

    // query fragments (B operand of S^T = K Q^T), resident in registers
    uint32_t qf[C::KSTEPS][NT][2];
    {
        const __nv_bfloat16 *qh = a.q + (static_cast<int64_t>(s) * a.num_q_heads + h * a.group) * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int g = nt * 8 + r;
            const bool live = g < a.group;
            const __nv_bfloat16 *qg = qh + g * D;
#pragma unroll
            for (int kk = 0; kk < C::KSTEPS; ++kk) {
                if constexpr (!FP8) {
                    // logical k = 2c, 2c+1 and 2c+8, 2c+9 of this 16-dim step
                    qf[kk][nt][0] = live ? __ldg(reinterpret_cast<const uint32_t *>(qg + kk * 16 + 2 * c)) : 0u;
                    qf[kk][nt][1] = live ? __ldg(reinterpret_cast<const uint32_t *>(qg + kk * 16 + 8 + 2 * c)) : 0u;
                } else if constexpr (!FQ) {
                    // permuted order: this thread's dims are c*16*CPT + 4*kk + {0,1,2,3}
                    uint2 w = live ? __ldg(reinterpret_cast<const uint2 *>(qg + c * 16 * C::CPT + 4 * kk))
                                   : make_uint2(0u, 0u);
                    float2 f0 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w.x));
                    float2 f1 = __bfloat1622float2(*reinterpret_cast<__nv_bfloat162 *>(&w.y));
                    qf[kk][nt][0] = pack2<true>(f0.x, f0.y);
                    qf[kk][nt][1] = pack2<true>(f1.x, f1.y);
                } else if (kk < C::KSTEPS / 2) {
                    // E4M3 codes; permuted order: 32-dim step kk takes this
                    // thread's dims c*16*CPT + 8*kk + {0..3} (logical k = 4c + i)
                    // and + {4..7} (logical k = 16 + 4c + i), as the K bytes below
                    const uint4 w = live ? __ldg(reinterpret_cast<const uint4 *>(qg + c * 16 * C::CPT + 8 * kk))
                                         : make_uint4(0u, 0u, 0u, 0u);
                    const uint2 q8 = quantize8_e4m3(w, a.q_scale);
                    qf[kk][nt][0] = q8.x;
                    qf[kk][nt][1] = q8.y;
                }
            }
        }
    }

    const int n_raw = a.context_lens[s];
    int n = n_raw;
    const int cap = a.max_blocks * BS;
    if (n > cap) {
        if (tid == 0 && part == 0 && h == 0) set_device_error(a.err, PA_DEVERR_BAD_CONTEXT);
        n = cap;
    }
    if (n < 0) n = 0;
    if (a.k_new && a.slot_out && n == 0 && part == 0 && h == 0 && tid == 0) a.slot_out[s] = -1;
    if (a.split && t_begin >= n) return;  // past this sequence's end: nothing to write
    const int t_end = min(t_begin + a.partition_size, n);
    const int npages = t_end > t_begin ? (t_end - t_begin + BS - 1) / BS : 0;

    if (a.k_new && n > 0 && n_raw <= cap && n - 1 >= t_begin && n - 1 < t_end) {
        // Append the newest token of sequence s (position n - 1, which this
        // partition holds) for KV head h, before any page copy is issued.
        const int pos = n - 1;
        const int32_t blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + pos / BS];
        if (blk >= 0 && blk < a.num_blocks) {
            if (tid < D / 8) {
                const int64_t src = (static_cast<int64_t>(s) * a.num_kv_heads + h) * (D / 8) + tid;
                const int64_t dst =
                    ((static_cast<int64_t>(blk) * a.num_kv_heads + h) * BS + pos % BS) * D + tid * 8;
                const uint4 kv = a.k_new[src], vv = a.v_new[src];
                if constexpr (!FP8) {
                    *reinterpret_cast<uint4 *>(a.k_cache_w + dst * 2) = kv;
                    *reinterpret_cast<uint4 *>(a.v_cache_w + dst * 2) = vv;
                } else {
                    *reinterpret_cast<uint2 *>(a.k_cache_w + dst) = quantize8_e4m3(kv, append_k_scale);
                    *reinterpret_cast<uint2 *>(a.v_cache_w + dst) = quantize8_e4m3(vv, append_v_scale);
                }
                // the row is read back below by this CTA's TMA (async proxy)
                fence_proxy_async_global();
            }
            if (h == 0 && tid == 0 && a.slot_out) a.slot_out[s] = blk * BS + pos % BS;
        } else {
            if (tid == 0) set_device_error(a.err, PA_DEVERR_BAD_BLOCK);
            if (h == 0 && tid == 0 && a.slot_out) a.slot_out[s] = -1;
        }
    } else if (a.k_new && a.slot_out && n_raw > cap && part == 0 && h == 0 && tid == 0) {
        a.slot_out[s] = -1;
    }

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < C::NSTAGE; ++i) mbar_init(smem_addr(&bars[i]), 1);
        mbar_init(smem_addr(&stall_bar), 1);
        fence_barrier_init();
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    __syncthreads();

    // ---- this warp's pages ----------------------------------------------------
    // The warp owns pages warp, warp + NW, ...; iteration i takes its pages
    // PPI*i .. PPI*i + PPI - 1 (MI m-tiles of 16 tokens) from one stage.
    constexpr int PPI = C::PPI, MI = C::MI;
    const int my_pages = npages > warp ? (npages - warp + NW - 1) / NW : 0;
    const int my_iters = (my_pages + PPI - 1) / PPI;
    int chunk_cur = 0;
    const uint64_t policy = l2_evict_first_policy();
    const int rows_total = a.num_blocks * a.num_kv_heads * BS;

    // Entry of the warp's k-th page; called by all lanes with k = 0, 1, 2, ...
    auto entry = [&](int k) -> int {
        const int ck = k >> 5;
        if (ck != chunk_cur) {
            ent_cur = ent_next;
            chunk_cur = ck;
            const int kk = (ck + 1) * 32 + lane;
            ent_next = kk < my_pages ? __ldg(bt + kk * NW) : -1;
        }
        return __shfl_sync(0xffffffffu, ent_cur, k & 31);
    };
    // All lanes: the physical blocks of iteration it's pages; lanes 0 ..
    // PPI-1 start their copies (pages past the warp's last are not copied:
    // their rows are masked and their V rows zeroed before use).
    auto fetch = [&](int it) {
        int blk[PPI];
#pragma unroll
        for (int p = 0; p < PPI; ++p) blk[p] = entry(PPI * it + p);
        const int live = min(PPI, my_pages - PPI * it);
        if (lane >= live) return;
        const int st = warp * SPW + it % SPW;
        const uint32_t bar = smem_addr(&bars[st]);
        // lane 0 arms the barrier for every live page; lane p copies page p
        if (lane == 0) mbar_arrive_expect_tx(bar, live * 2 * C::PAGE);
        const uint32_t kdst = ring + st * C::STAGE + lane * C::PAGE;
        const uint32_t vdst = kdst + PPI * C::PAGE;
        int b = blk[0];
#pragma unroll
        for (int p = 1; p < PPI; ++p)
            if (lane == p) b = blk[p];
        int y;
        if (b < 0 || b >= a.num_blocks) {
            set_device_error(a.err, PA_DEVERR_BAD_BLOCK);
            y = rows_total;  // wholly outside the tensor: the TMA fills zeros
        } else {
            y = (b * a.num_kv_heads + h) * BS;
        }
#pragma unroll
        for (int sl = 0; sl < C::NSLAB; ++sl) {
            tma_load_2d(kdst + sl * (BS * C::SLAB), &tmK, sl * (C::SLAB / C::ELEM), y, bar, policy);
            tma_load_2d(vdst + sl * (BS * C::SLAB), &tmV, sl * (C::SLAB / C::ELEM), y, bar, policy);
        }
    };

    const int prolog = my_iters < SPW ? my_iters : SPW;
    for (int it = 0; it < prolog; ++it) fetch(it);

    float o[C::DT][NT][4];
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[dt][nt][e] = 0.f;
    // Per group column: m_ref is the reference the probabilities are taken
    // against (it moves only when a tile's maximum exceeds it by more than
    // kLazy in base-2 units, so probabilities stay below 2^kLazy and the
    // accumulator is rescaled rarely), m_max the true running maximum, l
    // the sum of probabilities relative to m_ref.
    constexpr float kLazy = 8.f;
    float m_ref[NT][2], m_max[NT][2], l_run[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            m_ref[nt][j] = m_max[nt][j] = -INFINITY;
            l_run[nt][j] = 0.f;
        }

    // Token (within its 16-token m-tile) of MMA row r and of row r + 8.  The
    // E4M3 path reads V with a transposing byte-matrix load whose fragment
    // pairs rows 4c, 4c+1 and 4c+2, 4c+3; the sum over tokens is
    // order-free, so the scores take the matching order: MMA row 2c + e + 8h
    // holds token 4c + 2h + e.
    const int tok_r = FP8 ? (r >> 1) * 4 + (r & 1) : r;
    const int tok_dh = FP8 ? 2 : 8;

    // ---- main loop over this warp's pages ---------------------------------
    bool ok = true;
    int it_fail = 0;
    // Test hook: give up on a barrier that no copy completes, exactly as if
    // the first page never arrived (the copies already issued still land
    // and are drained below).
    if (a.stall_first_wait && my_iters > 0)
        ok = mbar_wait_bounded(smem_addr(&stall_bar), 0, a.wait_limit_ns);
    for (int it = 0; ok && it < my_iters; ++it) {
        const int st = warp * SPW + it % SPW;
        if (!mbar_wait_bounded(smem_addr(&bars[st]), (it / SPW) & 1, a.wait_limit_ns)) {
            ok = false;
            it_fail = it;
            break;
        }
        const uint32_t kbase = ring + st * C::STAGE;
        const uint32_t vbase = kbase + PPI * C::PAGE;
        int valid[PPI];
#pragma unroll
        for (int p = 0; p < PPI; ++p) {
            const int k = PPI * it + p;
            const int tok0 = (page0 + warp + k * NW) * BS;
            valid[p] = k < my_pages ? min(BS, t_end - tok0) : 0;
        }

        if (valid[PPI - 1] < BS) {
            // Rows past the context hold whatever the stage held (never read
            // as tokens): zero the V rows so 0-probability x garbage is 0.
            constexpr int CH = C::NSLAB * (C::SLAB / 16);
#pragma unroll
            for (int p = 0; p < PPI; ++p) {
                const uint32_t vb = vbase + p * C::PAGE;
                for (int i = lane; i < (BS - valid[p]) * CH; i += 32) {
                    const int row = valid[p] + i / CH;
                    const int rem = i % CH;
                    sts128_zero(vb + (rem / (C::SLAB / 16)) * (BS * C::SLAB) + row * C::SLAB +
                                (rem % (C::SLAB / 16)) * 16);
                }
            }
            // these generic-proxy stores precede the stage's next TMA write
            fence_proxy_async_smem();
            __syncwarp();
        }

        // S^T[t][g] for the iteration's tokens; m-tile mi is m-tile mi % MT
        // of page mi / MT
        float sc[MI][NT][4];
#pragma unroll
        for (int mi = 0; mi < MI; ++mi)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[mi][nt][e] = 0.f;

        if constexpr (!FP8) {
#pragma unroll
            for (int mi = 0; mi < MI; ++mi) {
                const uint32_t kb = kbase + (mi / C::MT) * C::PAGE;
                const int t = (mi % C::MT) * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4(swz<C, BS>(kb, t, (kk * 16 + (lane >> 4) * 8) * 2), a0, a1, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816<false>(sc[mi][nt], a0, a1, a2, a3, qf[kk][nt][0], qf[kk][nt][1]);
                }
            }
        } else if constexpr (FQ) {
            // E4M3 x E4M3: this thread's 8 bytes of a row per 32-dim step are
            // A fragment words as they lie in shared memory
#pragma unroll
            for (int mi = 0; mi < MI; ++mi) {
                const uint32_t kb = kbase + (mi / C::MT) * C::PAGE;
                const int t0 = (mi % C::MT) * 16 + tok_r, t1 = t0 + tok_dh;
                uint4 ra[C::CPT], rb[C::CPT];
#pragma unroll
                for (int j = 0; j < C::CPT; ++j) {
                    ra[j] = lds128(swz<C, BS>(kb, t0, (c * C::CPT + j) * 16));
                    rb[j] = lds128(swz<C, BS>(kb, t1, (c * C::CPT + j) * 16));
                }
                auto word = [](const uint4 &u, int i) { return i == 0 ? u.x : i == 1 ? u.y : i == 2 ? u.z : u.w; };
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS / 2; ++kk) {
                    const int w = 2 * kk;
                    const uint32_t a0 = word(ra[w / 4], w % 4), a2 = word(ra[w / 4], w % 4 + 1);
                    const uint32_t a1 = word(rb[w / 4], w % 4), a3 = word(rb[w / 4], w % 4 + 1);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16832_e4m3(sc[mi][nt], a0, a1, a2, a3, qf[kk][nt][0], qf[kk][nt][1]);
                }
            }
        } else {
#pragma unroll
            for (int mi = 0; mi < MI; ++mi) {
                const uint32_t kb = kbase + (mi / C::MT) * C::PAGE;
                const int t0 = (mi % C::MT) * 16 + tok_r, t1 = t0 + tok_dh;
                uint4 ra[C::CPT], rb[C::CPT];
#pragma unroll
                for (int j = 0; j < C::CPT; ++j) {
                    ra[j] = lds128(swz<C, BS>(kb, t0, (c * C::CPT + j) * 16));
                    rb[j] = lds128(swz<C, BS>(kb, t1, (c * C::CPT + j) * 16));
                }
#pragma unroll
                for (int kk = 0; kk < C::KSTEPS; ++kk) {
                    const uint4 &A = ra[kk / 4];
                    const uint4 &B = rb[kk / 4];
                    const uint32_t wa = (kk % 4 == 0) ? A.x : (kk % 4 == 1) ? A.y : (kk % 4 == 2) ? A.z : A.w;
                    const uint32_t wb = (kk % 4 == 0) ? B.x : (kk % 4 == 1) ? B.y : (kk % 4 == 2) ? B.z : B.w;
                    uint32_t a0, a1, a2, a3;
                    e4m3x4_to_f16x2x2(wa, a0, a2);  // row t0: k = 2c,2c+1 | 2c+8,2c+9
                    e4m3x4_to_f16x2x2(wb, a1, a3);  // row t1
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816<true>(sc[mi][nt], a0, a1, a2, a3, qf[kk][nt][0], qf[kk][nt][1]);
                }
            }
        }

        // online softmax over the iteration's tokens, per group column
        float mx[NT][2];
        bool grow = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float m = -INFINITY;
#pragma unroll
                for (int mi = 0; mi < MI; ++mi) {
                    const int lim = valid[mi / C::MT] - (mi % C::MT) * 16;
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        float x = sc[mi][nt][hi * 2 + j] * score_scale;
                        x = tok_r + hi * tok_dh < lim ? x : -INFINITY;
                        sc[mi][nt][hi * 2 + j] = x;
                        m = fmaxf(m, x);
                    }
                }
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
                m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
                mx[nt][j] = m;
                m_max[nt][j] = fmaxf(m_max[nt][j], m);
                grow |= m > m_ref[nt][j] + kLazy;
            }
        }
        if (__any_sync(0xffffffffu, grow)) {
            // move the reference to the running maximum and rescale
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const float m_new = fmaxf(m_ref[nt][j], mx[nt][j]);
                    const float alpha = fast_exp2(m_ref[nt][j] - m_new);
                    m_ref[nt][j] = m_new;
                    l_run[nt][j] *= alpha;
#pragma unroll
                    for (int dt = 0; dt < C::DT; ++dt) {
                        o[dt][nt][j] *= alpha;
                        o[dt][nt][j + 2] *= alpha;
                    }
                }
        }
        uint32_t pb[MI][NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                float sum = 0.f;
#pragma unroll
                for (int mi = 0; mi < MI; ++mi) {
#pragma unroll
                    for (int hi = 0; hi < 2; ++hi) {
                        const float pr = fast_exp2(sc[mi][nt][hi * 2 + j] - m_ref[nt][j]);
                        sc[mi][nt][hi * 2 + j] = pr;
                        sum += pr;
                    }
                }
                l_run[nt][j] += sum;
            }
#pragma unroll
            for (int mi = 0; mi < MI; ++mi) {
                pb[mi][nt][0] = movmatrix_trans(pack2<FP8>(sc[mi][nt][0], sc[mi][nt][1]));
                pb[mi][nt][1] = movmatrix_trans(pack2<FP8>(sc[mi][nt][2], sc[mi][nt][3]));
            }
        }

        // O^T += V^T P^T
        if constexpr (!FP8) {
#pragma unroll
            for (int mi = 0; mi < MI; ++mi) {
                const uint32_t vb = vbase + (mi / C::MT) * C::PAGE;
                const int t = (mi % C::MT) * 16 + (lane & 7) + (lane >> 4) * 8;
#pragma unroll
                for (int dt = 0; dt < C::DT; ++dt) {
                    uint32_t a0, a1, a2, a3;
                    ldsm_x4_trans(swz<C, BS>(vb, t, (dt * 16 + ((lane >> 3) & 1) * 8) * 2), a0, a1,
                                  a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816<false>(o[dt][nt], a0, a1, a2, a3, pb[mi][nt][0], pb[mi][nt][1]);
                }
            }
        } else {
            // Byte matrices of 16 tokens x 16 head dims, transposed: this
            // thread gets tokens 4c..4c+3 of dims r and r + 8, which widen to
            // the A fragment for MMA rows (2c, 2c+1 | 2c+8, 2c+9) = tokens
            // (4c, 4c+1 | 4c+2, 4c+3), the order the scores took.
#pragma unroll
            for (int mi = 0; mi < MI; ++mi) {
                const uint32_t vb = vbase + (mi / C::MT) * C::PAGE;
                const int t = (mi % C::MT) * 16 + (lane & 15);
#pragma unroll
                for (int cp = 0; cp < D / 32; ++cp) {
                    uint32_t w0, w1, w2, w3;
                    ldsm_x2_trans_b8(swz<C, BS>(vb, t, (2 * cp + (lane >> 4)) * 16), w0, w1, w2, w3);
                    uint32_t a0, a1, a2, a3;
                    e4m3x4_to_f16x2x2(w0, a0, a2);
                    e4m3x4_to_f16x2x2(w1, a1, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816<true>(o[2 * cp][nt], a0, a1, a2, a3, pb[mi][nt][0], pb[mi][nt][1]);
                    e4m3x4_to_f16x2x2(w2, a0, a2);
                    e4m3x4_to_f16x2x2(w3, a1, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
                        mma16816<true>(o[2 * cp + 1][nt], a0, a1, a2, a3, pb[mi][nt][0],
                                       pb[mi][nt][1]);
                }
            }
        }

        // hand the stage back to the TMA: refill with the iteration SPW
        // ahead.  The stage was only read by generic loads whose values the
        // MMAs above have consumed; once every lane is past them the copy
        // may overwrite it (stores made into it were fenced where made).
        __syncwarp();
        if (it + SPW < my_iters) fetch(it + SPW);
    }
    if (!ok) {
        // A copy never arrived: flag it, wait (bounded) for the copies still
        // in flight into this warp's stages, and fall through with zeros.
        if (lane == 0) set_device_error(a.err, PA_DEVERR_TIMEOUT);
        const int issued = min(my_iters, it_fail + SPW);
        for (int it = it_fail; it < issued; ++it)
            mbar_wait_bounded(smem_addr(&bars[warp * SPW + it % SPW]), (it / SPW) & 1, kWaitLimitNs);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            m_ref[nt][0] = m_ref[nt][1] = -INFINITY;
            m_max[nt][0] = m_max[nt][1] = -INFINITY;
            l_run[nt][0] = l_run[nt][1] = 0.f;
        }
    }

    // ---- merge the warps ----------------------------------------------------
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            float l = l_run[nt][j];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_run[nt][j] = l;
        }
    __syncthreads();  // every warp is done with the page ring
    float *osm = epi;                               // [NW][NP][OSTR]
    float *msm = osm + NW * C::NP * C::OSTR;        // [NW][NP] reference maxima
    float *lsm = msm + NW * C::NP;                  // [NW][NP]
    float *xsm = lsm + NW * C::NP;                  // [NW][NP] true maxima
    float *wsm = xsm + NW * C::NP;                  // [NW][NP]
    float *fin = wsm + NW * C::NP;                  // [2][NP]: true max, sum relative to it
#pragma unroll
    for (int dt = 0; dt < C::DT; ++dt) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int g = nt * 8 + 2 * c + (e & 1);
                const int d = dt * 16 + r + (e >> 1) * 8;
                osm[(warp * C::NP + g) * C::OSTR + d] = o[dt][nt][e];
            }
        }
    }
    if (r == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const int g = nt * 8 + 2 * c + j;
                msm[warp * C::NP + g] = m_ref[nt][j];
                lsm[warp * C::NP + g] = l_run[nt][j];
                xsm[warp * C::NP + g] = m_max[nt][j];
            }
    }
    __syncthreads();
    if (tid < C::NP) {
        const int g = tid;
        float M = -INFINITY, X = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            M = fmaxf(M, msm[w * C::NP + g]);
            X = fmaxf(X, xsm[w * C::NP + g]);
        }
        float L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) L += lsm[w * C::NP + g] * fast_exp2(msm[w * C::NP + g] - M);
        }
        const float inv = L > 0.f ? v_scale / L : 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w)
            wsm[w * C::NP + g] = L > 0.f ? fast_exp2(msm[w * C::NP + g] - M) * inv : 0.f;
        // the workspace holds the true maximum and the sum relative to it
        fin[g] = X;
        fin[C::NP + g] = L > 0.f ? L * fast_exp2(M - X) : 0.f;
    }
    __syncthreads();

    const int64_t row0 = static_cast<int64_t>(s) * a.num_q_heads + h * a.group;
    for (int i = tid; i < a.group * (D / 2); i += NW * 32) {
        const int g = i / (D / 2);
        const int d = (i % (D / 2)) * 2;
        float v0 = 0.f, v1 = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            const float wt = wsm[w * C::NP + g];
            const float *src = osm + (w * C::NP + g) * C::OSTR + d;
            v0 += wt * src[0];
            v1 += wt * src[1];
        }
        if (!a.split) {
            *reinterpret_cast<__nv_bfloat162 *>(a.out + (row0 + g) * D + d) = __floats2bfloat162_rn(v0, v1);
        } else {
            *reinterpret_cast<float2 *>(a.ws_o + ((row0 + g) * a.max_partitions + part) * D + d) =
                make_float2(v0, v1);
        }
    }
    if (a.split && tid < a.group) {
        const int64_t idx = (row0 + tid) * a.max_partitions + part;
        a.ws_m[idx] = fin[tid] * kLn2;  // natural-log units
        a.ws_l[idx] = fin[C::NP + tid];
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Tensor map over a cache viewed as [num_blocks * num_kv_heads * block_size
// rows][head_dim], one box = [block_size rows][min(row bytes, 128) bytes].
pa_status make_map(CUtensorMap *map, const void *cache, bool fp8, int head_dim, int64_t rows,
                   int block_size) {
    auto fn = encode_fn();
    if (!fn) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int elem = fp8 ? 1 : 2;
    const int row_bytes = head_dim * elem;
    const int slab = row_bytes >= 128 ? 128 : row_bytes;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(slab / elem), static_cast<cuuint32_t>(block_size)};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                      const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      slab == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled failed (CUresult %d)", static_cast<int>(res));
    return PA_OK;
}

// Launch shape (build-time): warps per CTA, and the shared-memory budget of
// the page ring, from which the pages in flight per warp follow.
#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 4
#endif
#ifndef PA_DECODE_RING_KB
#define PA_DECODE_RING_KB 64
#endif
// Groups above 8 (two MMA column tiles) at head dim 128 need so many
// registers that only two CTAs fit on an SM; their ring is larger at no
// cost in occupancy (more pages in flight per warp).  Except with a bf16
// cache of 16-token pages: those are held to three CTAs per SM and keep the
// 64 KB ring.
#ifndef PA_DECODE_RING_KB_WIDE
#define PA_DECODE_RING_KB_WIDE 96
#endif
constexpr int kWarps = PA_DECODE_WARPS;

template <int D, int NT, int BS, bool FP8>
constexpr int ring_bytes() {
    constexpr bool wide = D == 128 && NT == 2 && !(BS == 16 && !FP8);
    return (wide ? PA_DECODE_RING_KB_WIDE : PA_DECODE_RING_KB) * 1024;
}

template <int D, int BS, bool FP8, int NT>
constexpr int stages_per_warp() {
    constexpr int ppi = (FP8 && BS == 16) ? 2 : 1;  // Cfg::PPI
    constexpr int stage = 2 * ppi * BS * D * (FP8 ? 1 : 2);
    constexpr int spw = ring_bytes<D, NT, BS, FP8>() / (kWarps * stage);
    return spw < 1 ? 1 : spw;
}

template <int D, int BS, bool FP8, int NT, bool FQ>
static pa_status launch_decode(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                               dim3 grid, cudaStream_t stream) {
    constexpr int SPW = stages_per_warp<D, BS, FP8, NT>();
    using C = Cfg<D, BS, FP8, NT, kWarps, SPW>;
    auto kern = decode_kernel<D, BS, FP8, NT, kWarps, SPW, FQ>;
    // Raise the kernel's shared-memory limit once per device (the first call
    // on a device should precede any stream capture).
    static std::atomic<uint64_t> raised{0};
    int dev = 0;
    pa_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != PA_OK) return st;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(raised.load(std::memory_order_acquire) & bit)) {
        st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM),
                        "cudaFuncSetAttribute(decode)");
        if (st != PA_OK) return st;
        raised.fetch_or(bit, std::memory_order_release);
    }
    kern<<<grid, kWarps * 32, C::SMEM, stream>>>(tk, tv, a);
    return cuda_check(cudaGetLastError(), "decode launch");
}

template <int D, int BS, bool FP8, bool FQ>
static pa_status launch_nt(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeArgs &a,
                           dim3 grid, cudaStream_t stream) {
    if (a.group <= 8) return launch_decode<D, BS, FP8, 1, FQ>(tk, tv, a, grid, stream);
    return launch_decode<D, BS, FP8, 2, FQ>(tk, tv, a, grid, stream);
}

template <int D, int BS>
static pa_status launch_dtype(bool fp8, const CUtensorMap &tk, const CUtensorMap &tv,
                              const DecodeArgs &a, dim3 grid, cudaStream_t stream) {
    if (fp8 && a.q_scale > 0.f) return launch_nt<D, BS, true, true>(tk, tv, a, grid, stream);
    if (fp8) return launch_nt<D, BS, true, false>(tk, tv, a, grid, stream);
    return launch_nt<D, BS, false, false>(tk, tv, a, grid, stream);
}

struct DecodeShape {
    int num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, max_blocks;
    int partition_size;
    pa_kv_dtype kv_dtype;
};

static pa_status check_shape(const DecodeShape &sh, float kv_scale, float softmax_scale) {
    if (sh.num_seqs < 0 || sh.num_q_heads <= 0 || sh.num_kv_heads <= 0 || sh.num_blocks <= 0 ||
        sh.max_blocks <= 0 || sh.partition_size < 0)
        return fail(PA_ERR_INVALID_ARG,
                    "bad size (num_seqs=%d, num_q_heads=%d, num_kv_heads=%d, num_blocks=%d, "
                    "max_blocks_per_seq=%d, partition_size=%d)",
                    sh.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.num_blocks, sh.max_blocks,
                    sh.partition_size);
    if (sh.num_q_heads % sh.num_kv_heads != 0)
        return fail(PA_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d",
                    sh.num_q_heads, sh.num_kv_heads);
    if (sh.num_q_heads / sh.num_kv_heads > 16)
        return fail(PA_ERR_UNSUPPORTED, "query group of %d heads (supported: 1..16)",
                    sh.num_q_heads / sh.num_kv_heads);
    if (sh.head_dim != 64 && sh.head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", sh.head_dim);
    if (sh.block_size != 16 && sh.block_size != 32)
        return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: 16, 32)", sh.block_size);
    if (sh.kv_dtype != PA_KV_BF16 && sh.kv_dtype != PA_KV_FP8_E4M3)
        return fail(PA_ERR_UNSUPPORTED, "kv_dtype %d", static_cast<int>(sh.kv_dtype));
    if (sh.partition_size % sh.block_size != 0)
        return fail(PA_ERR_UNSUPPORTED, "partition_size %d is not a multiple of block_size %d",
                    sh.partition_size, sh.block_size);
    if (static_cast<int64_t>(sh.num_blocks) * sh.num_kv_heads * sh.block_size > 0x7fffffffLL)
        return fail(PA_ERR_UNSUPPORTED, "pool of %d blocks x %d heads x %d rows exceeds 2^31 rows",
                    sh.num_blocks, sh.num_kv_heads, sh.block_size);
    if (static_cast<int64_t>(sh.max_blocks) * sh.block_size > 0x7fffffffLL)
        return fail(PA_ERR_INVALID_ARG, "max_blocks_per_seq * block_size exceeds 2^31");
    if (sh.num_seqs > 65535 || sh.num_kv_heads > 65535)
        return fail(PA_ERR_UNSUPPORTED, "more than 65535 sequences or KV heads");
    if (!isfinite(softmax_scale)) return fail(PA_ERR_INVALID_ARG, "softmax_scale is not finite");
    if (sh.kv_dtype == PA_KV_FP8_E4M3 && !(kv_scale > 0.f && isfinite(kv_scale)))
        return fail(PA_ERR_INVALID_ARG, "fp8 kv_scale must be positive and finite");
    return PA_OK;
}

static int64_t max_partitions_of(int max_blocks, int block_size, int partition_size) {
    if (partition_size <= 0) return 1;
    int64_t tokens = static_cast<int64_t>(max_blocks) * block_size;
    return (tokens + partition_size - 1) / partition_size;
}

static size_t workspace_bytes_of(int num_seqs, int num_q_heads, int head_dim, int64_t parts) {
    return static_cast<size_t>(num_seqs) * num_q_heads * parts * (head_dim + 2) * sizeof(float);
}

// New-token rows appended by the decode kernel itself (pa_decode_step).
struct StepAppend {
    const void *k_new;  // null: attention only
    const void *v_new;
    int32_t *slot_out;
    const float *k_scales;  // optional per-KV-head E4M3 scales
    const float *v_scales;
    float q_scale;          // > 0: E4M3 query and E4M3 x E4M3 scores
};

// Launch the per-partition (split) or whole-context (unsplit) kernel.
static pa_status run_decode(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *context_lens,
                            const DecodeShape &sh, float kv_scale, float softmax_scale,
                            void *workspace, void *out, cudaStream_t stream,
                            const StepAppend *app = nullptr) {
    const bool split = sh.partition_size > 0;
    const int64_t parts = max_partitions_of(sh.max_blocks, sh.block_size, sh.partition_size);
    const bool fp8 = sh.kv_dtype == PA_KV_FP8_E4M3;
    const int64_t rows = static_cast<int64_t>(sh.num_blocks) * sh.num_kv_heads * sh.block_size;
    CUtensorMap tk, tv;
    pa_status st = make_map(&tk, k_cache, fp8, sh.head_dim, rows, sh.block_size);
    if (st != PA_OK) return st;
    st = make_map(&tv, v_cache, fp8, sh.head_dim, rows, sh.block_size);
    if (st != PA_OK) return st;
    unsigned int *err = device_error_word();
    if (!err) return fail(PA_ERR_CUDA, "cannot resolve the device error word");

    DecodeArgs a;
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.max_blocks = sh.max_blocks;
    a.num_blocks = sh.num_blocks;
    a.num_q_heads = sh.num_q_heads;
    a.num_kv_heads = sh.num_kv_heads;
    a.group = sh.num_q_heads / sh.num_kv_heads;
    a.partition_size = split ? sh.partition_size : sh.max_blocks * sh.block_size;
    a.max_partitions = static_cast<int>(parts);
    const float kscale = fp8 ? kv_scale : 1.f;
    a.score_scale = softmax_scale * kscale * 1.4426950408889634f;
    a.v_scale = fp8 ? kv_scale : 1.f;
    a.split = split ? 1 : 0;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.ws_o = static_cast<float *>(workspace);
    const int64_t wrows = static_cast<int64_t>(sh.num_seqs) * sh.num_q_heads;
    a.ws_m = split ? a.ws_o + wrows * parts * sh.head_dim : nullptr;
    a.ws_l = split ? a.ws_m + wrows * parts : nullptr;
    a.err = err;
    a.k_new = app ? static_cast<const uint4 *>(app->k_new) : nullptr;
    a.v_new = app ? static_cast<const uint4 *>(app->v_new) : nullptr;
    a.k_cache_w = a.k_new ? static_cast<uint8_t *>(const_cast<void *>(k_cache)) : nullptr;
    a.v_cache_w = a.k_new ? static_cast<uint8_t *>(const_cast<void *>(v_cache)) : nullptr;
    a.slot_out = a.k_new ? app->slot_out : nullptr;
    a.append_scale = kv_scale;
    a.k_scales = app ? app->k_scales : nullptr;
    a.v_scales = app ? app->v_scales : nullptr;
    a.softmax_log2 = softmax_scale * 1.4426950408889634f;
    a.q_scale = app ? app->q_scale : 0.f;
    a.wait_limit_ns = wait_limit_ns();
    a.stall_first_wait = stall_first_wait();

    if (parts > 0x7fffffffLL) return fail(PA_ERR_UNSUPPORTED, "too many partitions");
    dim3 grid(static_cast<unsigned>(split ? parts : 1), sh.num_kv_heads, sh.num_seqs);
    if (sh.head_dim == 128) {
        if (sh.block_size == 16) return launch_dtype<128, 16>(fp8, tk, tv, a, grid, stream);
        return launch_dtype<128, 32>(fp8, tk, tv, a, grid, stream);
    }
    if (sh.block_size == 16) return launch_dtype<64, 16>(fp8, tk, tv, a, grid, stream);
    return launch_dtype<64, 32>(fp8, tk, tv, a, grid, stream);
}

static pa_status check_pointers(const void *q, const void *k_cache, const void *v_cache,
                                const int32_t *block_tables, const int32_t *context_lens) {
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens)
        return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
        return fail(PA_ERR_INVALID_ARG, "q, k_cache and v_cache must be 16-byte aligned");
    return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_decode_max_partitions(int max_blocks_per_seq, int block_size, int partition_size) {
    if (max_blocks_per_seq <= 0 || block_size <= 0) return 0;
    int64_t p = max_partitions_of(max_blocks_per_seq, block_size, partition_size);
    return p > 0x7fffffffLL ? -1 : static_cast<int>(p);
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int head_dim,
                                int max_blocks_per_seq, int block_size, int partition_size) {
    if (partition_size <= 0 || num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 ||
        max_blocks_per_seq <= 0 || block_size <= 0)
        return 0;
    return workspace_bytes_of(num_seqs, num_q_heads, head_dim,
                              max_partitions_of(max_blocks_per_seq, block_size, partition_size));
}

pa_status pa_decode_partitions(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int num_seqs, int num_q_heads,
                               int num_kv_heads, int head_dim, int num_blocks, int block_size,
                               pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                               int partition_size, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
    clear_error();
    DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                   max_blocks_per_seq, partition_size, kv_dtype};
    pa_status st = check_shape(sh, kv_scale, softmax_scale);
    if (st != PA_OK) return st;
    if (partition_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "pa_decode_partitions needs partition_size > 0");
    if (num_seqs == 0) return PA_OK;
    st = check_pointers(q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, head_dim, max_blocks_per_seq,
                                           block_size, partition_size);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace %p of %zu bytes (need %zu, 16-byte aligned)",
                    workspace, workspace_bytes, need);
    return run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, kv_scale,
                      softmax_scale, workspace, nullptr, stream);
}

pa_status pa_decode_reduce(const void *workspace, size_t workspace_bytes,
                           const int32_t *context_lens, int num_seqs, int num_q_heads,
                           int head_dim, int max_blocks_per_seq, int block_size,
                           int partition_size, void *out, cudaStream_t stream) {
    clear_error();
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || block_size <= 0 ||
        partition_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "bad size (num_seqs=%d, num_q_heads=%d, max_blocks_per_seq=%d, "
                    "block_size=%d, partition_size=%d)", num_seqs, num_q_heads, max_blocks_per_seq,
                    block_size, partition_size);
    if (head_dim != 64 && head_dim != 128)
        return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
    if (num_seqs > 65535 || num_q_heads > 0x7fffffff)
        return fail(PA_ERR_UNSUPPORTED, "more than 65535 sequences");
    if (num_seqs == 0) return PA_OK;
    if (!context_lens || !out) return fail(PA_ERR_INVALID_ARG, "null pointer");
    if (!aligned16(out)) return fail(PA_ERR_INVALID_ARG, "out must be 16-byte aligned");
    int64_t parts = max_partitions_of(max_blocks_per_seq, block_size, partition_size);
    size_t need = workspace_bytes_of(num_seqs, num_q_heads, head_dim, parts);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace %p of %zu bytes (need %zu, 16-byte aligned)",
                    workspace, workspace_bytes, need);
    return launch_reduce(workspace, context_lens, num_seqs, num_q_heads, head_dim, partition_size,
                         static_cast<int>(parts), out, stream);
}

pa_status pa_decode(const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *context_lens, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int num_blocks, int block_size,
                    pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                    int partition_size, void *workspace, size_t workspace_bytes,
                    void *out, cudaStream_t stream) {
    clear_error();
    DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                   max_blocks_per_seq, partition_size, kv_dtype};
    pa_status st = check_shape(sh, kv_scale, softmax_scale);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    st = check_pointers(q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    if (!out || !aligned16(out)) return fail(PA_ERR_INVALID_ARG, "out must be non-null and 16-byte aligned");
    if (partition_size == 0)
        return run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, kv_scale,
                          softmax_scale, nullptr, out, stream);
    int64_t parts = max_partitions_of(max_blocks_per_seq, block_size, partition_size);
    size_t need = workspace_bytes_of(num_seqs, num_q_heads, head_dim, parts);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace %p of %zu bytes (need %zu, 16-byte aligned)",
                    workspace, workspace_bytes, need);
    st = run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, kv_scale, softmax_scale,
                    workspace, nullptr, stream);
    if (st != PA_OK) return st;
    return launch_reduce(workspace, context_lens, num_seqs, num_q_heads, head_dim, partition_size,
                         static_cast<int>(parts), out, stream);
}

pa_status pa_decode_step(const void *q, const void *k_new, const void *v_new, void *k_cache,
                         void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *context_lens, int num_seqs, int num_q_heads,
                         int num_kv_heads, int head_dim, int num_blocks, int block_size,
                         pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                         int partition_size, void *workspace, size_t workspace_bytes,
                         int32_t *slot_mapping, void *out, cudaStream_t stream) {
    clear_error();
    DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                   max_blocks_per_seq, partition_size, kv_dtype};
    pa_status st = check_shape(sh, kv_scale, softmax_scale);
    if (st != PA_OK) return st;
    if (num_seqs == 0) return PA_OK;
    st = check_pointers(q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    if (!k_new || !v_new) return fail(PA_ERR_INVALID_ARG, "null pointer (k_new / v_new)");
    if (!aligned16(k_new) || !aligned16(v_new))
        return fail(PA_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (!out || !aligned16(out)) return fail(PA_ERR_INVALID_ARG, "out must be non-null and 16-byte aligned");
    StepAppend app{k_new, v_new, slot_mapping, nullptr, nullptr};
    if (partition_size == 0)
        return run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, kv_scale,
                          softmax_scale, nullptr, out, stream, &app);
    int64_t parts = max_partitions_of(max_blocks_per_seq, block_size, partition_size);
    size_t need = workspace_bytes_of(num_seqs, num_q_heads, head_dim, parts);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace %p of %zu bytes (need %zu, 16-byte aligned)",
                    workspace, workspace_bytes, need);
    st = run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, kv_scale, softmax_scale,
                    workspace, nullptr, stream, &app);
    if (st != PA_OK) return st;
    return launch_reduce(workspace, context_lens, num_seqs, num_q_heads, head_dim, partition_size,
                         static_cast<int>(parts), out, stream);
}

}  // extern "C"

// The per-head-scaled E4M3 step; q_scale > 0 selects the E4M3 x E4M3 scores.
static pa_status step_scaled(const void *q, const void *k_new, const void *v_new, void *k_cache,
                             void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                             const int32_t *context_lens, int num_seqs, int num_q_heads,
                             int num_kv_heads, int head_dim, int num_blocks, int block_size,
                             const float *k_scales, const float *v_scales, float q_scale,
                             float softmax_scale, int partition_size, void *workspace,
                             size_t workspace_bytes, int32_t *slot_mapping, void *out,
                             cudaStream_t stream) {
    DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                   max_blocks_per_seq, partition_size, PA_KV_FP8_E4M3};
    pa_status st = check_shape(sh, 1.f, softmax_scale);
    if (st != PA_OK) return st;
    if (!k_scales || !v_scales) return fail(PA_ERR_INVALID_ARG, "null scale array");
    if (num_seqs == 0) return PA_OK;
    st = check_pointers(q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    if ((k_new == nullptr) != (v_new == nullptr))
        return fail(PA_ERR_INVALID_ARG, "k_new and v_new must both be given or both be NULL");
    if (k_new && (!aligned16(k_new) || !aligned16(v_new)))
        return fail(PA_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if (!out || !aligned16(out)) return fail(PA_ERR_INVALID_ARG, "out must be non-null and 16-byte aligned");
    StepAppend app{k_new, v_new, slot_mapping, k_scales, v_scales, q_scale};
    if (partition_size == 0)
        return run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, 1.f, softmax_scale,
                          nullptr, out, stream, &app);
    int64_t parts = max_partitions_of(max_blocks_per_seq, block_size, partition_size);
    size_t need = workspace_bytes_of(num_seqs, num_q_heads, head_dim, parts);
    if (!workspace || !aligned16(workspace) || workspace_bytes < need)
        return fail(PA_ERR_WORKSPACE, "workspace %p of %zu bytes (need %zu, 16-byte aligned)",
                    workspace, workspace_bytes, need);
    st = run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, 1.f, softmax_scale,
                    workspace, nullptr, stream, &app);
    if (st != PA_OK) return st;
    return launch_reduce(workspace, context_lens, num_seqs, num_q_heads, head_dim, partition_size,
                         static_cast<int>(parts), out, stream);
}

extern "C" {

pa_status pa_decode_step_scaled(const void *q, const void *k_new, const void *v_new,
                                void *k_cache, void *v_cache, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                int block_size, const float *k_scales, const float *v_scales,
                                float softmax_scale, int partition_size, void *workspace,
                                size_t workspace_bytes, int32_t *slot_mapping, void *out,
                                cudaStream_t stream) {
    clear_error();
    return step_scaled(q, k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                       block_size, k_scales, v_scales, 0.f, softmax_scale, partition_size, workspace,
                       workspace_bytes, slot_mapping, out, stream);
}

pa_status pa_decode_step_fp8_qk(const void *q, const void *k_new, const void *v_new,
                                void *k_cache, void *v_cache, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                int block_size, const float *k_scales, const float *v_scales,
                                float q_scale, float softmax_scale, int partition_size,
                                void *workspace, size_t workspace_bytes, int32_t *slot_mapping,
                                void *out, cudaStream_t stream) {
    clear_error();
    if (!(q_scale > 0.f) || !isfinite(q_scale))
        return fail(PA_ERR_INVALID_ARG, "q_scale %g must be positive and finite", static_cast<double>(q_scale));
    return step_scaled(q, k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                       context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                       block_size, k_scales, v_scales, q_scale, softmax_scale, partition_size,
                       workspace, workspace_bytes, slot_mapping, out, stream);
}

}  // extern "C"

namespace pa {

// Split-context decode into a caller-chosen scratch buffer of `capacity`
// bytes; used by the static-scratch entry point.  Same checks and kernels as
// pa_decode with partition_size > 0.
pa_status decode_split_into(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int num_blocks, int block_size,
                            pa_kv_dtype kv_dtype, float kv_scale, float softmax_scale,
                            int partition_size, void *scratch, size_t capacity, void *out,
                            cudaStream_t stream) {
    DecodeShape sh{num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                   max_blocks_per_seq, partition_size, kv_dtype};
    pa_status st = check_shape(sh, kv_scale, softmax_scale);
    if (st != PA_OK) return st;
    if (partition_size <= 0)
        return fail(PA_ERR_INVALID_ARG, "partition_size must be > 0 (the split path needs scratch)");
    if (num_seqs == 0) return PA_OK;
    st = check_pointers(q, k_cache, v_cache, block_tables, context_lens);
    if (st != PA_OK) return st;
    if (!out || !aligned16(out)) return fail(PA_ERR_INVALID_ARG, "out must be non-null and 16-byte aligned");
    int64_t parts = max_partitions_of(max_blocks_per_seq, block_size, partition_size);
    size_t need = workspace_bytes_of(num_seqs, num_q_heads, head_dim, parts);
    if (need > capacity)
        return fail(PA_ERR_WORKSPACE,
                    "this call needs %zu bytes of scratch but the library's static scratch holds "
                    "%zu; use fewer sequences, a larger partition_size, or pa_decode with a "
                    "workspace of your own", need, capacity);
    st = run_decode(q, k_cache, v_cache, block_tables, context_lens, sh, kv_scale, softmax_scale,
                    scratch, nullptr, stream);
    if (st != PA_OK) return st;
    return launch_reduce(scratch, context_lens, num_seqs, num_q_heads, head_dim, partition_size,
                         static_cast<int>(parts), out, stream);
}

}  // namespace pa
