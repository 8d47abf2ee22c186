// Chunked prefill on the 5th-generation tensor cores (tcgen05, tensor memory).
//
// Same computation as pa_prefill.cu (causal attention of each chunk token over
// its sequence's cached prefix and earlier chunk tokens, through the block
// table), organised for sm_103a's asynchronous tensor cores:
//  * One CTA per (query tile of 128 rows = (chunk token, query head of the KV
//    head's group) pairs, KV head, sequence), one CTA per SM (225 KB of
//    shared memory: the query tile and three K and three V stages; all 512
//    TMEM columns: two S accumulators, O, and two P buffers).
//  * Warp 8 streams the tile's queries (one 3-D TMA box per 64-dim slab) and
//    the K pages of each block of 128 keys; warp 10 streams the V pages.
//    Lane p issues page p's boxes (2-D TMA, hardware 128-byte swizzle), with
//    the block table read one block ahead.
//  * Warp 9 owns the tensor memory and one lane issues the MMAs:
//    S = Q K^T (M 128 x N 128 x K 128, both operands K-major in shared
//    memory) into one of two S accumulators, and O += P V (P read from
//    tensor memory, V read MN-major straight from the page layout) into the
//    O accumulator; each group is committed to an mbarrier.
//  * Warps 0-7 do the softmax: a query row is TMEM lane (warp % 4) * 32 +
//    lane, and warps w and w + 4 take its two 64-column halves (their
//    partial maxima meet in shared memory once per block).  They read S,
//    apply the causal mask, keep the row's sum against a reference max that
//    only moves when the row max outgrows it by 2^8 (so O is rescaled in
//    tensor memory rarely), and store P as bf16 pairs into one of two P
//    buffers in tensor memory.  While they work on block j the tensor cores
//    finish block j - 1's PV and compute S for block j + 1.
#include <cudaTypedefs.h>
#include <limits.h>
#include <math.h>

#include <atomic>

#include "pa_prefill.cuh"

namespace pa {

struct PrefillTcArgs {
    const int32_t *block_tables;
    const int32_t *context_lens;
    const int32_t *query_start;
    int max_blocks;
    int num_blocks;
    int num_q_heads;
    int num_kv_heads;
    int group;
    int tile_tokens;  // 128 / group
    float score_scale;
    __nv_bfloat16 *out;
    unsigned int *err;
};

constexpr int kTcRows = 128;          // query rows per tile (TMEM lanes)
constexpr int kTcKeys = 128;          // keys per block
constexpr int kTcTiles = 2;           // query tiles per CTA; both read every K/V stage
// warps 0-7 softmax (2 per row), 8 Q/K loads, 9 and 11 the MMAs of tiles 0
// and 1 (two issuing threads, on sub-partitions apart from each other and
// from the loaders, so neither tile's chain waits behind the other's), 10 V loads
constexpr int kTcThreads = 384;
constexpr int kTcSoftmaxThreads = 256;
constexpr int kTcLoadWarp = 8;
constexpr int kTcMmaWarp = 9;
constexpr int kTcVLoadWarp = 10;
constexpr int kTcMmaWarpB = 11;
constexpr int kTcSlab = 16384;        // one 64-dim slab of 128 rows x 128 B
constexpr int kTcTile = 2 * kTcSlab;  // 128 rows x 128 dims bf16
constexpr int kTcKStages = 3;
constexpr int kTcVStages = 2;
constexpr int kTcQOff = 0;                                   // one query tile after the other
constexpr int kTcKOff = kTcTiles * kTcTile;
constexpr int kTcVOff = kTcKOff + kTcKStages * kTcTile;
constexpr int kTcSmem = kTcVOff + kTcVStages * kTcTile + 1024;
// P is written against a reference max that only moves when the row max
// grows past it by more than this (base-2 units): P <= 2^8, and O is
// rescaled in tensor memory only then.
constexpr float kTcRescaleThreshold = 8.f;
// Tensor memory: S of tile T at columns [128 T, 128 T + 128), O of tile T at
// [256 + 128 T, ...); P of tile T (bf16 pairs, 64 columns) over the first
// half of its S once the softmax has read S.
constexpr int kTcTmemCols = 512;
constexpr int kTcOCol = 256;
constexpr uint64_t kTcWaitNs = 2000000000ull;

// Named barrier 1 over the softmax warps only.
__device__ __forceinline__ void softmax_bar() {
    asm volatile("bar.sync 1, %0;" ::"n"(kTcSoftmaxThreads) : "memory");
}

template <int BS>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const PrefillTcArgs a) {
    constexpr int NPG = kTcKeys / BS;  // pages per key block
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, drain[kTcTiles];
    __shared__ __align__(8) uint64_t k_full[kTcKStages], k_empty[kTcKStages], v_full[kTcVStages],
        v_empty[kTcVStages];
    __shared__ __align__(8) uint64_t s_full[kTcTiles], p_full[kTcTiles], pv_done[kTcTiles];
    __shared__ uint32_t tmem_base_s;
    __shared__ int failed_s;
    // per-row partial maxima of the two column halves (at the end: the
    // partial row sums)
    __shared__ float half_max[2][kTcRows];

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;

    const int pair = gridDim.x - 1 - blockIdx.x;  // tiles 2 pair and 2 pair + 1
    const int h = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q0 = a.query_start[s];
    const int chunk = a.query_start[s + 1] - q0;
    const int ctx = a.context_lens[s];
    int tok_begin[kTcTiles], kend[kTcTiles], nkb[kTcTiles];
#pragma unroll
    for (int T = 0; T < kTcTiles; ++T) tok_begin[T] = (kTcTiles * pair + T) * a.tile_tokens;
    // uniform exits, before any barrier or TMEM use
    if (ctx > a.max_blocks * BS || ctx < chunk) {
        if (tid == 0 && tok_begin[0] < chunk) set_device_error(a.err, PA_DEVERR_BAD_CONTEXT);
        return;
    }
    if (tok_begin[0] >= chunk) return;
    const int ntiles = tok_begin[1] < chunk ? 2 : 1;
    const int first_pos = ctx - chunk;
#pragma unroll
    for (int T = 0; T < kTcTiles; ++T) {
        kend[T] = first_pos + min(tok_begin[T] + a.tile_tokens, chunk);  // keys [0, kend)
        nkb[T] = (kend[T] + kTcKeys - 1) / kTcKeys;
    }
    // the later tile needs the most keys; the loads cover its blocks and both
    // tiles visit all of them (the earlier tile's extra block, at most one,
    // is fully masked), so every stage is released by every tile
    const int kend_c = kend[ntiles - 1];
    const int nkb_c = nkb[ntiles - 1];

    if (tid == 0) {
        mbar_init(smem_addr(&q_full), 1);
        for (int i = 0; i < kTcKStages; ++i) {
            mbar_init(smem_addr(&k_full[i]), 1);
            mbar_init(smem_addr(&k_empty[i]), ntiles);
        }
        for (int i = 0; i < kTcVStages; ++i) {
            mbar_init(smem_addr(&v_full[i]), 1);
            mbar_init(smem_addr(&v_empty[i]), ntiles);
        }
        for (int i = 0; i < kTcTiles; ++i) {
            mbar_init(smem_addr(&drain[i]), 1);
            mbar_init(smem_addr(&s_full[i]), 1);
            mbar_init(smem_addr(&p_full[i]), kTcSoftmaxThreads / 32);
            mbar_init(smem_addr(&pv_done[i]), 1);
        }
        failed_s = 0;
        fence_barrier_init();
        prefetch_tensormap(&tmQ);
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(&tmem_base_s)),
                     "r"(kTcTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    auto fail = [&]() {
        set_device_error(a.err, PA_DEVERR_TIMEOUT);
        atomicExch(&failed_s, 1);
    };

    // Loader lanes pg < NPG own page pg of a key block.  The block table
    // entry is fetched one block ahead and only checked when it is used, so
    // the fetch overlaps the current block's copies.
    const int32_t *bt = a.block_tables + static_cast<int64_t>(s) * a.max_blocks;
    const int rows_total = a.num_blocks * a.num_kv_heads * BS;
    constexpr int kPastKeys = INT_MIN;
    auto page_entry = [&](int kb) {
        const int pg_idx = kb * NPG + lane;
        return (lane < NPG && pg_idx * BS < kend_c) ? __ldg(bt + pg_idx) : kPastKeys;
    };
    // the page's first row in the cache; pages past the keys (and bad
    // entries, which are reported) read a row past the end: zeros
    auto page_row = [&](int blk) {
        if (blk == kPastKeys) return rows_total;
        if (blk < 0 || blk >= a.num_blocks) {
            set_device_error(a.err, PA_DEVERR_BAD_BLOCK);
            return rows_total;
        }
        return (blk * a.num_kv_heads + h) * BS;
    };

    if (warp == kTcLoadWarp) {
        // ---------------- Q and K loads ----------------
        const uint64_t policy = l2_evict_first_policy();
        if (lane == 0) {
            const uint32_t bar = smem_addr(&q_full);
            mbar_arrive_expect_tx(bar, ntiles * kTcTile);
            for (int T = 0; T < ntiles; ++T)
                for (int sl = 0; sl < 2; ++sl)
                    tma_load_3d(base + kTcQOff + T * kTcTile + sl * kTcSlab, &tmQ, sl * 64, h * a.group,
                                q0 + tok_begin[T], bar);
        }
        int e_next = page_entry(0);
        for (int kb = 0; kb < nkb_c; ++kb) {
            const int st = kb % kTcKStages, ph = (kb / kTcKStages) & 1;
            const int y = page_row(e_next);
            if (kb + 1 < nkb_c) e_next = page_entry(kb + 1);
            if (lane == 0) {
                if (!mbar_wait_bounded(smem_addr(&k_empty[st]), ph ^ 1, kTcWaitNs)) fail();
                mbar_arrive_expect_tx(smem_addr(&k_full[st]), kTcTile);
            }
            __syncwarp();
            if (lane < NPG) {
                for (int sl = 0; sl < 2; ++sl)
                    tma_load_2d(base + kTcKOff + st * kTcTile + sl * kTcSlab + lane * BS * 128, &tmK,
                                sl * 64, y, smem_addr(&k_full[st]), policy);
            }
        }
    } else if (warp == kTcVLoadWarp) {
        // ---------------- V loads: the same pages, from a second warp ----------------
        const uint64_t policy = l2_evict_first_policy();
        int e_next = page_entry(0);
        for (int kb = 0; kb < nkb_c; ++kb) {
            const int st = kb % kTcVStages, ph = (kb / kTcVStages) & 1;
            const int y = page_row(e_next);
            if (kb + 1 < nkb_c) e_next = page_entry(kb + 1);
            if (lane == 0) {
                if (!mbar_wait_bounded(smem_addr(&v_empty[st]), ph ^ 1, kTcWaitNs)) fail();
                mbar_arrive_expect_tx(smem_addr(&v_full[st]), kTcTile);
            }
            __syncwarp();
            if (lane < NPG) {
                for (int sl = 0; sl < 2; ++sl)
                    tma_load_2d(base + kTcVOff + st * kTcTile + sl * kTcSlab + lane * BS * 128, &tmV,
                                sl * 64, y, smem_addr(&v_full[st]), policy);
            }
        }
    } else if (warp == kTcMmaWarp || warp == kTcMmaWarpB) {
        // ---------------- MMA issue, one thread per tile ----------------
        // Per tile the chain is S(j) -> softmax -> PV(j) -> S(j + 1): P lives
        // in S's columns, so S(j + 1) waits until PV(j) has read it.  The
        // softmax warps alternate between the tiles, so each tile's PV and
        // next S run on the tensor cores while they work on the other tile.
        const int T = warp == kTcMmaWarp ? 0 : 1;
        if (lane == 0 && T < ntiles) {
            constexpr uint32_t idesc_qk = tc_idesc_bf16(kTcRows, kTcKeys, 0, 0);
            constexpr uint32_t idesc_pv = tc_idesc_bf16(kTcRows, 128, 0, 1);
            // A descriptor's start address is its low field (16-byte units,
            // no carry out within shared memory): every operand descriptor is
            // a base descriptor plus an offset, so issuing an MMA costs one add
            const uint64_t q_desc = tc_smem_desc(base + kTcQOff, 16, 1024, 2);
            const uint64_t k_desc = tc_smem_desc(base + kTcKOff, 16, 1024, 2);
            const uint64_t v_desc = tc_smem_desc(base + kTcVOff, kTcSlab, 1024, 2);
            bool ok = mbar_wait_bounded(smem_addr(&q_full), 0, kTcWaitNs);
            auto qk = [&](int T, int kb) {  // S_T = Q_T K(kb)^T
                const int ks = kb % kTcKStages;
                ok = ok && mbar_wait_bounded(smem_addr(&k_full[ks]), (kb / kTcKStages) & 1, kTcWaitNs);
                if (kb > 0) ok = ok && mbar_wait_bounded(smem_addr(&pv_done[T]), (kb - 1) & 1, kTcWaitNs);
                tc_fence_after();
                if (ok) {
                    const uint64_t a0 = q_desc + ((T * kTcTile) >> 4);
                    const uint64_t b0 = k_desc + ((ks * kTcTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 128 / 16; ++kk) {
                        const uint32_t off = ((kk >> 2) * kTcSlab + (kk & 3) * 32) >> 4;
                        tc_mma_bf16(tmem + T * 128, a0 + off, b0 + off, idesc_qk, kk > 0);
                    }
                }
                tc_commit(smem_addr(&s_full[T]));
            };
            auto pv = [&](int T, int kb) {  // O_T += P_T V(kb)
                const int vs = kb % kTcVStages;
                ok = ok && mbar_wait_bounded(smem_addr(&p_full[T]), kb & 1, kTcWaitNs);
                ok = ok && mbar_wait_bounded(smem_addr(&v_full[vs]), (kb / kTcVStages) & 1, kTcWaitNs);
                tc_fence_after();
                if (ok) {
                    const uint64_t b0 = v_desc + ((vs * kTcTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kTcKeys / 16; ++kk)
                        tc_mma_bf16_ts(tmem + kTcOCol + T * 128, tmem + T * 128 + kk * 8, b0 + ((kk * 16 * 128) >> 4),
                                       idesc_pv, kb > 0 || kk > 0);
                }
                tc_commit(smem_addr(&pv_done[T]));
            };
            qk(T, 0);
            tc_commit(smem_addr(&k_empty[0]));
            for (int kb = 0; kb < nkb_c; ++kb) {
                pv(T, kb);
                tc_commit(smem_addr(&v_empty[kb % kTcVStages]));
                if (kb + 1 < nkb_c) {
                    qk(T, kb + 1);
                    tc_commit(smem_addr(&k_empty[(kb + 1) % kTcKStages]));
                }
            }
            if (!ok) fail();
            // every MMA issued above is complete before the TMEM is released
            tc_commit(smem_addr(&drain[T]));
            mbar_wait_bounded(smem_addr(&drain[T]), 0, kTcWaitNs);
        }
    } else {
        // -------- softmax: two threads per query row, 64 columns each, --------
        // -------- the two tiles in turn                                 --------
        const int quarter = warp & 3, half = warp >> 2;
        const int row = quarter * 32 + lane;
        const int t = row / a.group, g = row % a.group;
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        const uint32_t col0 = half * 64;  // this thread's columns of S and O
        const float scale = a.score_scale;
        int pos[kTcTiles], warp_min_pos[kTcTiles];
        float m_ref[kTcTiles], l_run[kTcTiles];
#pragma unroll
        for (int T = 0; T < kTcTiles; ++T) {
            const bool live = T < ntiles && tok_begin[T] + t < chunk;
            pos[T] = live ? first_pos + tok_begin[T] + t : -1;
            // blocks ending at or before every row's position need no mask
            warp_min_pos[T] = __reduce_min_sync(0xffffffffu, pos[T]);
            m_ref[T] = -INFINITY;
            l_run[T] = 0.f;
        }
        bool ok = true;
        for (int kb = 0; kb < nkb_c; ++kb) {
#pragma unroll
            for (int T = 0; T < kTcTiles; ++T) {
                if (T >= ntiles) continue;  // uniform over the softmax warps
                const uint32_t tS = tmem + lane_addr + T * 128;
                const uint32_t tO = tmem + lane_addr + kTcOCol + T * 128 + col0;
                const int key0 = kb * kTcKeys + col0;
                const bool masked = kb * kTcKeys + kTcKeys - 1 > warp_min_pos[T];
                ok = ok && mbar_wait_bounded(smem_addr(&s_full[T]), kb & 1, kTcWaitNs);
                tc_fence_after();
                float v[64];
                {
                    float lo[32], hi[32];
                    tc_ld32(tS + col0, lo);
                    tc_ld32(tS + col0 + 32, hi);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] = lo[i];
                        v[32 + i] = hi[i];
                    }
                }
                if (masked) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = key0 + i <= pos[T] ? v[i] : -INFINITY;
                }
                // row max of this half: four independent chains of 3-input maxima
                float mq[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    mq[q] = fmax3(v[16 * q], v[16 * q + 1], v[16 * q + 2]);
#pragma unroll
                    for (int i = 3; i < 15; i += 2) mq[q] = fmax3(mq[q], v[16 * q + i], v[16 * q + i + 1]);
                    mq[q] = fmaxf(mq[q], v[16 * q + 15]);
                }
                float mx = fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]);
                // combine the two halves of the row (scale > 0 keeps the
                // order); past this barrier both halves have S in registers,
                // so P may overwrite it
                half_max[half][row] = mx;
                tc_fence_before();
                softmax_bar();
                tc_fence_after();
                mx = fmaxf(mx, half_max[half ^ 1][row]);
                const float mxs = mx * scale;
                // move the reference max only when the row max outgrew it;
                // O holds PV(kb - 1) here: S(kb) was computed after it
                bool rescale = false;
                float alpha = 1.f;
                if (mxs > m_ref[T] + kTcRescaleThreshold) {
                    alpha = fast_exp2(m_ref[T] - mxs);  // 0 when m_ref = -inf
                    m_ref[T] = mxs;
                    l_run[T] *= alpha;
                    rescale = kb > 0;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    float o0[32], o1[32];
                    tc_ld32(tO, o0);
                    tc_ld32(tO + 32, o1);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        o0[i] *= alpha;
                        o1[i] *= alpha;
                    }
                    tc_st32(tO, o0);
                    tc_st32(tO + 32, o1);
                    tc_wait_st();
                }
                // P = exp2(scale * s - m_ref) (bf16)
                const float neg = m_ref[T] == -INFINITY ? 0.f : -m_ref[T];
                float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int i = 0; i < 64; i += 2) {
                    ffma2(v[i], v[i + 1], scale, neg);
                    v[i] = fast_exp2(v[i]);  // masked: exp2(-inf) = 0
                    v[i + 1] = fast_exp2(v[i + 1]);
                    fadd2(sa[(i >> 1) & 3], sb[(i >> 1) & 3], v[i], v[i + 1]);
                }
                fadd2(sa[0], sb[0], sa[1], sb[1]);
                fadd2(sa[2], sb[2], sa[3], sb[3]);
                fadd2(sa[0], sb[0], sa[2], sb[2]);
                l_run[T] += sa[0] + sb[0];
                // both halves have read their partner's maximum: its slot is free
                softmax_bar();
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack2<false>(v[2 * i], v[2 * i + 1]);
                tc_st32(tS + half * 32, pk);
                tc_wait_st();
                if (kb == nkb_c - 1 && T == 0 && kend_c - kb * kTcKeys < kTcKeys) {
                    // keys past the context in the last block may hold
                    // anything: zero those V rows before the first PV reads
                    // them (P is 0 there, but 0 x garbage could be NaN)
                    const int vs = kb % kTcVStages;
                    ok = ok && mbar_wait_bounded(smem_addr(&v_full[vs]), (kb / kTcVStages) & 1, kTcWaitNs);
                    const int valid = kend_c - kb * kTcKeys;
                    const uint32_t vbase = base + kTcVOff + vs * kTcTile;
                    for (int r2 = valid + tid; r2 < kTcKeys; r2 += kTcSoftmaxThreads)
                        for (int sl = 0; sl < 2; ++sl)
                            for (int c16 = 0; c16 < 8; ++c16)
                                st_shared_zero16(vbase + sl * kTcSlab + r2 * 128 + c16 * 16);
                    fence_proxy_async_smem();
                    softmax_bar();  // every softmax warp zeroed its rows
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&p_full[T]));
            }
        }
        // every PV is done once the MMA threads' final commits land
        for (int T = 0; T < ntiles; ++T) ok = ok && mbar_wait_bounded(smem_addr(&drain[T]), 0, kTcWaitNs);
        tc_fence_after();
        if (!ok) fail();
#pragma unroll
        for (int T = 0; T < kTcTiles; ++T) {
            if (T >= ntiles) continue;
            half_max[half][row] = l_run[T];
            softmax_bar();
            const float l = half_max[0][row] + half_max[1][row];
            softmax_bar();  // both read before the next tile's sums overwrite them
            const float inv = l > 0.f ? 1.f / l : 0.f;
            const uint32_t tO = tmem + lane_addr + kTcOCol + T * 128 + col0;
            float o0[32], o1[32];
            tc_ld32(tO, o0);
            tc_ld32(tO + 32, o1);
            tc_wait_ld();
            if (pos[T] >= 0 && !failed_s) {
                __nv_bfloat16 *dst = a.out + ((static_cast<int64_t>(q0) + tok_begin[T] + t) * a.num_q_heads +
                                              h * a.group + g) * 128 + col0;
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 w0, w1;
                    w0.x = pack2<false>(o0[i] * inv, o0[i + 1] * inv);
                    w0.y = pack2<false>(o0[i + 2] * inv, o0[i + 3] * inv);
                    w0.z = pack2<false>(o0[i + 4] * inv, o0[i + 5] * inv);
                    w0.w = pack2<false>(o0[i + 6] * inv, o0[i + 7] * inv);
                    w1.x = pack2<false>(o1[i] * inv, o1[i + 1] * inv);
                    w1.y = pack2<false>(o1[i + 2] * inv, o1[i + 3] * inv);
                    w1.z = pack2<false>(o1[i + 4] * inv, o1[i + 5] * inv);
                    w1.w = pack2<false>(o1[i + 6] * inv, o1[i + 7] * inv);
                    *reinterpret_cast<uint4 *>(dst + i) = w0;
                    *reinterpret_cast<uint4 *>(dst + 32 + i) = w1;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTcTmemCols)
                     : "memory");
    }
}

// Queries [Tq][Hq][D] as a 3-D tensor (D, Hq, Tq); one box is 64 dims x
// `group` heads x `tile_tokens` tokens with the 128-byte swizzle.
static pa_status make_q_map(CUtensorMap *map, const void *q, int total_tokens, int num_q_heads,
                            int group, int tile_tokens) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(num_q_heads), static_cast<cuuint64_t>(total_tokens)};
    cuuint64_t strides[2] = {128 * 2, static_cast<cuuint64_t>(num_q_heads) * 128 * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tile_tokens)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "query tensor map failed (CUresult %d)", static_cast<int>(res));
    return PA_OK;
}

template <int BS>
static pa_status launch_tc(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const PrefillTcArgs &a, dim3 grid, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<BS>;
    static std::atomic<uint64_t> raised{0};
    int dev = 0;
    pa_status st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
    if (st != PA_OK) return st;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(raised.load(std::memory_order_acquire) & bit)) {
        st = cuda_check(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmem),
                        "cudaFuncSetAttribute(prefill tcgen05)");
        if (st != PA_OK) return st;
        raised.fetch_or(bit, std::memory_order_release);
    }
    kern<<<grid, kTcThreads, kTcSmem, stream>>>(tq, tk, tv, a);
    return cuda_check(cudaGetLastError(), "prefill tcgen05 launch");
}

// Called by pa_prefill for head_dim 128 (arguments already checked).
pa_status launch_prefill_tc(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                            int total_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                            int num_blocks, int block_size, float softmax_scale, void *out,
                            unsigned int *err, cudaStream_t stream) {
    const int group = num_q_heads / num_kv_heads;
    PrefillTcArgs a;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.query_start = query_start;
    a.max_blocks = max_blocks_per_seq;
    a.num_blocks = num_blocks;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.group = group;
    a.tile_tokens = kTcRows / group;
    a.score_scale = softmax_scale * 1.4426950408889634f;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
    CUtensorMap tq, tk, tv;
    pa_status st = make_q_map(&tq, q, total_tokens, num_q_heads, group, a.tile_tokens);
    if (st != PA_OK) return st;
    st = make_map(&tk, k_cache, false, 128, rows, block_size);
    if (st != PA_OK) return st;
    st = make_map(&tv, v_cache, false, 128, rows, block_size);
    if (st != PA_OK) return st;
    const int tiles = (max_query_len + a.tile_tokens - 1) / a.tile_tokens;
    dim3 grid((tiles + kTcTiles - 1) / kTcTiles, num_kv_heads, num_seqs);
    return block_size == 16 ? launch_tc<16>(tq, tk, tv, a, grid, stream)
                            : launch_tc<32>(tq, tk, tv, a, grid, stream);
}

}  // namespace pa
