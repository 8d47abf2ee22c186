// Chunked prefill on the 5th-generation tensor cores (tcgen05, tensor memory).
//
// Same computation as pa_prefill.cu (causal attention of each chunk token over
// its sequence's cached prefix and earlier chunk tokens, through the block
// table), organised for sm_103a's asynchronous tensor cores:
//  * One CTA per (two neighbouring query tiles, KV head, sequence).  A tile is
//    128 rows = (chunk token, query head of the KV head's group) pairs; both
//    tiles read every K/V stage, so each SM moves half the page bytes per
//    FLOP that one tile per CTA would.  One CTA per SM: at head dim 128,
//    225 KB of shared memory (both query tiles, five K and five V stages of
//    64 keys; at head dim 64, ten stages of half the size) and all 512 TMEM
//    columns (per tile: two S buffers and O).  A grid of under two waves
//    takes its sequences longest context first.
//  * Thread 0 requests the query tiles (3-D TMA) as soon as the barriers
//    exist.  Warp 8 streams the K pages of each block of 64 keys, warp 10
//    the V pages; lane p issues page p's 2-D TMA boxes (hardware 128-byte
//    swizzle), with the block table read one block ahead.
//    Warp 10 also zeroes the V rows past the context in the last block.
//  * Warp 9 + 2 T issues tile T's MMAs (tcgen05.mma.cta_group::1.kind::f16):
//    the whole warp runs the issue loop, so the operand arithmetic stays
//    warp-uniform, and the lane elect.sync picks issues every MMA and commit
//    (with all 32 lanes active always lane 0, so the commits track that
//    lane's MMAs).  S = Q K^T (M 128 x N 64 x K head dim; query and K both
//    K-major in shared memory), and O += P V (P read from tensor memory, V
//    read MN-major straight from the page layout).  S is double-buffered:
//    S(j) goes to buffer j % 2, and S(j + 2) is issued right after PV(j), so
//    the softmax finds S(j + 1) computed while it worked on S(j).  P(j) is
//    written over the first half of S(j)'s buffer; the MMAs of one thread
//    run in issue order, so S(j + 2) overwrites it only after PV(j) read
//    it.  Each group is committed to an mbarrier, and the commit after
//    PV(j) also releases block j's K/V stage.
//  * Warps 4 T .. 4 T + 3 do tile T's softmax, one query row (TMEM lane) per
//    thread: per block read S, apply the causal mask, keep the row's sum
//    against a reference max that only moves when the row max outgrows it
//    by 2^8 (so O is rescaled in tensor memory rarely), and store P as bf16
//    pairs over S, which PV(j) reads.
//  * Every wait lets the hardware suspend the waiting threads until the phase
//    completes (try_wait with a time hint) rather than spin: the MMA warps
//    share their SM sub-partitions with softmax warps, and a spinning waiter
//    takes issue slots from them.  The MMA and loader warps wait with all 32
//    lanes, so each parks and wakes as one (a lone waiting lane with the rest
//    of its warp held at a warp barrier made the issue that follows several
//    times slower).  Each wait is still bounded by the runtime limit (2 s by
//    default).
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
    float score_scale;       // softmax scale x log2(e) (x the E4M3 scale of K)
    float v_scale;           // the E4M3 scale of V, applied to the output (1 for bf16)
    const float *k_scales;   // E4M3: a K and a V scale per KV head (device), or null for
    const float *v_scales;   // the one scale folded into score_scale and v_scale
    uint64_t wait_limit_ns;  // give up on a wait after this long
    int stall_first_wait;    // test hook: the MMA threads' first wait is on a barrier nothing completes
    int num_seqs;
    int longest_first;       // sequences run longest context first (grids of under two waves, <= 32 sequences)
    __nv_bfloat16 *out;
    unsigned int *err;
};

constexpr int kTcRows = 128;          // query rows per tile (TMEM lanes)
constexpr int kTcKeys = 64;           // keys per block
constexpr int kTcTiles = 2;           // query tiles per CTA; both read every K/V stage
// warps 0-3 softmax of tile 0 and 4-7 of tile 1 (one query row per thread),
// 8 K loads, 9 and 11 the MMAs of tiles 0 and 1, 10 V loads (thread 0 requests the queries)
constexpr int kTcThreads = 384;
constexpr int kTcLoadWarp = 8;
constexpr int kTcMmaWarp = 9;
constexpr int kTcVLoadWarp = 10;
constexpr int kTcMmaWarpB = 11;
constexpr int kTcQSlab = 16384;       // 64 dims of a 128-row query tile
constexpr int kTcKVSlab = kTcKeys * 128;  // 64 dims of a 64-key block
constexpr int kTcQOff = 0;                            // one query tile after the other
// Shared memory for head dim D (64 or 128): every operand is stored as
// 64-dim slabs of 128-byte rows (the swizzle span).  At head dim 64 a stage
// is half the size, so the rings hold twice the blocks.
template <int D>
struct TcLayout {
    static constexpr int kSlabs = D / 64;
    static constexpr int kQTile = kSlabs * kTcQSlab;
    static constexpr int kKVStage = kSlabs * kTcKVSlab;
    static constexpr int kStages = D == 128 ? 5 : 10;  // K and V rings
    static constexpr int kKOff = kTcTiles * kQTile;
    static constexpr int kVOff = kKOff + kStages * kKVStage;
    static constexpr int kSmem = kVOff + kStages * kKVStage + 1024;
};
// P is written against a reference max that only moves when the row max
// grows past it by more than this (base-2 units): P <= 2^8, and O is
// rescaled in tensor memory only then.
constexpr float kTcRescaleThreshold = 8.f;
// Tensor memory, tile T at columns [256 T, 256 T + 256): S buffers [0, 64)
// and [64, 128) (P as bf16 pairs over the first 32 columns of its S), O
// [128, 256).
constexpr int kTcTmemCols = 512;
constexpr int kTcOCol = 128;
// Drain limit: after a wait gave up, the copies already issued are still
// waited for with this before the CTA ends.
constexpr uint64_t kTcWaitNs = 2000000000ull;

template <int D, int BS, bool FP8>
__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                      const PrefillTcArgs a) {
    constexpr int NPG = kTcKeys / BS;  // pages per key block
    using L = TcLayout<D>;
    constexpr int kSlabs = L::kSlabs, kTcQTile = L::kQTile, kTcKVStage = L::kKVStage, kTcStages = L::kStages;
    constexpr int kTcKOff = L::kKOff, kTcVOff = L::kVOff;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t q_full, v_zeroed;
    // kv_full[st]: both the K and the V pages of the stage's block have landed;
    // kv_empty[st]: every tile's PV of that block is done (its QK came
    // before), by a commit of each tile's MMA thread
    __shared__ __align__(8) uint64_t kv_full[kTcStages], kv_empty[kTcStages];
    // E4M3 caches: the stage's E4M3 pages have landed (kv_landed); each
    // tile's query row turned to fp16 (q_conv)
    __shared__ __align__(8) uint64_t kv_landed[2][kTcStages], q_conv[kTcTiles];
    // per tile: S written into buffer b (s_full[T][b]), P written over it
    // (p_full[T][b]), PV done (pv_done), every MMA done (drain).  With two
    // buffers the softmax may write P(j + 1) before the MMA thread saw P(j),
    // so P has a barrier per buffer too: neither barrier of a buffer can
    // complete twice before its waiter looked.
    __shared__ __align__(8) uint64_t s_full[kTcTiles][2], p_full[kTcTiles][2], pv_done[kTcTiles],
        drain[kTcTiles];
    __shared__ __align__(8) uint64_t stall_bar;  // never completed (wait-limit test hook)
    __shared__ uint32_t tmem_base_s;
    __shared__ int failed_s;

    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint64_t limit = a.wait_limit_ns;

    const int pair = gridDim.x - 1 - blockIdx.x;  // tiles 2 pair and 2 pair + 1
    const int h = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // With few CTAs per SM the last wave decides the launch's length: then
    // blockIdx.z takes the sequences longest context first (ties by index),
    // a sequence's tile pairs staying next to each other.  Every warp ranks
    // the (at most 32) contexts itself: lane j holds sequence j's.
    int s = blockIdx.z;
    if (a.longest_first) {
        const int cj = lane < a.num_seqs ? a.context_lens[lane] : INT_MIN;
        int rank = 0;
        for (int j = 0; j < a.num_seqs; ++j) {
            const int ck = __shfl_sync(0xffffffffu, cj, j);
            rank += ck > cj || (ck == cj && j < lane);
        }
        s = __ffs(__ballot_sync(0xffffffffu, lane < a.num_seqs && rank == static_cast<int>(blockIdx.z))) - 1;
    }
    const int q0 = a.query_start[s];
    const int chunk = a.query_start[s + 1] - q0;
    const int ctx = a.context_lens[s];
    const int tok_begin0 = kTcTiles * pair * a.tile_tokens;
    // uniform exits, before any barrier or TMEM use
    if (ctx > a.max_blocks * BS || ctx < chunk) {
        if (tid == 0 && tok_begin0 < chunk) set_device_error(a.err, PA_DEVERR_BAD_CONTEXT);
        return;
    }
    if (tok_begin0 >= chunk) return;
    const int ntiles = tok_begin0 + a.tile_tokens < chunk ? 2 : 1;
    const int first_pos = ctx - chunk;
    // keys [0, kend) cover the later tile's last row; both tiles visit every
    // block (rows past their own position are masked), so each stage is
    // released once per tile
    const int kend = first_pos + min(tok_begin0 + ntiles * a.tile_tokens, chunk);
    const int nkb = (kend + kTcKeys - 1) / kTcKeys;
    // Tile T's own blocks end at its last row's position: the earlier tile
    // skips a trailing block that only the later tile's rows reach (the
    // blocks a tile skips are among the last two, which no stage reuses, so
    // no release is missing).
    auto tile_blocks = [&](int T) {
        const int tile_end = min(tok_begin0 + (T + 1) * a.tile_tokens, chunk);
        return (first_pos + tile_end + kTcKeys - 1) / kTcKeys;
    };
    const bool partial = kend % kTcKeys != 0;  // the last block holds keys past the context

    // Loader lanes pg < NPG own page pg of a key block.  The block table
    // entry is fetched one block ahead and only checked when it is used, so
    // the fetch overlaps the current block's copies; the first block's
    // entries are fetched before the barrier and tensor-memory setup.
    const int32_t *bt = a.block_tables + static_cast<int64_t>(s) * a.max_blocks;
    constexpr int kPastKeys = INT_MIN;
    auto page_entry = [&](int kb) {
        const int pg_idx = kb * NPG + lane;
        return (lane < NPG && pg_idx * BS < kend) ? __ldg(bt + pg_idx) : kPastKeys;
    };
    const bool loader = warp == kTcLoadWarp || warp == kTcVLoadWarp;
    int e_first = loader ? page_entry(0) : kPastKeys;

    if (tid == 0) {
        mbar_init(smem_addr(&q_full), 1);
        mbar_init(smem_addr(&v_zeroed), 1);
        mbar_init(smem_addr(&stall_bar), 1);
        for (int i = 0; i < kTcStages; ++i) {
            mbar_init(smem_addr(&kv_full[i]), 2);  // the K loader and the V loader
            mbar_init(smem_addr(&kv_empty[i]), ntiles);
            mbar_init(smem_addr(&kv_landed[0][i]), 1);
            mbar_init(smem_addr(&kv_landed[1][i]), 1);
        }
        for (int t = 0; t < kTcTiles; ++t) {
            mbar_init(smem_addr(&s_full[t][0]), 1);
            mbar_init(smem_addr(&s_full[t][1]), 1);
            mbar_init(smem_addr(&p_full[t][0]), 4);  // one arrival per softmax warp
            mbar_init(smem_addr(&p_full[t][1]), 4);
            mbar_init(smem_addr(&pv_done[t]), 1);
            mbar_init(smem_addr(&drain[t]), 1);
            mbar_init(smem_addr(&q_conv[t]), 4);
        }
        failed_s = 0;
        fence_barrier_init();
        // the query tiles are requested before the tensor-memory setup
        mbar_arrive_expect_tx(smem_addr(&q_full), ntiles * kTcQTile);
        for (int T = 0; T < ntiles; ++T)
            for (int sl = 0; sl < kSlabs; ++sl)
                tma_load_3d(base + kTcQOff + T * kTcQTile + sl * kTcQSlab, &tmQ, sl * 64, h * a.group,
                            q0 + tok_begin0 + T * a.tile_tokens, smem_addr(&q_full));
        prefetch_tensormap(&tmK);
        prefetch_tensormap(&tmV);
        prefetch_tensormap(&tmO);
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

    const int rows_total = a.num_blocks * a.num_kv_heads * BS;
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

    if (loader) {
        if constexpr (FP8) {
            // ---- E4M3 pages: warp 8 loads K, warp 10 V, each into the second
            // 64-dim slab of its stages, and each widens its block in place to
            // fp16 rows (exact) in the layout bf16 pages would have, zeroing
            // rows past the context, two blocks after requesting it; only then
            // is the block given to the MMAs.  A stage wait for block kb needs
            // block kb - 5 widened, which happened two iterations before. ----
            constexpr int kLag = 2;
            const bool is_k = warp == kTcLoadWarp;
            const int w = is_k ? 0 : 1;
            const CUtensorMap *map = is_k ? &tmK : &tmV;
            const uint32_t ring = base + (is_k ? kTcKOff : kTcVOff);
            const uint64_t policy = l2_evict_first_policy();
            bool ok = true;
            auto widen = [&](int kb) {
                const int st = kb % kTcStages;
                ok = ok && __all_sync(0xffffffffu, mbar_wait_suspend(smem_addr(&kv_landed[w][st]),
                                                                     (kb / kTcStages) & 1, limit));
                // lane widens rows lane and lane + 32.  An E4M3 row is 128
                // bytes (chunk c = dims 16 c .. 16 c + 15 at chunk c ^ (row % 8));
                // its fp16 dims 64 s .. 64 s + 63 go to slab s, chunk f = dims
                // 8 f .. at chunk f ^ (row % 8).  Both rows are read whole
                // before either's slab-1 half is written over it.
                const uint32_t sb = ring + st * kTcKVStage;
                uint4 e[2][8];
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int r = lane + 32 * h2;
#pragma unroll
                    for (int c = 0; c < 8; ++c) e[h2][c] = lds128(sb + kTcKVSlab + r * 128 + ((c ^ (r & 7)) << 4));
                }
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int r = lane + 32 * h2;
                    const bool valid = kb * kTcKeys + r < kend;
                    const uint32_t sw = static_cast<uint32_t>(r & 7);
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
                        if (valid) {
                            e4m3x4_to_f16x2x2(e[h2][c].x, lo.x, lo.y);
                            e4m3x4_to_f16x2x2(e[h2][c].y, lo.z, lo.w);
                            e4m3x4_to_f16x2x2(e[h2][c].z, hi.x, hi.y);
                            e4m3x4_to_f16x2x2(e[h2][c].w, hi.z, hi.w);
                        }
                        const int f = 2 * c;
                        const uint32_t rb = sb + (f >> 3) * kTcKVSlab + r * 128;
                        st_shared16(rb + (((f & 7) ^ sw) << 4), lo);
                        st_shared16(rb + ((((f + 1) & 7) ^ sw) << 4), hi);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&kv_full[st]));
            };
            int e_next = e_first;
            for (int kb = 0; kb < nkb; ++kb) {
                const int st = kb % kTcStages, ph = (kb / kTcStages) & 1;
                const int y = page_row(e_next);
                if (kb + 1 < nkb) e_next = page_entry(kb + 1);
                const bool freed =
                    __all_sync(0xffffffffu, mbar_wait_suspend(smem_addr(&kv_empty[st]), ph ^ 1, limit));
                if (lane == 0) {
                    if (!freed) fail();
                    mbar_arrive_expect_tx(smem_addr(&kv_landed[w][st]), kTcKeys * 128);
                }
                __syncwarp();
                if (lane < NPG)
                    tma_load_2d(ring + st * kTcKVStage + kTcKVSlab + lane * BS * 128, map, 0, y,
                                smem_addr(&kv_landed[w][st]), policy);
                if (kb >= kLag) widen(kb - kLag);
            }
            for (int kb = max(0, nkb - kLag); kb < nkb; ++kb) widen(kb);
            if (!ok && lane == 0) fail();
            // a wait that gave up may leave copies in flight: only the last
            // kTcStages blocks' can be
            if (lane == 0)
                for (int kb = max(0, nkb - kTcStages); kb < nkb; ++kb)
                    mbar_wait_suspend(smem_addr(&kv_landed[w][kb % kTcStages]), (kb / kTcStages) & 1, kTcWaitNs);
        } else {
            // ------------- loads: warp 8 K, warp 10 V (thread 0 requested the queries) -------------
            const bool is_k = warp == kTcLoadWarp;
            const CUtensorMap *map = is_k ? &tmK : &tmV;
            const uint32_t ring = base + (is_k ? kTcKOff : kTcVOff);
            const uint64_t policy = l2_evict_first_policy();
            int e_next = e_first;
            for (int kb = 0; kb < nkb; ++kb) {
                const int st = kb % kTcStages, ph = (kb / kTcStages) & 1;
                const int y = page_row(e_next);
                if (kb + 1 < nkb) e_next = page_entry(kb + 1);
                const bool freed = __all_sync(0xffffffffu, mbar_wait_suspend(smem_addr(&kv_empty[st]), ph ^ 1, limit));
                if (lane == 0) {
                    if (!freed) fail();
                    mbar_arrive_expect_tx(smem_addr(&kv_full[st]), kTcKVStage);
                }
                __syncwarp();
                if (lane < NPG) {
                    for (int sl = 0; sl < kSlabs; ++sl)
                        tma_load_2d(ring + st * kTcKVStage + sl * kTcKVSlab + lane * BS * 128, map, sl * 64, y,
                                    smem_addr(&kv_full[st]), policy);
                }
            }
            if (!is_k && partial) {
                // keys past the context in the last block may hold anything:
                // zero those V rows before a PV reads them (P is 0 there, but
                // 0 x garbage could be NaN)
                const int kb = nkb - 1, st = kb % kTcStages;
                const bool landed = __all_sync(0xffffffffu, mbar_wait_suspend(smem_addr(&kv_full[st]), (kb / kTcStages) & 1, limit));
                if (!landed && lane == 0) fail();
                const uint32_t vbase = base + kTcVOff + st * kTcKVStage;
                for (int r2 = kend - kb * kTcKeys + lane; r2 < kTcKeys; r2 += 32)
                    for (int sl = 0; sl < kSlabs; ++sl)
                        for (int c16 = 0; c16 < 8; ++c16)
                            st_shared_zero16(vbase + sl * kTcKVSlab + r2 * 128 + c16 * 16);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&v_zeroed));
            }
            // Both loaders issue every block, so each stage's phase completes
            // once its copies land; issuing block kb needed block kb - kTcStages
            // released, so only the last kTcStages blocks can still be in flight.
            // Wait for them (2 s) before the CTA may end, whatever gave up.
            if (lane == 0)
                for (int kb = max(0, nkb - kTcStages); kb < nkb; ++kb)
                    mbar_wait_suspend(smem_addr(&kv_full[kb % kTcStages]), (kb / kTcStages) & 1, kTcWaitNs);
        }
    } else if (warp == kTcMmaWarp || warp == kTcMmaWarpB) {
        // ---------------- MMA issue, one thread per tile ----------------
        // S(0) and S(1) first; then per block j: PV(j) once P(j) is written,
        // and S(j + 2) into the buffer P(j) came from.
        const int T = warp == kTcMmaWarp ? 0 : 1;
        if (T < ntiles) {
            // E4M3 caches: fp16 products (the pages widen to fp16 exactly)
            constexpr uint32_t idesc_qk = FP8 ? tc_idesc_f16(kTcRows, kTcKeys, 0, 0) : tc_idesc_bf16(kTcRows, kTcKeys, 0, 0);
            constexpr uint32_t idesc_pv = FP8 ? tc_idesc_f16(kTcRows, D, 0, 1) : tc_idesc_bf16(kTcRows, D, 0, 1);
            // a descriptor's start address is its low field (16-byte units,
            // no carry out within shared memory): every operand descriptor is
            // a base descriptor plus an offset, so issuing an MMA costs one add
            const uint64_t q_desc = tc_smem_desc(base + kTcQOff + T * kTcQTile, 16, 1024, 2);
            const uint64_t k_desc = tc_smem_desc(base + kTcKOff, 16, 1024, 2);
            const uint64_t v_desc = tc_smem_desc(base + kTcVOff, kTcKVSlab, 1024, 2);
            const uint32_t tS = tmem + T * 256, tO = tS + kTcOCol;
            auto wait = [&](uint64_t &bar, uint32_t parity) {
                return __all_sync(0xffffffffu, mbar_wait_suspend(smem_addr(&bar), parity, limit)) != 0;
            };
            // test hook: give up at once on a barrier that nothing completes
            bool ok = !a.stall_first_wait || wait(stall_bar, 0);
            // E4M3 caches: the softmax warps turned the tile's query to fp16
            if constexpr (FP8) ok = ok && wait(q_conv[T], 0);
            else ok = ok && wait(q_full, 0);
            auto qk = [&](int kb) {  // S(kb) = Q K(kb)^T into buffer kb % 2
                const int ks = kb % kTcStages;
                // K and V of the block: V(kb) is in place for PV(kb) too
                ok = ok && wait(kv_full[ks], (kb / kTcStages) & 1);
                tc_fence_after();
                if (ok) {
                    const uint64_t b0 = k_desc + ((ks * kTcKVStage) >> 4);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {  // dims 16 kk .. 16 kk + 15
                        const int qoff = (kk >> 2) * kTcQSlab + (kk & 3) * 32;
                        const int koff = (kk >> 2) * kTcKVSlab + (kk & 3) * 32;
                        tc_mma_bf16_elect(tS + (kb & 1) * kTcKeys, q_desc + (qoff >> 4), b0 + (koff >> 4),
                                          idesc_qk, kk > 0);
                    }
                }
                tc_commit_elect(smem_addr(&s_full[T][kb & 1]));
            };
            const int nkb_t = tile_blocks(T);
            qk(0);
            if (nkb_t > 1) qk(1);
            for (int kb = 0; kb < nkb_t; ++kb) {
                const int vs = kb % kTcStages;
                ok = ok && wait(p_full[T][kb & 1], (kb >> 1) & 1);
                if (!FP8 && kb == nkb - 1 && partial) ok = ok && wait(v_zeroed, 0);
                tc_fence_after();
                if (ok) {  // O += P(kb) V(kb)
                    const uint64_t b0 = v_desc + ((vs * kTcKVStage) >> 4);
                    const uint32_t tP = tS + (kb & 1) * kTcKeys;
#pragma unroll
                    for (int kk = 0; kk < kTcKeys / 16; ++kk)
                        tc_mma_bf16_ts_elect(tO, tP + kk * 8, b0 + ((kk * 16 * 128) >> 4), idesc_pv,
                                             kb > 0 || kk > 0);
                }
                tc_commit_elect(smem_addr(&pv_done[T]));
                // this tile is done with block kb's stage once PV(kb) is
                tc_commit_elect(smem_addr(&kv_empty[vs]));
                if (kb + 2 < nkb_t) qk(kb + 2);
            }
            if (!ok && lane == 0) fail();
            // every MMA issued above is complete before the TMEM is released
            tc_commit_elect(smem_addr(&drain[T]));
            mbar_wait_suspend(smem_addr(&drain[T]), 0, kTcWaitNs);
            __syncwarp();
        }
    } else {
        // ------------- softmax: one query row per thread, 64 keys a block -------------
        const int T = warp >> 2;
        if (T < ntiles) {
            const int row = (warp & 3) * 32 + lane;
            const int t = row / a.group, g = row % a.group;
            const int tok_begin = tok_begin0 + T * a.tile_tokens;
            const bool live = tok_begin + t < chunk;
            const int pos = live ? first_pos + tok_begin + t : -1;
            // blocks ending at or before every row's position need no mask
            const int warp_min_pos = __reduce_min_sync(0xffffffffu, pos);
            const uint32_t lane_addr = static_cast<uint32_t>((warp & 3) * 32) << 16;
            const uint32_t tS = tmem + lane_addr + T * 256, tO = tS + kTcOCol;
            float scale = a.score_scale;
            if constexpr (FP8) {
                if (a.k_scales) scale *= __ldg(a.k_scales + h);
            }
            float m_ref = -INFINITY, l_run = 0.f;
            // the query tile has landed before its shared memory stages the output
            bool ok = mbar_wait_suspend(smem_addr(&q_full), 0, limit);
            if constexpr (FP8) {
                // the products run in fp16: each thread turns its query row
                // (bf16, exact in fp16 within its range) to fp16 in place
                for (int sl = 0; sl < kSlabs; ++sl)
                    for (int c = 0; c < 8; ++c) {
                        const uint32_t ad = base + kTcQOff + T * kTcQTile + sl * kTcQSlab + row * 128 + ((c ^ (row & 7)) << 4);
                        uint4 x = lds128(ad);
                        x.x = pack2<true>(__uint_as_float(x.x << 16), __uint_as_float(x.x & 0xffff0000u));
                        x.y = pack2<true>(__uint_as_float(x.y << 16), __uint_as_float(x.y & 0xffff0000u));
                        x.z = pack2<true>(__uint_as_float(x.z << 16), __uint_as_float(x.z & 0xffff0000u));
                        x.w = pack2<true>(__uint_as_float(x.w << 16), __uint_as_float(x.w & 0xffff0000u));
                        st_shared16(ad, x);
                    }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&q_conv[T]));
            }
            const int nkb_t = tile_blocks(T);
            for (int kb = 0; kb < nkb_t; ++kb) {
                const int key0 = kb * kTcKeys;
                const bool masked = key0 + kTcKeys - 1 > warp_min_pos;
                const uint32_t tSb = tS + (kb & 1) * kTcKeys;  // S(kb), then P(kb)
                ok = ok && mbar_wait_suspend(smem_addr(&s_full[T][kb & 1]), (kb >> 1) & 1, limit);
                tc_fence_after();
                float v[64];
                {
                    float lo[32], hi[32];
                    tc_ld32(tSb, lo);
                    tc_ld32(tSb + 32, hi);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] = lo[i];
                        v[32 + i] = hi[i];
                    }
                }
                if (masked) {
#pragma unroll
                    for (int i = 0; i < 64; ++i) v[i] = key0 + i <= pos ? v[i] : -INFINITY;
                }
                // row max of the block: four independent chains of 3-input maxima
                float mq[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    mq[q] = fmax3(v[16 * q], v[16 * q + 1], v[16 * q + 2]);
#pragma unroll
                    for (int i = 3; i < 15; i += 2) mq[q] = fmax3(mq[q], v[16 * q + i], v[16 * q + i + 1]);
                    mq[q] = fmaxf(mq[q], v[16 * q + 15]);
                }
                const float mxs = fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]) * scale;  // scale > 0 keeps the order
                // move the reference max only when the row max outgrew it
                bool rescale = false;
                float alpha = 1.f;
                if (mxs > m_ref + kTcRescaleThreshold) {
                    alpha = fast_exp2(m_ref - mxs);  // 0 when m_ref = -inf
                    m_ref = mxs;
                    l_run *= alpha;
                    rescale = kb > 0;
                }
                if (__any_sync(0xffffffffu, rescale)) {
                    // O must hold PV(kb - 1) before it is scaled.  PV(kb - 2)
                    // completed before S(kb) (issued after it) was committed,
                    // and PV(kb) waits for this P: the barrier is at most one
                    // phase away, so its parity is unambiguous.
                    ok = ok && mbar_wait_suspend(smem_addr(&pv_done[T]), (kb - 1) & 1, limit);
                    tc_fence_after();
#pragma unroll
                    for (int c = 0; c < D; c += 32) {
                        float o[32];
                        tc_ld32(tO + c, o);
                        tc_wait_ld();
#pragma unroll
                        for (int i = 0; i < 32; ++i) o[i] *= alpha;
                        tc_st32(tO + c, o);
                    }
                    tc_wait_st();
                }
                // P = exp2(scale * s - m_ref) (bf16), in P's columns
                const float neg = m_ref == -INFINITY ? 0.f : -m_ref;
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
                l_run += sa[0] + sb[0];
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) pk[i] = pack2<FP8>(v[2 * i], v[2 * i + 1]);
                // over S(kb), which this thread holds in registers; no MMA
                // writes this buffer before PV(kb), which waits for P
                tc_st32(tSb, pk);
                tc_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_addr(&p_full[T][kb & 1]));
            }
            // every PV is done once the tile's MMA thread's final commit lands
            ok = ok && mbar_wait_suspend(smem_addr(&drain[T]), 0, limit);
            tc_fence_after();
            if (!ok) fail();
            float v_scale = a.v_scale;
            if constexpr (FP8) {
                if (a.v_scales) v_scale = __ldg(a.v_scales + h);
            }
            const float inv = l_run > 0.f ? v_scale / l_run : 0.f;
            // A tile wholly inside its chunk leaves through shared memory (its
            // query tile's space, in the same swizzled layout) and two TMA
            // stores; a tile at the chunk's end is written row by row, so no
            // box reaches into the next sequence's rows.
            const bool full_tile = tok_begin + a.tile_tokens <= chunk;
            const uint32_t stage = base + kTcQOff + T * kTcQTile;
            __nv_bfloat16 *dst = a.out + ((static_cast<int64_t>(q0) + tok_begin + t) * a.num_q_heads +
                                          h * a.group + g) * D;
#pragma unroll
            for (int c = 0; c < D; c += 32) {
                float o[32];
                tc_ld32(tO + c, o);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 w;
                    w.x = pack2<false>(o[i] * inv, o[i + 1] * inv);
                    w.y = pack2<false>(o[i + 2] * inv, o[i + 3] * inv);
                    w.z = pack2<false>(o[i + 4] * inv, o[i + 5] * inv);
                    w.w = pack2<false>(o[i + 6] * inv, o[i + 7] * inv);
                    const int d0 = c + i;  // dims d0 .. d0 + 7
                    if (full_tile)
                        st_shared16(stage + (d0 >> 6) * kTcQSlab + row * 128 + ((((d0 & 63) >> 3) ^ (row & 7)) << 4), w);
                    else if (live && !failed_s)
                        *reinterpret_cast<uint4 *>(dst + d0) = w;
                }
            }
            if (full_tile) {
                fence_proxy_async_smem();
                asm volatile("bar.sync %0, 128;" ::"r"(1 + T) : "memory");  // the tile's four softmax warps
                if ((warp & 3) == 0 && lane == 0) {
                    for (int sl = 0; sl < kSlabs; ++sl)
                        tma_store_3d(&tmO, sl * 64, h * a.group, q0 + tok_begin, stage + sl * kTcQSlab);
                    tma_store_commit_and_wait_read();
                }
            }
        }
    }
    // the query tiles thread 0 requested have landed before the CTA ends
    if (tid == 0) mbar_wait_suspend(smem_addr(&q_full), 0, kTcWaitNs);
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
                            int head_dim, int group, int tile_tokens) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &qr) !=
            cudaSuccess ||
        qr != cudaDriverEntryPointSuccess)
        return fail(PA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    auto fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_q_heads),
                          static_cast<cuuint64_t>(total_tokens)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                             static_cast<cuuint64_t>(num_q_heads) * head_dim * 2};
    cuuint32_t box[3] = {64, static_cast<cuuint32_t>(group), static_cast<cuuint32_t>(tile_tokens)};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult res = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides, box,
                      estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "query tensor map failed (CUresult %d)", static_cast<int>(res));
    return PA_OK;
}

template <int D, int BS, bool FP8>
static pa_status launch_tc(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                           const CUtensorMap &to,
                           const PrefillTcArgs &a, dim3 grid, cudaStream_t stream) {
    auto kern = prefill_tc_kernel<D, BS, FP8>;
    constexpr int kTcSmem = TcLayout<D>::kSmem;
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
    kern<<<grid, kTcThreads, kTcSmem, stream>>>(tq, tk, tv, to, a);
    return cuda_check(cudaGetLastError(), "prefill tcgen05 launch");
}

// Called by pa_prefill for head_dim 64 and 128, bf16 caches, and for
// head_dim 128 with E4M3 caches (arguments already checked).
pa_status launch_prefill_tc(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *query_start, int num_seqs,
                            int total_tokens, int max_query_len, int num_q_heads, int num_kv_heads,
                            int head_dim, int num_blocks, int block_size, bool fp8, float kv_scale,
                            const float *k_scales, const float *v_scales, float softmax_scale, void *out,
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
    // E4M3: one scale folds into the score scale and the output; per-head
    // scales are read by each CTA for its KV head
    const bool per_head = fp8 && k_scales;
    a.score_scale = softmax_scale * 1.4426950408889634f * (fp8 && !per_head ? kv_scale : 1.f);
    a.v_scale = fp8 && !per_head ? kv_scale : 1.f;
    a.k_scales = per_head ? k_scales : nullptr;
    a.v_scales = per_head ? v_scales : nullptr;
    a.wait_limit_ns = wait_limit_ns();
    a.stall_first_wait = stall_first_wait();
    a.num_seqs = num_seqs;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = err;
    const int64_t rows = static_cast<int64_t>(num_blocks) * num_kv_heads * block_size;
    CUtensorMap tq, tk, tv, to;
    pa_status st = make_q_map(&tq, q, total_tokens, num_q_heads, head_dim, group, a.tile_tokens);
    if (st != PA_OK) return st;
    st = make_q_map(&to, out, total_tokens, num_q_heads, head_dim, group, a.tile_tokens);  // same geometry
    if (st != PA_OK) return st;
    st = make_map(&tk, k_cache, fp8, head_dim, rows, block_size);
    if (st != PA_OK) return st;
    st = make_map(&tv, v_cache, fp8, head_dim, rows, block_size);
    if (st != PA_OK) return st;
    const int tiles = (max_query_len + a.tile_tokens - 1) / a.tile_tokens;
    dim3 grid((tiles + kTcTiles - 1) / kTcTiles, num_kv_heads, num_seqs);
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return fail(PA_ERR_CUDA, "cannot read the SM count");
    a.longest_first = num_seqs <= 32 && static_cast<int64_t>(grid.x) * grid.y * grid.z < 2LL * sms;
    if (fp8)
        return block_size == 16 ? launch_tc<128, 16, true>(tq, tk, tv, to, a, grid, stream)
                                : launch_tc<128, 32, true>(tq, tk, tv, to, a, grid, stream);
    if (head_dim == 64)
        return block_size == 16 ? launch_tc<64, 16, false>(tq, tk, tv, to, a, grid, stream)
                                : launch_tc<64, 32, false>(tq, tk, tv, to, a, grid, stream);
    return block_size == 16 ? launch_tc<128, 16, false>(tq, tk, tv, to, a, grid, stream)
                            : launch_tc<128, 32, false>(tq, tk, tv, to, a, grid, stream);
}

}  // namespace pa
