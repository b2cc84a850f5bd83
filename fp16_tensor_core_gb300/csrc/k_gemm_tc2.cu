// k_gemm_tc2.cu -- CTA-pair variant of the tensor-core GEMM (M >= 256).
//
// Page shorthands: [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南";
// [DG-FP16] = the DeepGEMM FP16/WMMA deep-dive page.
//
// Same computation and epilogue as k_gemm_tc.cu ([FP8-guide] §2.3, §3.1-§3.3;
// [DG-FP16] §2.2), but two CTAs on two SMs (a cluster of 2) share one
// 256 x BN output tile.  Each CTA holds its own 128 rows of A and half of the
// tile's BN rows of B; one pair MMA (M = 256) reads A from both CTAs and B
// from both CTAs, and writes each CTA's 128 rows of the accumulator into that
// CTA's tensor memory.  Per SM this halves the B bytes that TMA writes into
// shared memory and that the MMA reads from it, the traffic that limits the
// single-CTA kernel with 128 x 256 tiles.
//
// From 12 K blocks on a stage holds two adjacent K blocks (KPS = 2): half
// the full/empty round trips per K block, which with one per stage set a
// floor on the time per K block above the MMA's own for tiles under 256
// wide.
//
// Signalling (all waits bounded):
//  * each CTA's producer loads its halves into its own shared memory; every
//    box completes on the even CTA's `full` barrier of the stage, whose
//    producer arms it for the bytes of both CTAs (of the stage's K blocks
//    within the item's K range);
//  * the even CTA's MMA thread issues the pair MMAs and frees a stage in both
//    CTAs with one multicast commit to `empty`; at the end of a tile it
//    commits to `acc_full` in both CTAs;
//  * both CTAs' epilogue warps release an accumulator buffer by arriving on
//    the even CTA's `acc_empty` (count 8: four warps per CTA);
//  * a final multicast commit to `drain` tells both CTAs that no pair MMA
//    still reads their shared memory or writes their tensor memory; only
//    then is tensor memory freed (collectively) and the CTAs exit;
//  * the epilogue (which overlaps the next tile's main loop) stages each
//    warp's 32 x 32 output boxes in a buffer of its own (TMA's 64- or 32-byte
//    swizzle) and writes them with bulk tensor stores -- whole lines, edges
//    clipped by the tensor map -- instead of one scattered 16-byte row piece
//    per lane, whose many partial-line writes slowed the concurrent main
//    loop by ~1 us per tile at 4096^3;
//  * once every CTA is on its last tile the grid lets the next kernel in the
//    stream be scheduled, so that its CTAs start as these exit.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "dg_internal.h"
#include "dg_ptx.cuh"
#include "gemm_common.cuh"

namespace dg {
namespace {

constexpr int kPairBM = 256;   // output rows of a pair tile
constexpr uint32_t kEpiBarrier = 1;   // named barrier of the four epilogue warps
constexpr int kHalfBM = 128;   // rows of it per CTA

// Staging boxes of the epilogue: one 32 x 32 box per epilogue warp.
constexpr int kStagingBytes = 4 * kBoxBytes;

// Stage count: what fits in 227 KB beside the barrier block (1 KB, keeping
// the staging boxes 1024-byte aligned) and the staging boxes, at most 8
// (4 with two K blocks per stage).
constexpr int pair_stages_for(int bn, int kps = 1) {
    const int st = (kSmemLimit - 1024 - 1024 - kStagingBytes) /
                   (kps * (kHalfBM * kBKBytes + (bn / 2) * kBKBytes));
    return st > 8 / kps ? 8 / kps : st;
}

// KPS: K blocks per pipeline stage (1 or 2, adjacent blocks loaded together).
template <int BN, int STAGES, bool kFp16In, int KPS = 1>
struct PairCfg {
    static constexpr int kBK = kFp16In ? 64 : 128;         // K elements per K block
    static constexpr int kABox = kHalfBM * kBKBytes;       // this CTA's 128 rows of A
    static constexpr int kBRows = BN / 2;                  // this CTA's rows of B
    static constexpr int kBBox = kBRows * kBKBytes;
    static constexpr int kABytes = KPS * kABox;
    static constexpr int kBBytes = KPS * kBBox;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTmemCols = pow2_at_least(2 * BN);
    static constexpr int kStagingOff = STAGES * kStageBytes + 1024;   // after the barriers
    static constexpr int kSmemBytes = 1024 + kStagingOff + kStagingBytes;
    static constexpr uint32_t kIdesc = idesc_f32acc(kPairBM, BN, 0, 0);
    static_assert(BN % 32 == 0 && BN >= 128 && BN <= 256, "BN");
    static_assert(kBBytes % 1024 == 0, "1024-byte aligned B stages (128-byte swizzle atoms)");
    static_assert(kTmemCols <= 512, "TMEM columns");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
};

// One work item of a pair: a tile t and its K blocks [kb0, kb1); part -1 is
// a whole tile, part s >= 0 the s-th K range of a split tile (part 0
// finishes the tile: it adds the other parts' partial tiles in part order).
struct PairItem {
    int t, kb0, kb1, part, r;   // r: index of a split tile (its slots, its counter)
};

// Params::tail_split value of the stream-K schedule.  The first
// floor(tiles / pairs) - 1 rounds run whole tiles round-robin, as without it
// (neighbouring pairs on neighbouring tiles, which share A and B in L2); the
// (tile, K block) units of the remaining tiles (between one and two rounds'
// worth) are cut into one equal contiguous range per pair, so every pair
// ends after the same MMA work.  A tile cut at the boundary between pairs
// b - 1 and b is split in two (index r = b): pair b runs its later K range
// first and publishes it, pair b - 1 runs its first K range last and
// finishes the tile.  Each pair's range spans at least one tile, so no tile
// is cut twice; the host chooses it only with at least two tiles per pair.
constexpr int kStreamK = -1;

// K ranges a split tile is cut into under a schedule.
__host__ __device__ constexpr int parts_of(int split) { return split == kStreamK ? 2 : split; }

// Item i of pair `pair` (false when the pair has no item i).  Without a
// split tail, tiles pair, pair + npairs, ...; with one (split >= 2), pairs
// < tail tiles x split hold part pair % split of tail tile pair / split.
// A pair holding a later part runs it first, so that its partial tile is
// published long before it is needed; the pair holding part 0 runs it last,
// after its tiles of the full waves, and finishes the tile.
__device__ __forceinline__ bool pair_item(int i, int pair, int npairs, int num_tiles, int num_kb,
                                          int split, PairItem& it) {
    it.kb0 = 0;
    it.kb1 = num_kb;
    it.part = -1;
    it.r = 0;
    if (split == kStreamK) {
        const int rounds = num_tiles / npairs - 1;   // whole-tile rounds first
        if (i < rounds) {
            it.t = pair + i * npairs;
            return true;
        }
        const int base = rounds * npairs;             // first tile of the stream-K part
        const int64_t units = static_cast<int64_t>(num_tiles - base) * num_kb;
        const int64_t u0 = static_cast<int64_t>(pair) * units / npairs;
        const int64_t u1 = static_cast<int64_t>(pair + 1) * units / npairs;
        const int t0 = static_cast<int>(u0 / num_kb);
        const int k0 = static_cast<int>(u0 - static_cast<int64_t>(t0) * num_kb);
        const int t1 = static_cast<int>((u1 - 1) / num_kb);              // last tile touched
        const int k1 = static_cast<int>(u1 - static_cast<int64_t>(t1) * num_kb);   // its end
        const int j = i - rounds;
        if (u1 <= u0 || t0 + j > t1) return false;
        it.t = base + t0 + j;
        if (j == 0 && k0 > 0) {              // later part of the tile cut at u0
            it.part = 1;
            it.kb0 = k0;
            it.r = pair;
        } else if (t0 + j == t1 && k1 < num_kb) {   // first part of the tile cut at u1
            it.part = 0;
            it.kb1 = k1;
            it.r = pair + 1;
        }
        return true;
    }
    if (split < 2) {
        it.t = pair + i * npairs;
        return it.t < num_tiles;
    }
    const int full_tiles = num_tiles / npairs * npairs;
    const int nfull = full_tiles / npairs;
    const bool has_part = pair < (num_tiles - full_tiles) * split;
    const int part = pair % split;
    int tail_at = -1;                        // position of the tail item
    if (has_part) tail_at = part > 0 ? 0 : nfull;
    if (i == tail_at) {
        it.r = pair / split;
        it.part = part;
        it.t = full_tiles + it.r;
        it.kb0 = part * num_kb / split;
        it.kb1 = (part + 1) * num_kb / split;
        return true;
    }
    const int f = (tail_at == 0) ? i - 1 : i;   // index among the pair's full tiles
    if (f < 0 || f >= nfull) return false;
    it.t = pair + f * npairs;
    return true;
}

// Acquire load of a split tail tile's arrival counter.
__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <int BN, int STAGES, bool kFp16In, int KPS = 1>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const __grid_constant__ CUtensorMap tmap_d, const Params p) {
    using C = PairCfg<BN, STAGES, kFp16In, KPS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * C::kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;   // [2]
    uint64_t* acc_empty = acc_full + 2;    // [2], used in the even CTA
    uint64_t* drain = acc_empty + 2;       // [1]
    uint64_t* fix_bar = drain + 1;         // [1] split tail: partial tiles staged in the ring
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(fix_bar + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 8);
        }
        mbar_init(drain, 1);
        mbar_init(fix_bar, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
    }
    // Both CTAs' barriers are initialised before either can signal the other.
    __syncwarp();
    cluster_sync_all();
    if (warp == 2) {
        tmem_alloc_pair<C::kTmemCols>(tmem_slot);
        tmem_relinquish_pair();
    }
    // Tensor memory exists in both CTAs before the even CTA's MMAs write it.
    tc_fence_before_sync();
    cluster_sync_all();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    const int num_m = (p.M + kPairBM - 1) / kPairBM;
    const int num_n = (p.N + BN - 1) / BN;
    const int num_tiles = num_m * num_n;
    const int num_kb = (p.K + C::kBK - 1) / C::kBK;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    // The producer's first item, its tile and the even CTA's barrier address
    // depend only on the launch: they are formed before the dependency wait,
    // while the preceding kernel drains (after it they took ~0.5 us of the
    // launch's critical path); the empty asm keeps them there.
    PairItem it0{};
    bool have0 = false;
    int mt0 = 0, nt0 = 0;
    uint32_t leader_full = 0;
    if (warp == 0 && lane == 0) {
        leader_full = map_to_rank(full, 0);
        have0 = pair_item(0, pair, npairs, num_tiles, num_kb, p.tail_split, it0);
        if (have0) tile_coords(it0.t, num_m, num_n, p.group_m, mt0, nt0);
        asm volatile("" :: "r"(leader_full), "r"(mt0), "r"(nt0), "r"(it0.kb0), "r"(it0.kb1),
                     "r"(have0 ? 1 : 0) : "memory");
    }
    pdl_wait();

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0, issued_phase = 0;
        bool skip = p.skip_first_load != 0 && blockIdx.x == 0;
        bool ok = true;
        bool first_lap = true;   // every stage starts free: no wait on the first lap
        PairItem it = it0;
        for (int i = 0;
             ok && (i == 0 ? have0 : pair_item(i, pair, npairs, num_tiles, num_kb, p.tail_split, it));
             ++i) {
            int mt = mt0, nt = nt0;
            if (i > 0) tile_coords(it.t, num_m, num_n, p.group_m, mt, nt);
            const int a_row = mt * kPairBM + static_cast<int>(rank) * kHalfBM;
            const int b_row = nt * BN + static_cast<int>(rank) * C::kBRows;
            for (int kb = it.kb0; kb < it.kb1; kb += KPS) {
                const int nk = min(KPS, it.kb1 - kb);   // the range's last stage may be half full
                if (!first_lap && !wait_bounded(&empty[stage], phase ^ 1u, ctl)) { ok = false; break; }
                if (skip) {
                    skip = false;            // leave this stage unloaded
                } else {
                    if (leader)
                        mbar_arrive_expect_tx(&full[stage], 2 * nk * (C::kABox + C::kBBox));
                    const uint32_t bar = leader_full + static_cast<uint32_t>(stage) * 8u;
#pragma unroll
                    for (int j = 0; j < KPS; ++j) {
                        if (j < nk) {
                            tma_load_2d_pair(sA + stage * C::kABytes + j * C::kABox, &tmap_a, bar,
                                             (kb + j) * C::kBK, a_row);
                            tma_load_2d_pair(sB + stage * C::kBBytes + j * C::kBBox, &tmap_b, bar,
                                             (kb + j) * C::kBK, b_row);
                        }
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1u; first_lap = false; }
            }
        }
        // The even CTA's barriers cover both CTAs' boxes: once every stage it
        // armed has completed, every box of both CTAs has landed.  (The odd
        // CTA's boxes were all consumed by MMAs before the final `drain`
        // commit, which the odd CTA waits for.)
        if (leader)
            for (int s = 0; s < STAGES; ++s)
                if (issued_mask & (1u << s))
                    wait_bounded_cluster(&full[s], (issued_phase >> s) & 1u, ctl, false);
    } else if (warp == 1 && lane == 0) {
        if (leader) {
            // -------------------------------------------- pair MMA issuer
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            PairItem it;
            for (int i = 0; ok && pair_item(i, pair, npairs, num_tiles, num_kb, p.tail_split, it); ++i) {
                if (!wait_bounded_cluster(&acc_empty[acc], acc_phase ^ 1u, ctl)) { ok = false; break; }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = it.kb0; kb < it.kb1; kb += KPS) {
                    const int nk = min(KPS, it.kb1 - kb);
                    if (!wait_bounded_cluster(&full[stage], phase, ctl)) { ok = false; break; }
                    tc_fence_after_sync();
#pragma unroll
                    for (int j = 0; j < KPS; ++j) {
                        if (j < nk) {
                            const uint32_t a0 = smem_addr(sA + stage * C::kABytes + j * C::kABox);
                            const uint32_t b0 = smem_addr(sB + stage * C::kBBytes + j * C::kBBox);
#pragma unroll
                            for (int kk = 0; kk < kBKBytes / 32; ++kk) {
                                const uint64_t ad = sdesc_k_major_sw128(a0 + kk * 32);
                                const uint64_t bd = sdesc_k_major_sw128(b0 + kk * 32);
                                const uint32_t accum = (kb > it.kb0 || j > 0 || kk > 0) ? 1u : 0u;
                                if constexpr (kFp16In)
                                    mma_f16_pair(d_tmem, ad, bd, C::kIdesc, accum);
                                else
                                    mma_f8f6f4_pair(d_tmem, ad, bd, C::kIdesc, accum);
                            }
                        }
                    }
                    mma_commit_pair_multicast(&empty[stage], 0x3);
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
                mma_commit_pair_multicast(&acc_full[acc], 0x3);
                if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            }
            // Both CTAs learn here that every pair MMA has completed.
            mma_commit_pair_multicast(drain, 0x3);
            wait_bounded(drain, 0, ctl, false);
        } else {
            // Odd CTA: its shared and tensor memory stay in use until the
            // even CTA's MMAs are done.
            wait_bounded_cluster(drain, 0, ctl, false);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        float alpha = 1.0f;
        if (p.sa != nullptr) alpha = (*p.sa) * (*p.sb);
        if (p.out_kind == kOutE4M3) alpha = __fdiv_rn(alpha, *p.sd);
        const uint32_t leader_acc_empty = map_to_rank(acc_empty, 0);
        uint32_t amax_bits = 0u;
        int acc = 0;
        uint32_t acc_phase = 0;
        const int r_local = q * 32 + lane;   // this thread's row of the CTA's 128
        constexpr int kSlotF4 = BN / 4 * kHalfBM;   // float4s of one partial tile
        constexpr int kSlotBytes = kSlotF4 * 16;
        constexpr int kCopyPiece = 16384;           // bulk copies of 16 KB
        static_assert(kSlotBytes % kCopyPiece == 0, "partial tile in whole pieces");
        static_assert(STAGES * C::kStageBytes >= kSlotBytes + 4 * (BN / 32) * kBoxBytes,
                      "a partial tile and every output box of a tile fit in the ring");
        // every other part's partial tile fits in the idle ring: staged loads
        const int nparts = parts_of(p.tail_split);   // K ranges of a split tile
        const bool staged_parts =
            static_cast<int64_t>(nparts - 1) * kSlotBytes <= STAGES * C::kStageBytes;
        PairItem it;
        for (int i = 0; pair_item(i, pair, npairs, num_tiles, num_kb, p.tail_split, it); ++i) {
            int mt, nt;
            tile_coords(it.t, num_m, num_n, p.group_m, mt, nt);
            // The next kernel in the stream may be scheduled once every CTA
            // is on its last item: its CTAs then start on SMs as these exit
            // (it still waits for this grid before touching memory).
            PairItem nx;
            const bool last_item = !pair_item(i + 1, pair, npairs, num_tiles, num_kb, p.tail_split, nx);
            if (p.early_release && warp == 4 && lane == 0 && last_item) pdl_launch_dependents();
            // The four warps continue or leave together (the split tail
            // below synchronises them on a named barrier).
            const bool got = wait_bounded_cluster(&acc_full[acc], acc_phase, ctl);
            if (!named_bar_and(kEpiBarrier, 128, got)) break;
            tc_fence_after_sync();
            const int row = mt * kPairBM + static_cast<int>(rank) * kHalfBM + q * 32 + lane;
            const int row0 = row - lane;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            // Split tail tile: this CTA's partial tile of part s lives in slot
            // (r * (split - 1) + s - 1) * 2 + rank, as FP32 column quads
            // ([BN / 4][128] float4: a warp's 32 rows are one 512-byte run).
            auto slot_of = [&](int s) {
                return reinterpret_cast<float4*>(p.tail_ws) +
                       static_cast<int64_t>((it.r * (nparts - 1) + s - 1) * 2 +
                                            static_cast<int>(rank)) * kSlotF4;
            };
            uint32_t* const counter = p.tail_counts + it.r * 2 + static_cast<int>(rank);
            bool ready = true;
            if (it.part > 0) {
                // A later part (the pair's first item; its next tiles'
                // main loop runs meanwhile): publish the partial tile with
                // coalesced stores (a warp's 32 rows of a column quad are one
                // 512-byte run), then count the arrival.
                float4* mine = slot_of(it.part);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_load_32cols(tbase + c * 32, r);
                    tmem_load_wait(r);
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        __stcg(mine + (c * 8 + g) * kHalfBM + r_local,
                               make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                           __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])));
                }
                named_bar_sync(kEpiBarrier, 128);   // every row of the CTA's half is out
                if (threadIdx.x == 128) {
                    __threadfence();
                    atomicAdd(counter, 1u);
                }
            } else if (it.part == 0) {
                // The first part finishes the tile: wait (bounded) until the
                // other parts have published theirs.
                bool arrived = true;
                if (threadIdx.x == 128) {
                    const uint32_t want = static_cast<uint32_t>(nparts - 1);
                    const uint64_t t0 = global_timer_ns();
                    while (ld_acquire_gpu(counter) < want) {
                        if (*ctl.abort_flag || global_timer_ns() - t0 > ctl.timeout_ns) {
                            *ctl.abort_flag = 1;
                            atomicOr(ctl.status, kStatusTimeout);
                            arrived = false;
                            break;
                        }
                    }
                }
                ready = named_bar_and(kEpiBarrier, 128, arrived);
                if (ready && staged_parts) {
                    // the other parts' partial tiles into the idle ring, in
                    // part order, on one barrier (used once per CTA)
                    if (threadIdx.x == 128) {
                        fence_proxy_async_global();
                        mbar_arrive_expect_tx(fix_bar, static_cast<uint32_t>(nparts - 1) *
                                                           kSlotBytes);
                        for (int s2 = 1; s2 < nparts; ++s2)
                            for (int piece = 0; piece < kSlotBytes; piece += kCopyPiece)
                                bulk_load_g2s(smem + (s2 - 1) * kSlotBytes + piece,
                                              reinterpret_cast<const uint8_t*>(slot_of(s2)) + piece,
                                              kCopyPiece, fix_bar);
                    }
                    const bool landed = wait_bounded(fix_bar, 0, ctl);
                    ready = named_bar_and(kEpiBarrier, 128, landed);
                    if (!ready && threadIdx.x == 128) wait_bounded(fix_bar, 0, ctl, false);
                }
            }
            // Adds the other parts' partials (in part order) to a chunk of
            // the first part's accumulator, from the ring when staged.
            auto add_parts = [&](int c, uint32_t (&r)[32]) {
                if (it.part != 0) return;
                for (int s = 1; s < nparts; ++s) {
                    const float4* w = staged_parts
                        ? reinterpret_cast<const float4*>(smem + (s - 1) * kSlotBytes)
                        : slot_of(s);
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        const float4 x = staged_parts ? w[(c * 8 + g) * kHalfBM + r_local]
                                                      : __ldcg(w + (c * 8 + g) * kHalfBM + r_local);
                        r[4 * g] = __float_as_uint(__uint_as_float(r[4 * g]) + x.x);
                        r[4 * g + 1] = __float_as_uint(__uint_as_float(r[4 * g + 1]) + x.y);
                        r[4 * g + 2] = __float_as_uint(__uint_as_float(r[4 * g + 2]) + x.z);
                        r[4 * g + 3] = __float_as_uint(__uint_as_float(r[4 * g + 3]) + x.w);
                    }
                }
            };
            if (it.part > 0 || !ready) {
                // nothing to store (a later part, or a wait that ran out)
            } else if (p.staged) {
                // Every tile: the warp's 32 x 32 boxes go through shared
                // memory and out by bulk tensor stores.  While later tiles'
                // main loops run, one staging box per warp (the next box is
                // written once the previous store has read the buffer); on
                // the CTA's last item, whose ring of stages is idle, every
                // box has a place of its own in the ring (after any staged
                // partial tiles), so the stores go out back to back.
                const int ring_base = (it.part == 0 && staged_parts)
                                          ? (nparts - 1) * kSlotBytes : 0;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_load_32cols(tbase + c * 32, r);
                    uint8_t* box = last_item
                        ? smem + ring_base + (q * (BN / 32) + c) * kBoxBytes
                        : smem + C::kStagingOff + q * kBoxBytes;
                    if (!last_item && lane == 0) bulk_wait_read_all();
                    __syncwarp();
                    tmem_load_wait(r);
                    add_parts(c, r);
                    const int col0 = nt * BN + c * 32;
                    amax_bits = max(amax_bits, stage_box(p, box, row, p.M, col0, r, alpha, lane));
                    if (last_item) continue;   // stored together below
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row0 < p.M && col0 < p.N) {
                        tma_store_2d(&tmap_d, box, col0, row0);
                        bulk_commit();
                    }
                }
                if (last_item) {
                    // every box of the warp is in the ring: one fence, then
                    // all of its stores
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row0 < p.M) {
                        for (int c = 0; c < BN / 32 && nt * BN + c * 32 < p.N; ++c)
                            tma_store_2d(&tmap_d, smem + ring_base + (q * (BN / 32) + c) * kBoxBytes,
                                         nt * BN + c * 32, row0);
                        bulk_commit();
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    __syncwarp();
                    tmem_load_32cols(tbase + c * 32, r);
                    tmem_load_wait(r);
                    add_parts(c, r);
                    amax_bits = max(amax_bits, store_chunk(p, row, p.M, nt * BN + c * 32, r, alpha));
                }
            }
            if (it.part == 0 && ready) {
                // every partial has been read: the counter is zero again for
                // the next launch
                named_bar_sync(kEpiBarrier, 128);
                if (threadIdx.x == 128) atomicExch(counter, 0u);
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
                if (leader)
                    mbar_arrive(&acc_empty[acc]);
                else
                    mbar_arrive_cluster(leader_acc_empty + static_cast<uint32_t>(acc) * 8u);
            }
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        // The staging boxes must have been written out before the CTA exits.
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        publish_amax(p, amax_bits);
    }

    // Warps 0 and 1 may arrive diverged (their lane 0 ran a role alone), so
    // the barriers before tensor memory is freed and the CTAs exit are the
    // non-aligned ones.
    tc_fence_before_sync();
    cta_sync_diverged();
    tc_fence_after_sync();
    if (warp == 2) tmem_dealloc_pair<C::kTmemCols>(tmem_base);
    // No arrival from one CTA may land in the other after it has exited.
    cluster_sync_all_diverged();
}

template <typename Kern>
cudaError_t launch_pair(Kern kern, dim3 grid, size_t smem, cudaStream_t s,
                        const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& td,
                        const Params& prm) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, ta, tb, td, prm);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int BN, int STAGES, bool kFp16In, int KPS = 1>
cudaError_t launch_pair_cfg(const TcLaunch& L, const Params& prm, cudaStream_t s) {
    using C = PairCfg<BN, STAGES, kFp16In, KPS>;
    auto kern = gemm_tc_pair_kernel<BN, STAGES, kFp16In, KPS>;
    static std::mutex mu;
    static int max_clusters[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int clusters;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (max_clusters[dev] == 0) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
            if (e != cudaSuccess) return e;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(2);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = C::kSmemBytes;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 2;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            int n = 0;
            e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            if (e != cudaSuccess) return e;
            if (n < 1) return cudaErrorInvalidConfiguration;
            max_clusters[dev] = n;
        }
        clusters = max_clusters[dev];
    }
    CUtensorMap ta, tb, td;
    if (!make_map(&ta, L.A, L.M, L.K, kFp16In, kHalfBM) ||
        !make_map(&tb, L.B, L.N, L.K, kFp16In, C::kBRows))
        return cudaErrorInvalidValue;
    Params prm2 = prm;
    // Split tail: when the last wave is partial, its tiles are cut into
    // `split` K ranges over the otherwise idle pairs (at least two per tile,
    // at most four, each range at least one K block), if the stream's
    // workspace holds their partial tiles.
    const int pairs = L.plan->tiles < clusters ? L.plan->tiles : clusters;
    prm2.tail_split = 1;
    // Stream-K: equal ranges of (tile, K block) units per pair, when every
    // pair covers at least two tiles' worth (a tile is cut at most once), the
    // tiles do not already divide evenly, and the workspace holds a partial
    // tile per boundary and CTA.
    const int64_t sk_need = static_cast<int64_t>(2) * pairs * BN * kHalfBM * sizeof(float);
    if (knobs().stream_k && L.tail_ws != nullptr && L.tail_counts != nullptr && pairs > 0 &&
        L.plan->tiles >= 2 * pairs && L.plan->tiles % pairs != 0 &&
        sk_need <= static_cast<int64_t>(L.tail_ws_bytes) && 2 * pairs <= kSkinnyMaxTiles) {
        prm2.tail_split = kStreamK;
        prm2.tail_ws = L.tail_ws;
        prm2.tail_counts = L.tail_counts;
        if (knobs().log)
            std::fprintf(stderr, "[dg] pair GEMM %dx%dx%d: stream-K over %d pairs, %d tiles\n",
                         L.M, L.N, L.K, pairs, L.plan->tiles);
    } else if (knobs().split_tail && L.tail_ws != nullptr && L.tail_counts != nullptr &&
               pairs > 0) {
        const int rem = L.plan->tiles % pairs;
        const int num_kb = (L.K + C::kBK - 1) / C::kBK;
        int split = rem > 0 ? pairs / rem : 0;
        if (split > 4) split = 4;
        const size_t need = static_cast<size_t>(rem) * (split > 1 ? split - 1 : 0) * 2 * BN *
                            kHalfBM * sizeof(float);
        if (split >= 2 && num_kb >= split && need <= L.tail_ws_bytes &&
            2 * rem <= kSkinnyMaxTiles) {
            prm2.tail_split = split;
            prm2.tail_ws = L.tail_ws;
            prm2.tail_counts = L.tail_counts;
        }
    }
    // Output map of the staged epilogue (else the epilogue stores directly).
    if (!prm2.staged || !make_out_map(&td, L)) {
        prm2.staged = 0;
        td = ta;
    }
    return launch_pair(kern, dim3(2 * pairs), C::kSmemBytes, s, ta, tb, td, prm2);
}

// One or two K blocks per stage, as the plan says (block_k = K elements per
// stage).
template <int BN, bool kFp16In>
cudaError_t launch_pair_bn(const TcLaunch& L, const Params& prm, cudaStream_t s) {
    if (L.plan->block_k == 2 * PairCfg<BN, 1, kFp16In>::kBK)
        return launch_pair_cfg<BN, pair_stages_for(BN, 2), kFp16In, 2>(L, prm, s);
    return launch_pair_cfg<BN, pair_stages_for(BN), kFp16In>(L, prm, s);
}

template <bool kFp16In>
cudaError_t launch_pair_in(const TcLaunch& L, const Params& prm, cudaStream_t s) {
    switch (L.plan->block_n) {
        case 128: return launch_pair_bn<128, kFp16In>(L, prm, s);
        case 160: return launch_pair_bn<160, kFp16In>(L, prm, s);
        case 192: return launch_pair_bn<192, kFp16In>(L, prm, s);
        case 224: return launch_pair_bn<224, kFp16In>(L, prm, s);
        default: return launch_pair_bn<256, kFp16In>(L, prm, s);
    }
}

}  // namespace

int pair_smem_for(int bn, int kps) {
    if (kps == 2) {
        switch (bn) {
            case 128: return PairCfg<128, pair_stages_for(128, 2), false, 2>::kSmemBytes;
            case 160: return PairCfg<160, pair_stages_for(160, 2), false, 2>::kSmemBytes;
            case 192: return PairCfg<192, pair_stages_for(192, 2), false, 2>::kSmemBytes;
            case 224: return PairCfg<224, pair_stages_for(224, 2), false, 2>::kSmemBytes;
            default: return PairCfg<256, pair_stages_for(256, 2), false, 2>::kSmemBytes;
        }
    }
    switch (bn) {
        case 128: return PairCfg<128, pair_stages_for(128), false>::kSmemBytes;
        case 160: return PairCfg<160, pair_stages_for(160), false>::kSmemBytes;
        case 192: return PairCfg<192, pair_stages_for(192), false>::kSmemBytes;
        case 224: return PairCfg<224, pair_stages_for(224), false>::kSmemBytes;
        default: return PairCfg<256, pair_stages_for(256), false>::kSmemBytes;
    }
}

int pair_stages(int bn, int kps) { return pair_stages_for(bn, kps); }

cudaError_t launch_gemm_tc_pair(const TcLaunch& L, const Params& prm, cudaStream_t s) {
    return L.fp16_in ? launch_pair_in<true>(L, prm, s) : launch_pair_in<false>(L, prm, s);
}

}  // namespace dg
