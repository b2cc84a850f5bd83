// k_gemm_tc.cu -- the tensor-core GEMM for M > 16 (E4M3 or FP16 inputs,
// FP32 accumulation in tensor memory, fused scale/convert epilogue).
//
// Page shorthands: [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南";
// [DG-FP16] = the DeepGEMM FP16/WMMA deep-dive page; [HGEMM-L2] =
// "HGEMM优化：深度学习中的矩阵乘法性能提升策略".
//
// What the pages prescribe, and how it maps onto sm_103a:
//  * block tiling of C with a K-blocked main loop ([FP8-guide] §3.1) ->
//    128 x BN output tiles, 128-byte K blocks, one tcgen05.mma (M=128,
//    N=BN, K=32 bytes) per 32 bytes of K, accumulating in tensor memory;
//  * loader warps separate from compute warps ([DG-FP16] §2.2) and a
//    multi-stage prefetch pipeline ([FP8-guide] §2.3, §4.4; [HGEMM-L2]
//    §3.2-§3.3) -> one TMA producer thread, one MMA-issuing thread and four
//    epilogue warps, joined by full/empty mbarriers over a STAGES-deep
//    shared-memory ring; single-wave plans up to 128 wide over at least 12
//    K blocks hold two adjacent K blocks per stage (256 contiguous bytes of
//    every operand row per request, half the barrier round trips);
//  * bank-conflict-free shared-memory layout ([DG-FP16] §3.2) -> TMA's
//    128-byte swizzle, which the MMA's shared-memory descriptors read
//    natively;
//  * scale_A * scale_B applied once to the accumulator on write-back, and
//    the output scale divided out for FP8 output ([FP8-guide] §3.2);
//  * M/N edges by predication and K tails by zero fill, in one kernel
//    ([FP8-guide] §3.3) -> TMA fills out-of-range box elements with zeros,
//    and epilogue stores are predicated on m < M, n < N; an operand that
//    ends inside a tile loads that last tile through a second tensor map
//    whose box is the rows left rounded up to 8, since rows of a box past
//    the tensor's end still cross into the SM.
// The kernel is persistent (one CTA per SM, tiles strided by the grid) and
// double-buffers the accumulator in tensor memory so that the epilogue of
// one tile overlaps the main loop of the next; the epilogue writes each
// warp's 32 x 32 output boxes through a staging box in shared memory with
// bulk tensor stores (whole lines; direct stores only for a grouped tile's
// rows that cross its group's end).  Every mbarrier wait is
// bounded: on a timeout the CTA raises its abort flag, records
// kStatusTimeout, lets in-flight copies and MMAs land, frees its tensor
// memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "dg_internal.h"
#include "dg_ptx.cuh"
#include "gemm_common.cuh"

namespace dg {
namespace {

constexpr int kBM = 128;

// Shared memory for the grouped variant's per-group tile prefix.
constexpr int kGroupSmem = 4 * (kMaxGroups + 1) + 12;

// Staging boxes of the epilogue: one 32 x 32 box per epilogue warp.
constexpr int kStagingBytes = 4 * kBoxBytes;

// Stage count = what fits in 227 KB beside the barrier block (1 KB, keeping
// the staging boxes 1024-byte aligned), the staging boxes and the grouped
// variant's tile prefix, at most 8 (4 with two K blocks per stage).
constexpr int stages_for(int bn, bool grouped = false, int kps = 1) {
    const int st = (kSmemLimit - 1024 - 1024 - kStagingBytes - (grouped ? kGroupSmem : 0)) /
                   (kps * (kBM * kBKBytes + bn * kBKBytes));
    return st > 8 / kps ? 8 / kps : st;
}

// KPS: K blocks per pipeline stage (1, or 2: each stage holds two adjacent
// 128-byte K blocks of every row, so a row's 256 bytes are requested
// together).
template <int BN, int STAGES, bool kFp16In, bool kGrouped = false, int KPS = 1>
struct Cfg {
    static constexpr int kBK = kFp16In ? 64 : 128;        // K elements per K block
    static constexpr int kABox = kBM * kBKBytes;          // 16 KB
    static constexpr int kBBox = BN * kBKBytes;
    static constexpr int kABytes = KPS * kABox;
    static constexpr int kBBytes = KPS * kBBox;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr uint32_t kTmemCols = pow2_at_least(2 * BN);  // two accumulators
    static constexpr int kBarBytes = 256;
    static constexpr int kStagingOff = STAGES * kStageBytes + 1024;   // after the barriers
    static constexpr int kGroupOff = kStagingOff + kStagingBytes;     // grouped: tile prefix
    static constexpr int kSmemBytes = 1024 + kGroupOff + (kGrouped ? kGroupSmem : 0);
    static constexpr uint32_t kIdesc = idesc_f32acc(kBM, BN, 0, 0);
    static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256,
                  "BN: MMA N (multiple of 16, <= 256) and 32-column epilogue chunks");
    static_assert(kTmemCols <= 512, "TMEM columns");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
    static_assert(kBBytes % 1024 == 0, "1024-byte aligned B stages (128-byte swizzle atoms)");
    static_assert(STAGES * kStageBytes >= 4 * (BN / 32) * kBoxBytes,
                  "every output box of a tile fits in the ring");
};

// Output tile t of this launch: A rows from a_row, B rows from b_row,
// output rows [a_row, row_end) and columns from col0.
struct Tile {
    int a_row, b_row, row_end, col0, g;
};

template <int BN, int STAGES, bool kFp16In, bool kGrouped = false, int KPS = 1>
__global__ void __launch_bounds__(kThreads, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmap_a,
               const __grid_constant__ CUtensorMap tmap_b,
               const __grid_constant__ CUtensorMap tmap_d,
               const __grid_constant__ CUtensorMap tmap_a_edge,
               const __grid_constant__ CUtensorMap tmap_b_edge, const Params p) {
    using C = Cfg<BN, STAGES, kFp16In, kGrouped, KPS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * C::kABytes;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * C::kStageBytes);
    uint64_t* empty = full + STAGES;
    uint64_t* acc_full = empty + STAGES;   // [2]
    uint64_t* acc_empty = acc_full + 2;    // [2]
    uint64_t* drain = acc_empty + 2;       // [1]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    // grouped only: tile_start[g] = first tile of group g (G + 1 entries)
    int* tile_start = reinterpret_cast<int*>(smem + C::kGroupOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_a);
        tma_prefetch_desc(&tmap_b);
        tma_prefetch_desc(&tmap_a_edge);
        tma_prefetch_desc(&tmap_b_edge);
    }
    if (warp == 2) {
        tmem_alloc<C::kTmemCols>(tmem_slot);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    const WaitCtl ctl{abort_flag, p.status, p.timeout_ns};
    const int num_m = (p.M + kBM - 1) / kBM;
    const int num_n = (p.N + BN - 1) / BN;
    int num_tiles = num_m * num_n;
    // pipeline steps per tile (KPS K blocks each; a block past K loads zeros)
    const int num_kb = ((p.K + C::kBK - 1) / C::kBK + KPS - 1) / KPS;
    // The prologue overlaps the preceding kernel's tail; the grouped tile
    // prefix reads the device offsets, so there the wait comes first, while
    // the plain kernel forms its first tile before it (below).
    if constexpr (kGrouped) pdl_wait();
    if constexpr (kGrouped) {
        // Tiles of group g: ceil(M_g / 128) x num_n, numbered group by group.
        // The offsets are validated here; invalid ones store nothing.
        if (warp == 3) {
            const int G = p.groups;
            bool valid = p.group_off[0] == 0 && p.group_off[G] == p.M;
            int base = 0;
            for (int g0 = 0; g0 < G; g0 += 32) {
                const int g = g0 + lane;
                int n_tiles = 0;
                if (g < G) {
                    const int m_g = p.group_off[g + 1] - p.group_off[g];
                    if (m_g < 0) valid = false;
                    n_tiles = (max(m_g, 0) + kBM - 1) / kBM * num_n;
                }
                int incl = n_tiles;   // inclusive warp scan
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                    if (lane >= o) incl += v;
                }
                if (g < G) tile_start[g] = base + incl - n_tiles;
                base += __shfl_sync(0xFFFFFFFFu, incl, 31);
            }
            valid = __all_sync(0xFFFFFFFFu, valid);
            if (lane == 0) {
                tile_start[G] = valid ? base : 0;
                if (!valid) atomicOr(p.status, kStatusBadArgument);
            }
            if (!valid)
                for (int g = lane; g < G; g += 32) tile_start[g] = 0;
        }
        __syncthreads();
        num_tiles = tile_start[p.groups];
    }
    // Tile coordinates for tile t (cursor g only moves forward: every role
    // visits its tiles in increasing t).
    auto tile_of = [&](int t, int& g) -> Tile {
        Tile T;
        if constexpr (kGrouped) {
            while (t >= tile_start[g + 1]) ++g;
            const int local = t - tile_start[g];
            const int mt = local / num_n, nt = local - mt * num_n;
            T.a_row = p.group_off[g] + mt * kBM;
            T.row_end = p.group_off[g + 1];
            T.b_row = g * p.N + nt * BN;
            T.col0 = nt * BN;
            T.g = g;
        } else {
            int mt, nt;
            tile_coords(t, num_m, num_n, p.group_m, mt, nt);
            T.a_row = mt * kBM;
            T.row_end = p.M;
            T.b_row = nt * BN;
            T.col0 = nt * BN;
            T.g = 0;
        }
        return T;
    };
    // The producer's first tile depends only on the launch: formed before the
    // dependency wait while the preceding kernel drains (the empty asm keeps
    // it there).
    Tile T0{};
    if constexpr (!kGrouped) {
        if (warp == 0 && lane == 0 && static_cast<int>(blockIdx.x) < num_tiles) {
            int g0 = 0;
            T0 = tile_of(static_cast<int>(blockIdx.x), g0);
            asm volatile("" :: "r"(T0.a_row), "r"(T0.b_row), "r"(T0.row_end), "r"(T0.col0) : "memory");
        }
        pdl_wait();
    }

    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0;          // stages with a load ever issued
        uint32_t issued_phase = 0;         // parity of each stage's last load
        bool skip = p.skip_first_load != 0 && blockIdx.x == 0;
        bool ok = true;
        bool first_lap = true;   // every stage starts free: no wait on the first lap
        int gcur = 0;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            const Tile T = (!kGrouped && t == static_cast<int>(blockIdx.x)) ? T0 : tile_of(t, gcur);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!first_lap && !wait_bounded(&empty[stage], phase ^ 1u, ctl)) { ok = false; break; }
                if (skip) {
                    skip = false;           // leave this stage unloaded
                } else {
                    // edge tiles load shorter boxes through their own maps
                    const bool ae = T.a_row >= p.a_edge_row, be = T.b_row >= p.b_edge_row;
                    mbar_arrive_expect_tx(&full[stage], KPS * ((ae ? p.a_edge_bytes : p.a_box_bytes) +
                                                               (be ? p.b_edge_bytes : p.b_box_bytes)));
#pragma unroll
                    for (int j = 0; j < KPS; ++j) {
                        const int x = (kb * KPS + j) * C::kBK;
                        tma_load_2d(sA + stage * C::kABytes + j * C::kABox,
                                    ae ? &tmap_a_edge : &tmap_a, &full[stage], x, T.a_row);
                        tma_load_2d(sB + stage * C::kBBytes + j * C::kBBox,
                                    be ? &tmap_b_edge : &tmap_b, &full[stage], x, T.b_row);
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                }
                if (++stage == STAGES) { stage = 0; phase ^= 1u; first_lap = false; }
            }
        }
        // Every load this thread issued must have landed before the CTA can
        // exit.  After a normal run they all have (the MMA thread consumed
        // each one) and these waits return at once; after an abort they let
        // copies still in flight finish.
        for (int s = 0; s < STAGES; ++s)
            if (issued_mask & (1u << s))
                wait_bounded(&full[s], (issued_phase >> s) & 1u, ctl, false);
    } else if (warp == 1 && lane == 0) {
        // ------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        bool issued_any = false;
        for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
            if (!wait_bounded(&acc_empty[acc], acc_phase ^ 1u, ctl)) { ok = false; break; }
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!wait_bounded(&full[stage], phase, ctl)) { ok = false; break; }
                tc_fence_after_sync();
#pragma unroll
                for (int j = 0; j < KPS; ++j) {
                    const uint32_t a0 = smem_addr(sA + stage * C::kABytes + j * C::kABox);
                    const uint32_t b0 = smem_addr(sB + stage * C::kBBytes + j * C::kBBox);
#pragma unroll
                    for (int kk = 0; kk < kBKBytes / 32; ++kk) {
                        const uint64_t ad = sdesc_k_major_sw128(a0 + kk * 32);
                        const uint64_t bd = sdesc_k_major_sw128(b0 + kk * 32);
                        const uint32_t accum = (kb > 0 || j > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (kFp16In)
                            mma_f16(d_tmem, ad, bd, C::kIdesc, accum);
                        else
                            mma_f8f6f4(d_tmem, ad, bd, C::kIdesc, accum);
                    }
                }
                issued_any = true;
                mma_commit(&empty[stage]);   // frees the stage when these MMAs finish
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            mma_commit(&acc_full[acc]);      // accumulator ready for the epilogue
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (issued_any) {
            // Tensor memory is freed below: wait for every MMA this thread
            // issued (normal end or abort alike).
            mma_commit(drain);
            wait_bounded(drain, 0, ctl, false);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        const int q = warp & 3;              // TMEM lane quarter of this warp
        auto alpha_of = [&](int g) {
            float a = 1.0f;
            if (p.sa != nullptr) a = p.sa[g] * p.sb[g];
            if (p.out_kind == kOutE4M3) a = __fdiv_rn(a, p.sd[g]);
            return a;
        };
        float alpha = alpha_of(0);
        int alpha_g = 0;
        uint32_t amax_bits = 0u;
        int acc = 0;
        uint32_t acc_phase = 0;
        int gcur = 0;
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            const Tile T = tile_of(t, gcur);
            if (T.g != alpha_g) {
                alpha = alpha_of(T.g);
                alpha_g = T.g;
            }
            // The next kernel in the stream may be scheduled once every CTA
            // is on its last tile (it still waits for this grid's memory).
            const bool last_tile = t + static_cast<int>(gridDim.x) >= num_tiles;
            if (p.early_release && last_tile && warp == 4 && lane == 0) pdl_launch_dependents();
            // Every lane waits; the vote reconverges the warp (tcgen05.ld is
            // .sync.aligned) and makes the whole warp leave together.
            const bool got = wait_bounded(&acc_full[acc], acc_phase, ctl);
            if (!__all_sync(0xFFFFFFFFu, got)) break;
            tc_fence_after_sync();
            const int row = T.a_row + q * 32 + lane;
            const int row0 = T.a_row + q * 32;
            const uint32_t tbase = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            // Staged bulk stores (whole lines, M / N edges clipped by the
            // tensor map) unless the warp's 32 rows cross a group's end,
            // which the tensor map cannot clip: those rows store directly.
            // One staging box per warp while later tiles' main loops run;
            // on the last tile the ring of stages is idle and every box has
            // a place of its own in it, so the stores go out back to back.
            const bool staged = p.staged && (!kGrouped || row0 + 32 <= T.row_end);
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
                uint32_t r[32];
                __syncwarp();
                tmem_load_32cols(tbase + c * 32, r);
                if (staged) {
                    uint8_t* box = last_tile ? smem + (q * (BN / 32) + c) * kBoxBytes
                                             : smem + C::kStagingOff + q * kBoxBytes;
                    if (!last_tile && lane == 0) bulk_wait_read_all();   // the box is free again
                    __syncwarp();
                    tmem_load_wait(r);
                    const int col0 = T.col0 + c * 32;
                    amax_bits = max(amax_bits, stage_box(p, box, row, T.row_end, col0, r, alpha, lane));
                    if (last_tile) continue;   // stored together below
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && row0 < T.row_end && col0 < p.N) {
                        tma_store_2d(&tmap_d, box, col0, row0);
                        bulk_commit();
                    }
                } else {
                    tmem_load_wait(r);
                    amax_bits = max(amax_bits, store_chunk(p, row, T.row_end, T.col0 + c * 32, r, alpha));
                }
            }
            if (staged && last_tile) {
                // every box of the warp is in the idle ring: one fence, then
                // all of its stores
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row0 < T.row_end) {
                    for (int c = 0; c < BN / 32 && T.col0 + c * 32 < p.N; ++c)
                        tma_store_2d(&tmap_d, smem + (q * (BN / 32) + c) * kBoxBytes, T.col0 + c * 32,
                                     row0);
                    bulk_commit();
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        // The staging box must have been written out before the CTA exits.
        if (lane == 0) bulk_wait_all();
        __syncwarp();
        publish_amax(p, amax_bits);
    }

    // Warps 0 and 1 may arrive diverged (their lane 0 ran a role alone): the
    // barrier before tensor memory is freed is the non-aligned one.
    tc_fence_before_sync();
    cta_sync_diverged();
    tc_fence_after_sync();
    if (warp == 2) tmem_dealloc<C::kTmemCols>(tmem_base);
}

// ------------------------------------------------------------- host side

template <int BN, int STAGES, bool kFp16In, bool kGrouped = false, int KPS = 1>
cudaError_t launch_cfg(const TcLaunch& L, const Params& prm, cudaStream_t s) {
    using C = Cfg<BN, STAGES, kFp16In, kGrouped, KPS>;
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!attr_done[dev]) {
            e = cudaFuncSetAttribute(gemm_tc_kernel<BN, STAGES, kFp16In, kGrouped, KPS>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
            if (e != cudaSuccess) return e;
            attr_done[dev] = true;
        }
    }
    CUtensorMap ta, tb, td;
    const int b_rows = kGrouped ? L.N * L.groups : L.N;   // grouped: B is (G*N) x K
    // Edge boxes: the last tile of an operand that ends inside a tile (128
    // rows of A, BN of B) loads boxes of the rows left rounded up to 8, so
    // no box reaches far past the tensor's end.  Those rows still cross
    // into the SM and slow every load: E4M3 17 x 11008 x 4096 17.3 -> 12.5
    // us, 33 x 12288 x 1040 9.9 -> 7.0, 48 x 11008 x 1040 9.3 -> 7.2 with
    // the short box; no change at 4096-deep K for 33..120 rows.
    // DG_TC_SHORT_BOX=0 keeps full boxes everywhere, =1 narrows only an
    // operand of at most 32 rows (sweeps).  Grouped B rows are slices of
    // one tall tensor: full boxes.
    const int sb = knobs().tc_short_box;
    auto edge = [&](int rows, int full, int* edge_row, int* edge_box) {
        const int left = rows % full;
        *edge_row = INT_MAX;
        *edge_box = full;
        if (kGrouped || left == 0 || sb == 0 || (sb == 1 && rows > 32)) return;
        *edge_row = rows - left;
        *edge_box = (left + 7) / 8 * 8;
    };
    int a_edge_row, a_edge_box, b_edge_row, b_edge_box;
    edge(L.M, kBM, &a_edge_row, &a_edge_box);
    edge(L.N, BN, &b_edge_row, &b_edge_box);
    // (an operand without an edge tile passes its full map twice: no
    // second encoding on the host)
    CUtensorMap tae, tbe;
    if (!make_map(&ta, L.A, L.M, L.K, kFp16In, kBM) ||
        !make_map(&tb, L.B, b_rows, L.K, kFp16In, BN))
        return cudaErrorInvalidValue;
    tae = ta;
    tbe = tb;
    if ((a_edge_row != INT_MAX && !make_map(&tae, L.A, L.M, L.K, kFp16In, a_edge_box)) ||
        (b_edge_row != INT_MAX && !make_map(&tbe, L.B, b_rows, L.K, kFp16In, b_edge_box)))
        return cudaErrorInvalidValue;
    Params prm2 = prm;
    prm2.a_box_bytes = kBM * kBKBytes;
    prm2.b_box_bytes = BN * kBKBytes;
    prm2.a_edge_bytes = a_edge_box * kBKBytes;
    prm2.b_edge_bytes = b_edge_box * kBKBytes;
    prm2.a_edge_row = a_edge_row;
    prm2.b_edge_row = b_edge_row;
    // Output map of the staged epilogue (else the epilogue stores directly).
    if (!prm2.staged || !make_out_map(&td, L)) {
        prm2.staged = 0;
        td = ta;
    }
    return launch_kernel(gemm_tc_kernel<BN, STAGES, kFp16In, kGrouped, KPS>, dim3(L.plan->grid),
                         dim3(kThreads), C::kSmemBytes, s, ta, tb, td, tae, tbe, prm2);
}

template <bool kFp16In>
cudaError_t launch_in(const TcLaunch& L, const Params& prm, cudaStream_t s) {
    switch (L.plan->block_n) {
        // two K blocks per stage: block_k is twice the K block
        case 64:
            if (L.plan->block_k == 2 * (kFp16In ? 64 : 128))
                return launch_cfg<64, stages_for(64, false, 2), kFp16In, false, 2>(L, prm, s);
            return launch_cfg<64, stages_for(64), kFp16In>(L, prm, s);
        case 96:
            if (L.plan->block_k == 2 * (kFp16In ? 64 : 128))
                return launch_cfg<96, stages_for(96, false, 2), kFp16In, false, 2>(L, prm, s);
            return launch_cfg<96, stages_for(96), kFp16In>(L, prm, s);
        case 128:
            if (L.plan->block_k == 2 * (kFp16In ? 64 : 128))
                return launch_cfg<128, stages_for(128, false, 2), kFp16In, false, 2>(L, prm, s);
            return launch_cfg<128, stages_for(128), kFp16In>(L, prm, s);
        case 160: return launch_cfg<160, stages_for(160), kFp16In>(L, prm, s);
        case 192: return launch_cfg<192, stages_for(192), kFp16In>(L, prm, s);
        case 224: return launch_cfg<224, stages_for(224), kFp16In>(L, prm, s);
        default: return launch_cfg<256, stages_for(256), kFp16In>(L, prm, s);
    }
}

int smem_for(int bn) {
    switch (bn) {
        case 64: return Cfg<64, stages_for(64), false>::kSmemBytes;
        case 96: return Cfg<96, stages_for(96), false>::kSmemBytes;
        case 128: return Cfg<128, stages_for(128), false>::kSmemBytes;
        case 160: return Cfg<160, stages_for(160), false>::kSmemBytes;
        case 192: return Cfg<192, stages_for(192), false>::kSmemBytes;
        case 224: return Cfg<224, stages_for(224), false>::kSmemBytes;
        default: return Cfg<256, stages_for(256), false>::kSmemBytes;
    }
}

}  // namespace

void plan_tc(int64_t M, int64_t N, int64_t K, bool fp16_in, int sm_count, dg_plan* p) {
    // Per-shape tile choice ([FP8-guide] §3.1, §3.3; [HGEMM-L2] §3.1):
    // estimate each candidate's time as (waves of tiles over the SMs) x
    // (tile width / relative MMA efficiency of that width) and keep the
    // cheapest; narrow tiles win when the grid would otherwise leave SMs
    // idle or strand a partial last wave.
    const int64_t num_m = (M + kBM - 1) / kBM;
    // Relative throughput per CTA of a 128 x BN tile.  Each 32-byte K step
    // reads 4 KB of A and BN*32 B of B from shared memory while the MMA runs
    // for BN/2 cycles, so narrow tiles need more shared-memory bandwidth per
    // flop (8192/BN + 64 B/clk).  Measured on GB300 (8192^3 E4M3): BN 256 ->
    // 1.0, 128 -> 0.72, 64 -> 0.36; the widths in between are interpolated
    // along that demand curve.  The 96-wide tile (last-but-one candidate)
    // takes part only in the one-wave rule below.
    constexpr int kCand = 7;
    const int cand[kCand] = {256, 224, 192, 160, 128, 96, 64};
    const double eff[kCand] = {1.0, 0.95, 0.88, 0.80, 0.72, 0.0, 0.36};
    int best = 256;
    double best_cost = 0.0;
    for (int i = 0; i < kCand; ++i) {
        if (cand[i] == 96) continue;
        const int bn = cand[i];
        const int64_t tiles = num_m * ((N + bn - 1) / bn);
        const int64_t waves = (tiles + sm_count - 1) / sm_count;
        const double cost = static_cast<double>(waves) * bn / eff[i];
        if (i == 0 || cost < best_cost) { best = bn; best_cost = cost; }
    }
    // A width that puts every tile in one wave (K up to 64 K blocks, up to
    // 32 for widths above 128): the launch is bound by latency and each
    // SM's own operand stream rather than by MMA efficiency, so the
    // narrowest such tile (most CTAs, fewest bytes per CTA) wins, and CTA
    // pairs only add cluster start-up.  Measured on GB300 (BF16 out,
    // graph-replayed), against the estimate below: 256^3 3.2 us (128 x 64)
    // vs 5.2 (pairs 256 x 128); 1024^3 5.9 vs 8.1; 129 x 1000 x 1040 6.8 vs
    // 7.7; 1024 x 1024 x 8192 20.9 vs 24.0; FP16 1024^3 8.1 vs 10.3;
    // 1024 x 4096 x 4096 15.5 vs 17.2 (128 x 224); equal at 256 x 12288 x
    // 4096.  DG_ONE_WAVE=0 turns the rule off and DG_ONE_WAVE_KB sets its
    // K-block limit (sweeps).
    const int64_t kblocks = (K + (fp16_in ? 64 : 128) - 1) / (fp16_in ? 64 : 128);
    const Knobs& kn = knobs();
    bool one_wave = false;
    if (kn.one_wave && kblocks <= kn.one_wave_kb) {
        for (int i = kCand - 1; i >= 0; --i) {   // narrowest first
            if (num_m * ((N + cand[i] - 1) / cand[i]) <= sm_count) {
                // past 32 K blocks a wide tile is MMA-bound enough for the
                // pairs' efficiency to win (2048^2 x 8192: 26.1 us as pairs
                // vs 27.6 as 128 x 256 single tiles)
                if (kblocks <= 32 || cand[i] <= 128) {
                    best = cand[i];
                    one_wave = true;
                }
                break;
            }
        }
    }
    // DG_FORCE_BLOCK_N=64|96|128|160|192|224|256 pins the tile width (sweeps).
    {
        const int v = kn.force_block_n;
        for (int i = 0; i < kCand; ++i)
            if (v == cand[i]) best = v;
    }
    const int64_t tiles = num_m * ((N + best - 1) / best);
    p->block_m = kBM;
    p->block_n = best;
    p->block_k = fp16_in ? 64 : 128;
    p->stages = stages_for(best);
    p->tiles = static_cast<int>(tiles);
    p->grid = static_cast<int>(tiles < sm_count ? tiles : sm_count);
    p->smem_bytes = smem_for(best);
    // Single-wave plans up to 128 wide over at least 12 K blocks take two K
    // blocks per stage: each stage then requests 256 contiguous bytes of
    // every row of B, which streams better, and the barrier round trips per
    // K block halve.  Measured on GB300 (graph-replayed, us, one -> two):
    // E4M3 32 x 12288 x 4096 12.87 -> 12.27, 128 x 12288 x 4096 13.28 ->
    // 12.82, 96 x 8192 x 2048 7.84 -> 6.86, 32 x 8192 x 3072 9.73 -> 8.27,
    // 48 x 12288 x 1536 7.28 -> 6.96, 256 x 4096 x 11008 26.59 -> 23.73,
    // 2048 x 1024 x 11008 27.12 -> 22.47, 512 x 2048 x 8192 20.40 -> 16.15;
    // FP16 1024 x 1024 x 8192 37.85 -> 32.20; over 9 K blocks no gain and up
    // to 4% lost on latency-bound shapes (129 x 1000 x 1040 5.33 -> 5.53).
    // DG_TC_KPS=1|2 pins one or two for every such plan (sweeps).
    const bool kps2 = kn.tc_kps == 2 || (kn.tc_kps == 0 && kblocks >= 12);
    if (tiles <= sm_count && kps2 && best <= 128) {
        p->block_k *= 2;
        p->stages = stages_for(best, false, 2);
        p->smem_bytes = best == 64 ? Cfg<64, stages_for(64, false, 2), false, false, 2>::kSmemBytes
                        : best == 96 ? Cfg<96, stages_for(96, false, 2), false, false, 2>::kSmemBytes
                                     : Cfg<128, stages_for(128, false, 2), false, false, 2>::kSmemBytes;
    }

    // CTA pairs (256 x BN tiles over sm_count / 2 clusters), for M >= 256.
    // Per-SM throughput relative to the single-CTA 128 x 256 tile: each SM
    // stores and reads only half of the tile's B rows.  Measured on GB300:
    // 8192^3 E4M3 3607 vs 3399 TFLOP/s (1.06).  With one K block per stage
    // a pair tile cost about the same whatever its N (4096^3 E4M3,
    // interleaved: 45.6 / 45.7 / 53.4 / 61.3 / 70.3 us at BN 256 / 224 /
    // 192 / 160 / 128 over 4 / 4 / 5 / 6 / 7 waves): the per-K-block
    // barrier round trip set the pace, so the narrower widths' relative
    // rates were below their share of 256; two K blocks per stage raise
    // them (below).  A partial last wave whose tiles the kernel splits along
    // K (two to four K ranges per tile over idle pairs) counts as that
    // fraction of a wave.  Pairs are used when their estimate is no worse;
    // DG_2CTA=0 disables them, DG_2CTA=1 forces them for M >= 256.
    const bool pairs_off = kn.two_cta == 0;
    const bool pairs_forced = kn.two_cta == 1;
    if (!pairs_off && (!one_wave || pairs_forced) && M >= 256 && sm_count >= 2) {
        const int64_t pm = (M + 255) / 256;
        const int slots = sm_count / 2;
        const int pcand[5] = {256, 224, 192, 160, 128};
        // Narrower widths with two K blocks per stage (12 K blocks on):
        // 4096^3 E4M3, 4 / 4 / 5 / 6 / 7 rounds: 43.5 / 42.5 / 46.9 / 51.2 /
        // 58.0 us at BN 256 / 224 / 192 / 160 / 128.  The plans this moves
        // from single-CTA to pair tiles of the same width, measured (us,
        // single -> pair): 3072 x 2240 x 11008 54.07 -> 50.65, 512 x 5120 x
        // 11008 28.00 -> 26.04, 1536 x 7168 x 8192 62.14 -> 59.94, 768 x
        // 7168 x 4096 22.51 -> 21.61, FP16 256 x 11008 x 4096 23.37 ->
        // 23.05; 256 x 12288 x 8192 25.97 -> 26.48 and 1024 x 5120 x 2048
        // 13.76 -> 13.92 the other way.
        const bool pk2 = kn.pair_kps == 2 || (kn.pair_kps == 0 && kblocks >= 12);
        const double peff[5] = {1.06, 0.95, pk2 ? 0.92 : 0.83, pk2 ? 0.84 : 0.72, pk2 ? 0.68 : 0.58};
        int pbest = 256;
        double pcost = 0.0;
        for (int i = 0; i < 5; ++i) {
            const int bn = pcand[i];
            const int64_t pt = pm * ((N + bn - 1) / bn);
            const int64_t full = pt / slots, rem = pt % slots;
            const int64_t split = rem > 0 ? std::min<int64_t>(slots / rem, 4) : 0;
            double waves = static_cast<double>(full);
            if (rem > 0)
                waves += (kn.split_tail && split >= 2 && kblocks >= split)
                             ? 1.0 / static_cast<double>(split) : 1.0;
            const double cost = waves * bn / peff[i];
            if (i == 0 || cost < pcost) { pbest = bn; pcost = cost; }
        }
        {
            const int v = kn.force_block_n;
            if (v == 128 || v == 160 || v == 192 || v == 224 || v == 256) pbest = v;
        }
        if (pairs_forced || pcost <= best_cost) {
            const int64_t pt = pm * ((N + pbest - 1) / pbest);
            p->block_m = 256;
            p->block_n = pbest;
            // Two K blocks per stage from 12 K blocks on, as for single-CTA
            // tiles: fewer barrier round trips per K block.  Measured on GB300
            // (graph-replayed, us, one -> two): E4M3 4096^3 45.92 -> 43.58,
            // HGEMM 4096^3 83.14 -> 79.59, 4096 x 4096 x 8192 85.31 ->
            // 82.31, FP16 1024 x 4096 x 4096 25.82 -> 24.83; the 8192^3 bench
            // step's GEMM 0.304-0.307 -> 0.298-0.301 ms.  DG_PAIR_KPS=1|2
            // pins either (sweeps).
            const int pkps = kn.pair_kps != 0 ? kn.pair_kps : (kblocks >= 12 ? 2 : 1);
            p->block_k = (fp16_in ? 64 : 128) * pkps;
            p->stages = pair_stages(pbest, pkps);
            p->tiles = static_cast<int>(pt);
            p->grid = static_cast<int>(2 * (pt < slots ? pt : slots));
            p->smem_bytes = pair_smem_for(pbest, pkps);
        }
    }
}

Params make_params(const TcLaunch& L) {
    Params prm;
    prm.D = L.D;
    prm.M = L.M;
    prm.N = L.N;
    prm.K = L.K;
    prm.sa = L.sa;
    prm.sb = L.sb;
    prm.sd = L.sd;
    prm.out_kind = L.out_kind;
    prm.out_elem = L.out_elem;
    prm.vec_ok = ((static_cast<int64_t>(L.N) * L.out_elem) % 16 == 0) ? 1 : 0;
    prm.staged = prm.vec_ok && knobs().staged_epilogue ? 1 : 0;   // confirmed by the launcher
    prm.early_release = knobs().early_release ? 1 : 0;
    prm.tail_split = 1;   // set by the CTA-pair launcher when the tail is split
    prm.tail_ws = nullptr;
    prm.tail_counts = nullptr;
    prm.status = L.status;
    prm.timeout_ns = wait_timeout_ns();
    prm.skip_first_load = take_skip_first_load() ? 1 : 0;
    prm.amax_out = L.amax_out;
    // Raster: groups of 32 M-tiles when there are many (8192^3: 3361 vs 3285
    // TFLOP/s at 16, measured), 8 otherwise (4096^3: 2865 vs 2830).
    prm.group_m = ((L.M + kBM - 1) / kBM) >= 48 ? 32 : 8;
    if (L.plan->block_m == 256) prm.group_m /= 2;   // pair tiles are 256 rows
    // DG_GROUP_M=<n> overrides the raster group size (sweeps).
    if (knobs().group_m != 0) prm.group_m = knobs().group_m;
    prm.group_off = L.group_off;
    prm.groups = L.groups;
    prm.a_box_bytes = kBM * kBKBytes;   // the single-CTA launcher sets the edge boxes
    prm.b_box_bytes = L.plan->block_n * kBKBytes;
    prm.a_edge_bytes = prm.a_box_bytes;
    prm.b_edge_bytes = prm.b_box_bytes;
    prm.a_edge_row = INT_MAX;
    prm.b_edge_row = INT_MAX;
    return prm;
}

cudaError_t launch_gemm_tc(const TcLaunch& L, cudaStream_t s) {
    const Params prm = make_params(L);
    if (L.plan->block_m == 256) return launch_gemm_tc_pair(L, prm, s);
    return L.fp16_in ? launch_in<true>(L, prm, s) : launch_in<false>(L, prm, s);
}

cudaError_t launch_gemm_tc_grouped(const TcLaunch& L, cudaStream_t s) {
    if (L.fp16_in || L.groups < 1 || L.groups > kMaxGroups) return cudaErrorInvalidValue;
    const Params prm = make_params(L);
    if (L.plan->block_n == 128)
        return launch_cfg<128, stages_for(128, true), false, true>(L, prm, s);
    return launch_cfg<256, stages_for(256, true), false, true>(L, prm, s);
}

}  // namespace dg
