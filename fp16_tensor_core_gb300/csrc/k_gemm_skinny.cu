// k_gemm_skinny.cu -- the tensor-core path for skinny GEMMs (M <= 128 with
// few output tiles): split-K over every SM, with the operands swapped so that
// the long side fills the 128-row MMA.
//
// Page shorthands: [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南";
// [DG-FP16] = the DeepGEMM FP16/WMMA deep-dive page.
//
// For a decode-style product (a handful of activation rows against a large
// weight matrix) the weight B is read once and the work is bound by HBM
// ([DG-FP16] §2.1, weight-aware tiling).  A 128 x BN output tile with
// M <= 16 would leave 7/8 of each MMA empty and give N/BN tiles -- too few
// to occupy 152 SMs.  Here instead:
//  * operands are swapped: the MMA computes D^T = B * A^T, its M side (128)
//    is 128 rows of B and its N side (NC = 16, 32, 64 or 128) the M rows of
//    A rounded up, zero-filled by TMA past M ([FP8-guide] §3.3's edge
//    handling);
//  * the K blocks of all tiles form one sequence of `units` (tile, k block)
//    that is cut into gridDim.x equal contiguous ranges, one per CTA, so every
//    SM streams the same number of bytes (split-K, balanced);
//  * a CTA's range splits at tile boundaries into segments.  A segment that
//    covers a whole tile writes D directly; otherwise the CTA stores its FP32
//    partial tile in a workspace slot and bumps the tile's arrival counter,
//    and the CTA that arrives last adds the partials in segment order (fixed,
//    so the result does not depend on arrival order), applies
//    scale_A * scale_B (/ scale_D for E4M3 out, [FP8-guide] §3.2), stores D
//    and resets the counter to zero.  No CTA waits for another.
// Pipeline: one TMA thread, one MMA thread, four epilogue warps, a ring of
// K blocks (16 KB of B + NC x 128 bytes of A each; 12 of them for NC = 16,
// 6 for NC = 128; 1 or 2 blocks per stage) and two NC-column accumulators in
// tensor memory.  Partial tiles are kept as FP32 column quads (16 bytes per
// row and 4 columns).  The finishing CTA adds them in segment order: from its
// idle ring, bulk-copied there, when the tile is its last segment and they
// fit, else four segments' quads at a time from L2; for its last tile, warps
// 0-3 (done with their own roles) take the odd 16-column chunks.  With at
// least two CTAs per tile the grid is a whole multiple of the tile count.
// Row ranges (DG_SPLITK_ROWS=1): when N fits 128 rows per SM, a tile may
// instead be a range of tile_rows = ceil(N / SMs) rows, one CTA per range
// over the whole of K (grid = tiles): every SM streams the same share of B
// with no tile split, so no partial tile, workspace or finishing pass.  TMA
// loads tile_rows rows of B per K block; the MMA still spans 128 rows, and
// the accumulator rows past tile_rows (stale shared memory) are never
// stored.  Measured on GB300 no faster than 128-row tiles at the decode QKV
// shape (16 x 12288 x 4096: 11.48 against 11.58 us) and much slower for
// short ranges over a long K (16 x 4096 x 11008, 27 rows per CTA: 22.1
// against 11.2 us, too few bytes per box in flight), so not the default.
// Launch overlap: before its
// dependency wait a CTA prefetches its first ring of B into L2, and right
// after it the grid lets the next kernel take over SMs as CTAs exit, so the
// start-up of one launch hides in the straggling tail of the one before.
// All mbarrier waits are bounded as in the other GEMMs.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "dg_internal.h"
#include "dg_ptx.cuh"
#include "gemm_common.cuh"

namespace dg {
namespace {

constexpr int kRows = kSkinnyTileRows;            // MMA M: rows of B per tile
constexpr int kWBytes = kRows * kBKBytes;         // 16 KB of B per K block
constexpr int kBarBytes = 512;
constexpr uint32_t kEpiBar = 1;                   // named barrier of the epilogue warps
constexpr uint32_t kEpiThreads = 128;
// Hand-off to warps 0-3 for a CTA's last tile: valid, tile, accumulator,
// first and last CTA of the tile, the first CTA's slot, staged.
constexpr int kHelpInts = 7;

// K blocks in flight per CTA for MMA N = nc (the rows of A, padded): as many
// as fit in 227 KB of shared memory, rounded down to an even number.
constexpr int ring_kblocks(int nc) {
    const int r = (kSmemLimit - 1024 - kBarBytes) / (kWBytes + nc * kBKBytes);
    const int even = r & ~1;
    return even > 12 ? 12 : even;
}

// Configuration for MMA N = NC (16, 32, 64 or 128 rows of A) with KPS
// consecutive K blocks per stage, loaded together so that each row of B is
// requested KPS x 128 contiguous bytes at a time.
template <int NC, int KPS>
struct SkCfg {
    static constexpr int kXBytes = NC * kBKBytes;           // A rows per K block
    static constexpr int kKBBytes = kWBytes + kXBytes;
    static constexpr int kRing = ring_kblocks(NC);
    static constexpr int kStages = kRing / KPS;
    static constexpr int kStageW = KPS * kWBytes;
    static constexpr int kStageX = KPS * kXBytes;
    static constexpr int kSmemBytes = 1024 + kRing * kKBBytes + kBarBytes;
    static constexpr uint32_t kTmemCols = pow2_at_least(2 * NC);   // two accumulators
    static constexpr uint32_t kIdesc = idesc_f32acc(kRows, NC, 0, 0);
    static_assert(NC % 16 == 0 && NC >= 16 && NC <= kSplitkMaxCols, "MMA N");
    static_assert(kRing % KPS == 0 && kStages <= 12, "ring");
    static_assert(kSmemBytes <= kSmemLimit, "shared memory");
    static_assert(kXBytes % 1024 == 0, "1024-byte aligned A blocks (128-byte swizzle atoms)");
    // barriers: full/empty per stage, 2 + 2 accumulator, drain, fix-up,
    // helpers; then the TMEM address, the abort flag, the last-arrival flag
    // and the helpers' hand-off block
    static_assert((2 * kStages + 7) * 8 + 3 * 4 + kHelpInts * 4 <= kBarBytes, "barrier block");
};

struct SkParams {
    void* D;
    int M, N, K;
    const float* sa;
    const float* sb;
    const float* sd;
    int out_kind;
    uint32_t* status;
    uint64_t timeout_ns;
    int skip_first_load;
    uint32_t* amax_out;
    float* partials;       // [2 * gridDim.x][NC / 4][128] float4: column quads
    uint32_t* counts;      // [tiles]
    int tiles;             // ceil(N / tile_rows)
    int tile_rows;         // rows of B per tile: 128, or a row range (<= 128)
    int kblocks;           // ceil(K / BK)
    int prefetch_kblocks;  // B boxes of its range a CTA moves into L2 up front
};

// CTA i's range of units is [range_start(i), range_start(i + 1)).
__device__ __forceinline__ int64_t range_start(int i, int G, int64_t units) {
    return static_cast<int64_t>(i) * units / G;
}

// The CTA whose range holds unit u.
__device__ __forceinline__ int cta_of_unit(int64_t u, int G, int64_t units) {
    return static_cast<int>(((u + 1) * G - 1) / units);
}

// Workspace slots: a CTA has at most two partial segments, its first (slot
// 2c) and its last (2c + 1).  In a split tile t, every CTA after the first
// one (c_first) starts its range inside t, so its segment there is its first
// (slot 2c); c_first's segment is its first only if its range starts exactly
// at the tile.

// Scale, convert and store rows c0 .. c0 + jn - 1 of A's side (m) at column
// n: one branch on the output type, then one strided store per row.
__device__ __forceinline__ void store_chunk16(const SkParams& p, int c0, int n, int jn,
                                              const float (&v)[16], float alpha) {
    const int64_t ld = p.N;
    const int64_t off = static_cast<int64_t>(c0) * ld + n;
    if (p.out_kind == kOutE4M3) {
        uint8_t* d = static_cast<uint8_t*>(p.D) + off;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < jn) d[j * ld] = static_cast<uint8_t>(f32x2_to_e4m3x2(v[j] * alpha, 0.0f) & 0xFFu);
    } else if (p.out_kind == kOutFP16) {
        uint16_t* d = static_cast<uint16_t*>(p.D) + off;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < jn) d[j * ld] = static_cast<uint16_t>(f32x2_to_f16x2(v[j] * alpha, 0.0f) & 0xFFFFu);
    } else {
        uint16_t* d = static_cast<uint16_t*>(p.D) + off;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (j < jn) d[j * ld] = static_cast<uint16_t>(f32x2_to_bf16x2(v[j] * alpha, 0.0f) & 0xFFFFu);
    }
}

// Adds up, scales and stores the 16-column chunks c0 = c0_begin,
// c0_begin + c0_step, ... (c0 < NC, c0 < M) of a finished tile for the
// calling thread's row r (its tensor-memory lane): the segments c_first ..
// c_last in that order, the own one (CTA me) from tensor memory, the others
// from the staged copies in shared memory or from their workspace slots.
// `first` holds chunk 0 when the CTA published its own partial.
template <int NC>
__device__ __forceinline__ void finish_chunks(const SkParams& p, uint8_t* smem, uint32_t tacc,
                                              int r, int n, int c0_begin, int c0_step, int me,
                                              int c_first, int c_last, int first_slot,
                                              bool staged, int quads, const float (&first)[16],
                                              float alpha, uint32_t& amax_bits) {
    const int others = c_last - c_first;
#pragma unroll 1
    for (int c0 = c0_begin; c0 < NC && c0 < p.M; c0 += c0_step) {
        float v[16];
        if (c_last > c_first && c0 == 0) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = first[j];
        } else {
            uint32_t raw[16];
            __syncwarp();
            tmem_load_16cols(tacc + static_cast<uint32_t>(c0), raw);
            tmem_load_wait(raw);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(raw[j]);
        }
        if (staged) {
            // Segments in order c_first .. c_last from the staged
            // copies, the own one written into its position first
            // (this thread reads back only what it wrote itself).
            float4* stage = reinterpret_cast<float4*>(smem) + (c0 >> 2) * kRows + r;
            const int seg_stride = quads * kRows;   // float4s per position
            float4* own = stage + (me - c_first) * seg_stride;
#pragma unroll
            for (int g = 0; g < 4; ++g)
                if (c0 + 4 * g < p.M)
                    own[g * kRows] = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2],
                                                 v[4 * g + 3]);
            float4 sum[4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                sum[g] = c0 + 4 * g < p.M ? stage[g * kRows]
                                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll 1
            for (int i = 1; i <= others; ++i) {
                const float4* w = stage + i * seg_stride;
#pragma unroll
                for (int g = 0; g < 4; ++g) {
                    if (c0 + 4 * g < p.M) {
                        const float4 x = w[g * kRows];
                        sum[g].x += x.x;
                        sum[g].y += x.y;
                        sum[g].z += x.z;
                        sum[g].w += x.w;
                    }
                }
            }
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                v[4 * g] = sum[g].x;
                v[4 * g + 1] = sum[g].y;
                v[4 * g + 2] = sum[g].z;
                v[4 * g + 3] = sum[g].w;
            }
        } else if (c_last > c_first) {
            // Sum the segments in order c_first .. c_last, the own
            // one from tensor memory, the others from their slots.
            // The slots of four segments are requested together
            // and then added in order, so the order (and the
            // result) is fixed while four loads are in flight.
            float sum[16];
#pragma unroll 1
            for (int cb = c_first; cb <= c_last; cb += 4) {
                float4 x[4][4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = cb + i;
                    const int slot = c == c_first ? first_slot : 2 * c;
                    const float4* w = reinterpret_cast<const float4*>(p.partials) +
                                      static_cast<int64_t>(slot) * (NC / 4) * kRows;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        x[i][g] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                        if (c <= c_last && c != me && c0 + 4 * g < p.M)
                            x[i][g] = __ldcg(w + ((c0 >> 2) + g) * kRows + r);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int c = cb + i;
                    if (c > c_last) break;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        float y[4] = {x[i][g].x, x[i][g].y, x[i][g].z, x[i][g].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int j = 4 * g + e;
                            const float val = c == me ? v[j] : y[e];
                            sum[j] = c == c_first ? val : sum[j] + val;
                        }
                    }
                }
            }
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = sum[j];
        }
        if (r < p.tile_rows && n < p.N) {
            const int jn = min(16, p.M - c0);   // rows of A in this chunk
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (j < jn) amax_bits = max(amax_bits, __float_as_uint(v[j]) & 0x7FFFFFFFu);
            store_chunk16(p, c0, n, jn, v, alpha);
        }
    }
}

template <bool kFp16In, int KPS, int NC>
__global__ void __launch_bounds__(kThreads, 1)
gemm_skinny_kernel(const __grid_constant__ CUtensorMap tmap_w,
                   const __grid_constant__ CUtensorMap tmap_x, const SkParams p) {
    constexpr int kBK = kFp16In ? 64 : 128;   // K elements per K block
    using C = SkCfg<NC, KPS>;
    constexpr int kStages = C::kStages;
    constexpr int kRingKBlocks = C::kRing;
    constexpr int kKBBytes = C::kKBBytes;
    constexpr int kXBytes = C::kXBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sW = smem;                          // B rows (MMA operand A)
    uint8_t* sX = smem + kStages * C::kStageW;   // A rows (MMA operand B)
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRingKBlocks * kKBBytes);
    uint64_t* empty = full + kStages;
    uint64_t* acc_full = empty + kStages;   // [2]
    uint64_t* acc_empty = acc_full + 2;     // [2]
    uint64_t* drain = acc_empty + 2;        // [1]
    uint64_t* fix_bar = drain + 1;          // [1] partial tiles staged for the fix-up
    uint64_t* help_bar = fix_bar + 1;       // [1] last tile handed to warps 0-3
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(help_bar + 1);
    int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
    volatile int* last_flag = abort_flag + 1;
    volatile int* help = last_flag + 1;     // [kHelpInts]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4);
        }
        mbar_init(drain, 1);
        mbar_init(fix_bar, 1);
        mbar_init(help_bar, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmap_w);
        tma_prefetch_desc(&tmap_x);
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
    const int G = gridDim.x;
    const int KB = p.kblocks;
    const int64_t units = static_cast<int64_t>(p.tiles) * KB;
    const int64_t u_begin = range_start(blockIdx.x, G, units);
    const int64_t n_units = range_start(blockIdx.x + 1, G, units) - u_begin;
    const int t_begin = static_cast<int>(u_begin / KB);
    const int kb_begin = static_cast<int>(u_begin - static_cast<int64_t>(t_begin) * KB);

    if (warp == 0 && lane == 0) {
        // Warm L2 with the start of this CTA's range of B while the preceding
        // kernel finishes (a prefetch only moves lines into L2).
        int t = t_begin, kb = kb_begin;
        for (int i = 0; i < p.prefetch_kblocks && i < n_units; ++i) {
            tma_prefetch_l2_2d(&tmap_w, kb * kBK, t * p.tile_rows);
            if (++kb == KB) { kb = 0; ++t; }
        }
    }
    pdl_wait();   // the prologue above overlaps the preceding kernel's tail
    // The next kernel may now take over each SM as soon as this grid's CTA
    // on it exits; it waits for the whole grid before touching memory.
    pdl_launch_dependents();

    // Every role walks the same segments: tile t from K block kb0 to kb_end.
    if (warp == 0 && lane == 0) {
        // ------------------------------------------------ TMA producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_mask = 0;
        uint32_t issued_phase = 0;
        bool skip = p.skip_first_load != 0 && blockIdx.x == 0;
        bool ok = true;
        bool first_lap = true;   // every stage starts free: no wait on the first lap
        // bytes of one K block: tile_rows rows of B (the box) and NC rows of A
        const uint32_t kb_bytes = static_cast<uint32_t>(p.tile_rows * kBKBytes + kXBytes);
        int t = t_begin, kb0 = kb_begin;
        for (int64_t left = n_units; left > 0 && ok; ++t, kb0 = 0) {
            const int kb_end = static_cast<int>(min(static_cast<int64_t>(KB), kb0 + left));
            left -= kb_end - kb0;
            for (int kb = kb0; kb < kb_end; kb += KPS) {
                const int nk = min(KPS, kb_end - kb);
                if (!first_lap && !wait_bounded(&empty[stage], phase ^ 1u, ctl)) { ok = false; break; }
                if (skip) {
                    skip = false;   // leave this stage unloaded
                } else {
                    mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(nk) * kb_bytes);
#pragma unroll
                    for (int i = 0; i < KPS; ++i) {
                        if (i < nk) {
                            tma_load_2d(sW + stage * C::kStageW + i * kWBytes, &tmap_w, &full[stage],
                                        (kb + i) * kBK, t * p.tile_rows);
                            tma_load_2d(sX + stage * C::kStageX + i * kXBytes, &tmap_x, &full[stage],
                                        (kb + i) * kBK, 0);
                        }
                    }
                    issued_mask |= 1u << stage;
                    issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
                }
                if (++stage == kStages) { stage = 0; phase ^= 1u; first_lap = false; }
            }
        }
        // Let every issued copy land before the CTA exits (immediate after a
        // normal run; after an abort, copies still in flight finish).
        for (int s = 0; s < kStages; ++s)
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
        int kb0 = kb_begin;
        for (int64_t left = n_units; left > 0 && ok; kb0 = 0) {
            const int kb_end = static_cast<int>(min(static_cast<int64_t>(KB), kb0 + left));
            left -= kb_end - kb0;
            if (!wait_bounded(&acc_empty[acc], acc_phase ^ 1u, ctl)) break;
            tc_fence_after_sync();
            const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NC);
            for (int kb = kb0; kb < kb_end; kb += KPS) {
                const int nk = min(KPS, kb_end - kb);
                if (!wait_bounded(&full[stage], phase, ctl)) { ok = false; break; }
                tc_fence_after_sync();
#pragma unroll
                for (int i = 0; i < KPS; ++i) {
                    if (i < nk) {
                        const uint32_t a0 = smem_addr(sW + stage * C::kStageW + i * kWBytes);
                        const uint32_t b0 = smem_addr(sX + stage * C::kStageX + i * kXBytes);
#pragma unroll
                        for (int kk = 0; kk < kBKBytes / 32; ++kk) {
                            const uint64_t ad = sdesc_k_major_sw128(a0 + kk * 32);
                            const uint64_t bd = sdesc_k_major_sw128(b0 + kk * 32);
                            const uint32_t accum = (kb > kb0 || i > 0 || kk > 0) ? 1u : 0u;
                            if constexpr (kFp16In)
                                mma_f16(d_tmem, ad, bd, C::kIdesc, accum);
                            else
                                mma_f8f6f4(d_tmem, ad, bd, C::kIdesc, accum);
                        }
                    }
                }
                issued_any = true;
                mma_commit(&empty[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            mma_commit(&acc_full[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
        }
        if (issued_any) {
            mma_commit(drain);
            wait_bounded(drain, 0, ctl, false);
        }
    } else if (warp >= 4) {
        // ------------------------------------------------ epilogue
        // Thread (q, lane) owns row r = 32 q + lane of each tile (its tensor-
        // memory lane) and that row's 16 accumulator columns, one per row of A.
        const int q = warp & 3;
        const int r = q * 32 + lane;
        const int me = static_cast<int>(blockIdx.x);
        float ab = 1.0f;
        if (p.sa != nullptr) ab = p.sa[0] * p.sb[0];
        const float alpha = p.out_kind == kOutE4M3 ? __fdiv_rn(ab, p.sd[0]) : ab;
        uint32_t amax_bits = 0u;
        bool released = false;   // the last tile handed to warps 0-3 (thread 128)
        int acc = 0;
        uint32_t acc_phase = 0;
        int t = t_begin, kb0 = kb_begin;
        for (int64_t left = n_units; left > 0; ++t, kb0 = 0) {
            const int kb_end = static_cast<int>(min(static_cast<int64_t>(KB), kb0 + left));
            left -= kb_end - kb0;
            // Which CTAs share tile t, and their slots (before the wait).
            const int64_t tile_u0 = static_cast<int64_t>(t) * KB;
            const int c_first = cta_of_unit(tile_u0, G, units);
            const int c_last = cta_of_unit(tile_u0 + KB - 1, G, units);
            const int first_slot =
                range_start(c_first, G, units) == tile_u0 ? 2 * c_first : 2 * c_first + 1;
            // The four warps continue or leave together (named barriers below).
            const bool got = wait_bounded(&acc_full[acc], acc_phase, ctl);
            if (!named_bar_and(kEpiBar, kEpiThreads, got)) break;
            tc_fence_after_sync();
            // Columns [c0, c0 + 16) of this row's accumulator, 16 at a time;
            // only chunks that hold rows of A (c0 < M) are read.
            const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                  static_cast<uint32_t>(acc * NC);
            const int n = t * p.tile_rows + r;
            float first[16];   // chunk 0, kept from the partial pass
            bool finish = true;
            int my_slot = 0;
            if (c_last > c_first) {
                // Split tile: publish this partial, count the arrival.
                my_slot = me == c_first ? first_slot : 2 * me;
                float4* ws = reinterpret_cast<float4*>(p.partials) +
                             static_cast<int64_t>(my_slot) * (NC / 4) * kRows;
#pragma unroll 1
                for (int c0 = 0; c0 < NC && c0 < p.M; c0 += 16) {
                    uint32_t raw[16];
                    __syncwarp();
                    tmem_load_16cols(tacc + static_cast<uint32_t>(c0), raw);
                    tmem_load_wait(raw);
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (c0 == 0) first[j] = __uint_as_float(raw[j]);
                    }
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        if (c0 + 4 * g < p.M)
                            __stcg(ws + ((c0 >> 2) + g) * kRows + r,
                                   make_float4(__uint_as_float(raw[4 * g]), __uint_as_float(raw[4 * g + 1]),
                                               __uint_as_float(raw[4 * g + 2]),
                                               __uint_as_float(raw[4 * g + 3])));
                    }
                }
                named_bar_sync(kEpiBar, kEpiThreads);
                if (threadIdx.x == 4 * 32) {
                    const uint32_t old = atom_add_acq_rel_gpu(&p.counts[t], 1u);
                    const bool last = old == static_cast<uint32_t>(c_last - c_first);
                    if (last) atomicExch(&p.counts[t], 0u);   // zero for the next launch
                    *last_flag = last ? 1 : 0;
                }
                named_bar_sync(kEpiBar, kEpiThreads);
                finish = *last_flag != 0;
            }
            // When this is the CTA's last segment its ring of K blocks is idle:
            // one thread bulk-copies every other segment's partial tile into
            // it on one barrier, and the sum below reads shared memory instead
            // of making L2 round trips for each 16 columns and each four
            // segments.  At NC = 16 with at most three other segments (one
            // chunk, one group of direct loads) the loads measured as fast.
            const int others = c_last - c_first;
            const int quads = (min(p.M, NC) + 3) >> 2;   // column quads that hold rows of A
            const uint32_t slot_bytes = static_cast<uint32_t>(quads) * kRows * 16u;
            const bool staged = (NC >= 32 || others >= 4) && finish && others > 0 && left == 0 &&
                                static_cast<int64_t>(others + 1) * slot_bytes <=
                                    static_cast<int64_t>(kRingKBlocks) * kKBBytes;
            if (staged) {
                if (threadIdx.x == 4 * 32) {
                    // the partials were published through the generic proxy
                    // and acquired by this thread's arrival atomic
                    fence_proxy_async_global();
                    mbar_arrive_expect_tx(fix_bar, static_cast<uint32_t>(others) * slot_bytes);
                    // segment c goes to position c - c_first; the own position
                    // is filled from tensor memory below
                    for (int c = c_first; c <= c_last; ++c) {
                        if (c == me) continue;
                        const int slot = c == c_first ? first_slot : 2 * c;
                        bulk_load_g2s(smem + static_cast<uint32_t>(c - c_first) * slot_bytes,
                                      reinterpret_cast<const float4*>(p.partials) +
                                          static_cast<int64_t>(slot) * (NC / 4) * kRows,
                                      slot_bytes, fix_bar);
                    }
                }
                const bool landed = wait_bounded(fix_bar, 0, ctl);
                if (!named_bar_and(kEpiBar, kEpiThreads, landed)) {
                    // let the copies land before the CTA's shared memory is released
                    if (threadIdx.x == 4 * 32) wait_bounded(fix_bar, 0, ctl, false);
                    break;
                }
            }
            // The CTA's last tile: with more than one chunk, warps 0-3 (idle
            // by now, each reading the same tensor-memory lanes as its twin
            // among warps 4-7) take the odd chunks.  The hand-off is an
            // mbarrier with bounded waits, released on every exit path.
            const bool helped = NC >= 32 && finish && left == 0;
            if (left == 0 && threadIdx.x == 4 * 32) {
                help[1] = t;
                help[2] = acc;
                help[3] = c_first;
                help[4] = c_last;
                help[5] = first_slot;
                help[6] = staged ? 1 : 0;
                help[0] = helped ? 1 : 0;
                mbar_arrive(help_bar);
                released = true;
            }
            if (finish)
                finish_chunks<NC>(p, smem, tacc, r, n, 0, helped ? 32 : 16, me, c_first, c_last,
                                  first_slot, staged, quads, first, alpha, amax_bits);
            // The accumulator is free once every chunk has been read.
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[acc]);
            if (++acc == 2) { acc = 0; acc_phase ^= 1u; }
            (void)my_slot;
        }
        // Every exit (including a timed-out wait) releases warps 0-3.
        if (threadIdx.x == 4 * 32 && !released) {
            help[0] = 0;
            mbar_arrive(help_bar);
        }
        // max |sa*sb*acc| of this warp's stored outputs (monotone rounding:
        // fl(max|acc| * c) is the exact maximum of fl(|acc| * c)).
        if (p.amax_out != nullptr) {
            __syncwarp();
            const uint32_t bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
            if (lane == 0 && bits != 0u)
                atomicMax(p.amax_out, __float_as_uint(__uint_as_float(bits) * ab) & 0x7FFFFFFFu);
        }
    }
    if constexpr (NC >= 32) {
        if (warp < 4) {
            // ------------------------------------------------ helpers
            // Warps 0-3, once their own roles are done, take the odd
            // 16-column chunks of the CTA's last tile when it finishes one.
            __syncwarp();
            const bool go = wait_bounded(help_bar, 0, ctl) && help[0] != 0;
            if (__all_sync(0xFFFFFFFFu, go)) {
                const int t = help[1], acc = help[2], c_first = help[3], c_last = help[4];
                const int first_slot = help[5];
                const bool staged = help[6] != 0;
                tc_fence_after_sync();
                const bool landed = !staged || wait_bounded(fix_bar, 0, ctl);
                if (__all_sync(0xFFFFFFFFu, landed)) {
                    const int q = warp;   // the same tensor-memory lanes as warp q + 4
                    const int r = q * 32 + lane;
                    const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                          static_cast<uint32_t>(acc * NC);
                    float ab = 1.0f;
                    if (p.sa != nullptr) ab = p.sa[0] * p.sb[0];
                    const float alpha = p.out_kind == kOutE4M3 ? __fdiv_rn(ab, p.sd[0]) : ab;
                    const int quads = (min(p.M, NC) + 3) >> 2;
                    const float none[16] = {};   // chunk 0 is not among the odd ones
                    uint32_t amax_bits = 0u;
                    finish_chunks<NC>(p, smem, tacc, r, t * p.tile_rows + r, 16, 32,
                                      static_cast<int>(blockIdx.x), c_first, c_last, first_slot,
                                      staged, quads, none, alpha, amax_bits);
                    if (p.amax_out != nullptr) {
                        __syncwarp();
                        const uint32_t bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
                        if (lane == 0 && bits != 0u)
                            atomicMax(p.amax_out,
                                      __float_as_uint(__uint_as_float(bits) * ab) & 0x7FFFFFFFu);
                    }
                }
            }
        }
    }

    // Warps whose lane 0 ran a role alone may arrive diverged: the barrier
    // before tensor memory is freed is the non-aligned one.
    tc_fence_before_sync();
    cta_sync_diverged();
    tc_fence_after_sync();
    if (warp == 2) tmem_dealloc<C::kTmemCols>(tmem_base);
}

// ------------------------------------------------------------- host side

// B boxes each CTA prefetches into L2 before its dependency wait:
// DG_SPLITK_PREFETCH=n (sweeps, 0..256), default one ring.
int splitk_prefetch_kblocks(int ring) {
    const int n = knobs().splitk_prefetch;
    return n >= 0 ? n : ring;
}

template <bool kFp16In, int KPS, int NC>
cudaError_t launch_sk(const TcLaunch& L, float* partials, uint32_t* counts, cudaStream_t s) {
    using C = SkCfg<NC, KPS>;
    static std::mutex mu;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        if (!attr_done[dev]) {
            e = cudaFuncSetAttribute(gemm_skinny_kernel<kFp16In, KPS, NC>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
            if (e != cudaSuccess) return e;
            attr_done[dev] = true;
        }
    }
    CUtensorMap tw, tx;
    const int tile_rows = L.plan->block_n;
    if (!make_map(&tw, L.B, L.N, L.K, kFp16In, tile_rows) ||
        !make_map(&tx, L.A, L.M, L.K, kFp16In, NC))
        return cudaErrorInvalidValue;
    SkParams prm;
    prm.D = L.D;
    prm.M = L.M;
    prm.N = L.N;
    prm.K = L.K;
    prm.sa = L.sa;
    prm.sb = L.sb;
    prm.sd = L.sd;
    prm.out_kind = L.out_kind;
    prm.status = L.status;
    prm.timeout_ns = wait_timeout_ns();
    prm.skip_first_load = take_skip_first_load() ? 1 : 0;
    prm.amax_out = L.amax_out;
    prm.partials = partials;
    prm.counts = counts;
    prm.tiles = L.plan->tiles;
    prm.tile_rows = tile_rows;
    const int bk = kFp16In ? 64 : 128;
    prm.kblocks = (L.K + bk - 1) / bk;
    prm.prefetch_kblocks = splitk_prefetch_kblocks(C::kRing);
    return launch_kernel(gemm_skinny_kernel<kFp16In, KPS, NC>, dim3(L.plan->grid), dim3(kThreads),
                         C::kSmemBytes, s, tw, tx, prm);
}

// K blocks per stage: DG_SPLITK_KPS=1|2 (sweeps), default 2.
int splitk_kps() { return knobs().splitk_kps; }

// MMA N for M rows of A: M rounded up to 16, 32, 64 or 128.
int nc_for(int64_t M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : 128; }

int smem_for_nc(int nc) {
    switch (nc) {
        case 16: return SkCfg<16, 2>::kSmemBytes;
        case 32: return SkCfg<32, 2>::kSmemBytes;
        case 64: return SkCfg<64, 2>::kSmemBytes;
        default: return SkCfg<128, 2>::kSmemBytes;
    }
}

template <bool kFp16In, int NC>
cudaError_t launch_nc(const TcLaunch& L, float* partials, uint32_t* counts, cudaStream_t s) {
    if (SkCfg<NC, 1>::kRing == L.plan->stages)
        return launch_sk<kFp16In, 1, NC>(L, partials, counts, s);
    return launch_sk<kFp16In, 2, NC>(L, partials, counts, s);
}

template <bool kFp16In>
cudaError_t launch_in(const TcLaunch& L, float* partials, uint32_t* counts, cudaStream_t s) {
    switch (nc_for(L.M)) {
        case 16: return launch_nc<kFp16In, 16>(L, partials, counts, s);
        case 32: return launch_nc<kFp16In, 32>(L, partials, counts, s);
        case 64: return launch_nc<kFp16In, 64>(L, partials, counts, s);
        default: return launch_nc<kFp16In, 128>(L, partials, counts, s);
    }
}

}  // namespace

void plan_skinny(int64_t M, int64_t N, int64_t K, bool fp16_in, int sm_count, dg_plan* p) {
    const int bk = fp16_in ? 64 : 128;
    const int nc = nc_for(M);
    // rows of B per tile: 128, or DG_SPLITK_TILE_ROWS (sweeps; the MMA still
    // spans 128 rows and the rows past the tile are not stored)
    const int tile_rows = knobs().splitk_tile_rows;
    const int64_t tiles = (N + tile_rows - 1) / tile_rows;
    const int64_t units = tiles * ((K + bk - 1) / bk);
    p->block_m = nc;
    p->block_n = tile_rows;
    p->block_k = bk;
    p->stages = ring_kblocks(nc) / splitk_kps();
    // Row ranges (see the file comment): N within 128 rows per SM.
    const int64_t range = (N + sm_count - 1) / sm_count;
    const int rows_knob = knobs().splitk_rows;
    if (range <= kRows && knobs().splitk_grid == 0 && rows_knob == 1) {
        p->block_n = static_cast<int>(range);
        p->tiles = static_cast<int>((N + range - 1) / range);
        p->grid = p->tiles;
        p->smem_bytes = smem_for_nc(nc);
        return;
    }
    p->tiles = static_cast<int>(tiles);
    // With room for at least two CTAs per tile, launch a whole multiple of
    // the tile count, so every CTA covers the same fraction of one tile (one
    // segment each, the same number of segments in every tile); otherwise
    // every SM, with ranges that cross tile edges.
    const int64_t per_tile = sm_count / tiles;
    const int64_t g = per_tile >= 2 ? per_tile * tiles : sm_count;
    p->grid = static_cast<int>(units < g ? units : g);
    if (const int64_t g = knobs().splitk_grid) {   // sweeps: CTAs per launch
        if (g <= sm_count && g <= units) p->grid = static_cast<int>(g);
    }
    p->smem_bytes = smem_for_nc(nc);
}

cudaError_t launch_gemm_skinny(const TcLaunch& L, float* partials, uint32_t* counts, int max_cols,
                               cudaStream_t s) {
    const int rows = L.plan->block_n;
    if (L.M < 1 || L.M > kSplitkMaxCols || nc_for(L.M) > max_cols || rows < 1 || rows > kRows ||
        L.plan->tiles > kSkinnyMaxTiles ||
        static_cast<int64_t>(L.plan->tiles) * rows < L.N)
        return cudaErrorInvalidValue;
    // Tiles may be split over CTAs (workspace needed) unless there is one CTA
    // per tile (grid = tiles: each CTA's range is exactly one tile).
    if (L.plan->grid != L.plan->tiles && (partials == nullptr || counts == nullptr))
        return cudaErrorInvalidValue;
    return L.fp16_in ? launch_in<true>(L, partials, counts, s)
                     : launch_in<false>(L, partials, counts, s);
}

}  // namespace dg
