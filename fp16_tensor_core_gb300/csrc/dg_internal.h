// dg_internal.h -- declarations shared by the library's translation units.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "dg.h"

namespace dg {

enum OutKind : int { kOutBF16 = 0, kOutE4M3 = 1, kOutFP16 = 2 };

inline int out_kind_of(dg_dtype t) {
    return t == DG_E4M3 ? kOutE4M3 : (t == DG_FP16 ? kOutFP16 : kOutBF16);
}
inline int elem_bytes(dg_dtype t) { return t == DG_E4M3 ? 1 : 2; }

// Split-K path for skinny GEMMs: 128 rows of B per tile, the M rows of A
// padded to MMA N = 16, 32, 64 or 128, K blocks of every tile spread evenly
// over the SMs.  Always used for M <= 16 (past the GEMV); for M <= 128 when
// the tiled kernels would leave SMs idle.
constexpr int kSkinnyMaxM = 16;
constexpr int kSplitkMaxCols = 128;
constexpr int kSkinnyTileRows = 128;
constexpr int kSkinnyMaxTiles = 8192;   // N <= 1,048,576

// Per-device state, created once per device on first use.
struct DeviceState {
    int device = -1;
    int sm_count = 0;
    uint32_t* status = nullptr;  // device status word (kStatus* bits)
    // Split-K workspace: two FP32 partial-tile slots of 128 x 128 per SM and
    // one arrival counter per tile (all zero between launches).
    float* splitk_partials = nullptr;
    uint32_t* splitk_counts = nullptr;
};

// Returns the current device's state, creating it on first use.
dg_status current_device_state(DeviceState** out);

// Tuning and diagnostic switches taken from DG_* environment variables.
// They are read once, on first use, and again only by dg_reload_env(); the
// per-call path reads this snapshot and never the environment.
struct Knobs {
    bool pdl = true;            // DG_PDL=0: no programmatic dependent launch
    bool log = false;           // DG_LOG=1: one stderr line per GEMM call
    int gemv_max_m = 2;         // DG_GEMV_MAX_M (0..16): largest M on the GEMV
    int gemv_rows = 0;          // DG_GEMV_ROWS (4, 8, 16): GEMV rows of B per CTA, M <= 2
    int splitk = -1;            // DG_SPLITK: 0 off, 1 for every M <= 128, else planned
    int splitk_grid = 0;        // DG_SPLITK_GRID: CTAs of a split-K launch
    int splitk_prefetch = -1;   // DG_SPLITK_PREFETCH (0..256): B boxes moved into L2 early
    int splitk_kps = 2;         // DG_SPLITK_KPS (1, 2): K blocks per split-K stage
    bool one_wave = true;       // DG_ONE_WAVE=0: no one-wave tile rule
    int64_t one_wave_kb = 64;   // DG_ONE_WAVE_KB: K-block limit of that rule
    int force_block_n = 0;      // DG_FORCE_BLOCK_N: tile width of the tiled kernels
    int two_cta = -1;           // DG_2CTA: 0 no CTA pairs, 1 pairs for every M >= 256
    int group_m = 0;            // DG_GROUP_M (1..4096): raster group of M tiles
    int mma_gemv = -1;          // DG_MMA_GEMV: 0 off, 1 for every M <= 16, else planned
    int mma_gemv_warps = 0;     // DG_MMA_GEMV_WARPS (2, 3, 4, 8): warps per CTA of that path
    bool staged_epilogue = true;  // DG_STAGED_EPI=0: tiled epilogues store rows directly
    bool split_tail = false;      // DG_SPLIT_TAIL=1: CTA pairs split a partial last wave along K
    // DG_STREAM_K=1: CTA pairs take equal ranges of (tile, K block) units
    bool stream_k = false;
    bool early_release = true;    // DG_EARLY_RELEASE=0: tiled kernels release the next one at exit
    // DG_SPLITK_ROWS=1: split-K plans take row ranges (one CTA per
    // ceil(N / SMs) rows of B over the whole of K, no split, no workspace)
    // wherever they fit; default 128-row tiles.
    int splitk_rows = 0;
    int splitk_tile_rows = 128;   // DG_SPLITK_TILE_ROWS=<16..128, multiple of 8> (sweeps)
    int tc_short_box = 2;         // DG_TC_SHORT_BOX (0, 1, 2): box rows of short operands
    int tc_kps = 0;               // DG_TC_KPS (1, 2; 0 planned): K blocks per stage, one-wave tiles
    int pair_kps = 0;             // DG_PAIR_KPS (1, 2; 0 planned): K blocks per stage, CTA pairs
};
const Knobs& knobs();

// Whether launches use programmatic dependent launch (knobs().pdl).
inline bool pdl_enabled() { return knobs().pdl; }

// Launches `kern` on `s`, with programmatic stream serialization when
// pdl_enabled(): the kernel may be scheduled while the preceding kernel in
// the stream drains, and waits (pdl_wait) before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Runtime knobs (host globals, read at launch time).
uint64_t wait_timeout_ns();
bool take_skip_first_load();

// Launchers; each returns the launch's cudaError_t.
cudaError_t launch_amax(const float* x, int64_t n, float* amax_out,
                        float* scale_out, int sm_count, cudaStream_t s,
                        bool pow2 = false);
cudaError_t launch_quantize_e4m3(const float* x, int64_t n, const float* scale,
                                 uint8_t* q, int sm_count, cudaStream_t s);
// rows_per_cta and chunks: rows of B per 4-warp CTA and 16-byte chunks per
// lane per row in flight, from the plan (4 x 8, 8 x 4, 16 x 3 or 16 x 2 at
// M <= 2; otherwise 8 x 4 for M <= 4 and 4 x 4 above).
cudaError_t launch_gemv(const void* A, const void* B, void* D, int M, int N,
                        int K, bool fp16_in, const float* sa, const float* sb,
                        const float* sd, int out_kind, uint32_t* amax_out,
                        int rows_per_cta, int chunks, cudaStream_t s);
// Quantise with a given scale and record max |x| (and optionally the next
// scale = amax / 448) in the same pass over x.
cudaError_t launch_quantize_e4m3_amax(const float* x, int64_t n, const float* scale, uint8_t* q,
                                      float* amax_out, float* next_scale_out, int sm_count,
                                      cudaStream_t s);
// FP16 dynamic-range scaling: out[0..3] = scale, sqrt(scale), 1/scale, 1
// (one-thread kernel), and out_i = fp16_rn(x_i * factor).
cudaError_t launch_fp16_range_scale(const float* amax_a, const float* amax_b, float* out,
                                    cudaStream_t s);
cudaError_t launch_convert_f16(const float* x, int64_t n, const float* factor, uint16_t* out,
                               int sm_count, cudaStream_t s);
// The conversion with a given factor that also records max |x| in the same
// pass (zeroing kernel first).
cudaError_t launch_convert_f16_amax(const float* x, int64_t n, const float* factor, uint16_t* out,
                                    float* amax_out, int sm_count, cudaStream_t s);
cudaError_t launch_convert_f16_amax_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                         const float* factor, uint16_t* out_a, uint16_t* out_b,
                                         float* amax_a, float* amax_b, int sm_count,
                                         cudaStream_t s);
cudaError_t launch_quantize_e4m3_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                      float* amax_a, float* amax_b, float* scale_a, float* scale_b,
                                      uint8_t* qa, uint8_t* qb, int sm_count, cudaStream_t s);
// Sets *bits = 0 on stream s (one-thread kernel).
cudaError_t launch_zero_word(uint32_t* bits, cudaStream_t s);

struct TcLaunch {
    const void* A;
    const void* B;
    void* D;
    int M, N, K;
    bool fp16_in;
    const float* sa;
    const float* sb;
    const float* sd;
    int out_kind;
    int out_elem;
    const dg_plan* plan;
    uint32_t* status;
    uint32_t* amax_out;   // optional running max |sa*sb*acc| (float bits)
    const int* group_off; // grouped GEMM: device offsets [groups + 1], else null
    int groups;
    // CTA-pair kernel: workspace for splitting the tiles of a partial last
    // wave along K (the split-K workspace of the stream), or null.
    float* tail_ws = nullptr;
    size_t tail_ws_bytes = 0;
    uint32_t* tail_counts = nullptr;
};
cudaError_t launch_gemm_tc(const TcLaunch& L, cudaStream_t s);
// Grouped variant (single-CTA tiles; L.plan->block_n is 128 or 256).
cudaError_t launch_gemm_tc_grouped(const TcLaunch& L, cudaStream_t s);
constexpr int kMaxGemmGroups = 1024;

// Decode-shape GEMM for 1 <= M <= 16 with the K sums on warp-level MMAs
// (plan path 5): one CTA per 16 rows of B, L.plan->stages warps per CTA.
cudaError_t launch_gemv_mma(const TcLaunch& L, cudaStream_t s);

// Skinny split-K tensor-core GEMM (plan path 4).
// partials must hold 2 * grid slots of nc_for(M) x 128 floats, with
// nc_for(M) <= max_cols.
cudaError_t launch_gemm_skinny(const TcLaunch& L, float* partials, uint32_t* counts, int max_cols,
                               cudaStream_t s);
void plan_skinny(int64_t M, int64_t N, int64_t K, bool fp16_in, int sm_count, dg_plan* p);

// Tile table for the tensor-core path (fills block_n, stages, smem, grid).
void plan_tc(int64_t M, int64_t N, int64_t K, bool fp16_in, int sm_count,
             dg_plan* p);

}  // namespace dg
