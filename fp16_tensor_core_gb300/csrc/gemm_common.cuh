// gemm_common.cuh -- pieces shared by the single-CTA and CTA-pair
// tensor-core GEMM kernels: launch parameters, tile raster, the fused
// scale/convert epilogue store and TMA tensor-map creation.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {

struct Params {
    void* D;
    int M, N, K;
    const float* sa;
    const float* sb;
    const float* sd;
    int out_kind;
    int out_elem;
    int vec_ok;
    uint32_t* status;
    uint64_t timeout_ns;
    int skip_first_load;
    int group_m;   // tiles are rastered in groups of group_m M-tiles sweeping N
    uint32_t* amax_out;  // optional: running max |sa*sb*acc| as float bits
    // Grouped GEMM: group g covers rows [group_off[g], group_off[g+1]) of A
    // and D and rows [g*N, g*N + N) of B; sa/sb/sd hold one scale per group.
    const int* group_off;
    int groups;
    int early_release;   // release the next kernel once every CTA is on its last tile
    int staged;          // epilogue through staging boxes and bulk tensor stores (tmap_d)
    // CTA-pair kernel, split tail: the tiles left after the last full wave
    // are cut into tail_split K ranges (>= 2; 1 = no split), one per pair.
    int tail_split;
    float* tail_ws;         // partial tiles: [slot][2 CTAs][BN / 4][128] float4
    uint32_t* tail_counts;  // per tail tile and CTA: arrivals of the later parts
    // Single-CTA kernel: bytes of one A box and one B box (128 and BN rows
    // x 128 bytes), and of the shorter boxes of the edge tiles: tiles whose
    // A rows start at a_edge_row or later (B rows at b_edge_row or later)
    // load through the edge maps, boxes of the rows left rounded up to 8
    // (INT_MAX: no edge).  The MMA still reads 128 and BN rows; the rows
    // past a box only reach output rows past M or columns past N, which are
    // not stored.
    int a_box_bytes;
    int b_box_bytes;
    int a_edge_bytes;
    int b_edge_bytes;
    int a_edge_row;
    int b_edge_row;
};

constexpr int kMaxGroups = 1024;

// CTA-pair kernel (k_gemm_tc2.cu): shared memory and stage count of the
// 256 x bn pair tile, and its launcher.
int pair_smem_for(int bn, int kps);   // kps: K blocks per stage (1 or 2)
int pair_stages(int bn, int kps);
cudaError_t launch_gemm_tc_pair(const TcLaunch& L, const Params& prm, cudaStream_t s);

namespace {

constexpr int kThreads = 256;   // warps: 0 TMA, 1 MMA, 2 TMEM owner, 3 idle, 4-7 epilogue
constexpr int kBKBytes = 128;   // one 128-byte swizzle row of K per stage

constexpr uint32_t pow2_at_least(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

// Shared memory per CTA available to a kernel (227 KB).
constexpr int kSmemLimit = 232448;


__device__ __forceinline__ void tile_coords(int t, int num_m, int num_n, int group_m, int& mt,
                                            int& nt) {
    const int group = group_m * num_n;
    const int g = t / group;
    const int first_m = g * group_m;
    const int gm = min(num_m - first_m, group_m);
    const int r = t - g * group;
    mt = first_m + r % gm;
    nt = r / gm;
}

__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Scale, convert and store 32 consecutive accumulator columns of one row.
// Returns max |acc| over the stored elements as ordered bits (the bit
// pattern of a non-negative float; NaN above every number), 0 if none.
__device__ __forceinline__ uint32_t store_chunk(const Params& p, int row, int row_end, int col0,
                                                const uint32_t (&r)[32], float alpha) {
    if (row >= row_end) return 0u;
    const int ncols = min(32, p.N - col0);
    if (ncols <= 0) return 0u;
    uint32_t amax_bits = 0u;
    if (p.amax_out != nullptr) {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < ncols) amax_bits = max(amax_bits, r[i] & 0x7FFFFFFFu);
    }
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * alpha;
    const int64_t off = static_cast<int64_t>(row) * p.N + col0;
    if (p.out_kind == kOutE4M3) {
        uint8_t* dst = static_cast<uint8_t*>(p.D) + off;
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            w[j] = static_cast<uint32_t>(f32x2_to_e4m3x2(v[4 * j], v[4 * j + 1])) |
                   (static_cast<uint32_t>(f32x2_to_e4m3x2(v[4 * j + 2], v[4 * j + 3])) << 16);
        if (ncols == 32 && p.vec_ok) {
            st_global_v4(dst, w[0], w[1], w[2], w[3]);
            st_global_v4(dst + 16, w[4], w[5], w[6], w[7]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncols) dst[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
        }
    } else {
        uint16_t* dst = static_cast<uint16_t*>(p.D) + off;
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            w[j] = p.out_kind == kOutFP16 ? f32x2_to_f16x2(v[2 * j], v[2 * j + 1])
                                          : f32x2_to_bf16x2(v[2 * j], v[2 * j + 1]);
        if (ncols == 32 && p.vec_ok) {
#pragma unroll
            for (int j = 0; j < 4; ++j)
                st_global_v4(dst + 8 * j, w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncols) dst[i] = static_cast<uint16_t>(w[i >> 1] >> (16 * (i & 1)));
        }
    }
    return amax_bits;
}

// Staged epilogue: each epilogue warp converts 32 rows x 32 columns of the
// accumulator into a box in shared memory laid out as the output tensor map
// expects (64-byte swizzle for 2-byte outputs, 32-byte for E4M3) and writes
// it with one bulk tensor store, which moves whole lines and clips rows >= M
// and columns >= N.
constexpr int kBoxBytes = 2048;   // 32 x 32 two-byte elements (E4M3 uses half)

// Thread `lane` converts accumulator row `row`, columns col0 .. col0 + 31,
// into its line of `box`.  Returns max |acc| over the columns < N of a row
// < row_end (ordered bits) when p.amax_out is set, else 0.
__device__ __forceinline__ uint32_t stage_box(const Params& p, uint8_t* box, int row, int row_end,
                                              int col0, const uint32_t (&r)[32], float alpha,
                                              int lane) {
    uint32_t amax_bits = 0u;
    if (p.amax_out != nullptr && row < row_end) {
        const int ncols = min(32, p.N - col0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < ncols) amax_bits = max(amax_bits, r[i] & 0x7FFFFFFFu);
    }
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]) * alpha;
    if (p.out_kind == kOutE4M3) {
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            w[j] = static_cast<uint32_t>(f32x2_to_e4m3x2(v[4 * j], v[4 * j + 1])) |
                   (static_cast<uint32_t>(f32x2_to_e4m3x2(v[4 * j + 2], v[4 * j + 3])) << 16);
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int ph = k ^ ((lane >> 2) & 1);   // 32-byte swizzle: 16-byte halves
            st_shared_v4(smem_addr(box + lane * 32 + ph * 16), w[4 * k], w[4 * k + 1], w[4 * k + 2],
                         w[4 * k + 3]);
        }
    } else {
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
            w[j] = p.out_kind == kOutFP16 ? f32x2_to_f16x2(v[2 * j], v[2 * j + 1])
                                          : f32x2_to_bf16x2(v[2 * j], v[2 * j + 1]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int ph = k ^ ((lane >> 1) & 3);   // 64-byte swizzle: 16-byte quarters
            st_shared_v4(smem_addr(box + lane * 64 + ph * 16), w[4 * k], w[4 * k + 1], w[4 * k + 2],
                         w[4 * k + 3]);
        }
    }
    return amax_bits;
}

// Waits until every bulk store this thread committed has finished reading
// shared memory (the staging box may then be rewritten).
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// The output tensor map of the staged epilogue: D (M x N of the output
// type), 32 x 32 boxes, swizzled to the width of one box line.  False if the
// rows of D are not 16-byte multiples (then the epilogue stores directly).
inline bool make_out_map(CUtensorMap* map, const TcLaunch& L);

// Publishes one warp's running max |acc| (ordered bits) as
// max |acc| * (sa * sb) into p.amax_out.  Rounding is monotone, so
// fl(max|acc| * c) = max fl(|acc| * c) exactly.  Whole warp, converged.
__device__ __forceinline__ void publish_amax(const Params& p, uint32_t amax_bits) {
    if (p.amax_out == nullptr) return;
    amax_bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
    if ((threadIdx.x & 31) == 0 && amax_bits != 0u) {
        float ab = 1.0f;
        if (p.sa != nullptr) ab = (*p.sa) * (*p.sb);
        const float v = __uint_as_float(amax_bits) * ab;
        atomicMax(p.amax_out, __float_as_uint(v) & 0x7FFFFFFFu);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D map over a rows x k row-major matrix, box = box_rows x 128 bytes,
// 128-byte swizzle, zero fill outside the matrix.
bool make_map(CUtensorMap* map, const void* base, int rows, int k, bool fp16, int box_rows) {
    auto encode = get_encode_fn();
    if (!encode) return false;
    const int elem = fp16 ? 2 : 1;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(k), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(k) * elem};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(kBKBytes / elem), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = encode(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8,
                              2, const_cast<void*>(base), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

inline bool make_out_map(CUtensorMap* map, const TcLaunch& L) {
    if ((static_cast<int64_t>(L.N) * L.out_elem) % 16 != 0) return false;
    auto encode = get_encode_fn();
    if (!encode) return false;
    const bool e4 = L.out_kind == kOutE4M3;
    const CUtensorMapDataType dt = e4 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                  : (L.out_kind == kOutFP16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                            : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.N), static_cast<cuuint64_t>(L.M)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.N) * L.out_elem};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, dt, 2, L.D, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  e4 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace dg
