// k_gemv.cu -- the small-M path (any M <= 16; the planner sends M <= 2
// here): a bandwidth-bound GEMV with the K sum split across the 32 lanes of
// a warp.
//
// Page shorthands: [DG-FP16] = the DeepGEMM FP16/WMMA deep-dive page;
// [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南".
//
// [DG-FP16] §2.1 (weight-aware tiling): for the decode QKV projection
// [1, 4096] x [4096, 12288] the weight B is long-lived and read once, so it
// is streamed from HBM without shared-memory staging; §4.1: the single A row
// is broadcast to every thread instead of 2-D tiling.  [FP8-guide] §2.3:
// 128-bit vector loads.  Here one warp owns R consecutive rows of B (N x K,
// K contiguous; R = 1, 2 or 4 at M <= 2, chosen by the planner so that the
// grid fits one wave; 2 for M <= 4, 1 above): lane l reads 16-byte chunks l,
// l+32, l+64, ... of each row (fully coalesced 512-byte warp loads, U per
// row in flight at once) and widens them to FP16 pairs; the matching A
// chunk (L1-resident, shared by every warp) is widened once and used for all
// R rows.  Products and sums use fma.rn.f32.f16 -- the exact product of two
// FP16 values rounded once into an FP32 accumulator, the same arithmetic as
// widening both to FP32 first.  The warp's partial sums meet in a shuffle
// reduction; the epilogue applies scale_A * scale_B ([FP8-guide] §3.2) and
// rounds to the output type.
#include <cuda_runtime.h>

#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

// 4-warp CTAs: the finer grid (1536 CTAs for N = 12288) evens out the last
// wave; measured 3% faster than 8-warp CTAs on the decode QKV shape.
constexpr int kWarps = 4;

// B is read exactly once: its lines are marked first for eviction from L2 so
// the stream does not push out data that other kernels reuse.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint4 ld_stream_u4(const uint4* p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(policy));
    return v;
}

// 16 bytes of operand as f16x2 words: E4M3 codes are widened to FP16 (exact:
// E4M3 is a subset of FP16); FP16 data is already in that form.
template <bool kFp16>
__device__ __forceinline__ void to_h2(const uint4& w, uint32_t (&h)[kFp16 ? 4 : 8]) {
    if constexpr (kFp16) {
        h[0] = w.x; h[1] = w.y; h[2] = w.z; h[3] = w.w;
    } else {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            h[2 * i] = e4m3x2_to_f16x2(static_cast<uint16_t>(ws[i] & 0xFFFFu));
            h[2 * i + 1] = e4m3x2_to_f16x2(static_cast<uint16_t>(ws[i] >> 16));
        }
    }
}

// A read-only float whose load is issued here, in program order with the
// (volatile) stream loads, rather than wherever the compiler would place it.
__device__ __forceinline__ float ld_f32_now(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// acc += a.lo * b.lo + a.hi * b.hi with FP16 inputs and FP32 accumulation:
// each fma.rn.f32.f16 forms the exact product and rounds once to FP32.
__device__ __forceinline__ float fma2_f16(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .f16 al, ah, bl, bh;\n\t"
        "mov.b32 {al, ah}, %1;\n\t"
        "mov.b32 {bl, bh}, %2;\n\t"
        "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
        "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
        : "+f"(acc) : "r"(a), "r"(b));
    return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// One warp owns R consecutive rows of B; each A chunk is widened once and
// used for all R rows.  U chunks per lane per row are in flight at once.
template <int MT, bool kFp16, int R, int U>
__global__ void __launch_bounds__(kWarps * 32)
gemv_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B, void* __restrict__ D,
            int M, int N, int K, const float* __restrict__ sa, const float* __restrict__ sb,
            const float* __restrict__ sd, int out_kind, uint32_t* __restrict__ amax_out) {
    constexpr int H = kFp16 ? 4 : 8;   // f16x2 words per 16-byte chunk
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n0 = (blockIdx.x * kWarps + warp) * R;
    if (n0 >= N) return;  // warp-uniform
    const int64_t row_bytes = static_cast<int64_t>(K) * (kFp16 ? 2 : 1);
    const int nch = static_cast<int>(row_bytes >> 4);
    const uint64_t policy = l2_evict_first_policy();
    // The scales are loaded before the stream starts, so that their latency
    // is not added to the end of every warp's (short) lifetime, and combined
    // only after the loop, so that nothing in the loop waits for them.
    float sav = 1.0f, sbv = 1.0f, sdv = 1.0f;
    if (sa != nullptr) {
        sav = ld_f32_now(sa);
        sbv = ld_f32_now(sb);
    }
    if (out_kind == kOutE4M3) sdv = ld_f32_now(sd);

    float acc[MT][R];
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < R; ++r) acc[m][r] = 0.0f;

    for (int c0 = 0; c0 < nch; c0 += 32 * U) {
        uint4 bw[R][U];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const uint4* brow = reinterpret_cast<const uint4*>(
                B + static_cast<int64_t>(min(n0 + r, N - 1)) * row_bytes);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + u * 32 + lane;
                bw[r][u] = (c < nch && n0 + r < N) ? ld_stream_u4(brow + c, policy) : make_uint4(0, 0, 0, 0);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < nch) {
                uint32_t bh[R][H];
#pragma unroll
                for (int r = 0; r < R; ++r) to_h2<kFp16>(bw[r][u], bh[r]);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (MT <= 2 || m < M) {   // M == MT for MT <= 2
                        const uint4 aw = __ldg(reinterpret_cast<const uint4*>(
                                                   A + static_cast<int64_t>(m) * row_bytes) + c);
                        uint32_t ah[H];
                        to_h2<kFp16>(aw, ah);
#pragma unroll
                        for (int r = 0; r < R; ++r)
#pragma unroll
                            for (int i = 0; i < H; ++i) acc[m][r] = fma2_f16(ah[i], bh[r][i], acc[m][r]);
                    }
                }
            }
        }
    }

    const float ab = sav * sbv;
    const float alpha = out_kind == kOutE4M3 ? __fdiv_rn(ab, sdv) : ab;
    float mine = 0.0f;
#pragma unroll
    for (int m = 0; m < MT; ++m)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float s = warp_sum(acc[m][r]);
            if (lane == m * R + r) mine = s;
        }
    const int m = lane / R, r = lane % R;
    const bool writes = m < M && m < MT && n0 + r < N;
    if (amax_out != nullptr) {
        // max |sa*sb*acc| over this warp's outputs; monotone rounding makes
        // fl(max|acc| * c) the exact maximum of fl(|acc| * c).
        const uint32_t bits = __reduce_max_sync(0xFFFFFFFFu, writes ? (__float_as_uint(mine) & 0x7FFFFFFFu) : 0u);
        if (lane == 0 && bits != 0u) {
            atomicMax(amax_out, __float_as_uint(__uint_as_float(bits) * ab) & 0x7FFFFFFFu);
        }
    }
    if (writes) {
        const float v = mine * alpha;
        const int64_t off = static_cast<int64_t>(m) * N + n0 + r;
        if (out_kind == kOutE4M3) {
            reinterpret_cast<uint8_t*>(D)[off] =
                static_cast<uint8_t>(f32x2_to_e4m3x2(v, 0.0f) & 0xFFu);
        } else if (out_kind == kOutFP16) {
            reinterpret_cast<uint16_t*>(D)[off] =
                static_cast<uint16_t>(f32x2_to_f16x2(v, 0.0f) & 0xFFFFu);
        } else {
            reinterpret_cast<uint16_t*>(D)[off] =
                static_cast<uint16_t>(f32x2_to_bf16x2(v, 0.0f) & 0xFFFFu);
        }
    }
}

template <int MT, bool kFp16, int R, int U>
cudaError_t launch_one(const void* A, const void* B, void* D, int M, int N, int K,
                       const float* sa, const float* sb, const float* sd, int out_kind,
                       uint32_t* amax_out, cudaStream_t s) {
    const int rows_per_block = kWarps * R;
    const dim3 grid((N + rows_per_block - 1) / rows_per_block), block(kWarps * 32);
    return launch_kernel(gemv_kernel<MT, kFp16, R, U>, grid, block, 0, s,
                         static_cast<const uint8_t*>(A), static_cast<const uint8_t*>(B), D, M, N, K,
                         sa, sb, sd, out_kind, amax_out);
}

template <bool kFp16>
cudaError_t launch_mt(int MT, const void* A, const void* B, void* D, int M, int N, int K,
                      const float* sa, const float* sb, const float* sd, int out_kind,
                      uint32_t* amax_out, int rows_per_cta, int chunks, cudaStream_t s) {
    // Rows of B per CTA and chunks in flight from the planner: 4 x 8 (1 row
    // per warp), 8 x 4 (2 rows), 16 x 3 or 16 x 2 (4 rows).  4 x 3 is
    // E4M3-only (QKV 1 x 12288 x 4096: 9.60 vs 9.73 us for 4 x 2).
    if (MT == 1 && rows_per_cta == 4)
        return launch_one<1, kFp16, 1, 8>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
    if constexpr (!kFp16) {
        if (MT == 1 && rows_per_cta == 16 && chunks == 3)
            return launch_one<1, kFp16, 4, 3>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
    }
    if (MT == 1 && rows_per_cta == 16)
        return launch_one<1, kFp16, 4, 2>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
    if (MT == 2 && rows_per_cta == 4)
        return launch_one<2, kFp16, 1, 8>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
    if (MT == 2 && rows_per_cta == 16)
        return launch_one<2, kFp16, 4, 2>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
    switch (MT) {
        case 1: return launch_one<1, kFp16, 2, 4>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
        case 2: return launch_one<2, kFp16, 2, 4>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
        case 4: return launch_one<4, kFp16, 2, 4>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
        case 8: return launch_one<8, kFp16, 1, 4>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
        default: return launch_one<16, kFp16, 1, 4>(A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out, s);
    }
}

}  // namespace

cudaError_t launch_gemv(const void* A, const void* B, void* D, int M, int N, int K, bool fp16_in,
                        const float* sa, const float* sb, const float* sd, int out_kind,
                        uint32_t* amax_out, int rows_per_cta, int chunks, cudaStream_t s) {
    if (M <= 0 || M > 16 || N <= 0 || K <= 0) return cudaErrorInvalidValue;
    const int MT = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16;
    return fp16_in ? launch_mt<true>(MT, A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out,
                                     rows_per_cta, chunks, s)
                   : launch_mt<false>(MT, A, B, D, M, N, K, sa, sb, sd, out_kind, amax_out,
                                      rows_per_cta, chunks, s);
}

}  // namespace dg
