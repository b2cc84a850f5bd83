// k_gemv.cu -- the M <= 16 path: a bandwidth-bound GEMV with the K sum split
// across the 32 lanes of a warp.
//
// Page shorthands: [DG-FP16] = the DeepGEMM FP16/WMMA deep-dive page;
// [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南".
//
// [DG-FP16] §2.1 (weight-aware tiling): for the decode QKV projection
// [1, 4096] x [4096, 12288] the weight B is long-lived and read once, so it
// is streamed from HBM without shared-memory staging; §4.1: the single A row
// is broadcast to every thread instead of 2-D tiling.  [FP8-guide] §2.3:
// 128-bit vector loads.  Here one warp owns one row n of B (N x K, K
// contiguous): lane l reads 16-byte chunks l, l+32, l+64, ... of that row
// (fully coalesced 512-byte warp loads, all of a 4 KB row in flight at
// once), multiplies them with the matching A chunks (L1-resident, shared by
// every warp) in FP32, and the warp's partial sums meet in a shuffle
// reduction.  The epilogue applies scale_A * scale_B ([FP8-guide] §3.2) and
// rounds to the output type.
#include <cuda_runtime.h>

#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int kWarps = 8;
constexpr int kUnroll = 8;  // 16-byte chunks per lane in flight

__device__ __forceinline__ uint4 ld_stream_u4(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// 16 bytes -> FP32 values (16 for E4M3 codes, 8 for FP16).  The conversion
// is exact in both cases (E4M3 and FP16 are subsets of FP32).
template <bool kFp16>
struct Chunk {
    static constexpr int kVals = kFp16 ? 8 : 16;
    float v[kVals];
    __device__ __forceinline__ void load(const uint4& w) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (kFp16) {
                const float2 f = f16x2_to_f32x2(ws[i]);
                v[2 * i] = f.x;
                v[2 * i + 1] = f.y;
            } else {
                const float2 a = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(ws[i] & 0xFFFFu)));
                const float2 b = f16x2_to_f32x2(e4m3x2_to_f16x2(static_cast<uint16_t>(ws[i] >> 16)));
                v[4 * i] = a.x;
                v[4 * i + 1] = a.y;
                v[4 * i + 2] = b.x;
                v[4 * i + 3] = b.y;
            }
        }
    }
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

template <int MT, bool kFp16>
__global__ void __launch_bounds__(kWarps * 32)
gemv_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B, void* __restrict__ D,
            int M, int N, int K, const float* __restrict__ sa, const float* __restrict__ sb,
            const float* __restrict__ sd, int out_kind) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n = blockIdx.x * kWarps + warp;
    if (n >= N) return;  // warp-uniform
    const int64_t row_bytes = static_cast<int64_t>(K) * (kFp16 ? 2 : 1);
    const int nch = static_cast<int>(row_bytes >> 4);
    const uint4* brow = reinterpret_cast<const uint4*>(B + static_cast<int64_t>(n) * row_bytes);

    float acc[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

    for (int c0 = 0; c0 < nch; c0 += 32 * kUnroll) {
        uint4 bw[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            bw[u] = c < nch ? ld_stream_u4(brow + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < nch) {
                Chunk<kFp16> bc;
                bc.load(bw[u]);
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < M) {
                        const uint4 aw = __ldg(reinterpret_cast<const uint4*>(
                                                   A + static_cast<int64_t>(m) * row_bytes) + c);
                        Chunk<kFp16> ac;
                        ac.load(aw);
#pragma unroll
                        for (int i = 0; i < Chunk<kFp16>::kVals; ++i)
                            acc[m] = fmaf(ac.v[i], bc.v[i], acc[m]);
                    }
                }
            }
        }
    }

#pragma unroll
    for (int m = 0; m < MT; ++m) acc[m] = warp_sum(acc[m]);

    float alpha = 1.0f;
    if (sa != nullptr) alpha = (*sa) * (*sb);
    if (out_kind == kOutE4M3) alpha = __fdiv_rn(alpha, *sd);

    float mine = 0.0f;
#pragma unroll
    for (int m = 0; m < MT; ++m)
        if (lane == m) mine = acc[m];
    if (lane < M) {
        const float v = mine * alpha;
        const int64_t off = static_cast<int64_t>(lane) * N + n;
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

template <bool kFp16>
cudaError_t launch_mt(int MT, const void* A, const void* B, void* D, int M, int N, int K,
                      const float* sa, const float* sb, const float* sd, int out_kind,
                      cudaStream_t s) {
    const dim3 grid((N + kWarps - 1) / kWarps), block(kWarps * 32);
    const auto* a = static_cast<const uint8_t*>(A);
    const auto* b = static_cast<const uint8_t*>(B);
    switch (MT) {
        case 1: gemv_kernel<1, kFp16><<<grid, block, 0, s>>>(a, b, D, M, N, K, sa, sb, sd, out_kind); break;
        case 2: gemv_kernel<2, kFp16><<<grid, block, 0, s>>>(a, b, D, M, N, K, sa, sb, sd, out_kind); break;
        case 4: gemv_kernel<4, kFp16><<<grid, block, 0, s>>>(a, b, D, M, N, K, sa, sb, sd, out_kind); break;
        case 8: gemv_kernel<8, kFp16><<<grid, block, 0, s>>>(a, b, D, M, N, K, sa, sb, sd, out_kind); break;
        default: gemv_kernel<16, kFp16><<<grid, block, 0, s>>>(a, b, D, M, N, K, sa, sb, sd, out_kind); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const void* A, const void* B, void* D, int M, int N, int K, bool fp16_in,
                        const float* sa, const float* sb, const float* sd, int out_kind,
                        cudaStream_t s) {
    const int MT = M <= 1 ? 1 : M <= 2 ? 2 : M <= 4 ? 4 : M <= 8 ? 8 : 16;
    return fp16_in ? launch_mt<true>(MT, A, B, D, M, N, K, sa, sb, sd, out_kind, s)
                   : launch_mt<false>(MT, A, B, D, M, N, K, sa, sb, sd, out_kind, s);
}

}  // namespace dg
