// k_gemv_mma.cu -- decode-shape GEMM (1 <= M <= 16) streamed straight from
// HBM into registers, with the K sums on the tensor cores (warp-level MMA).
//
// Page shorthands: [DG-FP16] = the DeepGEMM FP16/WMMA deep-dive page;
// [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南".
//
// [DG-FP16] §2.1 (weight-aware tiling for the decode QKV projection): the
// weight B is read once, so the kernel's only job is to stream it at HBM
// speed.  The CUDA-core GEMV does that for M <= 2, but its FMA count grows
// with M; the split-K tensor-core kernel spends ~4 us per launch on its
// cross-CTA fix-up.  Here each CTA owns 16 rows of B over the whole of K:
//  * its W warps split K into W contiguous ranges; per step a warp reads
//    16 rows x 64 bytes of B with one 16-byte load per lane and row half
//    (lane = 4 g + q reads rows g and g + 8 at byte 16 q of the step --
//    64 contiguous bytes per row, [FP8-guide] §2.3's 128-bit loads),
//    plus the matching 16 bytes of up to two rows of A (L1-resident);
//  * the products run on the tensor cores as D^T = B A^T: mma.sync
//    m16n8k32 (E4M3) or m16n8k16 (FP16), B rows as the MMA's M side, A's
//    rows (up to 8 per MMA) as its N side, FP32 accumulation ([FP8-guide]
//    §2.1).  A lane's 16 loaded bytes of a row are the operand of two MMAs
//    (4 bytes each for k-groups q and q + 4 of each); loading A with the
//    same byte offsets puts the same k under both operands, so the sum runs
//    over a permutation of k, which changes nothing;
//  * the W partial accumulators meet in shared memory and are added in warp
//    order (fixed, so the result is deterministic), scaled by
//    scale_A * scale_B (/ scale_D for E4M3 out, [FP8-guide] §3.2) and
//    stored.  No workspace, no cross-CTA traffic.
// Edges ([FP8-guide] §3.3): rows of B past N, rows of A past M and the K
// tail (K * element size is a multiple of 16 bytes, not of 64) are loaded as
// zeros by predicated loads; stores are predicated on m < M, n < N.
#include <cuda_runtime.h>

#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int kRowsPerCta = 16;   // the MMA's M side
constexpr int kStepBytes = 64;    // K bytes per row per warp step (4 lanes x 16 B)

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16 bytes of B, streamed once: not kept in L1, first out of L2.
__device__ __forceinline__ uint4 ld_stream(const void* p, uint64_t policy) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p), "l"(policy));
    return v;
}

__device__ __forceinline__ float ld_scalar(const float* p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// c += A (16 x 32 E4M3, row) * B (32 x 8 E4M3, col), FP32 accumulation.
__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// c += A (16 x 16 FP16, row) * B (16 x 8 FP16, col), FP32 accumulation.
__device__ __forceinline__ void mma_f16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// MT: MMAs per step (1: M <= 8, 2: M <= 16).  W: warps per CTA (K split).
// U: steps of B in flight per warp (2 U loads of 16 bytes per lane).
// Shapes: W = 2, 3, 4 with U = 8, 6, 4, register-capped for six resident
// CTAs per SM (912 on 152 SMs, so that N = 12288 / 16 = 768 CTAs fit one
// wave); W = 8, U = 4 for small N, capped for three.
template <int W>
constexpr int min_ctas_per_sm() { return W >= 8 ? 3 : 6; }
template <int W>
constexpr int batch_for() { return W == 2 ? 8 : W == 3 ? 6 : 4; }

template <int MT, bool kFp16, int W, int U>
__global__ void __launch_bounds__(W * 32, min_ctas_per_sm<W>())
gemv_mma_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B,
                void* __restrict__ D, int M, int N, int K, const float* __restrict__ sa,
                const float* __restrict__ sb, const float* __restrict__ sd, int out_kind,
                uint32_t* __restrict__ amax_out) {
    __shared__ float4 red[W][MT][32];   // per-warp partial accumulators
    __shared__ float scales[3];          // sa, sb, sd: loaded first, used last
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, q = lane & 3;
    const int r0 = blockIdx.x * kRowsPerCta;
    const int kbytes = K * (kFp16 ? 2 : 1);   // < 2^31 - 64 (checked by the launcher)
    const uint64_t policy = evict_first_policy();
    if (threadIdx.x == 0) {
        scales[0] = sa != nullptr ? ld_scalar(sa) : 1.0f;
        scales[1] = sa != nullptr ? ld_scalar(sb) : 1.0f;
        scales[2] = out_kind == kOutE4M3 ? ld_scalar(sd) : 1.0f;
    }

    // This warp's K range: steps [s_begin, s_end) of 64 bytes.  A lane's
    // 16-byte chunk at step offset `off` (bytes, relative to the range's
    // start) is loaded while off < its limit, and is zero otherwise: the K
    // tail, rows of B past N and rows of A past M (limit 0).
    const int steps = (kbytes + kStepBytes - 1) / kStepBytes;
    const int s_begin = steps * warp / W, s_end = steps * (warp + 1) / W;
    const int k0 = s_begin * kStepBytes + 16 * q;
    const int end = min(s_end * kStepBytes, kbytes) - k0;
    const int lim_b_lo = r0 + g < N ? end : 0, lim_b_hi = r0 + g + 8 < N ? end : 0;
    const int lim_a_lo = g < M ? end : 0, lim_a_hi = g + 8 < M ? end : 0;
    const uint8_t* pb_lo = B + static_cast<int64_t>(min(r0 + g, N - 1)) * kbytes + k0;
    const uint8_t* pb_hi = B + static_cast<int64_t>(min(r0 + g + 8, N - 1)) * kbytes + k0;
    const uint8_t* pa_lo = A + static_cast<int64_t>(min(g, M - 1)) * kbytes + k0;
    const uint8_t* pa_hi = A + static_cast<int64_t>(min(g + 8, M - 1)) * kbytes + k0;

    float c[MT][4];
#pragma unroll
    for (int j = 0; j < MT; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) c[j][i] = 0.0f;

    const uint4 zero = make_uint4(0, 0, 0, 0);
    const int span = (s_end - s_begin) * kStepBytes;
    for (int o = 0; o < span; o += U * kStepBytes) {
        // Only B is in flight across the batch; A (a few rows, L1-resident)
        // is read right before its MMAs, so the registers go to B.
        uint4 bl[U], bh[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int off = o + u * kStepBytes;
            bl[u] = off < lim_b_lo ? ld_stream(pb_lo + off, policy) : zero;
            bh[u] = off < lim_b_hi ? ld_stream(pb_hi + off, policy) : zero;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int off = o + u * kStepBytes;
            const uint4 al = off < lim_a_lo ? __ldg(reinterpret_cast<const uint4*>(pa_lo + off)) : zero;
            // two MMAs per 16 loaded bytes: words (x, y), then (z, w)
            if constexpr (kFp16) {
                mma_f16(c[0], bl[u].x, bh[u].x, bl[u].y, bh[u].y, al.x, al.y);
                mma_f16(c[0], bl[u].z, bh[u].z, bl[u].w, bh[u].w, al.z, al.w);
            } else {
                mma_e4m3(c[0], bl[u].x, bh[u].x, bl[u].y, bh[u].y, al.x, al.y);
                mma_e4m3(c[0], bl[u].z, bh[u].z, bl[u].w, bh[u].w, al.z, al.w);
            }
            if constexpr (MT == 2) {
                const uint4 ah =
                    off < lim_a_hi ? __ldg(reinterpret_cast<const uint4*>(pa_hi + off)) : zero;
                if constexpr (kFp16) {
                    mma_f16(c[1], bl[u].x, bh[u].x, bl[u].y, bh[u].y, ah.x, ah.y);
                    mma_f16(c[1], bl[u].z, bh[u].z, bl[u].w, bh[u].w, ah.z, ah.w);
                } else {
                    mma_e4m3(c[1], bl[u].x, bh[u].x, bl[u].y, bh[u].y, ah.x, ah.y);
                    mma_e4m3(c[1], bl[u].z, bh[u].z, bl[u].w, bh[u].w, ah.z, ah.w);
                }
            }
        }
    }

    // The W warps' partial sums, added in warp order.
#pragma unroll
    for (int j = 0; j < MT; ++j) red[warp][j][lane] = make_float4(c[j][0], c[j][1], c[j][2], c[j][3]);
    __syncthreads();
    if (warp != 0) return;
    float v[MT][4];
#pragma unroll
    for (int j = 0; j < MT; ++j) {
        float4 t = red[0][j][lane];
#pragma unroll
        for (int w = 1; w < W; ++w) {
            const float4 x = red[w][j][lane];
            t.x += x.x;
            t.y += x.y;
            t.z += x.z;
            t.w += x.w;
        }
        v[j][0] = t.x;
        v[j][1] = t.y;
        v[j][2] = t.z;
        v[j][3] = t.w;
    }
    // Lane (g, q) holds D^T rows n = r0 + g (v[.][0..1]) and r0 + g + 8
    // (v[.][2..3]) at columns m = 8 j + 2 q and 8 j + 2 q + 1.
    const float ab = scales[0] * scales[1];
    const float alpha = out_kind == kOutE4M3 ? __fdiv_rn(ab, scales[2]) : ab;
    uint32_t amax_bits = 0u;
#pragma unroll
    for (int j = 0; j < MT; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int n = r0 + g + ((i & 2) ? 8 : 0);
            const int m = 8 * j + 2 * q + (i & 1);
            if (n >= N || m >= M) continue;
            amax_bits = max(amax_bits, __float_as_uint(v[j][i]) & 0x7FFFFFFFu);
            const float y = v[j][i] * alpha;
            const int64_t off = static_cast<int64_t>(m) * N + n;
            if (out_kind == kOutE4M3)
                static_cast<uint8_t*>(D)[off] = static_cast<uint8_t>(f32x2_to_e4m3x2(y, 0.0f) & 0xFFu);
            else if (out_kind == kOutFP16)
                static_cast<uint16_t*>(D)[off] = static_cast<uint16_t>(f32x2_to_f16x2(y, 0.0f) & 0xFFFFu);
            else
                static_cast<uint16_t*>(D)[off] = static_cast<uint16_t>(f32x2_to_bf16x2(y, 0.0f) & 0xFFFFu);
        }
    }
    if (amax_out != nullptr) {
        // max |sa*sb*acc| of this CTA's outputs (monotone rounding: the
        // maximum of the scaled values is the scaled maximum)
        const uint32_t bits = __reduce_max_sync(0xFFFFFFFFu, amax_bits);
        if (lane == 0 && bits != 0u)
            atomicMax(amax_out, __float_as_uint(__uint_as_float(bits) * ab) & 0x7FFFFFFFu);
    }
}

template <int MT, bool kFp16, int W, int U>
cudaError_t launch_one(const TcLaunch& L, cudaStream_t s) {
    const dim3 grid((L.N + kRowsPerCta - 1) / kRowsPerCta), block(W * 32);
    return launch_kernel(gemv_mma_kernel<MT, kFp16, W, U>, grid, block, 0, s,
                         static_cast<const uint8_t*>(L.A), static_cast<const uint8_t*>(L.B), L.D,
                         L.M, L.N, L.K, L.sa, L.sb, L.sd, L.out_kind, L.amax_out);
}

template <int MT, bool kFp16>
cudaError_t launch_w(const TcLaunch& L, cudaStream_t s) {
    switch (L.plan->stages) {   // warps per CTA
        case 2: return launch_one<MT, kFp16, 2, batch_for<2>()>(L, s);
        case 3: return launch_one<MT, kFp16, 3, batch_for<3>()>(L, s);
        case 8: return launch_one<MT, kFp16, 8, batch_for<8>()>(L, s);
        default: return launch_one<MT, kFp16, 4, batch_for<4>()>(L, s);
    }
}

}  // namespace

cudaError_t launch_gemv_mma(const TcLaunch& L, cudaStream_t s) {
    if (L.M < 1 || L.M > 16 || L.N < 1 || L.K < 1 ||
        static_cast<int64_t>(L.K) * (L.fp16_in ? 2 : 1) > INT32_MAX - 64)
        return cudaErrorInvalidValue;
    if (L.M <= 8)
        return L.fp16_in ? launch_w<1, true>(L, s) : launch_w<1, false>(L, s);
    return L.fp16_in ? launch_w<2, true>(L, s) : launch_w<2, false>(L, s);
}

}  // namespace dg
