// k_scale.cu -- per-tensor amax, scale, the E4M3 quantiser, and the FP16
// dynamic-range scaling factors and conversion.
//
// [FP8-guide] = "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南".
// §3.2: one scale per tensor, scale = max |x| / 448; §4.3: the quantiser
// fp8 = clamp(round(x / scale), -448, 448).  [DG-FP16] = the DeepGEMM
// FP16/WMMA deep-dive page, §3.3: scale = min(1, 65504 / (max|A| max|B|)),
// operands times sqrt(scale) into FP16, result divided by scale.  The
// streaming kernels are bound by HBM: amax reads 4 B per element, the
// quantiser reads 4 B and writes 1 B, the FP16 conversion 4 B and 2 B.
#include <cuda_runtime.h>

#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int kAmaxThreads = 512;
constexpr int kQuantThreads = 256;

__device__ __forceinline__ float4 ld_stream_f4(const float4* p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// |x| as an ordered integer: for non-negative floats the bit pattern is
// monotone in the value, and every NaN pattern is above +Inf, so an unsigned
// max over (bits & 0x7fffffff) is max |x| with NaN propagating.
__device__ __forceinline__ uint32_t abs_bits(float v) {
    return __float_as_uint(v) & 0x7FFFFFFFu;
}
__device__ __forceinline__ uint32_t abs_bits4(float4 v) {
    return max(max(abs_bits(v.x), abs_bits(v.y)), max(abs_bits(v.z), abs_bits(v.w)));
}

// scale = amax / 448 (one IEEE binary32 division), 1 for an all-zero tensor.
__device__ __forceinline__ float scale_of_amax(float a) {
    return (a == 0.0f) ? 1.0f : __fdiv_rn(a, 448.0f);
}

// Power-of-two scale ([FP8-guide] §2.1): the smallest p = 2^e (e >= -149,
// so p is a binary32 value) with 448 * p >= amax, compared exactly in
// double; 1 for amax == 0, NaN for NaN, +Inf for +Inf.  Dividing by p is
// then exact: the quantiser only shifts exponents.
__device__ __forceinline__ float scale_pow2_of_amax(float a) {
    float p;
    if (a != a) {
        p = a;
    } else if (a == 0.0f) {
        p = 1.0f;
    } else if (a > 3.4028234663852886e38f) {
        p = a;
    } else {
        const int ebits = static_cast<int>((__float_as_uint(a) >> 23) & 0xFFu);
        int e = ebits == 0 ? -149 : max(-149, ebits - 127 - 10);
        const double ad = static_cast<double>(a);
        // 448 * 2^e for e >= -149 is an exact double; at most a few steps.
        for (int it = 0; it < 400; ++it) {
            const double pe = __longlong_as_double(static_cast<long long>(e + 1023) << 52);
            if (448.0 * pe >= ad) break;
            ++e;
        }
        p = static_cast<float>(__longlong_as_double(static_cast<long long>(e + 1023) << 52));
    }
    return p;
}

// Scale from the finished reduction, by the CTA that completes it: each CTA,
// after its atomicMax, counts its arrival in the scale word (zeroed before
// the launch); the last one reads the final maximum and writes the scale
// over the count.  One thread per CTA.
__device__ __forceinline__ void finish_scale(uint32_t* amax_bits, float* scale_out, bool pow2) {
    __threadfence();   // this CTA's maximum is visible before its arrival
    uint32_t* count = reinterpret_cast<uint32_t*>(scale_out);
    if (atomicAdd(count, 1u) == gridDim.x - 1) {
        __threadfence();
        const float a = __uint_as_float(atomicOr(amax_bits, 0u));
        *scale_out = pow2 ? scale_pow2_of_amax(a) : scale_of_amax(a);
    }
}

// This thread's max |x| (ordered bits) over its grid-stride share of x; the
// ragged tail (n mod 4 elements) is read by block `tail_block`.
__device__ __forceinline__ uint32_t amax_share(const float* __restrict__ x, int64_t n,
                                               unsigned tail_block) {
    const int64_t n4 = n >> 2;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    uint32_t m = 0;
    for (; i + 3 * stride < n4; i += 4 * stride) {
        const float4 v0 = ld_stream_f4(x4 + i);
        const float4 v1 = ld_stream_f4(x4 + i + stride);
        const float4 v2 = ld_stream_f4(x4 + i + 2 * stride);
        const float4 v3 = ld_stream_f4(x4 + i + 3 * stride);
        m = max(m, max(max(abs_bits4(v0), abs_bits4(v1)), max(abs_bits4(v2), abs_bits4(v3))));
    }
    for (; i < n4; i += stride) m = max(m, abs_bits4(ld_stream_f4(x4 + i)));
    if (blockIdx.x == tail_block && threadIdx.x < static_cast<unsigned>(n & 3))
        m = max(m, abs_bits(x[(n4 << 2) + threadIdx.x]));
    return m;
}

__global__ void __launch_bounds__(kAmaxThreads)
amax_kernel(const float* __restrict__ x, int64_t n, uint32_t* __restrict__ out_bits,
            float* __restrict__ scale_out, int pow2) {
    pdl_wait();
    uint32_t m = amax_share(x, n, 0);
    m = __reduce_max_sync(0xFFFFFFFFu, m);
    __shared__ uint32_t partial[kAmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) partial[warp] = m;
    __syncthreads();
    if (warp == 0) {
        m = lane < kAmaxThreads / 32 ? partial[lane] : 0u;
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        if (lane == 0 && m != 0u) atomicMax(out_bits, m);
        if (lane == 0 && scale_out != nullptr) finish_scale(out_bits, scale_out, pow2 != 0);
    }
}

// Power-of-two scale from a finished reduction (see scale_pow2_of_amax).
__global__ void scale_pow2_kernel(const float* __restrict__ amax, float* __restrict__ scale) {
    pdl_wait();
    *scale = scale_pow2_of_amax(*amax);
}

// Zeroes the running maximum before the reduction (and the arrival count in
// the scale word when the reduction's last CTA writes the scale).
__global__ void amax_init_kernel(uint32_t* __restrict__ out_bits, uint32_t* __restrict__ count,
                                 uint32_t* __restrict__ other) {
    pdl_wait();
    *out_bits = 0u;
    if (count != nullptr) *count = 0u;
    if (other != nullptr) *other = 0u;
}

// scale = amax / 448 from a finished reduction (see scale_of_amax).
__global__ void scale_kernel(const float* __restrict__ amax, float* __restrict__ scale) {
    pdl_wait();
    *scale = scale_of_amax(*amax);
}

__device__ __forceinline__ uint32_t quant4(float4 v, float s) {
    const uint32_t lo = f32x2_to_e4m3x2(__fdiv_rn(v.x, s), __fdiv_rn(v.y, s));
    const uint32_t hi = f32x2_to_e4m3x2(__fdiv_rn(v.z, s), __fdiv_rn(v.w, s));
    return lo | (hi << 16);
}

// amax and scale of both GEMM operands in one grid: every thread takes its
// grid-stride share of a, then of b (so the grid streams on from one tensor
// to the next without a launch boundary); each CTA adds its two maxima to
// the words, counts its arrival in scale_a's word (zeroed before), and the
// last CTA writes both scales, scale_a over the count last.
__global__ void __launch_bounds__(kAmaxThreads)
amax_pair_kernel(const float* __restrict__ xa, int64_t na, const float* __restrict__ xb, int64_t nb,
                 uint32_t* __restrict__ bits_a, uint32_t* __restrict__ bits_b,
                 float* __restrict__ scale_a, float* __restrict__ scale_b) {
    pdl_wait();
    uint32_t ma = amax_share(xa, na, 0);
    uint32_t mb = amax_share(xb, nb, gridDim.x > 1 ? 1u : 0u);
    ma = __reduce_max_sync(0xFFFFFFFFu, ma);
    mb = __reduce_max_sync(0xFFFFFFFFu, mb);
    __shared__ uint32_t pa[kAmaxThreads / 32], pb[kAmaxThreads / 32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (lane == 0) {
        pa[warp] = ma;
        pb[warp] = mb;
    }
    __syncthreads();
    if (warp == 0) {
        ma = lane < kAmaxThreads / 32 ? pa[lane] : 0u;
        mb = lane < kAmaxThreads / 32 ? pb[lane] : 0u;
        ma = __reduce_max_sync(0xFFFFFFFFu, ma);
        mb = __reduce_max_sync(0xFFFFFFFFu, mb);
        if (lane == 0) {
            if (ma != 0u) atomicMax(bits_a, ma);
            if (mb != 0u) atomicMax(bits_b, mb);
            __threadfence();   // both maxima visible before the arrival
            if (atomicAdd(reinterpret_cast<uint32_t*>(scale_a), 1u) == gridDim.x - 1) {
                __threadfence();
                *scale_b = scale_of_amax(__uint_as_float(atomicOr(bits_b, 0u)));
                *scale_a = scale_of_amax(__uint_as_float(atomicOr(bits_a, 0u)));
            }
        }
    }
}

// Quantisation of both GEMM operands in one grid, each with its own scale:
// the 512-element slabs of a, then of b, are dealt to warps as one sequence,
// taken from its end (a warp's slab lies wholly in one tensor); the ragged
// tails go to blocks 0 and 1 (0 alone for a one-CTA grid).
__global__ void __launch_bounds__(kQuantThreads)
quantize_pair_kernel(const float* __restrict__ xa, int64_t na, const float* __restrict__ sa_p,
                     uint8_t* __restrict__ qa, const float* __restrict__ xb, int64_t nb,
                     const float* __restrict__ sb_p, uint8_t* __restrict__ qb) {
    pdl_wait();
    const float sa = *sa_p, sb = *sb_p;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t ka = na >> 9, kb = nb >> 9;
    // Slabs from the end of b backwards: the amax pass before this one
    // streamed a then b front to back, so the first slabs taken here are
    // the ones it read last, still in L2.
    for (int64_t k = warp; k < ka + kb; k += nwarps) {
        const int64_t slab = ka + kb - 1 - k;
        const bool in_a = slab < ka;   // the same for the whole warp
        const float4* x4 = reinterpret_cast<const float4*>(in_a ? xa : xb);
        uint32_t* q4 = reinterpret_cast<uint32_t*>(in_a ? qa : qb);
        const float s = in_a ? sa : sb;
        const int64_t b = (in_a ? slab : slab - ka) * 128 + lane;
        const float4 v0 = ld_stream_f4(x4 + b);
        const float4 v1 = ld_stream_f4(x4 + b + 32);
        const float4 v2 = ld_stream_f4(x4 + b + 64);
        const float4 v3 = ld_stream_f4(x4 + b + 96);
        q4[b] = quant4(v0, s);
        q4[b + 32] = quant4(v1, s);
        q4[b + 64] = quant4(v2, s);
        q4[b + 96] = quant4(v3, s);
    }
    if (blockIdx.x == 0)
        for (int64_t i = (ka << 9) + threadIdx.x; i < na; i += blockDim.x)
            qa[i] = static_cast<uint8_t>(f32x2_to_e4m3x2(__fdiv_rn(xa[i], sa), 0.0f) & 0xFFu);
    if (blockIdx.x == (gridDim.x > 1 ? 1u : 0u))
        for (int64_t i = (kb << 9) + threadIdx.x; i < nb; i += blockDim.x)
            qb[i] = static_cast<uint8_t>(f32x2_to_e4m3x2(__fdiv_rn(xb[i], sb), 0.0f) & 0xFFu);
}


// Each warp iteration handles 512 consecutive elements: four fully coalesced
// 512-byte loads (lane j reads float4 j, j+32, j+64, j+96 of the slab) and
// four 128-byte stores of packed codes.
// kAmax: also the running max |x| (ordered bits, NaN above every number)
// into *amax_bits, for the scale of the next call (delayed scaling).
template <bool kAmax>
__global__ void __launch_bounds__(kQuantThreads)
quantize_kernel(const float* __restrict__ x, int64_t n, const float* __restrict__ scale_p,
                uint8_t* __restrict__ q, uint32_t* __restrict__ amax_bits,
                float* __restrict__ next_scale) {
    pdl_wait();
    const float s = *scale_p;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nslab = n >> 9;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint32_t* q4 = reinterpret_cast<uint32_t*>(q);
    uint32_t m = 0u;
    for (int64_t slab = warp; slab < nslab; slab += nwarps) {
        const int64_t b = slab * 128 + lane;
        const float4 v0 = ld_stream_f4(x4 + b);
        const float4 v1 = ld_stream_f4(x4 + b + 32);
        const float4 v2 = ld_stream_f4(x4 + b + 64);
        const float4 v3 = ld_stream_f4(x4 + b + 96);
        q4[b] = quant4(v0, s);
        q4[b + 32] = quant4(v1, s);
        q4[b + 64] = quant4(v2, s);
        q4[b + 96] = quant4(v3, s);
        if constexpr (kAmax)
            m = max(m, max(max(abs_bits4(v0), abs_bits4(v1)), max(abs_bits4(v2), abs_bits4(v3))));
    }
    // Ragged tail (< 512 elements): one element per thread of block 0.
    if (blockIdx.x == 0) {
        for (int64_t i = (nslab << 9) + threadIdx.x; i < n; i += blockDim.x) {
            const float v = x[i];
            q[i] = static_cast<uint8_t>(f32x2_to_e4m3x2(__fdiv_rn(v, s), 0.0f) & 0xFFu);
            if constexpr (kAmax) m = max(m, abs_bits(v));
        }
    }
    if constexpr (kAmax) {
        __shared__ uint32_t partial[kQuantThreads / 32];
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        const int w = threadIdx.x >> 5;
        if (lane == 0) partial[w] = m;
        __syncthreads();
        if (w == 0) {
            m = lane < kQuantThreads / 32 ? partial[lane] : 0u;
            m = __reduce_max_sync(0xFFFFFFFFu, m);
            if (lane == 0 && m != 0u) atomicMax(amax_bits, m);
            if (lane == 0 && next_scale != nullptr) finish_scale(amax_bits, next_scale, false);
        }
    }
}

// [DG-FP16] §3.3 factors: out = {scale, sqrt(scale), 1/scale, 1}.  The
// product of the two maxima and the quotient are formed in binary64 (no
// binary32 overflow) and rounded once; sqrt and the reciprocal are taken in
// binary64 from the binary32 scale and rounded once, which for these two
// operations is the correctly rounded binary32 result.
__global__ void fp16_range_scale_kernel(const float* __restrict__ amax_a,
                                        const float* __restrict__ amax_b,
                                        float* __restrict__ out) {
    pdl_wait();
    const float a = *amax_a, b = *amax_b;
    float sc;
    if (isnan(a) || isnan(b)) {
        sc = __int_as_float(0x7FC00000);
    } else {
        const double q = 65504.0 / (static_cast<double>(a) * static_cast<double>(b));
        sc = __double2float_rn(q < 1.0 ? q : 1.0);
    }
    out[0] = sc;
    out[1] = __double2float_rn(sqrt(static_cast<double>(sc)));
    out[2] = __double2float_rn(1.0 / static_cast<double>(sc));
    out[3] = 1.0f;
}

__device__ __forceinline__ uint2 half4(float4 v, float f) {
    return make_uint2(f32x2_to_f16x2(__fmul_rn(v.x, f), __fmul_rn(v.y, f)),
                      f32x2_to_f16x2(__fmul_rn(v.z, f), __fmul_rn(v.w, f)));
}

// out_i = fp16_rn(fl32(x_i * factor)): each warp converts 512-element slabs
// (four 512-byte loads, four 256-byte stores per slab); the ragged tail is
// converted by block 0.  kAmax: also the running max |x| (ordered bits) into
// *amax_bits, for the factors of the next call (delayed scaling).
template <bool kAmax>
__global__ void __launch_bounds__(kQuantThreads)
convert_f16_kernel(const float* __restrict__ x, int64_t n, const float* __restrict__ factor_p,
                   uint16_t* __restrict__ out, uint32_t* __restrict__ amax_bits) {
    pdl_wait();
    const float f = factor_p != nullptr ? *factor_p : 1.0f;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t nslab = n >> 9;
    const float4* x4 = reinterpret_cast<const float4*>(x);
    uint2* o4 = reinterpret_cast<uint2*>(out);
    uint32_t m = 0u;
    for (int64_t slab = warp; slab < nslab; slab += nwarps) {
        const int64_t b = slab * 128 + lane;
        const float4 v0 = ld_stream_f4(x4 + b);
        const float4 v1 = ld_stream_f4(x4 + b + 32);
        const float4 v2 = ld_stream_f4(x4 + b + 64);
        const float4 v3 = ld_stream_f4(x4 + b + 96);
        o4[b] = half4(v0, f);
        o4[b + 32] = half4(v1, f);
        o4[b + 64] = half4(v2, f);
        o4[b + 96] = half4(v3, f);
        if constexpr (kAmax)
            m = max(m, max(max(abs_bits4(v0), abs_bits4(v1)), max(abs_bits4(v2), abs_bits4(v3))));
    }
    if (blockIdx.x == 0) {
        for (int64_t i = (nslab << 9) + threadIdx.x; i < n; i += blockDim.x) {
            const float v = x[i];
            out[i] = static_cast<uint16_t>(f32x2_to_f16x2(__fmul_rn(v, f), 0.0f) & 0xFFFFu);
            if constexpr (kAmax) m = max(m, abs_bits(v));
        }
    }
    if constexpr (kAmax) {
        __shared__ uint32_t partial[kQuantThreads / 32];
        m = __reduce_max_sync(0xFFFFFFFFu, m);
        const int w = threadIdx.x >> 5;
        if (lane == 0) partial[w] = m;
        __syncthreads();
        if (w == 0) {
            m = lane < kQuantThreads / 32 ? partial[lane] : 0u;
            m = __reduce_max_sync(0xFFFFFFFFu, m);
            if (lane == 0 && m != 0u) atomicMax(amax_bits, m);
        }
    }
}

// Both operands of the scaled HGEMM in one launch ([DG-FP16] §3.3 multiplies
// each by the same factor): the 512-element slabs of a, then of b, are dealt
// to warps as one sequence (a warp's slab lies wholly in one tensor), each
// CTA keeps one running max |x| per tensor and adds both to the words;
// the ragged tails go to blocks 0 and 1 (0 alone for a one-CTA grid).
__global__ void __launch_bounds__(kQuantThreads)
convert_f16_pair_kernel(const float* __restrict__ xa, int64_t na, uint16_t* __restrict__ oa,
                        uint32_t* __restrict__ ma, const float* __restrict__ xb, int64_t nb,
                        uint16_t* __restrict__ ob, uint32_t* __restrict__ mb,
                        const float* __restrict__ factor_p) {
    pdl_wait();
    const float f = factor_p != nullptr ? *factor_p : 1.0f;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int64_t sa = na >> 9, sb = nb >> 9;
    uint32_t m_a = 0u, m_b = 0u;
    for (int64_t slab = warp; slab < sa + sb; slab += nwarps) {
        const bool in_a = slab < sa;   // the same for the whole warp
        const float4* x4 = reinterpret_cast<const float4*>(in_a ? xa : xb);
        uint2* o4 = reinterpret_cast<uint2*>(in_a ? oa : ob);
        const int64_t b = (in_a ? slab : slab - sa) * 128 + lane;
        const float4 v0 = ld_stream_f4(x4 + b);
        const float4 v1 = ld_stream_f4(x4 + b + 32);
        const float4 v2 = ld_stream_f4(x4 + b + 64);
        const float4 v3 = ld_stream_f4(x4 + b + 96);
        o4[b] = half4(v0, f);
        o4[b + 32] = half4(v1, f);
        o4[b + 64] = half4(v2, f);
        o4[b + 96] = half4(v3, f);
        const uint32_t mm = max(max(abs_bits4(v0), abs_bits4(v1)), max(abs_bits4(v2), abs_bits4(v3)));
        if (in_a) m_a = max(m_a, mm); else m_b = max(m_b, mm);
    }
    const unsigned tail_b = gridDim.x > 1 ? 1u : 0u;
    if (blockIdx.x == 0) {
        for (int64_t i = (sa << 9) + threadIdx.x; i < na; i += blockDim.x) {
            const float v = xa[i];
            oa[i] = static_cast<uint16_t>(f32x2_to_f16x2(__fmul_rn(v, f), 0.0f) & 0xFFFFu);
            m_a = max(m_a, abs_bits(v));
        }
    }
    if (blockIdx.x == tail_b) {
        for (int64_t i = (sb << 9) + threadIdx.x; i < nb; i += blockDim.x) {
            const float v = xb[i];
            ob[i] = static_cast<uint16_t>(f32x2_to_f16x2(__fmul_rn(v, f), 0.0f) & 0xFFFFu);
            m_b = max(m_b, abs_bits(v));
        }
    }
    __shared__ uint32_t part_a[kQuantThreads / 32], part_b[kQuantThreads / 32];
    m_a = __reduce_max_sync(0xFFFFFFFFu, m_a);
    m_b = __reduce_max_sync(0xFFFFFFFFu, m_b);
    const int w = threadIdx.x >> 5;
    if (lane == 0) {
        part_a[w] = m_a;
        part_b[w] = m_b;
    }
    __syncthreads();
    if (w == 0) {
        m_a = lane < kQuantThreads / 32 ? part_a[lane] : 0u;
        m_b = lane < kQuantThreads / 32 ? part_b[lane] : 0u;
        m_a = __reduce_max_sync(0xFFFFFFFFu, m_a);
        m_b = __reduce_max_sync(0xFFFFFFFFu, m_b);
        if (lane == 0 && m_a != 0u) atomicMax(ma, m_a);
        if (lane == 0 && m_b != 0u) atomicMax(mb, m_b);
    }
}

// Grid of the slab kernels (quantiser, FP16 conversion): one 512-element
// slab per warp, at most 8 CTAs of kQuantThreads per SM, at least one CTA.
int64_t slab_grid(int64_t n, int sm_count) {
    const int64_t slabs = n >> 9;
    const int warps_per_block = kQuantThreads / 32;
    int64_t blocks = (slabs + warps_per_block - 1) / warps_per_block;
    const int64_t cap = static_cast<int64_t>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : blocks;
}

}  // namespace

cudaError_t launch_fp16_range_scale(const float* amax_a, const float* amax_b, float* out,
                                    cudaStream_t s) {
    return launch_kernel(fp16_range_scale_kernel, dim3(1), dim3(1), 0, s, amax_a, amax_b, out);
}

cudaError_t launch_convert_f16(const float* x, int64_t n, const float* factor, uint16_t* out,
                               int sm_count, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = slab_grid(n, sm_count);
    return launch_kernel(convert_f16_kernel<false>, dim3(static_cast<unsigned>(blocks)),
                         dim3(kQuantThreads), 0, s, x, n, factor, out, static_cast<uint32_t*>(nullptr));
}

cudaError_t launch_convert_f16_amax(const float* x, int64_t n, const float* factor, uint16_t* out,
                                    float* amax_out, int sm_count, cudaStream_t s) {
    uint32_t* bits = reinterpret_cast<uint32_t*>(amax_out);
    cudaError_t e = launch_kernel(amax_init_kernel, dim3(1), dim3(1), 0, s, bits,
                                  static_cast<uint32_t*>(nullptr), static_cast<uint32_t*>(nullptr));
    if (e != cudaSuccess || n <= 0) return e;
    const int64_t blocks = slab_grid(n, sm_count);
    return launch_kernel(convert_f16_kernel<true>, dim3(static_cast<unsigned>(blocks)),
                         dim3(kQuantThreads), 0, s, x, n, factor, out, bits);
}

cudaError_t launch_convert_f16_amax_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                         const float* factor, uint16_t* out_a, uint16_t* out_b,
                                         float* amax_a, float* amax_b, int sm_count,
                                         cudaStream_t s) {
    uint32_t* bits_a = reinterpret_cast<uint32_t*>(amax_a);
    uint32_t* bits_b = reinterpret_cast<uint32_t*>(amax_b);
    // one one-thread kernel zeroes both maxima (the second word as the
    // "count" argument, which it also sets to zero)
    cudaError_t e = launch_kernel(amax_init_kernel, dim3(1), dim3(1), 0, s, bits_a, bits_b,
                                  static_cast<uint32_t*>(nullptr));
    if (e != cudaSuccess || na + nb <= 0) return e;
    const int64_t blocks = slab_grid(na + nb, sm_count);
    return launch_kernel(convert_f16_pair_kernel, dim3(static_cast<unsigned>(blocks)),
                         dim3(kQuantThreads), 0, s, a, na, out_a, bits_a, b, nb, out_b, bits_b,
                         factor);
}

cudaError_t launch_quantize_e4m3_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                      float* amax_a, float* amax_b, float* scale_a, float* scale_b,
                                      uint8_t* qa, uint8_t* qb, int sm_count, cudaStream_t s) {
    uint32_t* bits_a = reinterpret_cast<uint32_t*>(amax_a);
    uint32_t* bits_b = reinterpret_cast<uint32_t*>(amax_b);
    cudaError_t e = launch_kernel(amax_init_kernel, dim3(1), dim3(1), 0, s, bits_a, bits_b,
                                  reinterpret_cast<uint32_t*>(scale_a));
    if (e != cudaSuccess) return e;
    const int64_t n4 = ((na + 3) >> 2) + ((nb + 3) >> 2);
    int64_t blocks = (n4 + kAmaxThreads - 1) / kAmaxThreads;
    const int64_t cap = static_cast<int64_t>(sm_count) * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    e = launch_kernel(amax_pair_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kAmaxThreads), 0, s,
                      a, na, b, nb, bits_a, bits_b, scale_a, scale_b);
    if (e != cudaSuccess || na + nb <= 0) return e;
    const int64_t qblocks = slab_grid(na + nb, sm_count);
    return launch_kernel(quantize_pair_kernel, dim3(static_cast<unsigned>(qblocks)),
                         dim3(kQuantThreads), 0, s, a, na, static_cast<const float*>(scale_a), qa, b,
                         nb, static_cast<const float*>(scale_b), qb);
}

cudaError_t launch_amax(const float* x, int64_t n, float* amax_out, float* scale_out,
                        int sm_count, cudaStream_t s, bool pow2) {
    uint32_t* bits = reinterpret_cast<uint32_t*>(amax_out);
    // The reduction's last CTA writes the scale (two launches, not three)
    // unless there is no reduction or the scale and amax words coincide.
    float* fold = (n > 0 && scale_out != nullptr && scale_out != amax_out) ? scale_out : nullptr;
    cudaError_t e = launch_kernel(amax_init_kernel, dim3(1), dim3(1), 0, s, bits,
                                  reinterpret_cast<uint32_t*>(fold), static_cast<uint32_t*>(nullptr));
    if (e != cudaSuccess) return e;
    if (n > 0) {
        const int64_t n4 = (n + 3) >> 2;
        int64_t blocks = (n4 + kAmaxThreads - 1) / kAmaxThreads;
        const int64_t cap = static_cast<int64_t>(sm_count) * 4;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        e = launch_kernel(amax_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kAmaxThreads), 0, s,
                          x, n, bits, fold, pow2 ? 1 : 0);
        if (e != cudaSuccess) return e;
    }
    if (scale_out != nullptr && fold == nullptr)
        e = launch_kernel(pow2 ? scale_pow2_kernel : scale_kernel, dim3(1), dim3(1), 0, s,
                          static_cast<const float*>(amax_out), scale_out);
    return e;
}

cudaError_t launch_zero_word(uint32_t* bits, cudaStream_t s) {
    return launch_kernel(amax_init_kernel, dim3(1), dim3(1), 0, s, bits,
                         static_cast<uint32_t*>(nullptr), static_cast<uint32_t*>(nullptr));
}

cudaError_t launch_quantize_e4m3(const float* x, int64_t n, const float* scale, uint8_t* q,
                                 int sm_count, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = slab_grid(n, sm_count);
    return launch_kernel(quantize_kernel<false>, dim3(static_cast<unsigned>(blocks)),
                         dim3(kQuantThreads), 0, s, x, n, scale, q, static_cast<uint32_t*>(nullptr),
                         static_cast<float*>(nullptr));
}

cudaError_t launch_quantize_e4m3_amax(const float* x, int64_t n, const float* scale, uint8_t* q,
                                      float* amax_out, float* next_scale_out, int sm_count,
                                      cudaStream_t s) {
    uint32_t* bits = reinterpret_cast<uint32_t*>(amax_out);
    // The pass's last CTA writes the next scale (two launches, not three)
    // unless the next scale overwrites the scale this pass reads (in place)
    // or the amax word.
    float* fold = (n > 0 && next_scale_out != nullptr && next_scale_out != scale &&
                   next_scale_out != amax_out) ? next_scale_out : nullptr;
    cudaError_t e = launch_kernel(amax_init_kernel, dim3(1), dim3(1), 0, s, bits,
                                  reinterpret_cast<uint32_t*>(fold), static_cast<uint32_t*>(nullptr));
    if (e != cudaSuccess) return e;
    if (n > 0) {
        const int64_t blocks = slab_grid(n, sm_count);
        e = launch_kernel(quantize_kernel<true>, dim3(static_cast<unsigned>(blocks)),
                          dim3(kQuantThreads), 0, s, x, n, scale, q, bits, fold);
        if (e != cudaSuccess) return e;
    }
    if (next_scale_out != nullptr && fold == nullptr)
        e = launch_kernel(scale_kernel, dim3(1), dim3(1), 0, s,
                          static_cast<const float*>(amax_out), next_scale_out);
    return e;
}

}  // namespace dg
