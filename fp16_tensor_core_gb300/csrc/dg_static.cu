// dg_static.cu -- dg_fp8_gemm_splitk_static: the split-K skinny GEMM with its
// workspace in fixed static device arrays, so that a call never allocates.
//
// The regular entry points keep the split-K workspace in memory the library
// allocates once per device.  This variant runs the same kernel (same plan,
// same launcher, bit-identical results) on two file-scope device arrays of
// fixed size instead; the host looks their addresses up once per device.
#include <cuda_runtime.h>

#include <climits>
#include <cstdint>
#include <mutex>

#include "dg.h"
#include "dg_internal.h"

namespace dg {
namespace {

// Fixed capacity: up to 160 CTAs (two 16 x 128 FP32 partial slots each,
// 2.5 MiB) and up to 1024 tiles of 128 rows of B (N <= 131072), plus one
// status word for kernels that run without a caller-supplied one.
constexpr int kStaticMaxCtas = 160;
constexpr int kStaticMaxTiles = 1024;
constexpr size_t kStaticPartialFloats =
    static_cast<size_t>(2) * kStaticMaxCtas * kSkinnyMaxM * kSkinnyTileRows;

static __device__ __align__(256) float g_static_partials[kStaticPartialFloats];
static __device__ __align__(256) uint32_t g_static_counts[kStaticMaxTiles + 1];  // + status word

struct StaticAddrs {
    bool ready = false;
    float* partials = nullptr;
    uint32_t* counts = nullptr;
    int sm_count = 0;
};
constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
StaticAddrs g_static[kMaxDevices];

// The arrays' addresses on the current device (looked up on its first call).
dg_status static_addrs(StaticAddrs* out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return DG_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lk(g_static_mu);
    StaticAddrs& a = g_static[dev];
    if (!a.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DG_ERR_CUDA;
        if (major != 10 || minor != 3) return DG_ERR_UNSUPPORTED;
        void* p = nullptr;
        void* c = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_partials) != cudaSuccess ||
            cudaGetSymbolAddress(&c, g_static_counts) != cudaSuccess) {
            (void)cudaGetLastError();
            return DG_ERR_CUDA;
        }
        a.partials = static_cast<float*>(p);
        a.counts = static_cast<uint32_t*>(c);
        a.sm_count = sms < kStaticMaxCtas ? sms : kStaticMaxCtas;
        a.ready = true;
    }
    *out = a;
    return DG_OK;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" dg_status dg_fp8_gemm_splitk_static(const uint8_t* A, const uint8_t* B, void* D,
                                               int64_t M, int64_t N, int64_t K,
                                               const float* scale_a, const float* scale_b,
                                               const float* scale_d, dg_dtype out,
                                               uint32_t* status_out, dg_stream_t stream) {
    if (M < 0 || N < 0 || K < 0 || M > kSkinnyMaxM || N > INT_MAX || K > INT_MAX)
        return DG_ERR_INVALID_VALUE;
    if (out != DG_BF16 && out != DG_E4M3 && out != DG_FP16) return DG_ERR_INVALID_VALUE;
    if (N > static_cast<int64_t>(kStaticMaxTiles) * kSkinnyTileRows) return DG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(status_out) & 3u) != 0) return DG_ERR_MISALIGNED;
    if (M == 0 || N == 0) return DG_OK;
    if (D == nullptr) return DG_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr || scale_a == nullptr || scale_b == nullptr))
        return DG_ERR_INVALID_VALUE;
    if (K > 0 && out == DG_E4M3 && scale_d == nullptr) return DG_ERR_INVALID_VALUE;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (K % 16) != 0) return DG_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(scale_a) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(scale_b) & 3u) != 0 ||
        (out == DG_E4M3 && (reinterpret_cast<uintptr_t>(scale_d) & 3u) != 0))
        return DG_ERR_MISALIGNED;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0) {
        const size_t bytes = static_cast<size_t>(M * N) * (out == DG_E4M3 ? 1 : 2);
        return cudaMemsetAsync(D, 0, bytes, s) == cudaSuccess ? DG_OK : DG_ERR_CUDA;
    }
    StaticAddrs a;
    dg_status rc = static_addrs(&a);
    if (rc != DG_OK) return rc;
    dg_plan plan{};
    plan.path = 4;
    plan_skinny(M, N, K, false, a.sm_count, &plan);
    if (plan.grid > kStaticMaxCtas || plan.tiles > kStaticMaxTiles) return DG_ERR_INVALID_VALUE;
    // The arrival counters must start at zero.
    if (cudaMemsetAsync(a.counts, 0, sizeof(uint32_t) * static_cast<size_t>(plan.tiles), s) !=
        cudaSuccess)
        return DG_ERR_CUDA;
    TcLaunch L;
    L.A = A;
    L.B = B;
    L.D = D;
    L.M = static_cast<int>(M);
    L.N = static_cast<int>(N);
    L.K = static_cast<int>(K);
    L.fp16_in = false;
    L.sa = scale_a;
    L.sb = scale_b;
    L.sd = scale_d;
    L.out_kind = out_kind_of(out);
    L.out_elem = elem_bytes(out);
    L.plan = &plan;
    L.status = status_out != nullptr ? status_out : a.counts + kStaticMaxTiles;
    L.amax_out = nullptr;
    L.group_off = nullptr;
    L.groups = 0;
    return launch_gemm_skinny(L, a.partials, a.counts, kSkinnyMaxM, s) == cudaSuccess
               ? DG_OK
               : DG_ERR_CUDA;
}
