// dg_api.cu -- the C ABI declared in include/dg.h: argument validation,
// per-device state, path/tile selection and launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <unordered_map>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "dg.h"
#include "dg_internal.h"
#include "dg_ptx.cuh"

namespace dg {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceState g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices] = {};

// Split-K workspaces per device, one per stream that has run a split-K GEMM
// (calls on different streams may execute concurrently, so they must not
// share partial slots and arrival counters).  One stream at a time uses the
// workspace allocated with the device state; each other stream gets one of
// its own, up to kMaxStreamWorkspaces per device, until dg_release_stream.
struct SplitkWs {
    float* partials;
    uint32_t* counts;
};
constexpr size_t kMaxStreamWorkspaces = 16;
std::mutex g_ws_mu[kMaxDevices];
std::unordered_map<cudaStream_t, SplitkWs> g_ws[kMaxDevices];
bool g_dev_ws_taken[kMaxDevices] = {};   // the device-state workspace is in g_ws

size_t splitk_partial_bytes(int sm_count) {
    return sizeof(float) * 2 * static_cast<size_t>(sm_count) * kSplitkMaxCols * kSkinnyTileRows;
}
constexpr size_t kSplitkCountBytes = sizeof(uint32_t) * kSkinnyMaxTiles;

std::atomic<uint64_t> g_timeout_ns{2000000000ull};
std::atomic<int> g_skip_first_load{0};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// FP32 device scalars (scales, amax words) are read by 4-byte loads.
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline dg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DG_OK : DG_ERR_CUDA; }

}  // namespace

namespace {

// Integer value of environment variable `name` if set and within [lo, hi].
bool env_int(const char* name, int64_t lo, int64_t hi, int64_t* out) {
    const char* v = std::getenv(name);
    if (v == nullptr || v[0] == '\0') return false;
    char* end = nullptr;
    const long long x = std::strtoll(v, &end, 10);
    if (end == v || x < lo || x > hi) return false;
    *out = x;
    return true;
}

Knobs read_knobs() {
    Knobs k;
    int64_t v = 0;
    if (const char* e = std::getenv("DG_PDL")) k.pdl = e[0] != '0';
    if (const char* e = std::getenv("DG_LOG")) k.log = e[0] != '\0' && e[0] != '0';
    if (env_int("DG_GEMV_MAX_M", 0, 16, &v)) k.gemv_max_m = static_cast<int>(v);
    if (env_int("DG_GEMV_ROWS", 4, 16, &v) && (v == 4 || v == 8 || v == 16))
        k.gemv_rows = static_cast<int>(v);
    if (const char* e = std::getenv("DG_SPLITK")) k.splitk = e[0] == '0' ? 0 : e[0] == '1' ? 1 : -1;
    if (env_int("DG_SPLITK_GRID", 1, INT_MAX, &v)) k.splitk_grid = static_cast<int>(v);
    if (env_int("DG_SPLITK_PREFETCH", 0, 256, &v)) k.splitk_prefetch = static_cast<int>(v);
    if (env_int("DG_SPLITK_KPS", 1, 2, &v)) k.splitk_kps = static_cast<int>(v);
    if (const char* e = std::getenv("DG_ONE_WAVE")) k.one_wave = e[0] != '0';
    if (env_int("DG_ONE_WAVE_KB", INT64_MIN, INT64_MAX, &v)) k.one_wave_kb = v;
    if (env_int("DG_FORCE_BLOCK_N", 64, 256, &v)) k.force_block_n = static_cast<int>(v);
    if (const char* e = std::getenv("DG_2CTA")) k.two_cta = e[0] == '0' ? 0 : e[0] == '1' ? 1 : -1;
    if (env_int("DG_GROUP_M", 1, 4096, &v)) k.group_m = static_cast<int>(v);
    if (const char* e = std::getenv("DG_MMA_GEMV")) k.mma_gemv = e[0] == '0' ? 0 : e[0] == '1' ? 1 : -1;
    if (env_int("DG_MMA_GEMV_WARPS", 2, 8, &v) && (v == 2 || v == 3 || v == 4 || v == 8))
        k.mma_gemv_warps = static_cast<int>(v);
    if (const char* e = std::getenv("DG_STAGED_EPI")) k.staged_epilogue = e[0] != '0';
    if (const char* e = std::getenv("DG_SPLIT_TAIL")) k.split_tail = e[0] == '1';
    if (const char* e = std::getenv("DG_STREAM_K")) k.stream_k = e[0] == '1';
    if (const char* e = std::getenv("DG_EARLY_RELEASE")) k.early_release = e[0] != '0';
    if (const char* e = std::getenv("DG_SPLITK_ROWS")) k.splitk_rows = e[0] == '1' ? 1 : 0;
    if (env_int("DG_SPLITK_TILE_ROWS", 16, 128, &v) && v % 8 == 0)
        k.splitk_tile_rows = static_cast<int>(v);
    if (env_int("DG_TC_SHORT_BOX", 0, 2, &v)) k.tc_short_box = static_cast<int>(v);
    if (env_int("DG_TC_KPS", 1, 2, &v)) k.tc_kps = static_cast<int>(v);
    if (env_int("DG_PAIR_KPS", 1, 2, &v)) k.pair_kps = static_cast<int>(v);
    return k;
}

// The current snapshot.  dg_reload_env() publishes a new one and keeps the
// old one alive (a few bytes per reload), so a concurrent reader never sees
// freed memory.
std::atomic<const Knobs*> g_knobs{nullptr};
std::once_flag g_knobs_once;

}  // namespace

const Knobs& knobs() {
    const Knobs* k = g_knobs.load(std::memory_order_acquire);
    if (k != nullptr) return *k;
    std::call_once(g_knobs_once, [] {
        if (g_knobs.load(std::memory_order_acquire) == nullptr)
            g_knobs.store(new Knobs(read_knobs()), std::memory_order_release);
    });
    return *g_knobs.load(std::memory_order_acquire);
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

bool take_skip_first_load() { return g_skip_first_load.exchange(0) != 0; }

dg_status current_device_state(DeviceState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
        (void)cudaGetLastError();
        return DG_ERR_UNSUPPORTED;
    }
    if (dev >= kMaxDevices) return DG_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev_ready[dev]) {
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return DG_ERR_CUDA;
        if (prop.major != 10 || prop.minor != 3) return DG_ERR_UNSUPPORTED;
        DeviceState st;
        st.device = dev;
        st.sm_count = prop.multiProcessorCount;
        void* p = nullptr;
        if (cudaMalloc(&p, 16) != cudaSuccess) return DG_ERR_CUDA;
        if (cudaMemset(p, 0, 16) != cudaSuccess) {
            cudaFree(p);
            return DG_ERR_CUDA;
        }
        st.status = static_cast<uint32_t*>(p);
        // Split-K workspace (fixed size, so that nothing is allocated later,
        // e.g. while a stream is being captured into a graph).
        const size_t part_bytes = splitk_partial_bytes(st.sm_count);
        const size_t count_bytes = kSplitkCountBytes;
        void* w = nullptr;
        if (cudaMalloc(&w, part_bytes + count_bytes) != cudaSuccess) {
            cudaFree(p);
            return DG_ERR_CUDA;
        }
        if (cudaMemset(w, 0, part_bytes + count_bytes) != cudaSuccess) {
            cudaFree(w);
            cudaFree(p);
            return DG_ERR_CUDA;
        }
        st.splitk_partials = static_cast<float*>(w);
        st.splitk_counts = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(w) + part_bytes);
        g_dev[dev] = st;
        g_dev_ready[dev] = true;
    }
    *out = &g_dev[dev];
    return DG_OK;
}

namespace {

// DG_LOG=1: one line per GEMM call on stderr with the chosen path and tile.
void log_plan(const char* what, int64_t M, int64_t N, int64_t K, const dg_plan& p) {
    if (!knobs().log) return;
    static const char* const kPath[6] = {"no-op", "zero-fill", "gemv", "tensor-core",
                                         "split-k", "gemv-mma"};
    std::fprintf(stderr,
                 "dg: %s M=%lld N=%lld K=%lld path=%s tile=%dx%d stages=%d tiles=%d grid=%d\n",
                 what, static_cast<long long>(M), static_cast<long long>(N),
                 static_cast<long long>(K), kPath[p.path >= 0 && p.path <= 5 ? p.path : 0],
                 p.block_m, p.block_n, p.stages, p.tiles, p.grid);
}

// Launch-time estimates (microseconds) for choosing between the tiled and
// the split-K kernels at 17 <= M <= 128, fitted to graph-replayed GB300
// timings with B read from HBM (M = 16..128 against N = 1000..28672,
// K = 1040..14336; 45 shapes, the faster kernel chosen on 41, the four
// misses within 0.9 us).
//  * Tiled: ~3.4 us fixed, plus the larger of ~0.26 us per K block for
//    each wave of tiles (a CTA's pipeline refills at that rate whatever the
//    tile width) and all bytes at ~6.5 TB/s, plus ~0.12 us per 1000 output
//    elements of a tile (the epilogue's row-per-lane stores).
//  * Split-K: ~2.2 us fixed, B at ~5.8 TB/s (0.172 us per MB), ~0.235 us
//    per segment a tile is cut into (s = ceil(grid / tiles)), and for each
//    16 columns of A past the first, the finishing CTAs' extra pass over
//    the partial tiles: ~0.86 us plus ~0.058 us per segment.
double tiled_estimate_us(int64_t M, int64_t N, int64_t K, bool fp16_in, const dg_plan& p) {
    const double elem = fp16_in ? 2.0 : 1.0;
    const int64_t kb = fp16_in ? 64 : 128;   // one K block (a stage may hold two)
    const int64_t kblocks = (K + kb - 1) / kb;
    const int64_t waves = (p.tiles + p.grid - 1) / p.grid;
    const double all_mb = static_cast<double>(M + N) * static_cast<double>(K) * elem / 1e6;
    const double tile_rows = static_cast<double>(std::min<int64_t>(M, p.block_m));
    return 3.4 + std::max(0.26 * static_cast<double>(kblocks * waves), all_mb / 6.5) +
           0.121 * tile_rows * static_cast<double>(p.block_n) / 1000.0;
}

double splitk_estimate_us(int64_t M, int64_t N, int64_t K, bool fp16_in, const dg_plan& p) {
    const double elem = fp16_in ? 2.0 : 1.0;
    const int64_t chunks = (M + 15) / 16;
    const int64_t others = (p.grid + p.tiles - 1) / p.tiles;
    const double b_mb = static_cast<double>(N) * static_cast<double>(K) * elem / 1e6;
    return 2.2 + 0.172 * b_mb + 0.235 * static_cast<double>(others) +
           static_cast<double>(chunks - 1) * (0.86 + 0.058 * static_cast<double>(others));
}

// Shared path selection for dg_gemm_plan and the GEMM entry points.
dg_status make_plan(int64_t M, int64_t N, int64_t K, bool fp16_in, int sm_count, dg_plan* p) {
    *p = dg_plan{};
    if (M == 0 || N == 0) {
        p->path = 0;
        return DG_OK;
    }
    if (K == 0) {
        p->path = 1;
        return DG_OK;
    }
    // GEMV for M <= 2, split-K tensor cores up to M = 16.  Measured on GB300
    // for N = 12288 (B read from HBM, graph-replayed launches): at K = 4096
    // the GEMV takes 9.7 us at M = 1 and grows with M (its FMA count), the
    // split-K kernel a flat 11.1-11.5 us for M = 1..16; at K = 1024 4.4
    // against 6.9 us.  DG_GEMV_MAX_M (0..16) moves the crossover.
    const Knobs& kn = knobs();
    // Decode shapes on the warp-MMA GEMV (B streamed into registers, K sums
    // on warp-level MMAs, no workspace), one CTA per 16 rows of B.  Measured
    // on GB300 (graph-replayed, B from HBM; us): E4M3 x 12288 x 4096 at
    // M = 1 / 2 / 4 / 8: 9.3-9.5 / 9.5-10.0 / 9.7-10.1 / 9.9-10.2 against
    // 9.6 (GEMV) / 10.9 (GEMV) / 11.2-11.4 / 11.2-11.3 (split-K); x 4096 x
    // 4096: 5.0-5.2 against 5.1-6.7; x 1000 x 1040: 2.1-2.3 against 2.3-5.1.
    // With 9-16 rows of A an E4M3 step takes two MMAs, and the warp-level
    // MMA rate (about 1/16 of the tcgen05 one on this part) then sets the
    // time once N * K is large (16 x 12288 x 4096: 12.9 against 11.4 us on
    // split-K), so split-K keeps those; FP16 operands carry half the
    // products per byte and stay here (16 x 12288 x 4096: 20.8 against
    // 21.6 us).  M = 1 with E4M3 and more CTAs than one wave of four-warp
    // CTAs keeps the CUDA-core GEMV (1 x 28672 x 4096: 19.3 against 19.9).
    // Warps per CTA: 8 up to two CTAs per SM (small N), 4 up to six (one
    // wave), else 2; with two MMAs per step 2 from three CTAs per SM.
    const int64_t kbytes = K * (fp16_in ? 2 : 1);
    const int64_t mma_ctas = (N + 15) / 16;
    const int64_t sms = sm_count;
    bool use_mma = M <= 16 && kbytes <= INT32_MAX - 64 && mma_ctas <= INT_MAX;
    if (use_mma && kn.mma_gemv != 1) {
        use_mma = kn.mma_gemv != 0 &&
                  (fp16_in || M <= 8 || N * K <= (int64_t{1} << 22)) &&
                  !(M == 1 && !fp16_in && mma_ctas > 6 * sms);
    }
    if (use_mma) {
        p->path = 5;
        p->block_m = M <= 8 ? 8 : 16;
        p->block_n = 16;
        p->block_k = fp16_in ? 32 : 64;
        const int warps = mma_ctas <= 2 * sms ? 8 : (mma_ctas <= 6 * sms && M <= 8) ? 4 : 2;
        p->stages = kn.mma_gemv_warps != 0 ? kn.mma_gemv_warps : warps;
        p->grid = static_cast<int>(mma_ctas);
        p->tiles = static_cast<int>(mma_ctas);
        return DG_OK;
    }
    if (M <= kn.gemv_max_m) {
        p->path = 2;
        int rows = M <= 4 ? 8 : 4;   // 4 warps x (2 or 1) rows of B
        int chunks = 4;              // 16-byte chunks per lane per row in flight
        // M <= 2 with rows of B of at most 8 KB: the fewest rows per CTA whose
        // grid fits in one wave (at that layout's CTAs per SM, set by its
        // registers), so no partial second wave trails the stream; if none
        // fits, 8 for E4M3 and 4 for FP16.  Layouts per warp: 4 rows = 1 row x
        // 8 chunks, 8 = 2 x 4, 16 = 4 x 3 (E4M3, M = 1) or 4 x 2.  Measured on
        // GB300, graph-replayed (us, 8 rows -> chosen): E4M3 1 x 12288 x 4096
        // 10.10 -> 9.70 (4 x 2) -> 9.60 (4 x 3); 1 x 4096 x 4096 5.27 -> 5.09
        // (4 rows); 2 x 12288 x 4096 13.4 -> 10.9 (16); FP16 1 x 12288 x 4096
        // 22.3 -> 16.2 (16); 1 x 4096 x 4096 10.3 -> 7.2 (4); 1 x 28672 x 4096
        // 38.1 -> 33.8 (4, none fits); E4M3 1 x 28672 x 4096 and 1 x 8192 x
        // 8192 best at 8.
        const int64_t row_bytes = K * (fp16_in ? 2 : 1);
        if (M <= 2 && row_bytes <= 8192) {
            struct Layout { int rows, chunks, per_sm; };
            const Layout e4_m1[4] = {{4, 8, 8}, {8, 4, 8}, {16, 3, 6}, {16, 2, 8}};
            const Layout e4_m2[3] = {{4, 8, 8}, {8, 4, 8}, {16, 2, 6}};
            const Layout f16[3] = {{4, 8, 8}, {8, 4, 8}, {16, 2, M == 1 ? 8 : 7}};
            const Layout* cand = fp16_in ? f16 : (M == 1 ? e4_m1 : e4_m2);
            const int ncand = (!fp16_in && M == 1) ? 4 : 3;
            rows = fp16_in ? 4 : 8;
            chunks = fp16_in ? 8 : 4;
            for (int i = 0; i < ncand; ++i) {
                if ((N + cand[i].rows - 1) / cand[i].rows <=
                    static_cast<int64_t>(sm_count) * cand[i].per_sm) {
                    rows = cand[i].rows;
                    chunks = cand[i].chunks;
                    break;
                }
            }
        }
        if (kn.gemv_rows != 0 && M <= 2) {   // sweeps
            rows = kn.gemv_rows;
            chunks = rows == 4 ? 8 : rows == 8 ? 4 : 2;
        }
        p->grid = static_cast<int>((N + rows - 1) / rows);
        p->block_m = static_cast<int>(M);
        p->block_n = rows;
        p->block_k = fp16_in ? 8 * 32 : 16 * 32;
        p->stages = chunks;
        return DG_OK;
    }
    // Split-K with swapped operands (every SM streams an equal share of B)
    // for the remaining skinny shapes, and for 17 <= M <= 128 when the tiled
    // plan would keep fewer than 3/4 of the SMs busy and the time estimate
    // below favours it.  DG_SPLITK=0 turns it off, DG_SPLITK=1 uses it for
    // every M <= 128.
    //
    // Over a short K the tiled kernel wins instead once its tiles fill at
    // least half the SMs in one wave: a CTA then streams its few K blocks
    // straight into one tile, with no cross-CTA fix-up.  Measured on GB300
    // (E4M3, graph-replayed, us, split-K -> tiled): 16 x 12288 x 1040 8.24
    // -> 6.78, 9 x 12288 x 1040 8.20 -> 6.69, 16 x 14336 x 1040 8.70 ->
    // 7.13, 16 x 11008 x 2048 8.44 -> 8.03; split-K stays ahead at 32 K
    // blocks (16 x 12288 x 4096 11.6 against 12.8) and with fewer tiles
    // (16 x 4096 x 1040: 5.5 either way).
    const bool splitk_off = kn.splitk == 0;
    const bool splitk_forced = kn.splitk == 1;
    const int64_t sk_rows = kn.splitk_tile_rows;
    const bool splitk_fits = (N + sk_rows - 1) / sk_rows <= kSkinnyMaxTiles;
    const int64_t tiles = ((M + 127) / 128) * ((N + 63) / 64);
    if (tiles > INT_MAX) return DG_ERR_UNSUPPORTED;
    auto short_k_one_wave = [&](const dg_plan& t) {
        const int64_t bk = fp16_in ? 64 : 128;   // one K block (a stage may hold two)
        const int64_t kb = (K + bk - 1) / bk;
        return t.tiles <= t.grid && kb <= 16 && 2 * static_cast<int64_t>(t.tiles) >= sm_count;
    };
    if (!splitk_off && splitk_fits && M <= kSkinnyMaxM) {
        if (!splitk_forced) {
            dg_plan t{};
            t.path = 3;
            plan_tc(M, N, K, fp16_in, sm_count, &t);
            if (short_k_one_wave(t)) {
                *p = t;
                return DG_OK;
            }
        }
        p->path = 4;
        plan_skinny(M, N, K, fp16_in, sm_count, p);
        return DG_OK;
    }
    p->path = 3;
    plan_tc(M, N, K, fp16_in, sm_count, p);
    // Split-K is weighed only where the tiled plan keeps fewer than 3/4 of
    // the SMs busy.  Weighing it against the 96-wide one-wave plans too
    // (the 128-wide plans they replaced were weighed) was measured: 3-4%
    // gained at 17 / 32 x 11008 x 4096 E4M3, 8-20% lost at FP16 17 x 11008
    // x 1040, 32 x 12288 x 1040, 48 x 11008 x 4096 and E4M3 48 x 11008 x
    // 8192, where the split-K estimate is too low.
    const bool weigh = 4 * static_cast<int64_t>(p->grid) < 3 * static_cast<int64_t>(sm_count);
    if (!splitk_off && splitk_fits && M <= kSplitkMaxCols && (splitk_forced || weigh)) {
        dg_plan sk{};
        sk.path = 4;
        plan_skinny(M, N, K, fp16_in, sm_count, &sk);
        if (splitk_forced || splitk_estimate_us(M, N, K, fp16_in, sk) <
                                 tiled_estimate_us(M, N, K, fp16_in, *p))
            *p = sk;
    }
    return DG_OK;
}

dg_status check_sizes(int64_t M, int64_t N, int64_t K) {
    if (M < 0 || N < 0 || K < 0) return DG_ERR_INVALID_VALUE;
    if (M > INT_MAX || N > INT_MAX || K > INT_MAX) return DG_ERR_INVALID_VALUE;
    return DG_OK;
}

// Arguments of the E4M3 GEMM entry points (everything checked before any
// device work; a no-op shape needs no pointers).
dg_status check_fp8_gemm_args(const void* A, const void* B, const void* D, int64_t M,
                              int64_t N, int64_t K, const float* scale_a, const float* scale_b,
                              const float* scale_d, dg_dtype out) {
    const dg_status rc = check_sizes(M, N, K);
    if (rc != DG_OK) return rc;
    if (out != DG_BF16 && out != DG_E4M3 && out != DG_FP16) return DG_ERR_INVALID_VALUE;
    if (M > 0 && N > 0) {
        if (D == nullptr) return DG_ERR_INVALID_VALUE;
        if (K > 0 && (A == nullptr || B == nullptr || scale_a == nullptr || scale_b == nullptr))
            return DG_ERR_INVALID_VALUE;
        if (K > 0 && out == DG_E4M3 && scale_d == nullptr) return DG_ERR_INVALID_VALUE;
        if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (K % 16) != 0)
            return DG_ERR_MISALIGNED;
        if (!aligned4(scale_a) || !aligned4(scale_b) || (out == DG_E4M3 && !aligned4(scale_d)))
            return DG_ERR_MISALIGNED;
    }
    return DG_OK;
}

// Arguments of the FP16 GEMM entry points.
dg_status check_hgemm_args(const void* A, const void* B, const void* D, int64_t M, int64_t N,
                           int64_t K, dg_dtype out) {
    const dg_status rc = check_sizes(M, N, K);
    if (rc != DG_OK) return rc;
    if (out != DG_FP16 && out != DG_BF16) return DG_ERR_INVALID_VALUE;
    if (M > 0 && N > 0) {
        if (D == nullptr) return DG_ERR_INVALID_VALUE;
        if (K > 0 && (A == nullptr || B == nullptr)) return DG_ERR_INVALID_VALUE;
        if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (K % 8) != 0)
            return DG_ERR_MISALIGNED;
    }
    return DG_OK;
}

// The split-K workspace of `s` on the device of `st`: the device-state one
// if no other stream holds it, else one allocated on the stream's first
// split-K call (never while the stream is being captured into a graph).
// *out stays null when the stream already holds none and the per-device cap
// of allocated workspaces is reached.
dg_status splitk_workspace(const DeviceState* st, cudaStream_t s, SplitkWs* out,
                           bool may_allocate = true) {
    std::lock_guard<std::mutex> lk(g_ws_mu[st->device]);
    auto& map = g_ws[st->device];
    *out = SplitkWs{nullptr, nullptr};
    auto it = map.find(s);
    if (it != map.end()) {
        *out = it->second;
        return DG_OK;
    }
    if (!g_dev_ws_taken[st->device]) {
        map[s] = SplitkWs{st->splitk_partials, st->splitk_counts};
        g_dev_ws_taken[st->device] = true;
        *out = map[s];
        return DG_OK;
    }
    if (!may_allocate || map.size() > kMaxStreamWorkspaces) return DG_OK;   // none
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) != cudaSuccess) {
        (void)cudaGetLastError();
        return DG_ERR_CUDA;
    }
    if (cs != cudaStreamCaptureStatusNone) return DG_ERR_UNSUPPORTED;
    const size_t part_bytes = splitk_partial_bytes(st->sm_count);
    void* w = nullptr;
    if (cudaMalloc(&w, part_bytes + kSplitkCountBytes) != cudaSuccess) return DG_ERR_CUDA;
    if (cudaMemset(w, 0, part_bytes + kSplitkCountBytes) != cudaSuccess) {
        cudaFree(w);
        return DG_ERR_CUDA;
    }
    SplitkWs ws{static_cast<float*>(w),
                reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(w) + part_bytes)};
    map[s] = ws;
    *out = ws;
    return DG_OK;
}

dg_status run_gemm(const void* A, const void* B, void* D, int64_t M, int64_t N, int64_t K,
                   bool fp16_in, const float* sa, const float* sb, const float* sd,
                   dg_dtype out, cudaStream_t s, float* amax_d = nullptr) {
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    dg_plan plan;
    rc = make_plan(M, N, K, fp16_in, st->sm_count, &plan);
    if (rc != DG_OK) return rc;
    log_plan(fp16_in ? "hgemm" : "fp8_gemm", M, N, K, plan);
    const int ok = out_kind_of(out);
    uint32_t* amax_bits = reinterpret_cast<uint32_t*>(amax_d);
    if (amax_bits != nullptr) {
        // The running maximum starts at +0 (also the result for an empty or
        // K == 0 product).
        if (launch_zero_word(amax_bits, s) != cudaSuccess) return DG_ERR_CUDA;
    }
    switch (plan.path) {
        case 0:
            return DG_OK;
        case 1:
            return from_cuda(cudaMemsetAsync(D, 0, static_cast<size_t>(M * N * elem_bytes(out)), s));
        case 2:
            return from_cuda(launch_gemv(A, B, D, static_cast<int>(M), static_cast<int>(N),
                                         static_cast<int>(K), fp16_in, sa, sb, sd, ok, amax_bits,
                                         plan.block_n, plan.stages, s));
        case 5:
        case 4:
        default: {
            TcLaunch L;
            L.A = A;
            L.B = B;
            L.D = D;
            L.M = static_cast<int>(M);
            L.N = static_cast<int>(N);
            L.K = static_cast<int>(K);
            L.fp16_in = fp16_in;
            L.sa = sa;
            L.sb = sb;
            L.sd = sd;
            L.out_kind = ok;
            L.out_elem = elem_bytes(out);
            L.plan = &plan;
            L.status = st->status;
            L.amax_out = amax_bits;
            L.group_off = nullptr;
            L.groups = 0;
            if (plan.path == 5) return from_cuda(launch_gemv_mma(L, s));
            if (plan.path == 3 && plan.block_m == 256 &&
                (knobs().split_tail || knobs().stream_k)) {
                // CTA pairs may split tiles along K through the stream's
                // split-K workspace (none, e.g. while a new stream is being
                // captured: every tile runs whole).
                SplitkWs ws;
                if (splitk_workspace(st, s, &ws, /*may_allocate=*/knobs().stream_k) == DG_OK &&
                    ws.partials != nullptr) {
                    L.tail_ws = ws.partials;
                    L.tail_ws_bytes = splitk_partial_bytes(st->sm_count);
                    L.tail_counts = ws.counts;
                }
            }
            if (plan.path == 4 && plan.grid == plan.tiles) {
                // one CTA per tile (row ranges, or as many tiles as CTAs):
                // no partial tiles, so no workspace
                return from_cuda(launch_gemm_skinny(L, nullptr, nullptr, kSplitkMaxCols, s));
            }
            if (plan.path == 4) {
                SplitkWs ws;
                rc = splitk_workspace(st, s, &ws);
                if (rc != DG_OK) return rc;
                if (ws.partials != nullptr)
                    return from_cuda(
                        launch_gemm_skinny(L, ws.partials, ws.counts, kSplitkMaxCols, s));
                // No workspace left for this stream: the tiled kernel, which
                // needs none, computes the same product.
                plan = dg_plan{};
                plan.path = 3;
                plan_tc(M, N, K, fp16_in, st->sm_count, &plan);
                log_plan(fp16_in ? "hgemm (no split-K workspace)" : "fp8_gemm (no split-K workspace)",
                         M, N, K, plan);
            }
            return from_cuda(launch_gemm_tc(L, s));
        }
    }
}

}  // namespace
}  // namespace dg

using namespace dg;

extern "C" {

dg_status dg_amax(const float* x, int64_t n, float* amax_out, float* scale_out,
                  dg_stream_t stream) {
    if (n < 0 || amax_out == nullptr || (n > 0 && x == nullptr)) return DG_ERR_INVALID_VALUE;
    if (!aligned16(x)) return DG_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(amax_out) & 3u) != 0 ||
        (scale_out && (reinterpret_cast<uintptr_t>(scale_out) & 3u) != 0))
        return DG_ERR_MISALIGNED;
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_amax(x, n, amax_out, scale_out, st->sm_count,
                                 reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_amax_pow2(const float* x, int64_t n, float* amax_out, float* scale_out,
                       dg_stream_t stream) {
    if (n < 0 || amax_out == nullptr || scale_out == nullptr || (n > 0 && x == nullptr))
        return DG_ERR_INVALID_VALUE;
    if (!aligned16(x)) return DG_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(amax_out) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(scale_out) & 3u) != 0)
        return DG_ERR_MISALIGNED;
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_amax(x, n, amax_out, scale_out, st->sm_count,
                                 reinterpret_cast<cudaStream_t>(stream), true));
}

dg_status dg_quantize_e4m3(const float* x, int64_t n, const float* scale, uint8_t* q,
                           dg_stream_t stream) {
    if (n < 0 || scale == nullptr || (n > 0 && (x == nullptr || q == nullptr)))
        return DG_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
        return DG_ERR_MISALIGNED;
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_quantize_e4m3(x, n, scale, q, st->sm_count,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_quantize_e4m3_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                float* amax_a, float* amax_b, float* scale_a, float* scale_b,
                                uint8_t* qa, uint8_t* qb, dg_stream_t stream) {
    if (na < 0 || nb < 0 || amax_a == nullptr || amax_b == nullptr || scale_a == nullptr ||
        scale_b == nullptr || (na > 0 && (a == nullptr || qa == nullptr)) ||
        (nb > 0 && (b == nullptr || qb == nullptr)))
        return DG_ERR_INVALID_VALUE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(qa) || !aligned16(qb) || !aligned4(amax_a) ||
        !aligned4(amax_b) || !aligned4(scale_a) || !aligned4(scale_b))
        return DG_ERR_MISALIGNED;
    // four distinct words: two maxima, two scales (scale_a counts CTAs first)
    const float* w[4] = {amax_a, amax_b, scale_a, scale_b};
    for (int i = 0; i < 4; ++i)
        for (int j = i + 1; j < 4; ++j)
            if (w[i] == w[j]) return DG_ERR_INVALID_VALUE;
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_quantize_e4m3_pair(a, na, b, nb, amax_a, amax_b, scale_a, scale_b, qa,
                                               qb, st->sm_count,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_quantize_e4m3_amax(const float* x, int64_t n, const float* scale, uint8_t* q,
                                float* amax_out, float* next_scale_out, dg_stream_t stream) {
    if (n < 0 || scale == nullptr || amax_out == nullptr ||
        (n > 0 && (x == nullptr || q == nullptr)))
        return DG_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scale) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(amax_out) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(next_scale_out) & 3u) != 0)
        return DG_ERR_MISALIGNED;
    if (amax_out == scale) return DG_ERR_INVALID_VALUE;   // zeroed before the scale is read
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_quantize_e4m3_amax(x, n, scale, q, amax_out, next_scale_out,
                                               st->sm_count,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_fp8_gemm(const uint8_t* A, const uint8_t* B, void* D, int64_t M, int64_t N,
                      int64_t K, const float* scale_a, const float* scale_b,
                      const float* scale_d, dg_dtype out, dg_stream_t stream) {
    const dg_status rc = check_fp8_gemm_args(A, B, D, M, N, K, scale_a, scale_b, scale_d, out);
    if (rc != DG_OK) return rc;
    return run_gemm(A, B, D, M, N, K, false, scale_a, scale_b, scale_d, out,
                    reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_fp8_gemm_amax(const uint8_t* A, const uint8_t* B, void* D, int64_t M, int64_t N,
                           int64_t K, const float* scale_a, const float* scale_b,
                           const float* scale_d, dg_dtype out, float* amax_d,
                           dg_stream_t stream) {
    if (amax_d == nullptr) return DG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(amax_d) & 3u) != 0) return DG_ERR_MISALIGNED;
    const dg_status rc = check_fp8_gemm_args(A, B, D, M, N, K, scale_a, scale_b, scale_d, out);
    if (rc != DG_OK) return rc;
    return run_gemm(A, B, D, M, N, K, false, scale_a, scale_b, scale_d, out,
                    reinterpret_cast<cudaStream_t>(stream), amax_d);
}

dg_status dg_fp8_gemm_grouped(const uint8_t* A, const uint8_t* B, void* D, int64_t M, int64_t N,
                              int64_t K, int groups, const int32_t* group_offsets,
                              const float* scale_a, const float* scale_b, const float* scale_d,
                              dg_dtype out, dg_stream_t stream) {
    dg_status rc = check_sizes(M, N, K);
    if (rc != DG_OK) return rc;
    if (groups < 1 || groups > kMaxGemmGroups || group_offsets == nullptr) return DG_ERR_INVALID_VALUE;
    if (out != DG_BF16 && out != DG_E4M3 && out != DG_FP16) return DG_ERR_INVALID_VALUE;
    if (static_cast<int64_t>(groups) * N > INT_MAX) return DG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(group_offsets) & 3u) != 0) return DG_ERR_MISALIGNED;
    if (M == 0 || N == 0) return DG_OK;
    if (D == nullptr) return DG_ERR_INVALID_VALUE;
    if (K > 0 && (A == nullptr || B == nullptr || scale_a == nullptr || scale_b == nullptr))
        return DG_ERR_INVALID_VALUE;
    if (K > 0 && out == DG_E4M3 && scale_d == nullptr) return DG_ERR_INVALID_VALUE;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (K % 16) != 0) return DG_ERR_MISALIGNED;
    if (!aligned4(scale_a) || !aligned4(scale_b) || (out == DG_E4M3 && !aligned4(scale_d)))
        return DG_ERR_MISALIGNED;
    DeviceState* st = nullptr;
    rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (K == 0)
        return from_cuda(cudaMemsetAsync(D, 0, static_cast<size_t>(M * N * elem_bytes(out)), s));
    dg_plan plan{};
    plan.path = 3;
    plan.block_m = 128;
    plan.block_n = N >= 512 ? 256 : 128;
    plan.block_k = 128;
    // Upper bound on tiles: each group adds at most one partial 128-row tile.
    const int64_t num_n = (N + plan.block_n - 1) / plan.block_n;
    const int64_t tiles = ((M + 127) / 128 + groups) * num_n;
    if (tiles > INT_MAX) return DG_ERR_UNSUPPORTED;
    plan.tiles = static_cast<int>(tiles);
    plan.grid = static_cast<int>(tiles < st->sm_count ? tiles : st->sm_count);
    log_plan("fp8_gemm_grouped", M, N, K, plan);
    TcLaunch L{};
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
    L.status = st->status;
    L.amax_out = nullptr;
    L.group_off = group_offsets;
    L.groups = groups;
    return from_cuda(launch_gemm_tc_grouped(L, s));
}

dg_status dg_hgemm(const uint16_t* A, const uint16_t* B, void* D, int64_t M, int64_t N,
                   int64_t K, dg_dtype out, dg_stream_t stream) {
    const dg_status rc = check_hgemm_args(A, B, D, M, N, K, out);
    if (rc != DG_OK) return rc;
    return run_gemm(A, B, D, M, N, K, true, nullptr, nullptr, nullptr, out,
                    reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_hgemm_scaled(const uint16_t* A, const uint16_t* B, void* D, int64_t M, int64_t N,
                          int64_t K, const float* scale_a, const float* scale_b, dg_dtype out,
                          dg_stream_t stream) {
    if (scale_a == nullptr || scale_b == nullptr) return DG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(scale_a) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(scale_b) & 3u) != 0)
        return DG_ERR_MISALIGNED;
    const dg_status rc = check_hgemm_args(A, B, D, M, N, K, out);
    if (rc != DG_OK) return rc;
    return run_gemm(A, B, D, M, N, K, true, scale_a, scale_b, nullptr, out,
                    reinterpret_cast<cudaStream_t>(stream));
}

dg_status dg_fp16_range_scale(const float* amax_a, const float* amax_b, float* factors,
                              dg_stream_t stream) {
    if (amax_a == nullptr || amax_b == nullptr || factors == nullptr) return DG_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(amax_a) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(amax_b) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(factors) & 15u) != 0)
        return DG_ERR_MISALIGNED;
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_fp16_range_scale(amax_a, amax_b, factors,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_convert_f16(const float* x, int64_t n, const float* factor, uint16_t* out,
                         dg_stream_t stream) {
    if (n < 0 || (n > 0 && (x == nullptr || out == nullptr))) return DG_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(factor) & 3u) != 0)
        return DG_ERR_MISALIGNED;
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_convert_f16(x, n, factor, out, st->sm_count,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_convert_f16_amax(const float* x, int64_t n, const float* factor, uint16_t* out,
                              float* amax_out, dg_stream_t stream) {
    if (n < 0 || amax_out == nullptr || (n > 0 && (x == nullptr || out == nullptr)))
        return DG_ERR_INVALID_VALUE;
    if (!aligned16(x) || !aligned16(out) || !aligned4(factor) || !aligned4(amax_out))
        return DG_ERR_MISALIGNED;
    if (amax_out == factor) return DG_ERR_INVALID_VALUE;   // zeroed before the factor is read
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_convert_f16_amax(x, n, factor, out, amax_out, st->sm_count,
                                             reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_convert_f16_amax_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                   const float* factor, uint16_t* out_a, uint16_t* out_b,
                                   float* amax_a, float* amax_b, dg_stream_t stream) {
    if (na < 0 || nb < 0 || amax_a == nullptr || amax_b == nullptr ||
        (na > 0 && (a == nullptr || out_a == nullptr)) || (nb > 0 && (b == nullptr || out_b == nullptr)))
        return DG_ERR_INVALID_VALUE;
    if (!aligned16(a) || !aligned16(b) || !aligned16(out_a) || !aligned16(out_b) ||
        !aligned4(factor) || !aligned4(amax_a) || !aligned4(amax_b))
        return DG_ERR_MISALIGNED;
    // both words are zeroed before the pass reads the factor, and each
    // collects one tensor's maximum
    if (amax_a == amax_b || amax_a == factor || amax_b == factor) return DG_ERR_INVALID_VALUE;
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    return from_cuda(launch_convert_f16_amax_pair(a, na, b, nb, factor, out_a, out_b, amax_a, amax_b,
                                                  st->sm_count,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

dg_status dg_gemm_plan(int64_t M, int64_t N, int64_t K, dg_dtype in, dg_dtype out,
                       int sm_count, dg_plan* plan) {
    if (plan == nullptr) return DG_ERR_INVALID_VALUE;
    dg_status rc = check_sizes(M, N, K);
    if (rc != DG_OK) return rc;
    if (in != DG_E4M3 && in != DG_FP16) return DG_ERR_INVALID_VALUE;
    if (out != DG_BF16 && out != DG_E4M3 && out != DG_FP16) return DG_ERR_INVALID_VALUE;
    if (sm_count <= 0) {
        DeviceState* st = nullptr;
        rc = current_device_state(&st);
        if (rc != DG_OK) return rc;
        sm_count = st->sm_count;
    }
    return make_plan(M, N, K, in == DG_FP16, sm_count, plan);
}

dg_status dg_init(void) {
    DeviceState* st = nullptr;
    return current_device_state(&st);
}

dg_status dg_sync_status(dg_stream_t stream) {
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return DG_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, st->status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
        return DG_ERR_CUDA;
    if (word != 0) {
        if (cudaMemset(st->status, 0, sizeof(word)) != cudaSuccess) return DG_ERR_CUDA;
        if (word & kStatusTimeout) {
            // A CTA that gave up may have left split-K arrival counters
            // part-way: clear them (every launch expects zeros).
            if (cudaDeviceSynchronize() != cudaSuccess ||
                cudaMemset(st->splitk_counts, 0, kSplitkCountBytes) != cudaSuccess)
                return DG_ERR_CUDA;
            std::lock_guard<std::mutex> lk(g_ws_mu[st->device]);
            for (auto& kv : g_ws[st->device])
                if (cudaMemset(kv.second.counts, 0, kSplitkCountBytes) != cudaSuccess)
                    return DG_ERR_CUDA;
            return DG_ERR_TIMEOUT;
        }
        if (word & kStatusBadArgument) return DG_ERR_INVALID_VALUE;
    }
    return DG_OK;
}

dg_status dg_release_stream(dg_stream_t stream) {
    DeviceState* st = nullptr;
    dg_status rc = current_device_state(&st);
    if (rc != DG_OK) return rc;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lk(g_ws_mu[st->device]);
    auto& map = g_ws[st->device];
    auto it = map.find(s);
    if (it == map.end()) return DG_OK;
    // The stream's earlier split-K launches may still be running.
    if (cudaStreamSynchronize(s) != cudaSuccess) return DG_ERR_CUDA;
    if (it->second.partials == st->splitk_partials) {
        g_dev_ws_taken[st->device] = false;
    } else if (cudaFree(it->second.partials) != cudaSuccess) {
        return DG_ERR_CUDA;
    }
    map.erase(it);
    return DG_OK;
}

void dg_reload_env(void) {
    const Knobs* k = new Knobs(read_knobs());
    (void)knobs();   // the first snapshot exists before it is replaced
    g_knobs.store(k, std::memory_order_release);
}

void dg_set_wait_timeout_us(uint64_t us) {
    g_timeout_ns.store(us * 1000ull, std::memory_order_relaxed);
}

void dg_debug_skip_first_load(int enable) { g_skip_first_load.store(enable ? 1 : 0); }

const char* dg_status_string(dg_status s) {
    switch (s) {
        case DG_OK: return "DG_OK";
        case DG_ERR_INVALID_VALUE: return "DG_ERR_INVALID_VALUE";
        case DG_ERR_MISALIGNED: return "DG_ERR_MISALIGNED";
        case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED";
        case DG_ERR_CUDA: return "DG_ERR_CUDA";
        case DG_ERR_TIMEOUT: return "DG_ERR_TIMEOUT";
    }
    return "DG_ERR_UNKNOWN";
}

int dg_version(void) { return 100; }

}  // extern "C"
