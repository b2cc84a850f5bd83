/*
 * dg.h -- C ABI of libdg: per-tensor-scaled E4M3 GEMM, FP16 GEMM and the
 * E4M3 quantiser on one NVIDIA GB300 (sm_103a).
 *
 * Page shorthands used in the citations:
 *   [FP8-guide] "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南"
 *               (sheratonhq.com/news/156926), sections as numbered there.
 *   [DG-FP16]   the DeepGEMM FP16/WMMA deep-dive page (hnwysp.cn/news/84236).
 *   [HGEMM-L2]  "HGEMM优化：深度学习中的矩阵乘法性能提升策略"
 *               (jsqmd.com/news/710660).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.    Every data pointer is DEVICE memory on the current CUDA device,
 *            owned by the caller.  The library allocates nothing per call and
 *            takes no workspace argument.  The first call on a device (or
 *            dg_init) allocates a 16-byte device status word and a split-K
 *            workspace (two 128 x 128 FP32 partial tiles per SM and 8192
 *            counters, 20 MB on 152 SMs) that live until exit.  Split-K
 *            GEMMs (plan path 4) issued on a second, third, ... stream get a
 *            workspace of their own (same size) on that stream's first such
 *            call, so calls on different streams may run concurrently; that
 *            first call must not happen while the stream is being captured
 *            into a graph (it returns DG_ERR_UNSUPPORTED then).  A stream
 *            keeps its workspace until dg_release_stream(stream) or exit.
 *            At most 16 streams per device hold an allocated one at a time;
 *            past that, split-K shapes on further streams run on the tiled
 *            tensor-core kernel (no workspace, same tolerance).  A graph
 *            captured on a stream refers to that stream's workspace: do not
 *            replay it concurrently with another replay of itself or with
 *            split-K work (or DG_SPLIT_TAIL / DG_STREAM_K pair GEMMs) on the
 *            capturing stream; replays in stream order are fine.
 * Layout.    Dense, row-major, no leading-dimension arguments: A is M x K,
 *            B is N x K (both K contiguous, the "TN" form), D is M x N.
 * Alignment. Every data pointer must be 16-byte aligned, every FP32 device
 *            scalar (scales, amax words) 4-byte aligned, and K * element
 *            size must be a multiple of 16 bytes; otherwise the call returns
 *            DG_ERR_MISALIGNED and launches nothing (there is no slow path).
 * Streams.   Work is enqueued on `stream` (NULL = the legacy default stream)
 *            and nothing synchronises the host.  Scales are device pointers
 *            so that amax -> quantise -> GEMM needs no host round trip.
 * Errors.    Argument errors return a status and launch nothing.  A failed
 *            launch returns DG_ERR_CUDA.  Every wait inside a kernel is
 *            bounded; a wait that runs out records DG_ERR_TIMEOUT in the
 *            device status word, the kernel returns cleanly, and
 *            dg_sync_status() reports it.
 * Aliasing.  Outputs must not overlap inputs.
 * Threads.   Entry points are thread-safe; per-device set-up runs once.
 */
#ifndef DG_H
#define DG_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that the header needs no CUDA
 * include. */
typedef struct CUstream_st* dg_stream_t;

typedef enum {
    DG_OK = 0,
    DG_ERR_INVALID_VALUE = 1, /* null pointer, negative size, bad dtype     */
    DG_ERR_MISALIGNED = 2,    /* pointer or row pitch not 16-byte aligned   */
    DG_ERR_UNSUPPORTED = 3,   /* no CUDA device of compute capability 10.3  */
    DG_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed          */
    DG_ERR_TIMEOUT = 5        /* a bounded in-kernel wait ran out           */
} dg_status;

typedef enum {
    DG_BF16 = 0, /* bfloat16, round to nearest even                        */
    DG_E4M3 = 1, /* E4M3 "fn": bias 7, max 448, no Inf, RNE, saturating    */
    DG_FP16 = 2  /* IEEE binary16, round to nearest even                   */
} dg_dtype;

/* amax and scale.  [FP8-guide] §3.2: the per-tensor scale is the largest
 * absolute value of the tensor divided by 448, the largest E4M3 value.
 *   x          FP32[n], device, 16-byte aligned.
 *   amax_out   FP32[1], device: max_i |x_i|; NaN if any x_i is NaN; 0 for
 *              n == 0.
 *   scale_out  FP32[1], device, may be NULL: amax / 448 as one binary32
 *              division, or 1 when amax == 0.
 * Two kernel launches on the stream: a one-thread kernel that zeroes
 * amax_out (and scale_out, which counts the reduction's CTAs until the
 * last one writes the scale over the count), and the reduction.  When
 * n == 0 or scale_out == amax_out, a third one-thread kernel forms the
 * scale after the reduction instead.  scale_out holds no scale while the
 * call runs. */
dg_status dg_amax(const float* x, int64_t n, float* amax_out, float* scale_out,
                  dg_stream_t stream);

/* amax and a power-of-two scale.  [FP8-guide] §2.1: instead of amax/448
 * itself, take a power of two just above it, so that scaling and unscaling
 * are exponent shifts (division by the scale is exact).
 *   amax_out   FP32[1], device: as dg_amax.
 *   scale_out  FP32[1], device, required: the smallest power of two p
 *              (2^-149 <= p) with 448 * p >= amax, compared exactly; 1 when
 *              amax == 0; NaN for NaN and +Inf for +Inf inputs.
 * The tensor's largest magnitude quantises into (224, 448]: no saturation,
 * at most one binade of the E4M3 range unused.  Errors as dg_amax. */
dg_status dg_amax_pow2(const float* x, int64_t n, float* amax_out,
                       float* scale_out, dg_stream_t stream);

/* E4M3 quantiser.  [FP8-guide] §4.3: fp8 = clamp(round(x / scale), -448,
 * 448), implemented as q_i = E4M3(fl32(x_i / *scale)) with an IEEE binary32
 * division and round-to-nearest-even, saturating to +-448; NaN -> 0x7F.
 *   x      FP32[n], device, 16-byte aligned.
 *   scale  FP32[1], device.
 *   q      uint8[n] E4M3 codes, device, 16-byte aligned; same order as x. */
dg_status dg_quantize_e4m3(const float* x, int64_t n, const float* scale,
                           uint8_t* q, dg_stream_t stream);

/* Both operands of the E4M3 GEMM prepared in one call: amax and scale of a
 * and of b (as dg_amax), then each quantised with its own scale (as
 * dg_quantize_e4m3).  [FP8-guide] §3.2 scales each operand by its own
 * amax / 448 before the GEMM.  Three kernel launches: a one-thread kernel
 * zeroes the two maxima (and scale_a, which counts the reduction's CTAs
 * until the last one writes both scales), one grid takes the maxima of a
 * and then b, one grid quantises a and b.  The results are bit-identical to
 * dg_amax + dg_quantize_e4m3 on each tensor; the grids stream on from one
 * tensor to the next without a launch boundary between them.
 *   a, b          FP32[na], FP32[nb], device, 16-byte aligned (na, nb >= 0)
 *   amax_a/_b     FP32 device words: max |a|, max |b| (NaN propagates)
 *   scale_a/_b    FP32 device words: amax / 448, or 1 when amax == 0
 *   qa, qb        uint8[na], uint8[nb] E4M3 codes, 16-byte aligned
 * The four words must be distinct and 4-byte aligned (DG_ERR_INVALID_VALUE,
 * DG_ERR_MISALIGNED). */
dg_status dg_quantize_e4m3_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                float* amax_a, float* amax_b, float* scale_a, float* scale_b,
                                uint8_t* qa, uint8_t* qb, dg_stream_t stream);

/* Per-tensor-scaled E4M3 GEMM.  [FP8-guide] §2.1, §3.2, §3.3:
 *   D[m,n] = out( scale_a * scale_b * sum_k A[m,k] * B[n,k] )
 * with FP8 inputs, FP32 accumulation and the scales applied once to the
 * accumulator on write-back.  For out == DG_E4M3 the value is divided by
 * *scale_d before the saturating E4M3 rounding.
 *   A        uint8 E4M3 codes, M x K row-major, device.
 *   B        uint8 E4M3 codes, N x K row-major (K contiguous), device.
 *   D        M x N row-major of `out` (DG_BF16, DG_E4M3 or DG_FP16), device.
 *            Elements outside [0,M) x [0,N) are never touched.
 *   scale_a, scale_b  FP32[1], device.
 *   scale_d  FP32[1], device; required iff out == DG_E4M3, else ignored.
 *   M, N, K  >= 0 and < 2^31.  M == 0 or N == 0 is a no-op; K == 0 writes
 *            zeros.  K must be a multiple of 16 (row pitch alignment).
 * Paths (dg_gemm_plan reports the one taken): M <= 8 a bandwidth-bound
 * GEMV that streams B into registers and sums K on warp-level MMAs (up to
 * M = 16 for FP16 operands or small N * K; the CUDA-core GEMV for M = 1 when
 * N is too large for one wave of its CTAs) ([DG-FP16] §2.1 and §4.1, the
 * decode QKV projection); 9 <= M <= 16 a split-K tensor-core kernel
 * (operands swapped, K spread over every SM), or over a short K the tiled
 * kernel when its tiles fill at least half the SMs in one wave; larger M
 * the tiled tensor-core kernel with a tile chosen per shape, or for
 * 17 <= M <= 128 the split-K kernel where the tiled one would leave SMs
 * idle and a time estimate favours split-K (few rows of A against a long
 * K).  K tails are zero-filled by the tensor-memory loads and M/N edges are
 * predicated or clipped stores ([FP8-guide] §3.3).
 */
dg_status dg_fp8_gemm(const uint8_t* A, const uint8_t* B, void* D, int64_t M,
                      int64_t N, int64_t K, const float* scale_a,
                      const float* scale_b, const float* scale_d, dg_dtype out,
                      dg_stream_t stream);

/* dg_fp8_gemm that also reports the output's largest magnitude, for delayed
 * output scaling.  [FP8-guide] §3.2: calibration records each GEMM's largest
 * absolute output, and the output scale is that value over 448.  Besides
 * everything dg_fp8_gemm does, this call writes
 *   *amax_d = max over m < M, n < N of |scale_a * scale_b * acc[m,n]|
 * -- the unrounded output before the division by scale_d and the output
 * rounding -- in binary32 (NaN-propagating; +0 when M, N or K is 0), so that
 * the next call's output scale can be fl32(*amax_d / 448) with no host round
 * trip.  The maximum is taken on the epilogue's registers: no extra pass
 * over D.
 *   amax_d  FP32[1], device, 4-byte aligned; zeroed by the call (a
 *           one-thread kernel) before the GEMM runs.
 * Other arguments, layouts and errors as dg_fp8_gemm; amax_d == NULL is
 * DG_ERR_INVALID_VALUE. */
dg_status dg_fp8_gemm_amax(const uint8_t* A, const uint8_t* B, void* D,
                           int64_t M, int64_t N, int64_t K,
                           const float* scale_a, const float* scale_b,
                           const float* scale_d, dg_dtype out, float* amax_d,
                           dg_stream_t stream);

/* Grouped per-tensor-scaled E4M3 GEMM: a batch of GEMMs that share N and K
 * (the expert projections of a mixture-of-experts layer) in one launch.
 * [DG-FP16] §1 (an MoE forward pass as the workload) and [FP8-guide] §4.4
 * (merge many small GEMMs into one launch).  Group g, 0 <= g < groups,
 * computes rows [off[g], off[g+1]) of D:
 *   D[m,n] = out( scale_a[g] * scale_b[g] * sum_k A[m,k] * B[g*N + n, k] )
 * (divided by scale_d[g] before the rounding when out == DG_E4M3).
 *   A      M x K E4M3 codes, the groups' rows stacked, device.
 *   B      (groups * N) x K E4M3 codes: group g's N x K matrix at rows g*N.
 *   D      M x N of `out`, device.
 *   group_offsets  int32[groups + 1], device, 4-byte aligned:
 *          0 = off[0] <= off[1] <= ... <= off[groups] = M.  Read by the
 *          kernel (no host round trip, no padding of group sizes; empty
 *          groups allowed).  Offsets that break these rules make the kernel
 *          store nothing and dg_sync_status report DG_ERR_INVALID_VALUE.
 *   scale_a, scale_b  FP32[groups], device; scale_d FP32[groups], device,
 *          required iff out == DG_E4M3.
 *   groups 1 .. 1024.
 * Layout, alignment and other errors as dg_fp8_gemm.  The tiles are 128 x
 * BN per group (one tensor-core kernel, tiles of all groups scheduled over
 * all SMs). */
dg_status dg_fp8_gemm_grouped(const uint8_t* A, const uint8_t* B, void* D,
                              int64_t M, int64_t N, int64_t K, int groups,
                              const int32_t* group_offsets,
                              const float* scale_a, const float* scale_b,
                              const float* scale_d, dg_dtype out,
                              dg_stream_t stream);

/* dg_quantize_e4m3 with a scale recorded earlier (delayed scaling), fused
 * with the amax of this tensor for the next call: one pass over x writes
 * q[i] = e4m3(fl32(x[i] / scale[0])) and amax_out[0] = max |x| (NaN
 * propagates), then, if next_scale_out is not NULL, next_scale_out[0] =
 * amax / 448 (1 when amax == 0) — the same rules as dg_amax and
 * dg_quantize_e4m3.  [FP8-guide] §3.2: the calibration run records each
 * tensor's largest magnitude and the scale comes from it; here the record
 * of one call scales the next, so amax and quantisation share one read.
 * next_scale_out may be the same buffer as scale (it is then written by a
 * one-thread kernel after the pass; otherwise the pass's last CTA writes
 * it, the word counting the CTAs until then); amax_out must not be scale.
 * Pointers as dg_quantize_e4m3 and dg_amax. */
dg_status dg_quantize_e4m3_amax(const float* x, int64_t n, const float* scale,
                                uint8_t* q, float* amax_out,
                                float* next_scale_out, dg_stream_t stream);

/* dg_fp8_gemm for skinny shapes (1 <= M <= 16) that never allocates: the
 * split-K tensor-core kernel (plan path 4) runs with its workspace in fixed
 * static device arrays of the library (2.5 MiB of FP32 partial tiles and
 * 1025 32-bit words) instead of memory the library allocates.  The pages
 * have no counterpart.  It is for callers that cannot let a library call
 * cudaMalloc: a process whose own pool allocator has already reserved the
 * device memory, code running while a stream is captured in global mode
 * (where cudaMalloc is refused), or a latency-bound loop that cannot take
 * cudaMalloc's implicit synchronisation.  For the same arguments the
 * result is bit-identical to dg_fp8_gemm on the split-K path.
 *   A, B, D, M, N, K, scale_a, scale_b, scale_d, out, stream: as
 *          dg_fp8_gemm, with M <= 16 and N <= 131072 (1024 tiles of 128
 *          rows of B); larger sizes return DG_ERR_INVALID_VALUE.
 *   status_out  optional device uint32, 4-byte aligned: the kernel ORs its
 *          error bits into it (1 = a bounded wait ran out, the output is
 *          incomplete).  It is the only way to learn of a timeout on this
 *          entry point: dg_sync_status does not see these bits, and with
 *          status_out NULL they go to a library word nobody reads.
 * Each call first zeroes the arrival counters of the static workspace on
 * `stream` (cudaMemsetAsync), then launches the kernel.  Calls share that one
 * workspace per device: two calls whose executions overlap (different
 * streams without ordering between them) race and give wrong results.  The
 * first call on each device looks the arrays' addresses up and sets the
 * kernel's shared-memory limit; make that first call before capturing a
 * stream into a CUDA graph.  No memory is allocated or freed by this call.
 */
dg_status dg_fp8_gemm_splitk_static(const uint8_t* A, const uint8_t* B, void* D,
                                    int64_t M, int64_t N, int64_t K,
                                    const float* scale_a, const float* scale_b,
                                    const float* scale_d, dg_dtype out,
                                    uint32_t* status_out, dg_stream_t stream);

/* FP16 GEMM (HGEMM), FP32 accumulation, no scaling.  [HGEMM-L2] §1.3 (FP16
 * inputs, FP32 accumulator) and §3; same layouts and edge rules as
 * dg_fp8_gemm.  A, B hold IEEE binary16 bit patterns.  K must be a multiple
 * of 8.  out is DG_FP16 or DG_BF16. */
dg_status dg_hgemm(const uint16_t* A, const uint16_t* B, void* D, int64_t M,
                   int64_t N, int64_t K, dg_dtype out, dg_stream_t stream);

/* HGEMM with per-tensor scales in the epilogue: D = out(scale_a * scale_b *
 * A * B^T), FP32 accumulation.  As dg_hgemm otherwise; scale_a, scale_b are
 * FP32 device scalars (both required, 4-byte aligned).  With the factors of
 * dg_fp16_range_scale (scale_a = &factors[2], scale_b = &factors[3]) this is
 * the last step of [DG-FP16] §3.3's dynamic-range scaling: the result is
 * divided by the scale the operands were multiplied with (as 1/scale). */
dg_status dg_hgemm_scaled(const uint16_t* A, const uint16_t* B, void* D,
                          int64_t M, int64_t N, int64_t K,
                          const float* scale_a, const float* scale_b,
                          dg_dtype out, dg_stream_t stream);

/* [DG-FP16] §3.3 dynamic-range-aware scaling for FP16 operands: from the
 * two maxima (e.g. dg_amax of A and of B, FP32 device scalars) it writes
 * factors[0..3] = { scale, sqrt(scale), 1/scale, 1 } with
 * scale = min(1, 65504 / (amax_a * amax_b)): the product and quotient are
 * formed in binary64 and rounded once to binary32; sqrt and the reciprocal
 * are correctly rounded binary32 values of that scale.  1 when a maximum is
 * 0; NaN when one is NaN.  factors: device, 4 floats, 16-byte aligned,
 * caller-owned.  The scale bounds every |a * b| * scale by 65504; a single
 * operand value still overflows FP16 after the sqrt(scale) multiply if
 * max|A| / max|B| (or its inverse) exceeds 65504. */
dg_status dg_fp16_range_scale(const float* amax_a, const float* amax_b,
                              float* factors, dg_stream_t stream);

/* out[i] = fp16_rn(fl32(x[i] * factor[0])), IEEE round-to-nearest-even,
 * overflow to +-Inf, NaN stays NaN.  x: n FP32, out: n binary16 bit
 * patterns, both device, 16-byte aligned, caller-owned; factor: FP32 device
 * scalar (NULL = 1), e.g. &factors[1] of dg_fp16_range_scale.  An HBM
 * stream (6 B per element). */
dg_status dg_convert_f16(const float* x, int64_t n, const float* factor,
                         uint16_t* out, dg_stream_t stream);

/* dg_convert_f16 with a factor recorded earlier (delayed scaling), fused
 * with the amax of this tensor for the next call: one pass over x writes
 * out[i] = fp16_rn(fl32(x[i] * factor[0])) and amax_out[0] = max |x|
 * (NaN propagates; 0 for n == 0).  [DG-FP16] §3.3 forms the scale from the
 * two operands' maxima; recording them while converting (as [FP8-guide]
 * §3.2's calibration records each tensor's maximum) lets the factors of the
 * next call come from dg_fp16_range_scale on these maxima, so each operand
 * is read once per call instead of twice.  amax_out: FP32 device word,
 * 4-byte aligned, zeroed by the call (a one-thread kernel) before the pass;
 * it must not be the factor word.  Other arguments and errors as
 * dg_convert_f16; factor NULL = 1. */
dg_status dg_convert_f16_amax(const float* x, int64_t n, const float* factor,
                              uint16_t* out, float* amax_out,
                              dg_stream_t stream);

/* dg_convert_f16_amax for both operands of the scaled HGEMM in one pass:
 * out_a[i] = fp16_rn(fl32(a[i] * factor[0])), out_b[i] likewise from b, and
 * amax_a[0] = max |a|, amax_b[0] = max |b|.  [DG-FP16] §3.3 multiplies both
 * operands by the same factor (the square root of the range scale); the
 * next call's factors come from dg_fp16_range_scale(amax_a, amax_b, ...).
 * Two kernel launches: a one-thread kernel zeroes both maxima, then one
 * grid converts a and b (half the launches of two dg_convert_f16_amax
 * calls).  amax_a and amax_b: distinct FP32 device words, 4-byte aligned,
 * neither the factor word (DG_ERR_INVALID_VALUE).  Other arguments and
 * errors as dg_convert_f16_amax; na or nb may be 0. */
dg_status dg_convert_f16_amax_pair(const float* a, int64_t na, const float* b, int64_t nb,
                                   const float* factor, uint16_t* out_a, uint16_t* out_b,
                                   float* amax_a, float* amax_b, dg_stream_t stream);

/* Tile / path selection for a GEMM shape, host only (launches nothing).
 * [FP8-guide] §2.2, §3.1, §3.3 (per-shape tile choice, smaller tiles where
 * edge waste is high) and [HGEMM-L2] §3.1-§3.3 (tile and stage count chosen
 * from M, N, K); here the choice comes from a compiled table instead of a
 * JIT.  in is DG_E4M3 or DG_FP16.  sm_count <= 0 queries the current device.
 */
typedef struct {
    int path;       /* 0 no-op, 1 zero-fill (K == 0), 2 GEMV, 3 tensor core,
                       4 split-K tensor core for M <= 16 (unless a short K
                       lets one wave of tiles fill half the SMs), and for
                       M <= 128 where it is estimated faster (operands
                       swapped: block_m = 16, 32, 64 or 128 padded rows of
                       A, block_n = 128 rows of B per tile, K blocks of all
                       tiles spread over grid CTAs; with DG_SPLITK_ROWS=1
                       and N <= 128 x SMs, block_n = ceil(N / SMs) rows of
                       B per CTA over the whole of K, grid = tiles, no
                       workspace), 5 warp-MMA GEMV for
                       M <= 16 (block_n = 16 rows of B per CTA, the K sum
                       split over `stages` warps, block_k = K elements per
                       warp step)                                           */
    int block_m;    /* output rows per tile (tensor-core paths)             */
    int block_n;    /* output columns per tile                              */
    int block_k;    /* K elements per pipeline stage                        */
    int stages;     /* shared-memory pipeline depth; for the GEMV (path 2)
                       the 16-byte chunks per lane per row of B in flight   */
    int grid;       /* CTAs launched                                        */
    int tiles;      /* output tiles (tensor-core paths)                     */
    int smem_bytes; /* dynamic shared memory per CTA                        */
} dg_plan;

dg_status dg_gemm_plan(int64_t M, int64_t N, int64_t K, dg_dtype in,
                       dg_dtype out, int sm_count, dg_plan* plan);

/* Per-device set-up for the current device: checks compute capability 10.3
 * and allocates the device status word.  Optional (every entry point does it
 * on first use); call it before capturing a stream into a CUDA graph. */
dg_status dg_init(void);

/* Synchronises `stream`, then returns and clears the current device's
 * status word: DG_ERR_TIMEOUT if a kernel's bounded wait ran out since the
 * last call, DG_ERR_CUDA if the synchronisation failed, else DG_OK. */
dg_status dg_sync_status(dg_stream_t stream);

/* Gives back the split-K workspace that `stream` holds on the current
 * device (see Memory above): synchronises the stream, then frees the
 * workspace (or returns the device's own to the pool).  Call it before
 * destroying a stream that ran split-K GEMMs; a later split-K call on the
 * stream takes a workspace again.  A stream that holds none: DG_OK, no
 * synchronisation.  DG_ERR_CUDA if the synchronisation or the free fails.
 * Not while the stream is being captured, nor concurrently with GEMM calls
 * on the same stream. */
dg_status dg_release_stream(dg_stream_t stream);

/* Re-reads the DG_* tuning variables of the environment (tile, path and
 * launch switches used for sweeps and tests).  They are otherwise read
 * once, at the library's first call; no call reads the environment
 * again.  Applies to calls made afterwards.  None changes what is
 * computed, only which kernel and launch shape compute it (the results
 * stay within the same tolerance; values outside the ranges below are
 * ignored):
 *   DG_LOG=1              one stderr line per GEMM call (path and tile)
 *   DG_PDL=0              no programmatic dependent launch (launch overlap)
 *   DG_MMA_GEMV=0|1       warp-MMA GEMV off / for every M <= 16 (plan path 5)
 *   DG_MMA_GEMV_WARPS=n   its warps per CTA (2, 3, 4 or 8)
 *   DG_GEMV_MAX_M=n       largest M on the CUDA-core GEMV (0..16; default 2)
 *   DG_GEMV_ROWS=n        its rows of B per CTA at M <= 2 (4, 8 or 16)
 *   DG_SPLITK=0|1         split-K off / for every M <= 128
 *   DG_SPLITK_GRID=n      CTAs of a split-K launch
 *   DG_SPLITK_KPS=1|2     K blocks per split-K pipeline stage (default 2)
 *   DG_SPLITK_PREFETCH=n  B boxes a split-K CTA moves into L2 before its
 *                         dependency wait (0..256; default one ring)
 *   DG_SPLITK_ROWS=1      split-K in row ranges: ceil(N / SMs) rows of B
 *                         per CTA over the whole of K, no workspace
 *   DG_SPLITK_TILE_ROWS=n rows of B per split-K tile (16..128, a multiple
 *                         of 8; default 128)
 *   DG_2CTA=0|1           CTA pairs off / for every M >= 256
 *   DG_FORCE_BLOCK_N=n    tile width of the tiled kernels (64..256)
 *   DG_GROUP_M=n          raster group of M tiles (1..4096)
 *   DG_PAIR_KPS=1|2       CTA-pair tiles: one or two K blocks per pipeline
 *                         stage (default: two from 12 K blocks on)
 *   DG_TC_KPS=1|2         one-wave single-CTA plans up to 128 wide: one or
 *                         two K blocks per pipeline stage (default: two
 *                         from 12 K blocks on)
 *   DG_TC_SHORT_BOX=0|1|2 single-CTA tiled kernel: operand boxes of full
 *                         height / of the operand's rows rounded up to 8
 *                         when it has at most 32 / whenever it is shorter
 *                         than its box (default)
 *   DG_ONE_WAVE=0         no one-wave tile rule; DG_ONE_WAVE_KB=n its
 *                         K-block limit (default 64)
 *   DG_STAGED_EPI=0       tiled epilogues store rows directly instead of
 *                         through staging boxes and bulk tensor stores
 *   DG_EARLY_RELEASE=0    tiled kernels release the next launch at exit
 *                         instead of once every CTA is on its last tile
 *   DG_SPLIT_TAIL=1       CTA pairs split the tiles of a partial last
 *                         round along K over the idle pairs
 *   DG_STREAM_K=1         CTA pairs run whole-tile rounds, then equal
 *                         (tile, K block) ranges over the last rounds
 * DG_SPLIT_TAIL and DG_STREAM_K use the stream's split-K workspace (see
 * Memory above); without one the tiles run whole. */
void dg_reload_env(void);

/* Upper bound, in microseconds, on any single in-kernel wait (default
 * 2 000 000).  Applies to launches made after the call. */
void dg_set_wait_timeout_us(uint64_t us);

/* Test hook: when non-zero, the next tensor-core GEMM launch leaves the
 * first shared-memory stage of its first tile unloaded, so that the MMA
 * warp's wait on it runs out (bounded) and the kernel reports
 * DG_ERR_TIMEOUT.  Resets itself after one launch. */
void dg_debug_skip_first_load(int enable);

/* Human-readable name of a status code (static storage). */
const char* dg_status_string(dg_status s);

/* Library version, major * 10000 + minor * 100 + patch. */
int dg_version(void);

#ifdef __cplusplus
}
#endif
#endif /* DG_H */
