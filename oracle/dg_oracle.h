/*
 * dg_oracle.h -- plain, slow CPU oracle for the per-tensor-scaled E4M3 GEMM,
 * its FP16 sibling (HGEMM) and the E4M3 quantiser.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this code; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no source, header, table or constant with
 * the CUDA library: every table here is built from the number-format
 * definitions at first use.
 *
 * Page shorthands used in the citations below:
 *   [FP8-guide]  "DeepGEMM实战：FP8矩阵乘法与JIT编译优化指南"
 *                (sheratonhq.com/news/156926), sections as numbered there.
 *   [DG-FP16]    the DeepGEMM FP16/WMMA deep-dive page (hnwysp.cn/news/84236).
 *   [HGEMM-L2]   "HGEMM优化：深度学习中的矩阵乘法性能提升策略"
 *                (jsqmd.com/news/710660).
 *
 * Every function is a direct transcription of a definition; there is no
 * blocking, reordering or fusion beyond what the definition states.
 */
#ifndef DG_ORACLE_H
#define DG_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* E4M3 ("fn" variant: bias 7, no infinities, S.1111.111 is NaN, max 448).
 * [FP8-guide] §2.1 (4 exponent / 3 mantissa bits), §3.2 and §4.3 (448 is
 * the largest E4M3 value). */
double  dgo_e4m3_decode(uint8_t code);
/* Nearest E4M3 value, ties to even mantissa, saturating at +-448, NaN->0x7F.
 * [FP8-guide] §4.3: fp8 = clamp(round(x/scale), -448, 448). */
uint8_t dgo_e4m3_encode(double y);

/* IEEE binary16 and bfloat16 decoders built from the format definitions. */
double   dgo_fp16_decode(uint16_t h);
double   dgo_bf16_decode(uint16_t h);
/* bfloat16 round-to-nearest-even of a binary32 value (used for the oracle's
 * own BF16 output in the tolerance-soundness check). */
uint16_t dgo_bf16_encode(float x);
/* binary16 round-to-nearest-even of a double, overflow to +-Inf. */
uint16_t dgo_fp16_encode(double y);

/* amax = max_i |x_i|; any NaN makes the result NaN. [FP8-guide] §3.2. */
float dgo_amax(const float* x, int64_t n);
/* scale = fl32(amax / 448); 1 when amax == 0.  [FP8-guide] §3.2. */
float dgo_scale_from_amax(float amax);
/* Power-of-two scale: the smallest power of two p (a binary32 value, at
 * least 2^-149) with 448 * p >= amax, compared exactly; 1 when amax == 0,
 * NaN for NaN, +Inf for +Inf.  [FP8-guide] §2.1: a power of two just above
 * the range, so that scaling and unscaling are exponent shifts. */
float dgo_scale_pow2_from_amax(float amax);
/* FP16 dynamic-range scaling, [DG-FP16] §3.3 (mixed-precision pitfalls):
 * scale = min(1, 65504 / (max|A| * max|B|)); A and B are multiplied by
 * sqrt(scale) before they become FP16, and the result is divided by scale.
 * out[0] = scale, with the product and the quotient formed in binary64 (no
 * binary32 overflow of max|A| * max|B|) and rounded once to binary32; 1 when
 * the product is 0; NaN when either amax is NaN.
 * out[1] = fl32(sqrt(scale)), out[2] = fl32(1 / scale), out[3] = 1. */
void  dgo_fp16_range_scale(float amax_a, float amax_b, float out[4]);
/* out_i = fp16_rn(fl32(x_i * factor)): binary32 product, then one
 * round-to-nearest-even to binary16 (overflow to +-Inf, NaN stays NaN). */
void  dgo_convert_f16(const float* x, int64_t n, float factor, uint16_t* out);
/* q_i = e4m3(fl32(x_i / scale)), binary32 division.  [FP8-guide] §4.3. */
void  dgo_quantize_e4m3(const float* x, int64_t n, float scale, uint8_t* q);

/* R[m,n] = sum_k dec(A[m,k]) * dec(B[n,k]) and S[m,n] = sum_k |...|, both
 * accumulated in double over ascending k.  A is M x K, B is N x K, both
 * row-major (K contiguous).  R, S are M x N row-major; S may be NULL.
 * nthreads <= 0 uses every online core.  [FP8-guide] §2.1, §3.2. */
void dgo_gemm_e4m3(const uint8_t* A, const uint8_t* B, int64_t M, int64_t N,
                   int64_t K, double* R, double* S, int nthreads);
/* The same sums at cnt selected (m,n) positions. */
void dgo_gemm_e4m3_at(const uint8_t* A, const uint8_t* B, int64_t K,
                      const int64_t* ms, const int64_t* ns, int64_t cnt,
                      double* R, double* S);
/* Same contraction for binary16 inputs ([HGEMM-L2] §1.3: FP16 inputs with an
 * FP32-or-wider accumulator). */
void dgo_hgemm(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
               int64_t K, double* R, double* S, int nthreads);
void dgo_hgemm_at(const uint16_t* A, const uint16_t* B, int64_t K,
                  const int64_t* ms, const int64_t* ns, int64_t cnt,
                  double* R, double* S);

/* Epilogue references ([FP8-guide] §3.2: multiply the accumulator by
 * scale_A*scale_B on write-back; for FP8 output divide by the output scale).
 *   dref[i] = R[i] * sA * sB                 (double)
 *   e[i]    = e4m3(R[i] * sA * sB / sD)       (one rounding, double math) */
void dgo_epilogue_scale(const double* R, int64_t cnt, float sA, float sB,
                        double* dref);
void dgo_epilogue_e4m3(const double* R, int64_t cnt, float sA, float sB,
                       float sD, uint8_t* e);

/* Independent exact cross-check: the same E4M3 contraction as integer sums
 * of codes in units of 2^-18 (every E4M3 value is an integer multiple of
 * 2^-9).  Returns 0 on success, -1 if any input code is NaN. */
int dgo_gemm_e4m3_exact_i64(const uint8_t* A, const uint8_t* B, int64_t M,
                            int64_t N, int64_t K, int64_t* R_units);

#ifdef __cplusplus
}
#endif
#endif /* DG_ORACLE_H */
