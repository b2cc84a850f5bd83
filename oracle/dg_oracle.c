/*
 * dg_oracle.c -- plain, slow CPU oracle (see dg_oracle.h for the contract
 * and the page shorthands [FP8-guide], [DG-FP16], [HGEMM-L2]).
 *
 * TEST INFRASTRUCTURE ONLY: the product library never links or calls this.
 * Built with -ffp-contract=off and without fast-math so that every double
 * and float operation below is one IEEE-754 operation, rounded once, in the
 * order written.
 */
#define _GNU_SOURCE
#include "dg_oracle.h"

#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* Number-format tables, built once from the format definitions.            */
/* ------------------------------------------------------------------------ */

static double g_e4m3[256];
static double g_fp16[65536];
static pthread_once_t g_once = PTHREAD_ONCE_INIT;

static void build_tables(void) {
    /* E4M3: s | eeee | mmm, exponent bias 7.  e == 0 is subnormal
     * (value m/8 * 2^(1-7) = m * 2^-9); 1111.111 is NaN; no infinities.
     * [FP8-guide] §2.1 names the 4/3 split, §4.3 the 448 maximum, which
     * (1 + 6/8) * 2^(15-7) = 448 fixes as the bias-7, no-Inf variant. */
    for (int c = 0; c < 256; ++c) {
        int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
        double v;
        if (e == 15 && m == 7)
            v = NAN;
        else if (e == 0)
            v = ldexp((double)m, -9);
        else
            v = ldexp(1.0 + m / 8.0, e - 7);
        g_e4m3[c] = s ? -v : v;
    }
    /* IEEE binary16: s | 5-bit exponent (bias 15) | 10-bit fraction. */
    for (int h = 0; h < 65536; ++h) {
        int s = h >> 15, e = (h >> 10) & 0x1F, m = h & 0x3FF;
        double v;
        if (e == 31)
            v = m ? NAN : INFINITY;
        else if (e == 0)
            v = ldexp((double)m, -24);
        else
            v = ldexp(1.0 + m / 1024.0, e - 15);
        g_fp16[h] = s ? -v : v;
    }
}

static inline void ensure_tables(void) { pthread_once(&g_once, build_tables); }

double dgo_e4m3_decode(uint8_t code) {
    ensure_tables();
    return g_e4m3[code];
}

/* Round |y| to the nearest of the 127 non-negative finite E4M3 values
 * (codes 0x00..0x7E, ascending), ties to the code with even mantissa, by a
 * linear scan compared exactly in double.  |y| >= 448 and +-Inf saturate to
 * 448 (the clamp of [FP8-guide] §4.3); NaN maps to 0x7F. */
uint8_t dgo_e4m3_encode(double y) {
    ensure_tables();
    if (isnan(y)) return 0x7F;
    int neg = signbit(y) ? 1 : 0;
    double a = fabs(y);
    int mag;
    if (a >= 448.0) {
        mag = 0x7E;
    } else {
        int lo = 0;
        for (int c = 1; c <= 0x7E; ++c)
            if (g_e4m3[c] <= a) lo = c;
        if (g_e4m3[lo] == a) {
            mag = lo;
        } else {
            /* a lies strictly between codes lo and lo+1 (lo+1 <= 0x7E since
             * a < 448).  Both differences are exact (Sterbenz). */
            double dlo = a - g_e4m3[lo];
            double dhi = g_e4m3[lo + 1] - a;
            if (dlo < dhi)
                mag = lo;
            else if (dhi < dlo)
                mag = lo + 1;
            else
                mag = (lo & 1) ? lo + 1 : lo; /* even mantissa = even code */
        }
    }
    return (uint8_t)(neg ? (0x80 | mag) : mag);
}

double dgo_fp16_decode(uint16_t h) {
    ensure_tables();
    return g_fp16[h];
}

/* bfloat16: s | 8-bit exponent (bias 127) | 7-bit fraction. */
double dgo_bf16_decode(uint16_t h) {
    int s = h >> 15, e = (h >> 7) & 0xFF, m = h & 0x7F;
    double v;
    if (e == 255)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -133);
    else
        v = ldexp(1.0 + m / 128.0, e - 127);
    return s ? -v : v;
}

/* Round a finite, non-zero |y| to a grid whose spacing is 2^(E-p) inside the
 * binade [2^E, 2^(E+1)), with E clamped below at emin (gradual underflow).
 * nearbyint() rounds half to even in the default rounding mode. */
static double round_to_format(double a, int p, int emin) {
    int ex;
    (void)frexp(a, &ex);         /* a = f * 2^ex, f in [0.5, 1) */
    int E = ex - 1;
    if (E < emin) E = emin;
    double q = ldexp(1.0, E - p); /* spacing of representable values */
    return nearbyint(a / q) * q;  /* a / q is exact (power-of-two scaling) */
}

uint16_t dgo_bf16_encode(float x) {
    if (isnan(x)) return 0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    double a = fabs((double)x);
    uint16_t bits;
    if (a == 0.0) {
        bits = 0;
    } else {
        double v = isinf(a) ? INFINITY : round_to_format(a, 7, -126);
        if (v >= ldexp(1.0, 128)) {
            bits = 0x7F80;
        } else if (v < ldexp(1.0, -126)) {
            bits = (uint16_t)(v / ldexp(1.0, -133)); /* subnormal fraction */
        } else {
            int ex;
            (void)frexp(v, &ex);
            int E = ex - 1;
            int m = (int)(v / ldexp(1.0, E - 7)) - 128;
            bits = (uint16_t)(((E + 127) << 7) | m);
        }
    }
    return (uint16_t)(neg ? (0x8000 | bits) : bits);
}

uint16_t dgo_fp16_encode(double y) {
    if (isnan(y)) return 0x7E00;
    int neg = signbit(y) ? 1 : 0;
    double a = fabs(y);
    uint16_t bits;
    if (a == 0.0) {
        bits = 0;
    } else {
        double v = isinf(a) ? INFINITY : round_to_format(a, 10, -14);
        if (v >= 65536.0) {
            bits = 0x7C00;
        } else if (v < ldexp(1.0, -14)) {
            bits = (uint16_t)(v / ldexp(1.0, -24));
        } else {
            int ex;
            (void)frexp(v, &ex);
            int E = ex - 1;
            int m = (int)(v / ldexp(1.0, E - 10)) - 1024;
            bits = (uint16_t)(((E + 15) << 10) | m);
        }
    }
    return (uint16_t)(neg ? (0x8000 | bits) : bits);
}

/* ------------------------------------------------------------------------ */
/* Per-tensor scaling and the quantiser.                                     */
/* ------------------------------------------------------------------------ */

/* [FP8-guide] §3.2: record the maximum absolute value of the tensor.  NaN
 * anywhere propagates (reading: a NaN input must not be silently dropped). */
float dgo_amax(const float* x, int64_t n) {
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (isnan(a)) return NAN;
        if (a > m) m = a;
    }
    return m;
}

/* [FP8-guide] §3.2: scale = max_val / 448.0 (448 = largest E4M3 value).
 * An all-zero tensor gets scale 1 (reading: the page is silent). */
float dgo_scale_from_amax(float amax) {
    if (amax == 0.0f) return 1.0f;
    return amax / 448.0f; /* one binary32 division */
}

/* [FP8-guide] §2.1: instead of amax/448 itself, a power of two slightly
 * larger, so that dividing by the scale is exact.  Smallest p = 2^e, e >=
 * -149, with 448 * p >= amax; both sides exact in double. */
float dgo_scale_pow2_from_amax(float amax) {
    if (isnan(amax)) return NAN;
    if (amax == 0.0f) return 1.0f;
    if (isinf(amax)) return INFINITY;
    const double a = (double)amax;
    int e = -149;
    while (448.0 * ldexp(1.0, e) < a) ++e;
    return (float)ldexp(1.0, e);
}

/* [DG-FP16] §3.3: before the launch, take the largest magnitudes of A and
 * B, form scale = min(1, 65504 / (max_abs_A * max_abs_B)), multiply A and B
 * by sqrt(scale) and divide the result by scale, so that no FP16 value
 * overflows on the way in.  The scale is formed in binary64 and rounded once
 * to binary32; sqrt and the reciprocal are taken in binary64 from that
 * binary32 value and rounded once (for sqrt and division this equals the
 * correctly rounded binary32 operation). */
void dgo_fp16_range_scale(float amax_a, float amax_b, float out[4]) {
    float s;
    if (isnan(amax_a) || isnan(amax_b)) {
        s = NAN;
    } else {
        const double prod = (double)amax_a * (double)amax_b;
        const double q = 65504.0 / prod;          /* +Inf when prod == 0 */
        s = (float)(q < 1.0 ? q : 1.0);
    }
    out[0] = s;
    out[1] = (float)sqrt((double)s);
    out[2] = (float)(1.0 / (double)s);
    out[3] = 1.0f;
}

void dgo_convert_f16(const float* x, int64_t n, float factor, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) {
        const float y = x[i] * factor;            /* one binary32 rounding */
        out[i] = dgo_fp16_encode((double)y);
    }
}

/* [FP8-guide] §4.3: fp8 = clamp(round(x / scale), -448, 448), read as
 * round-to-nearest-even onto the E4M3 grid after a binary32 division. */
static void quantize_range(const float* x, int64_t lo, int64_t hi, float scale,
                           uint8_t* q) {
    for (int64_t i = lo; i < hi; ++i) {
        float y = x[i] / scale;
        q[i] = dgo_e4m3_encode((double)y);
    }
}

typedef struct {
    const float* x;
    int64_t lo, hi;
    float scale;
    uint8_t* q;
} qjob_t;

static void* quantize_worker(void* p) {
    qjob_t* j = (qjob_t*)p;
    quantize_range(j->x, j->lo, j->hi, j->scale, j->q);
    return NULL;
}

static int online_cores(void);

/* Elements are independent, so large inputs are split into contiguous
 * slices over threads; each element sees exactly the same two steps. */
void dgo_quantize_e4m3(const float* x, int64_t n, float scale, uint8_t* q) {
    ensure_tables();
    int nt = n >= (1 << 20) ? online_cores() : 1;
    if (nt > 256) nt = 256;
    if (nt <= 1) {
        quantize_range(x, 0, n, scale, q);
        return;
    }
    qjob_t jobs[256];
    pthread_t th[256];
    int started[256];
    int64_t per = (n + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        int64_t lo = (int64_t)t * per, hi = lo + per;
        if (lo > n) lo = n;
        if (hi > n) hi = n;
        jobs[t] = (qjob_t){x, lo, hi, scale, q};
        started[t] = pthread_create(&th[t], NULL, quantize_worker, &jobs[t]) == 0;
        if (!started[t]) quantize_worker(&jobs[t]);
    }
    for (int t = 0; t < nt; ++t)
        if (started[t]) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* Contractions: FP64 triple loops, threaded over output elements.           */
/* ------------------------------------------------------------------------ */

static int online_cores(void) {
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int c = CPU_COUNT(&set);
        if (c > 0) return c;
    }
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

typedef struct {
    const void* A;
    const void* B;
    int64_t N, K;
    int64_t lo, hi;   /* flattened output index range m*N+n */
    double* R;
    double* S;
    int is_fp16;
} job_t;

static void* gemm_worker(void* p) {
    job_t* j = (job_t*)p;
    const double* tab = j->is_fp16 ? g_fp16 : g_e4m3;
    for (int64_t idx = j->lo; idx < j->hi; ++idx) {
        int64_t m = idx / j->N, n = idx % j->N;
        double r = 0.0, s = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
            double a, b;
            if (j->is_fp16) {
                a = tab[((const uint16_t*)j->A)[m * j->K + k]];
                b = tab[((const uint16_t*)j->B)[n * j->K + k]];
            } else {
                a = tab[((const uint8_t*)j->A)[m * j->K + k]];
                b = tab[((const uint8_t*)j->B)[n * j->K + k]];
            }
            double prod = a * b;
            r += prod;
            s += fabs(prod);
        }
        j->R[idx] = r;
        if (j->S) j->S[idx] = s;
    }
    return NULL;
}

static void run_gemm(const void* A, const void* B, int64_t M, int64_t N,
                     int64_t K, double* R, double* S, int nthreads, int fp16) {
    ensure_tables();
    int64_t total = M * N;
    if (total <= 0) return;
    if (nthreads <= 0) nthreads = online_cores();
    if ((int64_t)nthreads > total) nthreads = (int)total;
    if (nthreads > 256) nthreads = 256;
    job_t jobs[256];
    pthread_t th[256];
    int joined[256];
    int64_t per = (total + nthreads - 1) / nthreads;
    int launched = 0;
    for (int t = 0; t < nthreads; ++t) {
        int64_t lo = (int64_t)t * per, hi = lo + per;
        if (lo >= total) break;
        if (hi > total) hi = total;
        jobs[t] = (job_t){A, B, N, K, lo, hi, R, S, fp16};
        joined[t] = 0;
        if (pthread_create(&th[t], NULL, gemm_worker, &jobs[t]) != 0) {
            gemm_worker(&jobs[t]); /* no thread: do the slice inline */
            joined[t] = 1;
        }
        launched = t + 1;
    }
    for (int t = 0; t < launched; ++t)
        if (!joined[t]) pthread_join(th[t], NULL);
}

void dgo_gemm_e4m3(const uint8_t* A, const uint8_t* B, int64_t M, int64_t N,
                   int64_t K, double* R, double* S, int nthreads) {
    run_gemm(A, B, M, N, K, R, S, nthreads, 0);
}

void dgo_hgemm(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
               int64_t K, double* R, double* S, int nthreads) {
    run_gemm(A, B, M, N, K, R, S, nthreads, 1);
}

void dgo_gemm_e4m3_at(const uint8_t* A, const uint8_t* B, int64_t K,
                      const int64_t* ms, const int64_t* ns, int64_t cnt,
                      double* R, double* S) {
    ensure_tables();
    for (int64_t i = 0; i < cnt; ++i) {
        double r = 0.0, s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double prod = g_e4m3[A[ms[i] * K + k]] * g_e4m3[B[ns[i] * K + k]];
            r += prod;
            s += fabs(prod);
        }
        R[i] = r;
        if (S) S[i] = s;
    }
}

void dgo_hgemm_at(const uint16_t* A, const uint16_t* B, int64_t K,
                  const int64_t* ms, const int64_t* ns, int64_t cnt,
                  double* R, double* S) {
    ensure_tables();
    for (int64_t i = 0; i < cnt; ++i) {
        double r = 0.0, s = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double prod = g_fp16[A[ms[i] * K + k]] * g_fp16[B[ns[i] * K + k]];
            r += prod;
            s += fabs(prod);
        }
        R[i] = r;
        if (S) S[i] = s;
    }
}

/* ------------------------------------------------------------------------ */
/* Epilogue references.  [FP8-guide] §3.2 gives the chain FP8 in, input    */
/* scales, FP32 accumulation, output scale, FP8 out: the accumulator is      */
/* multiplied by scale_A * scale_B when written back, and FP8 output is      */
/* divided by the output scale (the section names the output-scale step both */
/* a multiply and a divide; the divide is taken, so that output quantisation */
/* is the same map as the input quantiser of §4.3).                          */
/* ------------------------------------------------------------------------ */

void dgo_epilogue_scale(const double* R, int64_t cnt, float sA, float sB,
                        double* dref) {
    for (int64_t i = 0; i < cnt; ++i) dref[i] = R[i] * (double)sA * (double)sB;
}

void dgo_epilogue_e4m3(const double* R, int64_t cnt, float sA, float sB,
                       float sD, uint8_t* e) {
    for (int64_t i = 0; i < cnt; ++i)
        e[i] = dgo_e4m3_encode(R[i] * (double)sA * (double)sB / (double)sD);
}

/* ------------------------------------------------------------------------ */
/* Independent integer formulation (pins the double contraction).           */
/* ------------------------------------------------------------------------ */

/* E4M3 code -> signed integer k with value k * 2^-9, straight from the bit
 * fields (no table): subnormal m * 2^-9 -> k = m; normal
 * (8 + m) * 2^(e - 10) -> k = (8 + m) << (e - 1). */
static int code_units(uint8_t c, int64_t* k) {
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 15 && m == 7) return -1;
    int64_t v = (e == 0) ? (int64_t)m : ((int64_t)(8 + m) << (e - 1));
    *k = s ? -v : v;
    return 0;
}

int dgo_gemm_e4m3_exact_i64(const uint8_t* A, const uint8_t* B, int64_t M,
                            int64_t N, int64_t K, int64_t* R_units) {
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            int64_t acc = 0;
            for (int64_t k = 0; k < K; ++k) {
                int64_t ka, kb;
                if (code_units(A[m * K + k], &ka) || code_units(B[n * K + k], &kb))
                    return -1;
                acc += ka * kb;
            }
            R_units[m * N + n] = acc;
        }
    return 0;
}
