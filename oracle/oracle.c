/*
 * oracle.c -- plain, slow, obviously correct CPU statement of what the
 * streamed AllGather+GEMM computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only tests/, __graft_entry__.smoke() and the cpu_baseline /
 * reference legs of bench.py use it.  It shares no source, header, table or
 * helper with the CUDA library, and it includes no CUDA header.
 *
 * Sources (web pages, by title and section):
 *  [PTO]  "AllGather + GEMM 通算融合算子示例" (PTO-ISA allgather_gemm README),
 *         section 计算功能: n_ranks ranks each hold rows
 *         [rank*M/n, (rank+1)*M/n) of A (M x K, fp16); B (K x N, fp16) is
 *         replicated; after the AllGather every rank computes C = A x B,
 *         M x N, fp32.
 *  [CAT]  "AllGather矩阵乘法反量化算子设计文档" (CANN/catccos
 *         AllGatherMatmulDequant), sections 1.1, 1.2 and 2.2: int8 A gathered,
 *         result_int32 = matmul(A, B) + bias (bias int32 [N]),
 *         result_fp32 = result_int32 * scale (per-channel fp32 [N], no
 *         per-token scale), output_fp16 = cast_to_fp16(result_fp32).
 *  [TRI]  "全聚合-通用矩阵乘法（Allgather Gemm）" (Triton-distributed),
 *         torch_allgather_gemm golden: all_gather the shards, concatenate
 *         them along dim 0 in rank order, then matmul.
 *  [MGPU] "Collective matrix multiplication" (Pallas:MGPU), 使用 Pallas 实现:
 *         the same gathered GEMM with bfloat16 operands (the page's default
 *         dtype); the bf16 variant below is the [PTO] GEMM with bf16 inputs.
 *
 * Precision: the fp16 and bf16 GEMMs are evaluated in fp64 (every fp16 or
 * bf16 value and every product of two of them is exact in fp64; the k-ordered
 * sum rounds in fp64).  The int8 GEMM is exact in int64.  The dequant step follows [CAT]
 * 2.2 literally: the int32 result is rounded to fp32, multiplied by the fp32
 * scale in fp32 (correctly rounded), and the fp32 value is rounded to fp16.
 * All roundings are round-to-nearest-even and are written out below from the
 * IEEE 754 definitions of binary16 and binary32 (no reliance on the C
 * compiler's float conversions).
 *
 * Pins (tests/test_oracle_pins.py): IEEE encode/decode against numpy's
 * conversions and hand-picked boundary values; GEMM against one-hot and
 * permutation B, rank-1 closed forms, exact big-integer brute force on tiny
 * shapes and torch float64 on CPU; bf16 encode/decode against float32 bit
 * patterns and boundary values, the bf16 GEMM against one-hot B, rank-1 and
 * dyadic closed forms and torch's bfloat16 -> float64 matmul; int8 path
 * against Python integers and the
 * all-127 closed form; dequant against the all-ones debug mode of [CAT] 8.6.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARGS (-1)
#define ORACLE_ERR_INT32_RANGE (-2)
#define ORACLE_ERR_NOMEM (-3)

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 / binary32                                              */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int efield = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (efield == 0)
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-24 */
    else if (efield == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 1024), efield - 25); /* 1.frac * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int efield = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (efield == 0)
        v = ldexp((double)frac, -133); /* subnormal: frac * 2^-133 */
    else if (efield == 255)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 128), efield - 134); /* 1.frac * 2^(e-127) */
    return sign ? -v : v;
}

/*
 * Round a double to the nearest value with `p` significant bits whose
 * exponent is at least `emin` (values below 2^emin keep the fixed spacing
 * 2^(emin-p+1), i.e. gradual underflow), ties to even.  Returns the rounded
 * magnitude as a double (exact: the target formats are subsets of binary64).
 * Overflow is left to the caller.
 */
static double round_rne(double a, int p, int emin)
{
    int e2;
    double q, n, r;
    if (a == 0.0)
        return 0.0;
    frexp(a, &e2);           /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;          /* a in [2^e, 2^(e+1)) */
    if (e < emin)
        e = emin;            /* subnormal range: fixed spacing */
    double ulp = ldexp(1.0, e - (p - 1));
    q = a / ulp;             /* exact: division by a power of two */
    n = floor(q);
    r = q - n;               /* exact fractional part */
    if (r > 0.5 || (r == 0.5 && fmod(n, 2.0) != 0.0))
        n += 1.0;
    return n * ulp;          /* exact */
}

/* binary16 round-to-nearest-even from a double; overflow -> +-inf. */
uint16_t oracle_f64_to_f16_rn(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | 0x7e00);
    double v = round_rne(a, 11, -14);
    if (v >= 65536.0)        /* 2^16: beyond the largest finite 65504 */
        return (uint16_t)(sign | 0x7c00);
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -14)) /* subnormal: fraction = v / 2^-24 */
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -24)));
    int e2;
    frexp(v, &e2);
    int e = e2 - 1;          /* v in [2^e, 2^(e+1)), -14 <= e <= 15 */
    uint16_t frac = (uint16_t)(v / ldexp(1.0, e - 10) - 1024.0);
    return (uint16_t)(sign | ((uint16_t)(e + 15) << 10) | frac);
}

/* bfloat16 round-to-nearest-even from a double; overflow -> +-inf. */
uint16_t oracle_f64_to_bf16_rn(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(sign | 0x7fc0);
    double v = round_rne(a, 8, -126);
    if (v >= ldexp(1.0, 128)) /* beyond the largest finite (2 - 2^-7) * 2^127 */
        return (uint16_t)(sign | 0x7f80);
    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -126)) /* subnormal: fraction = v / 2^-133 */
        return (uint16_t)(sign | (uint16_t)(v / ldexp(1.0, -133)));
    int e2;
    frexp(v, &e2);
    int e = e2 - 1;           /* v in [2^e, 2^(e+1)), -126 <= e <= 127 */
    uint16_t frac = (uint16_t)(v / ldexp(1.0, e - 7) - 128.0);
    return (uint16_t)(sign | ((uint16_t)(e + 127) << 7) | frac);
}

/* binary32 round-to-nearest-even from a double; overflow -> +-inf. */
float oracle_f64_to_f32_rn(double x)
{
    if (isnan(x))
        return NAN;
    double a = fabs(x);
    double v = round_rne(a, 24, -126);
    /* largest finite binary32 is (2 - 2^-23) * 2^127 */
    if (v > ldexp(2.0 - ldexp(1.0, -23), 127))
        v = INFINITY;
    return (float)(signbit(x) ? -v : v); /* exact: v is representable */
}

/* ------------------------------------------------------------------------ */
/* AllGather                                                                 */
/* ------------------------------------------------------------------------ */

/*
 * [PTO] 计算功能 / [TRI] torch_allgather_gemm: the gathered A is the shards
 * concatenated along rows in rank order; rank s owns global rows
 * [s*R, (s+1)*R).  Row m of A is row (m mod R) of shard (m / R), whatever
 * order the shards are transferred or consumed in.
 */
static const void *gathered_row(const void *const *shards, int64_t R,
                                int64_t K, int64_t m, size_t elem)
{
    int64_t s = m / R;
    int64_t r = m % R;
    return (const char *)shards[s] + (size_t)(r * K) * elem;
}

/* Copy the gathered A (S*R x K, element size `elem`) into `out`. */
int oracle_allgather(int S, int64_t R, int64_t K, size_t elem,
                     const void *const *shards, void *out)
{
    if (S < 1 || R < 0 || K < 0 || !shards || !out)
        return ORACLE_ERR_ARGS;
    for (int64_t m = 0; m < (int64_t)S * R; ++m) {
        const unsigned char *src = gathered_row(shards, R, K, m, elem);
        unsigned char *dst = (unsigned char *)out + (size_t)(m * K) * elem;
        for (size_t i = 0; i < (size_t)K * elem; ++i)
            dst[i] = src[i];
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* fp16 AllGather + GEMM  ([PTO] 计算功能)                                   */
/* ------------------------------------------------------------------------ */

/*
 * C (S*R x N, row-major, fp64) = AllGather(shards) x B.
 * shards[s]: R x K fp16 bit patterns, row-major.  B: K x N fp16, row-major.
 * Loop order i-k-j: every C[m][n] is summed in ascending k, in fp64.
 */
int oracle_ag_gemm_f16(int S, int64_t R, int64_t K, int64_t N,
                       const uint16_t *const *shards, const uint16_t *B,
                       double *C)
{
    if (S < 1 || R < 0 || K < 0 || N < 0 || !shards || !B || !C)
        return ORACLE_ERR_ARGS;
    int64_t M = (int64_t)S * R;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *a = gathered_row((const void *const *)shards, R, K,
                                         m, sizeof(uint16_t));
        double *c = C + m * N;
        for (int64_t n = 0; n < N; ++n)
            c[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double av = oracle_f16_to_f64(a[k]);
            const uint16_t *b = B + k * N;
            for (int64_t n = 0; n < N; ++n)
                c[n] += av * oracle_f16_to_f64(b[n]);
        }
    }
    return ORACLE_OK;
}

/* The same definition evaluated only at the points (rows[i], cols[i]). */
int oracle_ag_gemm_f16_at(int S, int64_t R, int64_t K, int64_t N,
                          const uint16_t *const *shards, const uint16_t *B,
                          int64_t npts, const int64_t *rows,
                          const int64_t *cols, double *out)
{
    if (S < 1 || !shards || !B || !rows || !cols || !out)
        return ORACLE_ERR_ARGS;
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = rows[i], n = cols[i];
        if (m < 0 || m >= (int64_t)S * R || n < 0 || n >= N)
            return ORACLE_ERR_ARGS;
        const uint16_t *a = gathered_row((const void *const *)shards, R, K,
                                         m, sizeof(uint16_t));
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += oracle_f16_to_f64(a[k]) * oracle_f16_to_f64(B[k * N + n]);
        out[i] = acc;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* bf16 AllGather + GEMM  ([PTO] 计算功能 with [MGPU]'s bfloat16 operands)    */
/* ------------------------------------------------------------------------ */

/* As oracle_ag_gemm_f16, the elements being bfloat16 bit patterns. */
int oracle_ag_gemm_bf16(int S, int64_t R, int64_t K, int64_t N,
                        const uint16_t *const *shards, const uint16_t *B,
                        double *C)
{
    if (S < 1 || R < 0 || K < 0 || N < 0 || !shards || !B || !C)
        return ORACLE_ERR_ARGS;
    int64_t M = (int64_t)S * R;
    for (int64_t m = 0; m < M; ++m) {
        const uint16_t *a = gathered_row((const void *const *)shards, R, K,
                                         m, sizeof(uint16_t));
        double *c = C + m * N;
        for (int64_t n = 0; n < N; ++n)
            c[n] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double av = oracle_bf16_to_f64(a[k]);
            const uint16_t *b = B + k * N;
            for (int64_t n = 0; n < N; ++n)
                c[n] += av * oracle_bf16_to_f64(b[n]);
        }
    }
    return ORACLE_OK;
}

/* The same definition evaluated only at the points (rows[i], cols[i]). */
int oracle_ag_gemm_bf16_at(int S, int64_t R, int64_t K, int64_t N,
                           const uint16_t *const *shards, const uint16_t *B,
                           int64_t npts, const int64_t *rows,
                           const int64_t *cols, double *out)
{
    if (S < 1 || !shards || !B || !rows || !cols || !out)
        return ORACLE_ERR_ARGS;
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = rows[i], n = cols[i];
        if (m < 0 || m >= (int64_t)S * R || n < 0 || n >= N)
            return ORACLE_ERR_ARGS;
        const uint16_t *a = gathered_row((const void *const *)shards, R, K,
                                         m, sizeof(uint16_t));
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += oracle_bf16_to_f64(a[k]) * oracle_bf16_to_f64(B[k * N + n]);
        out[i] = acc;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------------ */
/* int8 AllGatherMatmulDequant  ([CAT] 1.1, 1.2, 2.2)                        */
/* ------------------------------------------------------------------------ */

/* [CAT] 2.2: result_fp32 = result_int32 * scale; output_fp16 = fp16(...) */
static uint16_t dequant_one(int32_t c, float scale)
{
    double cf = (double)oracle_f64_to_f32_rn((double)c);  /* int32 -> fp32 */
    /* fp32 x fp32: the exact product has <= 48 significant bits, so the
     * double product is exact and one rounding gives the fp32 multiply. */
    double prod = (double)oracle_f64_to_f32_rn(cf * (double)scale);
    return oracle_f64_to_f16_rn(prod);
}

/* One output element: exact int64 dot product, plus bias. */
static int64_t i8_dot_bias(const int8_t *a, const int8_t *B, int64_t K,
                           int64_t N, int64_t n, int32_t bias_n)
{
    int64_t acc = 0;
    for (int64_t k = 0; k < K; ++k)
        acc += (int64_t)a[k] * (int64_t)B[k * N + n];
    return acc + (int64_t)bias_n;
}

/*
 * C_i32 (S*R x N) = AllGather(shards) x B + bias  (exact; error if any value
 * leaves the int32 range), D (S*R x N, fp16 bits) = dequant(C_i32, scale).
 */
int oracle_ag_gemm_dequant(int S, int64_t R, int64_t K, int64_t N,
                           const int8_t *const *shards, const int8_t *B,
                           const int32_t *bias, const float *scale,
                           int32_t *C_i32, uint16_t *D)
{
    if (S < 1 || R < 0 || K < 0 || N < 0 || !shards || !B || !bias ||
        !scale || !C_i32 || !D)
        return ORACLE_ERR_ARGS;
    int64_t M = (int64_t)S * R;
    int64_t *acc = (int64_t *)malloc(sizeof(int64_t) * (size_t)(N ? N : 1));
    if (!acc)
        return ORACLE_ERR_NOMEM;
    int rc = ORACLE_OK;
    for (int64_t m = 0; m < M && rc == ORACLE_OK; ++m) {
        const int8_t *a = gathered_row((const void *const *)shards, R, K, m,
                                       sizeof(int8_t));
        for (int64_t n = 0; n < N; ++n)
            acc[n] = 0;
        for (int64_t k = 0; k < K; ++k) {
            int64_t av = a[k];
            const int8_t *b = B + k * N;
            for (int64_t n = 0; n < N; ++n)
                acc[n] += av * (int64_t)b[n];
        }
        for (int64_t n = 0; n < N; ++n) {
            int64_t c = acc[n] + (int64_t)bias[n];
            if (c < INT32_MIN || c > INT32_MAX) {
                rc = ORACLE_ERR_INT32_RANGE;
                break;
            }
            C_i32[m * N + n] = (int32_t)c;
            D[m * N + n] = dequant_one((int32_t)c, scale[n]);
        }
    }
    free(acc);
    return rc;
}

/* The same definition evaluated only at the points (rows[i], cols[i]). */
int oracle_ag_gemm_dequant_at(int S, int64_t R, int64_t K, int64_t N,
                              const int8_t *const *shards, const int8_t *B,
                              const int32_t *bias, const float *scale,
                              int64_t npts, const int64_t *rows,
                              const int64_t *cols, int32_t *C_i32,
                              uint16_t *D)
{
    if (S < 1 || !shards || !B || !bias || !scale || !rows || !cols ||
        !C_i32 || !D)
        return ORACLE_ERR_ARGS;
    for (int64_t i = 0; i < npts; ++i) {
        int64_t m = rows[i], n = cols[i];
        if (m < 0 || m >= (int64_t)S * R || n < 0 || n >= N)
            return ORACLE_ERR_ARGS;
        const int8_t *a = gathered_row((const void *const *)shards, R, K, m,
                                       sizeof(int8_t));
        int64_t c = i8_dot_bias(a, B, K, N, n, bias[n]);
        if (c < INT32_MIN || c > INT32_MAX)
            return ORACLE_ERR_INT32_RANGE;
        C_i32[i] = (int32_t)c;
        D[i] = dequant_one((int32_t)c, scale[n]);
    }
    return ORACLE_OK;
}

/* Element-wise dequant of given int32 values (used to pin the epilogue). */
int oracle_dequant(int64_t count, const int32_t *c, const float *scale,
                   uint16_t *D)
{
    if (count < 0 || (count && (!c || !scale || !D)))
        return ORACLE_ERR_ARGS;
    for (int64_t i = 0; i < count; ++i)
        D[i] = dequant_one(c[i], scale[i]);
    return ORACLE_OK;
}

/* Element-wise conversions exposed for pinning against numpy. */
void oracle_f64_to_f16_rn_array(int64_t count, const double *x, uint16_t *h)
{
    for (int64_t i = 0; i < count; ++i)
        h[i] = oracle_f64_to_f16_rn(x[i]);
}

void oracle_f16_to_f64_array(int64_t count, const uint16_t *h, double *x)
{
    for (int64_t i = 0; i < count; ++i)
        x[i] = oracle_f16_to_f64(h[i]);
}

void oracle_f64_to_f32_rn_array(int64_t count, const double *x, float *f)
{
    for (int64_t i = 0; i < count; ++i)
        f[i] = oracle_f64_to_f32_rn(x[i]);
}

void oracle_f64_to_bf16_rn_array(int64_t count, const double *x, uint16_t *h)
{
    for (int64_t i = 0; i < count; ++i)
        h[i] = oracle_f64_to_bf16_rn(x[i]);
}

void oracle_bf16_to_f64_array(int64_t count, const uint16_t *h, double *x)
{
    for (int64_t i = 0; i < count; ++i)
        x[i] = oracle_bf16_to_f64(h[i]);
}
