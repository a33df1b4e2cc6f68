/*
 * oracle.c -- plain, slow, CPU reference for the small-M FP8 block-scaled
 * linear layer  Y[M,N] = dequant(Aq[M,K]) . dequant(Wq[N,K])^T.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test-suite, the smoke check and the benchmark's CPU-baseline leg load
 * it.  It shares no code, header, table or constant generator with the CUDA
 * library; the two see only the same seeded raw inputs.
 *
 * Sources for what is computed (page title, then section):
 *  - "A 23% faster GPU kernel, and a model that did not move", section "Why
 *    this shape is hard": the weight carries one scale per 128x128 block and
 *    the long (K) dimension is reduced.
 *  - "The profiler said the kernel ran zero times", sections "What the trace
 *    showed" (inputs are cast to FP8 at run time) and "The output layer, which
 *    did run" (the 248,320 x 5,120 output layer, one scale per 128x128 block).
 *  - "Kernel-Level Optimisations for LLM Inference and Training", section
 *    "Quantisation kernels": E4M3 = 4-bit exponent, 3-bit mantissa, used for
 *    weights and activations.
 *
 * Where the pages are silent the plainest reading is taken:
 *  - E4M3 is the "fn" variant: bias 7, no infinities, 0x7F/0xFF are NaN,
 *    largest finite magnitude 448, subnormal step 2^-9.
 *  - Encoding rounds to nearest, ties to the even code, and saturates to
 *    +-448 (values beyond the largest finite never become NaN); the sign of a
 *    value that rounds to zero is kept (code 0x80 for negative zero).
 *  - A group (1x128 of the activations) or block (128x128 of the weights)
 *    has scale s = fl32(amax / 448) with IEEE fp32 division, stored as the
 *    dequantisation factor; if amax == 0 the scale is 1.0.  The code is
 *    enc(fl32(x / s)), again with IEEE fp32 division.
 *  - Activations are grouped 1x128 per token.
 *  - A ragged last weight block (N not a multiple of 128) takes its amax over
 *    the rows that exist.
 *  - Y = sum over 128-wide K blocks kb of s_a[m,kb] * s_w[n/128,kb] * P_kb,
 *    P_kb = sum_{k in kb} dec(Aq[m,k]) * dec(Wq[n,k]), all in fp64; P_kb is
 *    exact in fp64.  The error bound reference is
 *    sum_k |s_a dec(Aq)| * |s_w dec(Wq)|.
 *
 * Build with -ffp-contract=off and no fast-math so that every float
 * expression is a single IEEE operation.
 *
 * ORACLE_MUTANT (default 0) plants one deliberate mistake per value; the
 * test-suite builds those copies separately and checks that its pins reject
 * each of them.  The default build has none of them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ------------------------------------------------------------------ */
/* E4M3 decode: straight from the format's field definition.          */
/* ------------------------------------------------------------------ */
double oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 0xF;
    int mant = code & 0x7;
    double mag;
    if (expo == 0xF && mant == 0x7)
        return NAN;                          /* 0x7F and 0xFF */
    if (expo == 0)
#if ORACLE_MUTANT == 2
        mag = ldexp((double)mant / 8.0, -7); /* mutant: wrong subnormal exponent */
#else
        mag = ldexp((double)mant / 8.0, -6); /* subnormal: f/8 * 2^(1-7) */
#endif
    else
        mag = ldexp(1.0 + (double)mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

void oracle_e4m3_decode_table(double *out256)
{
    for (int c = 0; c < 256; ++c)
        out256[c] = oracle_e4m3_decode((uint8_t)c);
}

/* ------------------------------------------------------------------ */
/* E4M3 encode of a finite fp32 value: nearest finite code, ties to the */
/* code whose mantissa LSB is 0, saturating at 448, sign kept.          */
/* ------------------------------------------------------------------ */
uint8_t oracle_e4m3_encode(float v)
{
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs((double)v);
    if (isnan(v))
        return 0x7F;                    /* outside the contract */
#if ORACLE_MUTANT == 11
    if (a >= 464.0)
        return sign | 0x7F;             /* mutant: overflow to NaN */
#endif
    if (a >= 448.0)
        return sign | 0x7E;             /* satfinite */
    /* Largest non-negative code c in [0, 0x7E] with dec(c) <= a.  The
       positive finite codes are ordered like their values. */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_decode((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid - 1;
    }
    /* a < 448 so lo < 0x7E here.  The midpoint of two neighbours is exact
       in fp64. */
    double below = oracle_e4m3_decode((uint8_t)lo);
    double above = oracle_e4m3_decode((uint8_t)(lo + 1));
    double mid = 0.5 * (below + above);
    int code;
    if (a < mid)
        code = lo;
    else if (a > mid)
        code = lo + 1;
    else
#if ORACLE_MUTANT == 1
        code = lo + 1;                  /* mutant: ties away from zero */
#else
        code = (lo & 1) ? lo + 1 : lo;  /* code LSB is the mantissa LSB */
#endif
#if ORACLE_MUTANT == 10
    if (code == 0)
        sign = 0;                       /* mutant: sign of zero dropped */
#endif
    return sign | (uint8_t)code;
}

/* bf16 bits -> fp32 value (exact). */
static float bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------ */
/* fp64 -> bf16, one rounding, to nearest with ties to even.            */
/* ------------------------------------------------------------------ */
uint16_t oracle_round_bf16(double v)
{
    if (isnan(v))
        return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0x0000;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                        /* a = f * 2^e, 0.5 <= f < 1 */
    /* bf16 keeps 8 significant bits; below 2^-126 the spacing is fixed at
       2^-133 (subnormals). */
#if ORACLE_MUTANT == 7
    a = (double)(float)a;                /* mutant: rounds through fp32 first */
    frexp(a, &e);
#endif
    int q = e - 8;                       /* weight of the last kept bit */
    if (q < -133)
        q = -133;
    double t = ldexp(a, -q);             /* exact scaling */
    double r = floor(t);
    double frac = t - r;                 /* exact: t has a finite expansion */
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    double rounded = ldexp(r, q);
    if (rounded >= ldexp(1.0, 128))
        return sign | 0x7F80;            /* overflow to infinity */
    float f = (float)rounded;            /* exact: at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFF);
}

/* ------------------------------------------------------------------ */
/* Group / block quantisation.                                          */
/* ------------------------------------------------------------------ */

/* Scale of a group whose largest magnitude is amax. */
static float group_scale(float amax)
{
    if (amax == 0.0f)
        return 1.0f;
#if ORACLE_MUTANT == 3
    return amax / 240.0f;               /* mutant: another format's maximum */
#else
    return amax / 448.0f;               /* one IEEE fp32 division */
#endif
}

/* Activations: X bf16 [M rows, row stride ldx elements], K % 128 == 0.
   Writes xq [M*K] (row stride K) and xs [M * K/128] (row-major [M][K/128]).
   Returns 0, or -1 on a bad shape. */
int oracle_quant_act(const uint16_t *x, int M, int K, int ldx,
                     uint8_t *xq, float *xs)
{
    if (M < 0 || K < 0 || K % 128 != 0 || ldx < K)
        return -1;
    int kg = K / 128;
    for (int m = 0; m < M; ++m) {
        for (int g = 0; g < kg; ++g) {
            const uint16_t *src = x + (size_t)m * ldx + (size_t)g * 128;
            float amax = 0.0f;
            for (int j = 0; j < 128; ++j) {
                float a = fabsf(bf16_to_f32(src[j]));
                if (a > amax)
                    amax = a;
            }
            float s = group_scale(amax);
            xs[(size_t)m * kg + g] = s;
            for (int j = 0; j < 128; ++j) {
                float t = bf16_to_f32(src[j]) / s;
                xq[(size_t)m * K + (size_t)g * 128 + j] = oracle_e4m3_encode(t);
            }
        }
    }
    return 0;
}

/* Weights: W [N rows, K cols] row-major, dtype 0 = fp32, 1 = bf16 bits.
   Writes wq [N*K] and ws [ceil(N/128) * K/128].  Returns 0 or -1. */
int oracle_quant_weight(const void *w, int dtype, int N, int K,
                        uint8_t *wq, float *ws)
{
    if (N < 0 || K < 0 || K % 128 != 0 || (dtype != 0 && dtype != 1))
        return -1;
    int kg = K / 128;
    int nblk = (N + 127) / 128;
    const float *wf = (const float *)w;
    const uint16_t *wb = (const uint16_t *)w;
    for (int nb = 0; nb < nblk; ++nb) {
        int r0 = nb * 128;
        int r1 = r0 + 128 < N ? r0 + 128 : N;
        for (int kb = 0; kb < kg; ++kb) {
            float amax = 0.0f;
            for (int r = r0; r < r1; ++r)
                for (int j = 0; j < 128; ++j) {
                    size_t i = (size_t)r * K + (size_t)kb * 128 + j;
                    float v = dtype == 0 ? wf[i] : bf16_to_f32(wb[i]);
#if ORACLE_MUTANT == 8
                    float a = v;                /* mutant: signed maximum */
#else
                    float a = fabsf(v);
#endif
                    if (a > amax)
                        amax = a;
                }
            float s = group_scale(amax);
            ws[(size_t)nb * kg + kb] = s;
            for (int r = r0; r < r1; ++r)
                for (int j = 0; j < 128; ++j) {
                    size_t i = (size_t)r * K + (size_t)kb * 128 + j;
                    float v = dtype == 0 ? wf[i] : bf16_to_f32(wb[i]);
                    wq[i] = oracle_e4m3_encode(v / s);
                }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Block-scaled GEMM in fp64.                                           */
/* ------------------------------------------------------------------ */

typedef struct {
    /* fp8 GEMM operands */
    const uint8_t *aq;
    const float *as;
    const uint8_t *wq;
    const float *ws;
    /* bf16 GEMM operands */
    const uint16_t *xb;
    const uint16_t *wb;
    /* MX GEMM scale bytes (codes in aq / wq) */
    const uint8_t *as8;
    const uint8_t *ws8;
    int M, N, K;
    const int *cols;   /* optional list of output columns */
    int ncols;
    double *y;         /* [M][ncols] */
    double *bound;     /* [M][ncols] */
    int j0, j1;        /* this worker's column range */
    double table[256];
} gemm_job;

static void fp8_columns(gemm_job *g)
{
    int kg = g->K / 128;
    int kb_end = kg;
#if ORACLE_MUTANT == 4
    kb_end = kg - 1;                                   /* mutant: last block dropped */
#endif
    for (int j = g->j0; j < g->j1; ++j) {
        int n = g->cols ? g->cols[j] : j;
        const uint8_t *wrow = g->wq + (size_t)n * g->K;
        const float *wsc = g->ws + (size_t)(n / 128) * kg;
        for (int m = 0; m < g->M; ++m) {
            const uint8_t *arow = g->aq + (size_t)m * g->K;
            const float *asc = g->as + (size_t)m * kg;
            double y = 0.0, bound = 0.0;
            for (int kb = 0; kb < kb_end; ++kb) {
                double p = 0.0, pabs = 0.0;
                for (int k = kb * 128; k < kb * 128 + 128; ++k) {
#if ORACLE_MUTANT == 9
                    /* mutant: weight read as if stored [K][N] */
                    double prod = g->table[arow[k]] * g->table[g->wq[(size_t)k * g->N + n]];
#else
                    double prod = g->table[arow[k]] * g->table[wrow[k]];
#endif
                    p += prod;
                    pabs += fabs(prod);
                }
#if ORACLE_MUTANT == 5
                /* mutant: weight scales read as if stored [K/128][N/128] */
                double sc = (double)asc[kb] *
                            (double)g->ws[(size_t)kb * ((g->N + 127) / 128) + n / 128];
#elif ORACLE_MUTANT == 6
                /* mutant: activation scales read as if stored [K/128][M] */
                double sc = (double)g->as[(size_t)kb * g->M + m] * (double)wsc[kb];
#else
                double sc = (double)asc[kb] * (double)wsc[kb];
#endif
                y += sc * p;
                bound += fabs(sc) * pabs;
            }
            g->y[(size_t)m * g->ncols + j] = y;
            g->bound[(size_t)m * g->ncols + j] = bound;
        }
    }
}

static void bf16_columns(gemm_job *g)
{
    for (int j = g->j0; j < g->j1; ++j) {
        int n = g->cols ? g->cols[j] : j;
        const uint16_t *wrow = g->wb + (size_t)n * g->K;
        for (int m = 0; m < g->M; ++m) {
            const uint16_t *xrow = g->xb + (size_t)m * g->K;
            double y = 0.0, bound = 0.0;
            for (int k = 0; k < g->K; ++k) {
                double prod = (double)bf16_to_f32(xrow[k]) *
                              (double)bf16_to_f32(wrow[k]);
                y += prod;
                bound += fabs(prod);
            }
            g->y[(size_t)m * g->ncols + j] = y;
            g->bound[(size_t)m * g->ncols + j] = bound;
        }
    }
}

/* MX product: 32-wide blocks, scale 2^(byte - 127) per block and operand. */
static void mx_columns(gemm_job *g)
{
    int kb32 = g->K / 32;
    for (int j = g->j0; j < g->j1; ++j) {
        int n = g->cols ? g->cols[j] : j;
        const uint8_t *wrow = g->wq + (size_t)n * g->K;
        const uint8_t *wsc = g->ws8 + (size_t)n * kb32;
        for (int m = 0; m < g->M; ++m) {
            const uint8_t *arow = g->aq + (size_t)m * g->K;
            const uint8_t *asc = g->as8 + (size_t)m * kb32;
            double y = 0.0, bound = 0.0;
            for (int b = 0; b < kb32; ++b) {
                double p = 0.0, pabs = 0.0;
                for (int k = b * 32; k < b * 32 + 32; ++k) {
                    double prod = g->table[arow[k]] * g->table[wrow[k]];
                    p += prod;
                    pabs += fabs(prod);
                }
                double sc = ldexp(1.0, (int)asc[b] - 127 + (int)wsc[b] - 127);
                y += sc * p;
                bound += sc * pabs;
            }
            g->y[(size_t)m * g->ncols + j] = y;
            g->bound[(size_t)m * g->ncols + j] = bound;
        }
    }
}

static void *fp8_worker(void *p) { fp8_columns((gemm_job *)p); return NULL; }
static void *mx_worker(void *p) { mx_columns((gemm_job *)p); return NULL; }
static void *bf16_worker(void *p) { bf16_columns((gemm_job *)p); return NULL; }

/* Split the output columns over nthreads workers.  Each output element is
   computed by exactly one worker in a fixed order, so the result does not
   depend on the thread count. */
static int run_columns(gemm_job *proto, int nthreads, void *(*fn)(void *))
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    if (nthreads > proto->ncols)
        nthreads = proto->ncols > 0 ? proto->ncols : 1;
    gemm_job *jobs = (gemm_job *)malloc(sizeof(gemm_job) * (size_t)nthreads);
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return -2;
    }
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].j0 = (int)((long long)proto->ncols * t / nthreads);
        jobs[t].j1 = (int)((long long)proto->ncols * (t + 1) / nthreads);
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, fn, &jobs[t]) != 0)
            break;
        started = t;
    }
    fn(&jobs[0]);
    for (int t = 1; t <= started; ++t)
        pthread_join(tid[t], NULL);
    /* Any worker that failed to start runs here, in the calling thread. */
    for (int t = started + 1; t < nthreads; ++t)
        fn(&jobs[t]);
    free(jobs);
    free(tid);
    return 0;
}

/* y[m][j] and bound[m][j] for output columns n = cols[j] (or n = j when cols
   is NULL and ncols == N).  Operands are the quantised tensors in the
   layouts written by oracle_quant_act / oracle_quant_weight. */
int oracle_gemm_fp8(const uint8_t *aq, const float *as,
                    const uint8_t *wq, const float *ws,
                    int M, int N, int K, const int *cols, int ncols,
                    double *y, double *bound, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || K % 128 != 0 || ncols < 0)
        return -1;
    if (cols) {
        for (int j = 0; j < ncols; ++j)
            if (cols[j] < 0 || cols[j] >= N)
                return -1;
    } else if (ncols != N) {
        return -1;
    }
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.aq = aq; g.as = as; g.wq = wq; g.ws = ws;
    g.M = M; g.N = N; g.K = K; g.cols = cols; g.ncols = ncols;
    g.y = y; g.bound = bound;
    oracle_e4m3_decode_table(g.table);
    return run_columns(&g, nthreads, fp8_worker);
}

/* Plain bf16 x bf16 product with fp64 accumulation: y = sum_k x[m,k] w[n,k]. */
int oracle_gemm_bf16(const uint16_t *x, const uint16_t *w,
                     int M, int N, int K, const int *cols, int ncols,
                     double *y, double *bound, int nthreads)
{
    if (M < 0 || N < 0 || K < 0 || ncols < 0)
        return -1;
    if (cols) {
        for (int j = 0; j < ncols; ++j)
            if (cols[j] < 0 || cols[j] >= N)
                return -1;
    } else if (ncols != N) {
        return -1;
    }
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.xb = x; g.wb = w;
    g.M = M; g.N = N; g.K = K; g.cols = cols; g.ncols = ncols;
    g.y = y; g.bound = bound;
    return run_columns(&g, nthreads, bf16_worker);
}

/* fp32 -> bf16 bits, round to nearest even (used to form the bf16 copy of an
   fp32 weight matrix for the 16-bit comparison layer). */
uint16_t oracle_f32_to_bf16(float v)
{
    return oracle_round_bf16((double)v);
}

/* ------------------------------------------------------------------ */
/* Greedy token choice over the output layer's logits.                  */
/* ------------------------------------------------------------------ */
/* The output layer feeds the greedy choice of the next token ("The profiler
   said the kernel ran zero times", section "The output layer, which did
   run").  Reading taken: for each token row m of the bf16 logits
   Y [M rows, row stride ldy] (bit patterns), token[m] = the column n < N of
   the largest value, compared as numbers (+0 equals -0); among equal values
   the lowest n.  logit[m] (optional) = that largest value, with a zero
   reported as +0.  NaN logits are outside the contract: -1. */
int oracle_greedy(const uint16_t *y, int M, int N, int ldy, int32_t *token, float *logit)
{
    if (M < 0 || N < 1 || ldy < N)
        return -1;
    for (int m = 0; m < M; ++m) {
        const uint16_t *row = y + (size_t)m * ldy;
        int best = 0;
        float bv = bf16_to_f32(row[0]);
        for (int n = 0; n < N; ++n) {
            float v = bf16_to_f32(row[n]);
            if (isnan(v))
                return -1;
#if ORACLE_MUTANT == 12
            if (v >= bv) {                 /* mutant: ties go to the highest column */
#elif ORACLE_MUTANT == 13
            if (v > bv || (v == bv && signbit(bv) && !signbit(v))) { /* mutant: -0 below +0 */
#else
            if (v > bv) {
#endif
                best = n;
                bv = v;
            }
        }
        token[m] = best;
        if (logit)
            logit[m] = bv == 0.0f ? 0.0f : bv;
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* MX (microscaling) E4M3: 32 consecutive values along K share one      */
/* power-of-two scale stored as an 8-bit biased exponent (UE8M0).        */
/* ------------------------------------------------------------------ */
/* The pages only name the MX formats ("Kernel-Level Optimisations for LLM
   Inference and Training", on CUTLASS).  Reading taken, the conversion of
   the OCP Microscaling Formats specification: per block of 32 values, with
   amax the largest magnitude, the shared exponent is
   e = floor(log2(amax)) - 8 (8 = the exponent of E4M3's largest normal,
   448 = 1.75 * 2^8), clamped to [-127, 127]; the scale is X = 2^e, stored as
   the byte e + 127; each element is E4M3(v / X), nearest-even and
   saturating at 448 (v / X is exact: X is a power of two).  A block of
   zeros takes e = 0.  Input: rows x K values, fp32 (dtype 0) or bf16 bit
   patterns (dtype 1), K % 32 == 0.  Output: codes [rows][K], scale bytes
   [rows][K/32]. */
int oracle_mx_quant(const void *x, int dtype, int rows, int K, uint8_t *codes, uint8_t *scale_bytes)
{
    if (rows < 0 || K <= 0 || K % 32 != 0 || (dtype != 0 && dtype != 1))
        return -1;
    for (int r = 0; r < rows; ++r) {
        for (int b = 0; b < K / 32; ++b) {
            float v[32];
            float amax = 0.0f;
            for (int j = 0; j < 32; ++j) {
                size_t i = (size_t)r * K + (size_t)b * 32 + j;
                v[j] = dtype == 0 ? ((const float *)x)[i] : bf16_to_f32(((const uint16_t *)x)[i]);
                if (isnan(v[j]) || isinf(v[j]))
                    return -1;
                if (fabsf(v[j]) > amax)
                    amax = fabsf(v[j]);
            }
            int e = 0;
            if (amax > 0.0f) {
                int ex;
                frexp((double)amax, &ex);       /* amax = f * 2^ex, f in [0.5, 1) */
#if ORACLE_MUTANT == 14
                e = (ex - 1) - 7;               /* mutant: another element maximum exponent */
#elif ORACLE_MUTANT == 15
                e = ex - 8;                     /* mutant: ceiling instead of floor of log2 */
#else
                e = (ex - 1) - 8;
#endif
                if (e < -127)
                    e = -127;
                if (e > 127)
                    e = 127;
            }
            scale_bytes[(size_t)r * (K / 32) + b] = (uint8_t)(e + 127);
            for (int j = 0; j < 32; ++j) {
                /* exact in fp64; representable in fp32 whenever it is not
                   far below the smallest E4M3 step, where it rounds to zero
                   either way */
                float t = (float)ldexp((double)v[j], -e);
                codes[(size_t)r * K + (size_t)b * 32 + j] = oracle_e4m3_encode(t);
            }
        }
    }
    return 0;
}

/* y[m][j] = sum over 32-wide blocks b of 2^(ea[m,b] + ew[n,b]) *
   sum_{k in b} dec(aq[m,k]) * dec(wq[n,k]), n = cols[j] (or j), in fp64
   (exact: every block sum is exact and the scales are powers of two);
   bound = the same with |products|. */
int oracle_mx_gemm(const uint8_t *aq, const uint8_t *as8, const uint8_t *wq, const uint8_t *ws8,
                   int M, int N, int K, const int *cols, int ncols, double *y, double *bound, int nthreads)
{
    if (M < 0 || N < 0 || K <= 0 || K % 32 != 0 || ncols < 0)
        return -1;
    if (cols) {
        for (int j = 0; j < ncols; ++j)
            if (cols[j] < 0 || cols[j] >= N)
                return -1;
    } else if (ncols != N) {
        return -1;
    }
    gemm_job g;
    memset(&g, 0, sizeof g);
    g.aq = aq; g.as8 = as8; g.wq = wq; g.ws8 = ws8;
    g.M = M; g.N = N; g.K = K; g.cols = cols; g.ncols = ncols;
    g.y = y; g.bound = bound;
    oracle_e4m3_decode_table(g.table);
    return run_columns(&g, nthreads, mx_worker);
}
