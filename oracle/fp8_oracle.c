/*
 * CPU oracle for the FP8 GEMM path.  TEST INFRASTRUCTURE ONLY: the tests,
 * the smoke check and the bench's CPU-baseline leg use it; the library never
 * does.  It shares no code, header or table with the CUDA path.
 *
 * What it computes (plain definitions, fp64):
 *
 *   dense   D[m,n]   = bf16_rne( sum_k dec(A[m,k]) * dec(B[n,k]) )
 *   masked  D[g,m,n] = bf16_rne( sum_k dec(A[g,m,k]) * dec(B[g,n,k]) )
 *                       for m < masked_m[g]; other rows of D untouched.
 *   scaled  the same with the exact sum multiplied by per-tensor or
 *           per-channel FP32 scales sa * sb before the one rounding.
 *   block-scaled  every product a_k b_k multiplied by the UE8M0 scales of
 *           the K group (of 32 or 128 elements) that k falls in, for its
 *           row of A and its row of B, before the sum.
 *   contiguous  D[r,n] = bf16_rne( sum_k dec(A[r,k]) * dec(B[g,n,k]) ) for the
 *           rows r of group g in a concatenated [M_total, K] token array.
 *   epilogue  round_mode(act(alpha * S + beta * C + bias)) of any of the
 *           above sums S, with BF16 rounding to nearest even, toward zero,
 *           toward +infinity or toward -infinity.
 *
 * Sources:
 *  - "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
 *    (sheratonhq.com/news/187119), §1.3: A and B are FP8 (E4M3/E5M2
 *    selectable), the accumulator is FP32; §3.1: E4M3 is 4 exponent + 3
 *    mantissa bits, E5M2 is 5 + 2.
 *  - "一次“转置”，半张算力：DeepSeek SwapAB 漂流史" (hwcomputing.csdn.net),
 *    §3.1/§3.3: the masked grouped GEMM m_grouped_fp8_gemm_nt_masked, where
 *    only the first valid_m token rows of each group are real.
 *
 * Readings (the pages give only the bit splits of the two formats):
 *  - FP8 codes follow the OCP 8-bit float definitions as NVIDIA hardware
 *    implements them: E4M3 has bias 7, no infinity and NaN only at S.1111.111;
 *    E5M2 has bias 15, IEEE-style infinities and NaNs at exponent 31.
 *  - The GPU accumulates in FP32 in hardware order; the oracle accumulates the
 *    exact products in double in ascending k (each product of two FP8 values is
 *    exact in double) and rounds once to BF16, round-to-nearest-even.
 */
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_E4M3 0
#define ORACLE_E5M2 1

/* ---- FP8 decode, from the closed form of each format ------------------ */

/* E4M3: s | e(4) | m(3), bias 7.
 *   e == 0          : (-1)^s * (m/8) * 2^-6       (subnormal, incl. +-0)
 *   e == 15, m == 7 : NaN                         (no infinities)
 *   otherwise       : (-1)^s * (1 + m/8) * 2^(e-7)
 * E5M2: s | e(5) | m(2), bias 15.
 *   e == 0          : (-1)^s * (m/4) * 2^-14
 *   e == 31         : +-inf if m == 0, else NaN
 *   otherwise       : (-1)^s * (1 + m/4) * 2^(e-15)
 */
double oracle_decode_fp8(uint8_t code, int fmt)
{
    int s = (code >> 7) & 1;
    double v;
    if (fmt == ORACLE_E4M3) {
        int e = (code >> 3) & 0xF;
        int m = code & 0x7;
        if (e == 15 && m == 7)
            return NAN;
        if (e == 0)
            v = ((double)m / 8.0) * ldexp(1.0, -6);
        else
            v = (1.0 + (double)m / 8.0) * ldexp(1.0, e - 7);
    } else {
        int e = (code >> 2) & 0x1F;
        int m = code & 0x3;
        if (e == 31)
            return m == 0 ? (s ? -INFINITY : INFINITY) : NAN;
        if (e == 0)
            v = ((double)m / 4.0) * ldexp(1.0, -14);
        else
            v = (1.0 + (double)m / 4.0) * ldexp(1.0, e - 15);
    }
    return s ? -v : v;
}

/* Fill a 256-entry table with oracle_decode_fp8 of every code. */
void oracle_decode_table(int fmt, double *out256)
{
    for (int c = 0; c < 256; ++c)
        out256[c] = oracle_decode_fp8((uint8_t)c, fmt);
}

/* ---- BF16 rounding ----------------------------------------------------- */

/* Round a double to the nearest BF16 (1 sign, 8 exponent, 7 stored mantissa
 * bits, bias 127), ties to even, overflow to infinity, gradual underflow.
 * Written from the format definition: find the binade of |x|, divide by the
 * spacing of that binade (a power of two, so exact), round the quotient to an
 * integer with ties to even, and re-pack. */
uint16_t oracle_round_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;

    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1)         */
    int E = e2 - 1;               /* floor(log2 a)                       */
    if (E < -126)
        E = -126;                 /* below the normal range: fixed spacing */
    double spacing = ldexp(1.0, E - 7);
    double q = a / spacing;       /* exact: division by a power of two   */
    double f = floor(q);
    double rem = q - f;           /* exact                               */
    if (rem > 0.5 || (rem == 0.5 && fmod(f, 2.0) != 0.0))
        f += 1.0;

    if (f >= 256.0) {             /* rounded up into the next binade     */
        f = 128.0;
        E += 1;
    }
    if (f < 128.0)                /* subnormal (only possible at E=-126) */
        return sign | (uint16_t)f;
    if (E > 127)
        return sign | 0x7F80;     /* overflow                            */
    return sign | (uint16_t)(((E + 127) << 7) | ((int)f - 128));
}

/* Round a double to BF16 with a given rounding direction: 0 nearest-even
 * (as above), 1 toward zero, 2 toward +infinity, 3 toward -infinity.  Same
 * construction: the quotient by the binade's spacing is truncated, then
 * bumped by one unit when the direction asks for it; a finite value beyond
 * the largest BF16 goes to infinity only when rounding away from zero in its
 * direction, otherwise to the largest finite value (IEEE 754 directed
 * rounding). */
uint16_t oracle_round_bf16_mode(double x, int mode)
{
    if (mode == 0)
        return oracle_round_bf16(x);
    if (isnan(x))
        return 0x7FC0;
    int neg = signbit(x) ? 1 : 0;
    uint16_t sign = neg ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    if (isinf(a))
        return sign | 0x7F80;
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;
    if (E < -126)
        E = -126;
    double spacing = ldexp(1.0, E - 7);
    double q = a / spacing;
    double f = floor(q);
    int inexact = (q - f) != 0.0;
    /* away from zero: toward +inf for positives, toward -inf for negatives */
    int away = (mode == 2 && !neg) || (mode == 3 && neg);
    if (inexact && away)
        f += 1.0;
    if (f >= 256.0) {
        f = 128.0;
        E += 1;
    }
    if (f < 128.0)
        return sign | (uint16_t)f;
    if (E > 127)
        return away ? (uint16_t)(sign | 0x7F80) : (uint16_t)(sign | 0x7F7F);
    return sign | (uint16_t)(((E + 127) << 7) | ((int)f - 128));
}

/* BF16 code -> double (exact). */
double oracle_bf16_to_double(uint16_t h)
{
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int m = h & 0x7F;
    double v;
    if (e == 0xFF)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = (double)m * ldexp(1.0, -133);
    else
        v = (double)(128 + m) * ldexp(1.0, e - 134);
    return s ? -v : v;
}

/* ---- threading helper (splits output rows; no change to arithmetic) --- */

static int oracle_cpu_count(void)
{
#ifdef CPU_COUNT
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int c = CPU_COUNT(&set);
        if (c > 0)
            return c;
    }
#endif
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

int oracle_default_threads(void) { return oracle_cpu_count(); }

typedef void (*row_fn)(void *ctx, int64_t row);

typedef struct {
    row_fn fn;
    void *ctx;
    int64_t rows;
    int64_t next;
    pthread_mutex_t lock;
} row_pool;

static void *row_worker(void *arg)
{
    row_pool *p = (row_pool *)arg;
    for (;;) {
        pthread_mutex_lock(&p->lock);
        int64_t r = p->next++;
        pthread_mutex_unlock(&p->lock);
        if (r >= p->rows)
            break;
        p->fn(p->ctx, r);
    }
    return NULL;
}

static void run_rows(row_fn fn, void *ctx, int64_t rows, int nthreads)
{
    if (nthreads <= 0)
        nthreads = oracle_cpu_count();
    if (nthreads > rows)
        nthreads = (int)(rows > 0 ? rows : 1);
    row_pool p;
    p.fn = fn;
    p.ctx = ctx;
    p.rows = rows;
    p.next = 0;
    pthread_mutex_init(&p.lock, NULL);
    if (nthreads <= 1) {
        row_worker(&p);
    } else {
        pthread_t *t = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; ++i)
            pthread_create(&t[i], NULL, row_worker, &p);
        for (int i = 0; i < nthreads; ++i)
            pthread_join(t[i], NULL);
        free(t);
    }
    pthread_mutex_destroy(&p.lock);
}

/* ---- the contraction --------------------------------------------------- */

/* One output element: the exact dot product of row a (K codes, format fa)
 * with row b (K codes, format fb), summed in double in ascending k.  Also
 * returns sum_k |a_k * b_k|, which scales the tolerance of the GPU result. */
static double dot_row(const uint8_t *a, const uint8_t *b, int64_t K,
                      const double *ta, const double *tb, double *absdot)
{
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double p = ta[a[k]] * tb[b[k]];
        s += p;
        sa += fabs(p);
    }
    *absdot = sa;
    return s;
}

typedef struct {
    const uint8_t *A, *B;
    int64_t M, N, K;
    double ta[256], tb[256];
    uint16_t *D;       /* [M,N] bf16 codes, may be NULL */
    double *exact;     /* [M,N] double sums, may be NULL */
    double *absdot;    /* [M,N], may be NULL */
} gemm_ctx;

static void gemm_row(void *vctx, int64_t m)
{
    gemm_ctx *c = (gemm_ctx *)vctx;
    const uint8_t *a = c->A + m * c->K;
    for (int64_t n = 0; n < c->N; ++n) {
        double ad;
        double s = dot_row(a, c->B + n * c->K, c->K, c->ta, c->tb, &ad);
        int64_t o = m * c->N + n;
        if (c->D)
            c->D[o] = oracle_round_bf16(s);
        if (c->exact)
            c->exact[o] = s;
        if (c->absdot)
            c->absdot[o] = ad;
    }
}

/* Dense D[M,N] = A[M,K] * B[N,K]^T.  A and B are row-major with K
 * contiguous (the "NT" layout).  nthreads <= 0 uses every core available. */
void oracle_gemm_nt(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N,
                    int64_t K, int fa, int fb, uint16_t *D, double *exact,
                    double *absdot, int nthreads)
{
    gemm_ctx c;
    c.A = A;
    c.B = B;
    c.M = M;
    c.N = N;
    c.K = K;
    oracle_decode_table(fa, c.ta);
    oracle_decode_table(fb, c.tb);
    c.D = D;
    c.exact = exact;
    c.absdot = absdot;
    run_rows(gemm_row, &c, M, nthreads);
}

/* Selected elements of the dense product: out[i] = D[ms[i], ns[i]]. */
void oracle_gemm_nt_entries(const uint8_t *A, const uint8_t *B, int64_t K,
                            int fa, int fb, const int64_t *ms,
                            const int64_t *ns, int64_t count, uint16_t *D,
                            double *exact, double *absdot)
{
    double ta[256], tb[256];
    oracle_decode_table(fa, ta);
    oracle_decode_table(fb, tb);
    for (int64_t i = 0; i < count; ++i) {
        double ad;
        double s = dot_row(A + ms[i] * K, B + ns[i] * K, K, ta, tb, &ad);
        if (D)
            D[i] = oracle_round_bf16(s);
        if (exact)
            exact[i] = s;
        if (absdot)
            absdot[i] = ad;
    }
}

typedef struct {
    const uint8_t *A, *B;
    const int32_t *masked_m;
    int64_t G, M_max, N, K;
    double ta[256], tb[256];
    uint16_t *D;
    double *absdot;
} grouped_ctx;

/* One (group, row) pair; rows at or beyond the group's valid count are left
 * exactly as the caller passed them. */
static void grouped_row(void *vctx, int64_t gm)
{
    grouped_ctx *c = (grouped_ctx *)vctx;
    int64_t g = gm / c->M_max, m = gm % c->M_max;
    if (m >= (int64_t)c->masked_m[g])
        return;
    const uint8_t *a = c->A + (g * c->M_max + m) * c->K;
    const uint8_t *b = c->B + g * c->N * c->K;
    for (int64_t n = 0; n < c->N; ++n) {
        double ad;
        double s = dot_row(a, b + n * c->K, c->K, c->ta, c->tb, &ad);
        int64_t o = (g * c->M_max + m) * c->N + n;
        c->D[o] = oracle_round_bf16(s);
        if (c->absdot)
            c->absdot[o] = ad;
    }
}

/* Masked grouped D[g,m,n] for m < masked_m[g]; A[G,M_max,K], B[G,N,K],
 * D[G,M_max,N].  masked_m values must already lie in [0, M_max]. */
void oracle_gemm_grouped_masked(const uint8_t *A, const uint8_t *B,
                                const int32_t *masked_m, int64_t G,
                                int64_t M_max, int64_t N, int64_t K, int fa,
                                int fb, uint16_t *D, double *absdot,
                                int nthreads)
{
    grouped_ctx c;
    c.A = A;
    c.B = B;
    c.masked_m = masked_m;
    c.G = G;
    c.M_max = M_max;
    c.N = N;
    c.K = K;
    oracle_decode_table(fa, c.ta);
    oracle_decode_table(fb, c.tb);
    c.D = D;
    c.absdot = absdot;
    run_rows(grouped_row, &c, G * M_max, nthreads);
}

/* ---- scaled variants ------------------------------------------------------
 * "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" §3.1: the
 * scale is computed beforehand and multiplied back at the output; §5.2: the
 * scale may be per tensor or per channel.  Here
 *     D[m,n] = bf16_rne( sa(m) * sb(n) * sum_k dec(A[m,k]) * dec(B[n,k]) )
 * with sa(m) = scale_a[0] (sa_len == 1) or scale_a[m] (sa_len == M), and
 * sb(n) = scale_b[0] or scale_b[n].  The product is formed in double and
 * rounded once.  absdot (if given) receives |sa(m) sb(n)| * sum_k |a_k b_k|. */
void oracle_gemm_nt_scaled(const uint8_t *A, const uint8_t *B, int64_t M, int64_t N,
                           int64_t K, int fa, int fb, const float *scale_a,
                           int64_t sa_len, const float *scale_b, int64_t sb_len,
                           uint16_t *D, double *absdot, int nthreads)
{
    double *exact = (double *)malloc(sizeof(double) * (size_t)(M * N));
    double *ad = (double *)malloc(sizeof(double) * (size_t)(M * N));
    oracle_gemm_nt(A, B, M, N, K, fa, fb, NULL, exact, ad, nthreads);
    for (int64_t m = 0; m < M; ++m) {
        double sa = (double)scale_a[sa_len == 1 ? 0 : m];
        for (int64_t n = 0; n < N; ++n) {
            double sb = (double)scale_b[sb_len == 1 ? 0 : n];
            int64_t o = m * N + n;
            D[o] = oracle_round_bf16(sa * sb * exact[o]);
            if (absdot)
                absdot[o] = fabs(sa * sb) * ad[o];
        }
    }
    free(exact);
    free(ad);
}

/* Masked grouped, scaled: sa(g,m) = scale_a[g] (sa_len == G) or
 * scale_a[g*M_max + m] (sa_len == G*M_max); sb(g,n) = scale_b[g] or
 * scale_b[g*N + n].  Rows m >= masked_m[g] are left untouched. */
void oracle_gemm_grouped_masked_scaled(const uint8_t *A, const uint8_t *B,
                                       const int32_t *masked_m, int64_t G,
                                       int64_t M_max, int64_t N, int64_t K, int fa,
                                       int fb, const float *scale_a, int64_t sa_len,
                                       const float *scale_b, int64_t sb_len,
                                       uint16_t *D, double *absdot, int nthreads)
{
    for (int64_t g = 0; g < G; ++g) {
        int64_t m_g = masked_m[g];
        if (m_g <= 0)
            continue;
        double *exact = (double *)malloc(sizeof(double) * (size_t)(m_g * N));
        double *ad = (double *)malloc(sizeof(double) * (size_t)(m_g * N));
        oracle_gemm_nt(A + g * M_max * K, B + g * N * K, m_g, N, K, fa, fb, NULL, exact, ad,
                       nthreads);
        for (int64_t m = 0; m < m_g; ++m) {
            double sa = (double)scale_a[sa_len == G ? g : g * M_max + m];
            for (int64_t n = 0; n < N; ++n) {
                double sb = (double)scale_b[sb_len == G ? g : g * N + n];
                int64_t o = (g * M_max + m) * N + n;
                D[o] = oracle_round_bf16(sa * sb * exact[m * N + n]);
                if (absdot)
                    absdot[o] = fabs(sa * sb) * ad[m * N + n];
            }
        }
        free(exact);
        free(ad);
    }
}

/* ---- block-scaled variant ---------------------------------------------------
 * "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" §5.2: scales
 * may be kept per group of 128 elements; "一次“转置”，半张算力：DeepSeek SwapAB
 * 漂流史" §5 (timeline) gives the SM100 form as UE8M0 ("packed") scale
 * factors and §3.4 shows the Blackwell MMA consuming A- and B-side scale
 * factors.  Reading: with gran in {32, 128} and KS = ceil(K/gran),
 *     D[g,m,n] = bf16_rne( sum_k dec(A[g,m,k]) dec(B[g,n,k])
 *                          * 2^(SA[g][k/gran][m] - 127) * 2^(SB[g][k/gran][n] - 127) )
 * SA is [G][KS][lda] bytes (row m of A at byte m of each K group's vector),
 * SB is [G][KS][ldb].  A UE8M0 code is a power of two 2^(e-127); code 255 is
 * NaN (OCP microscaling formats).  Every product is exact in double; the sum
 * is taken in ascending k and rounded once.  absdot receives
 * sum_k |a_k b_k| * scales.
 *
 * accbound (may be NULL) receives 2^-23 * sum_i |S_i|, S_i the running sum
 * after the i-th slice of 32 consecutive k (the K of one tensor-core MMA
 * instruction on 8-bit operands, "一次“转置”，半张算力" §1.1; a shorter last
 * slice counts as one).  It bounds the error of a hardware accumulator that
 * adds each instruction's result into an FP32 running sum with at most one
 * FP32 ulp (2^-23 relative) of error per addition, whatever its rounding
 * direction.  "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践"
 * §5.1: FP32 accumulation still carries the rounding error of its order,
 * largest when intermediate sums are much larger than the result, and the
 * tensor core's accumulation path is fixed in hardware; block scales make
 * exactly that case (products of one K group up to 2^28 times another's). */
static double ue8m0_value(uint8_t e)
{
    return e == 255 ? NAN : ldexp(1.0, (int)e - 127);
}

typedef struct {
    const uint8_t *A, *B, *SA, *SB;
    const int32_t *masked_m;   /* NULL: every row */
    int64_t G, M_max, N, K, lda, ldb, gran, KS;
    double ta[256], tb[256];
    uint16_t *D;
    double *exact;     /* sums before rounding, may be NULL */
    double *absdot;
    double *accbound;  /* 2^-23 * sum of |running sum| at 32-element slice ends, may be NULL */
} bs_ctx;

static void blockscaled_row(void *vctx, int64_t gm)
{
    bs_ctx *c = (bs_ctx *)vctx;
    int64_t g = gm / c->M_max, m = gm % c->M_max;
    if (c->masked_m && m >= (int64_t)c->masked_m[g])
        return;
    const uint8_t *a = c->A + (g * c->M_max + m) * c->K;
    const uint8_t *sa = c->SA + g * c->KS * c->lda + m;
    for (int64_t n = 0; n < c->N; ++n) {
        const uint8_t *b = c->B + (g * c->N + n) * c->K;
        const uint8_t *sb = c->SB + g * c->KS * c->ldb + n;
        double s = 0.0, ad = 0.0, runs = 0.0;
        for (int64_t kg = 0; kg < c->KS; ++kg) {
            double f = ue8m0_value(sa[kg * c->lda]) * ue8m0_value(sb[kg * c->ldb]);
            int64_t k1 = (kg + 1) * c->gran < c->K ? (kg + 1) * c->gran : c->K;
            for (int64_t k = kg * c->gran; k < k1; ++k) {
                double p = c->ta[a[k]] * c->tb[b[k]] * f;
                s += p;
                ad += fabs(p);
                if ((k + 1) % 32 == 0 || k + 1 == c->K)
                    runs += fabs(s);
            }
        }
        int64_t o = (g * c->M_max + m) * c->N + n;
        c->D[o] = oracle_round_bf16(s);
        if (c->exact)
            c->exact[o] = s;
        if (c->absdot)
            c->absdot[o] = ad;
        if (c->accbound)
            c->accbound[o] = ldexp(runs, -23);
    }
}

/* Grouped form; dense is G = 1, masked_m = NULL.  A[G,M_max,K],
 * B[G,N,K], D[G,M_max,N]; rows m >= masked_m[g] of D are left untouched. */
void oracle_gemm_blockscaled(const uint8_t *A, const uint8_t *B, const int32_t *masked_m,
                             int64_t G, int64_t M_max, int64_t N, int64_t K, int fa, int fb,
                             const uint8_t *SA, int64_t lda, const uint8_t *SB, int64_t ldb,
                             int64_t gran, uint16_t *D, double *exact, double *absdot, double *accbound,
                             int nthreads)
{
    bs_ctx c;
    c.A = A;
    c.B = B;
    c.SA = SA;
    c.SB = SB;
    c.masked_m = masked_m;
    c.G = G;
    c.M_max = M_max;
    c.N = N;
    c.K = K;
    c.lda = lda;
    c.ldb = ldb;
    c.gran = gran;
    c.KS = (K + gran - 1) / gran;
    oracle_decode_table(fa, c.ta);
    oracle_decode_table(fb, c.tb);
    c.D = D;
    c.exact = exact;
    c.absdot = absdot;
    c.accbound = accbound;
    run_rows(blockscaled_row, &c, G * M_max, nthreads);
}

/* ---- fused epilogue ----------------------------------------------------------
 * "DeepGEMM：基于 Hopper Tensor Core 的 FP8 矩阵乘法内核优化实践" §3.3: the
 * epilogue computes C = alpha * A B + beta * C + bias (bias per output
 * channel) with an optional ReLU inside the GEMM, and the final rounding may
 * be to nearest even, toward zero or toward +infinity.  Reading: for each
 * output element with product value S (the exact sum, already multiplied by
 * any output or block scales),
 *     out = round_mode( act( alpha * S + beta * C[row, n] + bias[group, n] ) )
 * with C a BF16 array shaped like D (NULL: the term is absent), bias FP32
 * [groups][N] (NULL: absent), act 0 = none, 1 = ReLU (x < 0 becomes +0; NaN
 * stays NaN), evaluated in double and rounded once.  Row r belongs to group
 * r / rows_per_group; with masked_m (NULL: every row) rows at or beyond
 * masked_m[group] keep D's bits.  absdot receives
 * |alpha| * absS + |beta * C| + |bias|. */
void oracle_epilogue(const double *S, const double *absS, int64_t rows, int64_t rows_per_group,
                     int64_t N, const int32_t *masked_m, double alpha, double beta, const uint16_t *C,
                     const float *bias, int act, int mode, uint16_t *D, double *absdot)
{
    for (int64_t r = 0; r < rows; ++r) {
        int64_t g = r / rows_per_group;
        if (masked_m && (r % rows_per_group) >= (int64_t)masked_m[g])
            continue;
        for (int64_t n = 0; n < N; ++n) {
            int64_t o = r * N + n;
            double c = C ? oracle_bf16_to_double(C[o]) : 0.0;
            double b = bias ? (double)bias[g * N + n] : 0.0;
            double v = alpha * S[o] + beta * c + b;
            if (act == 1 && v < 0.0)
                v = 0.0;
            D[o] = oracle_round_bf16_mode(v, mode);
            if (absdot)
                absdot[o] = fabs(alpha) * absS[o] + fabs(beta * c) + fabs(b);
        }
    }
}

/* ---- contiguous grouped layout ------------------------------------------------
 * "一次“转置”，半张算力：DeepSeek SwapAB 漂流史" §3.1 names the masked grouped
 * form and its §5 timeline counts four grouped layouts on SM100 without
 * describing the others.  Reading for the contiguous form: the token rows of all groups
 * are concatenated along M in group order, group g owning rows
 * offsets[g] .. offsets[g+1]-1 of A [M_total, K] and of D [M_total, N], and
 * multiplying B[g] [N, K]:
 *     D[r, n] = bf16_rne( sum_k dec(A[r, k]) * dec(B[g, n, k]) ),  offsets[g] <= r < offsets[g+1]
 * Rows outside every group keep D's bits.  offsets is nondecreasing with
 * 0 <= offsets[0] and offsets[G] <= M_total. */
typedef struct {
    const uint8_t *A, *B;
    const int32_t *offsets;
    int64_t G, N, K;
    double ta[256], tb[256];
    uint16_t *D;
    double *exact, *absdot;
} contig_ctx;

static void contig_row(void *vctx, int64_t r)
{
    contig_ctx *c = (contig_ctx *)vctx;
    int64_t g = -1;
    for (int64_t i = 0; i < c->G; ++i)
        if (r >= (int64_t)c->offsets[i] && r < (int64_t)c->offsets[i + 1]) {
            g = i;
            break;
        }
    if (g < 0)
        return;
    const uint8_t *a = c->A + r * c->K;
    for (int64_t n = 0; n < c->N; ++n) {
        double ad;
        double s = dot_row(a, c->B + (g * c->N + n) * c->K, c->K, c->ta, c->tb, &ad);
        int64_t o = r * c->N + n;
        c->D[o] = oracle_round_bf16(s);
        if (c->exact)
            c->exact[o] = s;
        if (c->absdot)
            c->absdot[o] = ad;
    }
}

void oracle_gemm_grouped_contiguous(const uint8_t *A, const uint8_t *B, const int32_t *offsets, int64_t G,
                                    int64_t M_total, int64_t N, int64_t K, int fa, int fb, uint16_t *D,
                                    double *exact, double *absdot, int nthreads)
{
    contig_ctx c;
    c.A = A;
    c.B = B;
    c.offsets = offsets;
    c.G = G;
    c.N = N;
    c.K = K;
    oracle_decode_table(fa, c.ta);
    oracle_decode_table(fb, c.tb);
    c.D = D;
    c.exact = exact;
    c.absdot = absdot;
    run_rows(contig_row, &c, M_total, nthreads);
}
