/*
 * Seeded synthetic inputs for the FP8 GEMM tests and bench.
 *
 * This module is shared by the CPU oracle's tests and the GPU path's tests;
 * it holds none of the GEMM arithmetic (no decode, accumulation or output
 * rounding).  It turns a seed and an element index into an FP8 byte:
 *
 *   u      = SplitMix64 output for counter (seed, index)   -> uniform [0,1)
 *   value  = lo + (hi - lo) * u                 (uniform workloads), or
 *            mean + std * sqrt(-2 ln u1) cos(2 pi u2)  (Box-Muller normal)
 *   byte   = FP8 code nearest to value, ties to even, magnitudes beyond the
 *            largest finite code saturate to it
 *
 * Every element depends only on (seed, index), so any slice of a tensor can
 * be regenerated on its own and the fill can be split across threads.
 *
 * SplitMix64 is the generator published by Steele, Lea and Flood
 * ("Fast splittable pseudorandom number generators", OOPSLA 2014): state
 * advances by the golden-ratio increment 0x9E3779B97F4A7C15 and each output
 * is the state passed through the variant-13 finaliser of MurmurHash3.
 */
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdint.h>
#include <stdlib.h>
#include <unistd.h>

#define SYNTH_E4M3 0
#define SYNTH_E5M2 1

static const uint64_t GOLDEN = 0x9E3779B97F4A7C15ULL;

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Output number `i` (0-based) of a SplitMix64 stream started at `seed`:
 * the state after i+1 increments, finalised. */
uint64_t synth_splitmix64_at(uint64_t seed, uint64_t i)
{
    return mix64(seed + (i + 1) * GOLDEN);
}

/* Uniform double in [0,1) from the top 53 bits. */
static inline double unit_from(uint64_t r)
{
    return (double)(r >> 11) * (1.0 / 9007199254740992.0);
}

double synth_uniform_at(uint64_t seed, uint64_t i)
{
    return unit_from(synth_splitmix64_at(seed, i));
}

/* Standard normal for element i: Box-Muller on outputs 2i and 2i+1. */
double synth_normal_at(uint64_t seed, uint64_t i)
{
    double u1 = unit_from(synth_splitmix64_at(seed, 2 * i));
    double u2 = unit_from(synth_splitmix64_at(seed, 2 * i + 1));
    if (u1 <= 0.0)
        u1 = 1.0 / 9007199254740992.0;   /* keep log finite */
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* Nearest FP8 code to x, ties to even mantissa, saturating at the largest
 * finite magnitude (448 for E4M3, 57344 for E5M2).  Values smaller than half
 * the smallest subnormal round to a signed zero.  NaN input gives the
 * format's canonical NaN (never produced by the workloads). */
uint8_t synth_encode_fp8(double x, int fmt)
{
    const int mbits = fmt == SYNTH_E4M3 ? 3 : 2;
    const int bias = fmt == SYNTH_E4M3 ? 7 : 15;
    const int emin = 1 - bias;                   /* exponent of the smallest normal */
    const double maxv = fmt == SYNTH_E4M3 ? 448.0 : 57344.0;
    const uint8_t maxcode = fmt == SYNTH_E4M3 ? 0x7E : 0x7B;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return 0x7F;
    double a = fabs(x);
    if (a >= maxv)
        return sign | maxcode;
    if (a == 0.0)
        return sign;
    int e2;
    (void)frexp(a, &e2);
    int E = e2 - 1;                              /* floor(log2 a) */
    if (E < emin)
        E = emin;
    double q = ldexp(a, mbits - E);              /* significand scaled to an integer grid */
    double f = floor(q);
    double rem = q - f;
    if (rem > 0.5 || (rem == 0.5 && fmod(f, 2.0) != 0.0))
        f += 1.0;
    int top = 1 << (mbits + 1);
    if ((int)f >= top) {                         /* carried into the next binade */
        f = (double)(1 << mbits);
        E += 1;
    }
    int r = (int)f;
    if (r < (1 << mbits))                        /* subnormal (E == emin) or zero */
        return sign | (uint8_t)r;
    int code = ((E + bias) << mbits) | (r - (1 << mbits));
    if (code > maxcode)
        code = maxcode;
    return sign | (uint8_t)code;
}

/* ---- bulk fills, split across threads ---------------------------------- */

typedef struct {
    uint8_t *out;
    int64_t begin, end;
    uint64_t seed;
    int kind;            /* 0 uniform, 1 normal */
    double p0, p1;       /* lo,hi  or  mean,std */
    int fmt;
} fill_job;

static void *fill_worker(void *arg)
{
    fill_job *j = (fill_job *)arg;
    for (int64_t i = j->begin; i < j->end; ++i) {
        double v;
        if (j->kind == 0)
            v = j->p0 + (j->p1 - j->p0) * synth_uniform_at(j->seed, (uint64_t)i);
        else
            v = j->p0 + j->p1 * synth_normal_at(j->seed, (uint64_t)i);
        j->out[i - j->begin] = synth_encode_fp8(v, j->fmt);
    }
    return NULL;
}

static int cpu_count(void)
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

static void fill(uint8_t *out, int64_t first, int64_t n, uint64_t seed,
                 int kind, double p0, double p1, int fmt, int nthreads)
{
    if (n <= 0)
        return;
    if (nthreads <= 0)
        nthreads = cpu_count();
    if (nthreads > 64)
        nthreads = 64;
    int64_t per = (n + nthreads - 1) / nthreads;
    if (per < 65536) {
        per = 65536;
    }
    int jobs = (int)((n + per - 1) / per);
    fill_job js[64];
    pthread_t ts[64];
    for (int t = 0; t < jobs; ++t) {
        int64_t b = first + (int64_t)t * per;
        int64_t e = b + per;
        if (e > first + n)
            e = first + n;
        js[t].out = out + (b - first);
        js[t].begin = b;
        js[t].end = e;
        js[t].seed = seed;
        js[t].kind = kind;
        js[t].p0 = p0;
        js[t].p1 = p1;
        js[t].fmt = fmt;
    }
    if (jobs == 1) {
        fill_worker(&js[0]);
        return;
    }
    for (int t = 0; t < jobs; ++t)
        pthread_create(&ts[t], NULL, fill_worker, &js[t]);
    for (int t = 0; t < jobs; ++t)
        pthread_join(ts[t], NULL);
}

/* Elements [first, first+n) of a tensor of FP8 codes from U[lo,hi). */
void synth_fill_uniform_fp8(uint8_t *out, int64_t first, int64_t n,
                            uint64_t seed, double lo, double hi, int fmt,
                            int nthreads)
{
    fill(out, first, n, seed, 0, lo, hi, fmt, nthreads);
}

/* Elements [first, first+n) of a tensor of FP8 codes from N(mean, std^2). */
void synth_fill_normal_fp8(uint8_t *out, int64_t first, int64_t n,
                           uint64_t seed, double mean, double std, int fmt,
                           int nthreads)
{
    fill(out, first, n, seed, 1, mean, std, fmt, nthreads);
}

/* Integers uniform on [lo, hi] (inclusive) for element i: floor of a
 * uniform draw scaled to the range. */
void synth_fill_uniform_int(int32_t *out, int64_t n, uint64_t seed, int32_t lo,
                            int32_t hi)
{
    double span = (double)hi - (double)lo + 1.0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t v = lo + (int64_t)floor(span * synth_uniform_at(seed, (uint64_t)i));
        if (v > hi)
            v = hi;
        out[i] = (int32_t)v;
    }
}

/* Raw 16-bit patterns (canaries for never-written output rows). */
void synth_fill_u16(uint16_t *out, int64_t n, uint64_t seed)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (uint16_t)(synth_splitmix64_at(seed, (uint64_t)i) >> 48);
}
