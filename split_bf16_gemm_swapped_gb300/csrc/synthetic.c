/*
 * Seeded synthetic bf16 inputs for the split-K decode GEMM.
 *
 * This file only draws numbers; it holds none of the GEMM's arithmetic and is
 * shared by the CUDA path's tests/benchmark and the CPU oracle's callers as
 * the common source of inputs.
 *
 * Generator (counter based, so any element can be drawn independently and the
 * output does not depend on the thread count):
 *   word(s, i)  = the (i+1)-th output of SplitMix64 seeded with
 *                 key(s) = mix64(16*seed + stream); SplitMix64 is the
 *                 generator of Steele, Lea and Flood (OOPSLA 2014): state
 *                 advances by 0x9E3779B97F4A7C15 and is passed through mix64.
 *   uniforms    u1 = (word(2j) >> 11 + 1) * 2^-53 in (0, 1],
 *               u2 = (word(2j+1) >> 11) * 2^-53 in [0, 1).
 *   normals     Box-Muller: r = sqrt(-2 ln u1); element 2j is r cos(2 pi u2),
 *               element 2j+1 is r sin(2 pi u2).
 *   value       x = sigma * z, times `outlier_scale` where the uniform drawn
 *               from stream `outlier_stream` at the same index is below
 *               `outlier_p`.
 *   bf16        x is rounded once, directly from binary64 to bf16, to
 *               nearest with ties to even (no intermediate binary32).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SM64_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return mix64(seed * 16u + stream);
}

static inline uint64_t word_at(uint64_t key, uint64_t i)
{
    return mix64(key + (i + 1u) * SM64_GAMMA);
}

static inline double uniform_open0(uint64_t w)  /* (0, 1] */
{
    return (double)((w >> 11) + 1u) * 0x1p-53;
}

static inline double uniform_closed0(uint64_t w)  /* [0, 1) */
{
    return (double)(w >> 11) * 0x1p-53;
}

/*
 * binary64 -> bf16 bits, one rounding to nearest-even.  A bf16 number keeps 8
 * significant bits, a binary64 53: for |x| in bf16's normal range the 45 low
 * significand bits of x are rounded away on its bit pattern (adding half an
 * ulp minus one, plus the kept lsb, carries into the exponent when needed),
 * which leaves a binary64 that binary32 holds exactly.  Below 2^-126 the
 * spacing is the fixed 2^-133, so x * 2^133 is rounded to an integer with the
 * default (nearest-even) mode.  Past the largest finite bf16: infinity.
 */
static inline uint16_t to_bf16_bits(double x)
{
    const double ax = fabs(x);
    double r;
    if (ax < 0x1p-126) {
        r = nearbyint(x * 0x1p133) * 0x1p-133;
    } else {
        uint64_t u;
        memcpy(&u, &x, sizeof u);
        u += 0x00000FFFFFFFFFFFULL + ((u >> 45) & 1u);
        u &= ~0x00001FFFFFFFFFFFULL;
        memcpy(&r, &u, sizeof r);
    }
    float f = fabs(r) >= 0x1p128 ? copysignf(INFINITY, (float)x) : (float)r;
    uint32_t b;
    memcpy(&b, &f, sizeof b);
    return (uint16_t)(b >> 16);
}

struct syn_job {
    uint16_t *out;
    uint64_t begin, end;
    uint64_t key, okey;
    double sigma, outlier_p, outlier_scale;
};

static void fill_range(const struct syn_job *j)
{
    const double two_pi = 6.283185307179586476925286766559;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        uint64_t pair = i >> 1;
        double u1 = uniform_open0(word_at(j->key, 2u * pair));
        double u2 = uniform_closed0(word_at(j->key, 2u * pair + 1u));
        double r = sqrt(-2.0 * log(u1));
        double z = (i & 1u) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
        double x = j->sigma * z;
        if (j->outlier_p > 0.0 &&
            uniform_closed0(word_at(j->okey, i)) < j->outlier_p) {
            x *= j->outlier_scale;
        }
        j->out[i - j->begin] = to_bf16_bits(x);
    }
}

static void *fill_worker(void *arg)
{
    fill_range((const struct syn_job *)arg);
    return NULL;
}

/*
 * Writes elements [offset, offset + count) of the sequence into out[0..count).
 * Returns the number of host threads used.
 */
int synthetic_normal_bf16(uint16_t *out, uint64_t offset, uint64_t count,
                          uint64_t seed, uint64_t stream, double sigma,
                          double outlier_p, double outlier_scale,
                          uint64_t outlier_stream, int threads)
{
    struct syn_job base;
    base.out = out;
    base.begin = offset;
    base.end = offset + count;
    base.key = stream_key(seed, stream);
    base.okey = stream_key(seed, outlier_stream);
    base.sigma = sigma;
    base.outlier_p = outlier_p;
    base.outlier_scale = outlier_scale;
    if (threads < 1) threads = 1;
    if (threads == 1 || count < (uint64_t)threads * 4096u) {
        fill_range(&base);
        return 1;
    }
    pthread_t *tid = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
    int *live = (int *)calloc((size_t)threads, sizeof(int));
    struct syn_job *jobs = (struct syn_job *)calloc((size_t)threads, sizeof *jobs);
    if (!tid || !live || !jobs) {
        free(tid);
        free(live);
        free(jobs);
        fill_range(&base);
        return 1;
    }
    int started = 0;
    for (int t = 0; t < threads; ++t) {
        jobs[t] = base;
        jobs[t].begin = offset + count * (uint64_t)t / (uint64_t)threads;
        jobs[t].end = offset + count * (uint64_t)(t + 1) / (uint64_t)threads;
        jobs[t].out = out + (jobs[t].begin - offset);
        if (pthread_create(&tid[t], NULL, fill_worker, &jobs[t]) == 0) {
            live[t] = 1;
            ++started;
        } else {
            fill_range(&jobs[t]);
        }
    }
    for (int t = 0; t < threads; ++t) {
        if (live[t]) pthread_join(tid[t], NULL);
    }
    free(tid);
    free(live);
    free(jobs);
    return started > 0 ? started : 1;
}

/* The raw SplitMix64 word, exposed so tests can check the generator itself. */
uint64_t synthetic_word(uint64_t seed, uint64_t stream, uint64_t i)
{
    return word_at(stream_key(seed, stream), i);
}

/*
 * Uniform bytes: out[i] = lo + (word i of (seed, stream)) mod span, for
 * elements [offset, offset + count) -- random 4-bit weight codes (two per
 * byte, span 256) and 8-bit scale codes (a range of exponents).  Single
 * threaded: these tensors are a quarter and a 64th of the bf16 weights.
 */
void synthetic_bytes(uint8_t *out, uint64_t offset, uint64_t count, uint64_t seed, uint64_t stream,
                     unsigned lo, unsigned span)
{
    const uint64_t key = stream_key(seed, stream);
    if (span == 0u) span = 1u;
    for (uint64_t i = 0; i < count; ++i) {
        out[i] = (uint8_t)(lo + (unsigned)(word_at(key, offset + i) % (uint64_t)span));
    }
}
