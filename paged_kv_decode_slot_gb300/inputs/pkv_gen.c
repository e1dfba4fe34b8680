/*
 * pkv_gen.c - seeded synthetic inputs for the paged decode-attention workloads.
 *
 * This file holds random-number generation only: it draws the numbers that
 * fill a workload (queries, cache pools, new tokens, context lengths, block
 * permutations) and rounds them to bf16.  It contains none of the attention
 * arithmetic; the CUDA library and the float64 oracle both receive its output
 * as plain input bytes and share nothing else.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used as a counter-based generator: draw i
 * of stream (seed, stream) is the SplitMix64 output for state
 * key + (i + 1) * golden_gamma, where key is itself a SplitMix64 output of
 * (seed, stream).  Any element can therefore be produced independently, so
 * the result does not depend on the thread count.
 *
 * Normals: Box-Muller (Box and Muller, 1958), z = sqrt(-2 ln u1) cos(2 pi u2),
 * with u1, u2 the draws 2i and 2i+1 mapped to (0, 1].  Element i uses one
 * pair.  float -> bf16 is round-to-nearest-even on the bit pattern.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>
#include <unistd.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ull

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static uint64_t stream_key(uint64_t seed, uint64_t stream)
{
    return mix64(mix64(seed + GOLDEN_GAMMA) ^ (stream * 0xD1B54A32D192ED03ull + 1u));
}

static uint64_t draw_u64(uint64_t key, uint64_t i)
{
    return mix64(key + (i + 1u) * GOLDEN_GAMMA);
}

/* uniform in (0, 1]: 53 random bits, shifted away from zero */
static double draw_unit(uint64_t key, uint64_t i)
{
    return (double)((draw_u64(key, i) >> 11) + 1u) * (1.0 / 9007199254740992.0);
}

static double draw_normal(uint64_t key, uint64_t i)
{
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = draw_unit(key, 2u * i);
    double u2 = draw_unit(key, 2u * i + 1u);
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static uint16_t float_to_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)0x7FC0u; /* quiet NaN */
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

typedef struct {
    uint64_t key, offset, begin, end;
    float mult;
    uint16_t *out;
} normal_job;

static void *normal_worker(void *arg)
{
    normal_job *j = (normal_job *)arg;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        float v = (float)draw_normal(j->key, j->offset + i) * j->mult;
        j->out[i] = float_to_bf16_rne(v);
    }
    return 0;
}

static int pick_threads(int nthreads, uint64_t n)
{
    if (nthreads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = c > 0 ? (int)c : 1;
    }
    if (nthreads > 256) nthreads = 256;
    if ((uint64_t)nthreads > n / 65536u + 1u) nthreads = (int)(n / 65536u + 1u);
    return nthreads < 1 ? 1 : nthreads;
}

/*
 * out[i] = bf16(mult * N(0,1) draw number (offset + i) of stream (seed, stream)),
 * for i in [0, n).  mult is applied in float before rounding.
 */
int pkvgen_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, uint64_t n,
                       float mult, uint16_t *out, int nthreads)
{
    if (!out && n) return -1;
    uint64_t key = stream_key(seed, stream);
    int nt = pick_threads(nthreads, n);
    normal_job jobs[256];
    pthread_t tids[256];
    for (int t = 0; t < nt; ++t) {
        jobs[t].key = key;
        jobs[t].offset = offset;
        jobs[t].begin = n * (uint64_t)t / (uint64_t)nt;
        jobs[t].end = n * (uint64_t)(t + 1) / (uint64_t)nt;
        jobs[t].mult = mult;
        jobs[t].out = out;
    }
    int started = 0;
    for (int t = 1; t < nt; ++t) {
        if (pthread_create(&tids[t], 0, normal_worker, &jobs[t]) != 0) break;
        started = t;
    }
    normal_worker(&jobs[0]);
    for (int t = started + 1; t < nt; ++t) normal_worker(&jobs[t]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], 0);
    return 0;
}

/* out[i] = lo + floor(u * (hi - lo + 1)), u uniform in [0, 1): integers in [lo, hi]. */
int pkvgen_uniform_int(uint64_t seed, uint64_t stream, uint64_t n, int64_t lo, int64_t hi,
                       int64_t *out)
{
    if (hi < lo || (!out && n)) return -1;
    uint64_t key = stream_key(seed, stream);
    uint64_t span = (uint64_t)(hi - lo) + 1u;
    for (uint64_t i = 0; i < n; ++i) {
        double u = (double)(draw_u64(key, i) >> 11) * (1.0 / 9007199254740992.0);
        uint64_t k = (uint64_t)(u * (double)span);
        if (k >= span) k = span - 1u;
        out[i] = lo + (int64_t)k;
    }
    return 0;
}

/* out = a uniformly random permutation of 0..n-1 (Fisher-Yates, Durstenfeld's form). */
int pkvgen_permutation(uint64_t seed, uint64_t stream, int64_t n, int64_t *out)
{
    if (n < 0 || (!out && n)) return -1;
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = i;
    for (int64_t i = n - 1; i > 0; --i) {
        double u = (double)(draw_u64(key, (uint64_t)i) >> 11) * (1.0 / 9007199254740992.0);
        int64_t j = (int64_t)(u * (double)(i + 1));
        if (j > i) j = i;
        int64_t tmp = out[i];
        out[i] = out[j];
        out[j] = tmp;
    }
    return 0;
}
