/*
 * Seeded N(0,1) float32 samples — the same generator as seeded_inputs/__init__.py,
 * in C so that multi-gigabyte inputs take seconds. Holds no attention arithmetic.
 *
 * SplitMix64 (Steele, Lea and Flood, OOPSLA 2014): output n of a stream with state s0 is
 * mix64(s0 + (n + 1) * 0x9E3779B97F4A7C15). Uniforms on (0, 1] take the top 53 bits.
 * Box-Muller in double turns counters (2i, 2i+1) into elements 2i (cosine branch) and
 * 2i+1 (sine branch); the double is rounded to float32 by the C conversion (nearest even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

static uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double uniform01(uint64_t s0, uint64_t n) {
    const uint64_t x = mix64(s0 + (n + 1) * 0x9E3779B97F4A7C15ull);
    return ((double)(x >> 11) + 1.0) * 0x1.0p-53;
}

typedef struct {
    uint64_t s0;
    int64_t count, lo, hi; /* pair range [lo, hi) */
    float* out;
} gen_job;

static void* gen_worker(void* arg) {
    const gen_job* j = (const gen_job*)arg;
    const double two_pi = 6.283185307179586476925286766559;
    for (int64_t i = j->lo; i < j->hi; ++i) {
        const double u1 = uniform01(j->s0, (uint64_t)(2 * i));
        const double u2 = uniform01(j->s0, (uint64_t)(2 * i + 1));
        const double r = sqrt(-2.0 * log(u1));
        const double th = two_pi * u2;
        j->out[2 * i] = (float)(r * cos(th));
        if (2 * i + 1 < j->count) j->out[2 * i + 1] = (float)(r * sin(th));
    }
    return NULL;
}

/* count samples of stream `stream` under `seed` into out; returns 0 or -1. */
int si_normal_f32(uint64_t seed, uint64_t stream, int64_t count, float* out, int nthreads) {
    if (count < 0 || (!out && count > 0) || nthreads < 1) return -1;
    const uint64_t s0 = mix64(seed * 65536ull + stream);
    const int64_t pairs = (count + 1) / 2;
    if (nthreads > 64) nthreads = 64;
    if ((int64_t)nthreads > pairs) nthreads = pairs > 0 ? (int)pairs : 1;
    gen_job jobs[64];
    pthread_t th[64];
    int started[64] = {0};
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].s0 = s0;
        jobs[t].count = count;
        jobs[t].lo = pairs * t / nthreads;
        jobs[t].hi = pairs * (t + 1) / nthreads;
        jobs[t].out = out;
        if (t > 0) started[t] = pthread_create(&th[t], NULL, gen_worker, &jobs[t]) == 0;
        if (t > 0 && !started[t]) gen_worker(&jobs[t]);
    }
    if (nthreads > 0) gen_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (started[t]) pthread_join(th[t], NULL);
    return 0;
}
