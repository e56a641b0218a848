/*
 * Seeded synthetic tensors for tests and benchmarks.
 *
 * This module only draws numbers. It holds none of the arithmetic of the
 * sharding, reduction or tensor-parallel MLP it feeds, and both the CUDA
 * library and the CPU oracle receive the very same bytes from it.
 *
 * Counter-based draws: value i of a stream depends only on (seed, i), so the
 * result does not depend on how the work is split across threads.
 *   - splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014) turns (seed, counter) into 64 random bits;
 *   - the top 53 bits give u in [0, 1);
 *   - normals use the Box-Muller transform on the pair of uniforms drawn at
 *     counters 2j and 2j+1: r = sqrt(-2 ln(1 - u0)), t = 2 pi u1,
 *     element 2j = r cos t, element 2j+1 = r sin t (scaled by std);
 *   - uniforms on [lo, hi) are lo + (hi - lo) u.
 * Values are formed in double, cast to float (round to nearest even) and,
 * for bf16, rounded from that float to bf16 (nearest even).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static uint64_t mix64(uint64_t seed, uint64_t counter)
{
    uint64_t z = seed + (counter + 1u) * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

static double unit53(uint64_t bits) { return (double)(bits >> 11) * (1.0 / 9007199254740992.0); }

static uint16_t f32_to_bf16_rne(float f)
{
    uint32_t b;
    memcpy(&b, &f, 4);
    if ((b & 0x7F800000u) == 0x7F800000u && (b & 0x007FFFFFu)) return (uint16_t)((b >> 16) | 0x0040u);
    b += 0x7FFFu + ((b >> 16) & 1u);
    return (uint16_t)(b >> 16);
}

enum { SYN_NORMAL = 0, SYN_UNIFORM = 1 };
enum { SYN_F32 = 0, SYN_BF16 = 1, SYN_F64 = 2 };

typedef struct {
    int kind, dtype;
    uint64_t seed;
    double a, b; /* normal: mean, std; uniform: lo, hi */
    int64_t begin, end; /* element range handled by this worker */
    void* out;
} job_t;

static void put(const job_t* j, int64_t i, double v)
{
    if (j->dtype == SYN_F64) ((double*)j->out)[i] = v;
    else if (j->dtype == SYN_F32) ((float*)j->out)[i] = (float)v;
    else ((uint16_t*)j->out)[i] = f32_to_bf16_rne((float)v);
}

static void* run(void* arg)
{
    const job_t* j = (const job_t*)arg;
    if (j->kind == SYN_UNIFORM) {
        for (int64_t i = j->begin; i < j->end; ++i)
            put(j, i, j->a + (j->b - j->a) * unit53(mix64(j->seed, (uint64_t)i)));
    } else {
        const double two_pi = 6.283185307179586476925286766559;
        for (int64_t i = j->begin; i < j->end; ++i) {
            int64_t pair = i >> 1;
            double u0 = unit53(mix64(j->seed, (uint64_t)(2 * pair)));
            double u1 = unit53(mix64(j->seed, (uint64_t)(2 * pair + 1)));
            double r = sqrt(-2.0 * log(1.0 - u0));
            double t = two_pi * u1;
            double z = (i & 1) ? r * sin(t) : r * cos(t);
            put(j, i, j->a + j->b * z);
        }
    }
    return 0;
}

/* Fill out[0..n) with draws of the given kind; returns 0 on success. */
int synth_fill(int kind, int dtype, uint64_t seed, double a, double b, int64_t n, void* out, int nthreads)
{
    if (n < 0 || (n > 0 && !out) || kind < 0 || kind > 1 || dtype < 0 || dtype > 2) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 64) nthreads = 64;
    if (n < (int64_t)1 << 16) nthreads = 1;
    pthread_t th[64];
    job_t jobs[64];
    int64_t per = ((n + nthreads - 1) / nthreads + 1) & ~(int64_t)1;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t].kind = kind;
        jobs[t].dtype = dtype;
        jobs[t].seed = seed;
        jobs[t].a = a;
        jobs[t].b = b;
        jobs[t].begin = (int64_t)t * per < n ? (int64_t)t * per : n;
        jobs[t].end = (int64_t)(t + 1) * per < n ? (int64_t)(t + 1) * per : n;
        jobs[t].out = out;
    }
    for (int t = 1; t < nthreads; ++t) {
        if (jobs[t].begin >= jobs[t].end) break;
        if (pthread_create(&th[t], 0, run, &jobs[t]) != 0) break;
        started = t;
    }
    run(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(th[t], 0);
    for (int t = started + 1; t < nthreads; ++t) /* workers that could not start */
        if (jobs[t].begin < jobs[t].end) run(&jobs[t]);
    return 0;
}
