/*
 * Seeded synthetic inputs for the attention workloads.
 *
 * This file holds random-number generation only: no attention arithmetic.
 * Both the CUDA path (through the tests and the benchmark) and the CPU oracle
 * consume the bytes it writes, so the two sides always see identical inputs.
 *
 * Generator: splitmix64 used as a counter-based stream. Output number i
 * (0-based) of the stream with seed s is the splitmix64 finaliser applied to
 * s + (i+1) * 0x9E3779B97F4A7C15, which is exactly the i-th value of the
 * sequential splitmix64 generator started from state s. Normals come from the
 * Box-Muller transform on consecutive pairs of outputs, computed in double,
 * multiplied by a caller factor, rounded to fp32 and then to bf16 with
 * round-to-nearest-even.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1u) * SYNTH_GOLDEN;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

uint64_t synth_splitmix64_at(uint64_t seed, uint64_t i) { return splitmix64_at(seed, i); }

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t bits;
    memcpy(&bits, &f, 4);
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu)) return 0x7FC0u; /* NaN */
    uint32_t rounding = 0x7FFFu + ((bits >> 16) & 1u);
    return (uint16_t)((bits + rounding) >> 16);
}

uint16_t synth_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }

/* Box-Muller pair j of the stream: element 2j is r*cos(2*pi*u2), element 2j+1 is r*sin. */
static inline double normal_at(uint64_t seed, int64_t idx) {
    const int64_t j = idx >> 1;
    const uint64_t a = splitmix64_at(seed, (uint64_t)(2 * j));
    const uint64_t b = splitmix64_at(seed, (uint64_t)(2 * j + 1));
    const double u1 = (double)((a >> 11) + 1u) * 0x1.0p-53; /* (0, 1] */
    const double u2 = (double)(b >> 11) * 0x1.0p-53;        /* [0, 1) */
    const double r = sqrt(-2.0 * log(u1));
    const double t = 6.283185307179586476925286766559 * u2;
    return (idx & 1) ? r * sin(t) : r * cos(t);
}

typedef struct {
    uint16_t* out;
    int64_t begin, end;
    uint64_t seed;
    double mult;
} normal_job_t;

static void* normal_worker(void* p) {
    normal_job_t* job = (normal_job_t*)p;
    for (int64_t i = job->begin; i < job->end; ++i) {
        const float f = (float)(normal_at(job->seed, i) * job->mult);
        job->out[i] = f32_to_bf16_rne(f);
    }
    return NULL;
}

/* Fill out[0..n) with bf16 bit patterns of mult * N(0,1), element i from stream index i. */
int synth_normal_bf16(uint16_t* out, int64_t n, uint64_t seed, double mult, int n_threads) {
    if (!out || n < 0) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if (n < 65536) n_threads = 1;
    pthread_t th[256];
    normal_job_t jobs[256];
    const int64_t chunk = ((n + n_threads - 1) / n_threads + 1) & ~(int64_t)1;
    int started = 0;
    for (int t = 0; t < n_threads; ++t) {
        int64_t b = (int64_t)t * chunk, e = b + chunk;
        if (b > n) b = n;
        if (e > n) e = n;
        jobs[t] = (normal_job_t){out, b, e, seed, mult};
        if (n_threads == 1) {
            normal_worker(&jobs[t]);
        } else if (pthread_create(&th[t], NULL, normal_worker, &jobs[t]) == 0) {
            ++started;
        } else {
            normal_worker(&jobs[t]); /* run inline if a thread cannot be made */
            th[t] = 0;
            jobs[t].out = NULL;
        }
    }
    if (n_threads > 1)
        for (int t = 0; t < n_threads; ++t)
            if (jobs[t].out) pthread_join(th[t], NULL);
    (void)started;
    return 0;
}

/* out[i] = lo + (stream value i mod (hi - lo + 1)), inclusive range [lo, hi]. */
int synth_uniform_int(int32_t* out, int64_t n, uint64_t seed, int32_t lo, int32_t hi) {
    if (!out || n < 0 || hi < lo) return -1;
    const uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo + 1);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)((int64_t)lo + (int64_t)(splitmix64_at(seed, (uint64_t)i) % span));
    return 0;
}

/* Seeded Fisher-Yates shuffle of 0..n-1; the swap partner at step i uses stream value (n-1-i). */
int synth_permutation(int32_t* out, int64_t n, uint64_t seed) {
    if (!out || n < 0) return -1;
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i > 0; --i) {
        const int64_t j = (int64_t)(splitmix64_at(seed, (uint64_t)(n - 1 - i)) % (uint64_t)(i + 1));
        const int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
    return 0;
}
