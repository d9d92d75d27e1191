/*
 * CPU model of the software exponential used on the FMA pipes.
 *
 * TEST INFRASTRUCTURE ONLY (see attn_oracle.c). Shares no code with the CUDA path.
 *
 * Steps, in the order of "FlashAttention-4: Blackwell algorithm-pipeline
 * co-design", section "hybrid exponential" (steps one to three and the boundary
 * paragraph), and "FlashAttention4 精读" section 3.1.3:
 *   1. clamp x >= -127 (below that 2^x underflows fp32);
 *   2. Cody-Waite split x = n + f, n = floor(x), f in [0, 1); n is obtained with
 *      the magic bias C = 1.5 * 2^23 = 12582912 as (x + C) - C where the add
 *      rounds toward minus infinity;
 *   3. 2^f by the cubic p(f) = ((p3 f + p2) f + p1) f + p0 in Horner form, three
 *      fp32 fused multiply-adds, coefficients p0 = 1, p1 = 0.6951, p2 = 0.2276,
 *      p3 = 0.0771 (the four-digit values printed in the hybrid-exponential section);
 *   4. 2^n * q by adding n << 23 to the bit pattern of q (q in [1, 2) has exponent
 *      field 127, so the sum is the exponent field of 2^n q).
 *
 * The round-toward-minus-infinity add of step 2 is modelled exactly without
 * touching the FPU rounding mode: the round-to-nearest sum t = x + C lies on the
 * integer grid (ulp(C) = 1); t - C is exact, and if it exceeds x the nearest
 * rounding went up, so the round-down result is one less.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

static const float P0 = 1.0f, P1 = 0.6951f, P2 = 0.2276f, P3 = 0.0771f;
static const float MAGIC = 12582912.0f; /* 1.5 * 2^23 */

float oracle_floor_magic(float x) {
    volatile float t = x + MAGIC; /* round to nearest */
    float n = t - MAGIC;          /* exact */
    if (n > x) n -= 1.0f;         /* nearest rounded up: the round-down sum is one lower */
    return n;
}

float oracle_exp2_cubic(float f) { return fmaf(fmaf(fmaf(P3, f, P2), f, P1), f, P0); }

float oracle_exp2_poly(float x) {
    if (x != x) return x;
    x = fmaxf(x, -127.0f);
    const float n = oracle_floor_magic(x);
    const float f = x - n;
    const float q = oracle_exp2_cubic(f);
    uint32_t qb;
    memcpy(&qb, &q, 4);
    const int32_t ni = (int32_t)n;
    const uint32_t rb = qb + ((uint32_t)ni << 23);
    float r;
    memcpy(&r, &rb, 4);
    return r;
}

void oracle_exp2_poly_batch(const float* x, float* y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = oracle_exp2_poly(x[i]);
}

/* ---- error sweeps of the cubic against exp2 in double ---- */

typedef struct {
    uint32_t lo, hi;      /* bit-pattern range [lo, hi) of fp32 inputs, or grid indices */
    int grid;             /* 0: bit patterns; 1: f = i / 2^24 */
    double max_rel, sum_rel;
    uint64_t count;
    float argmax;
} sweep_job_t;

static void* sweep_worker(void* p) {
    sweep_job_t* J = (sweep_job_t*)p;
    double mx = 0.0, sum = 0.0;
    float arg = 0.0f;
    for (uint32_t i = J->lo; i < J->hi; ++i) {
        float f;
        if (J->grid) {
            f = (float)i * 0x1.0p-24f;
        } else {
            memcpy(&f, &i, 4);
        }
        const double exact = exp2((double)f);
        const double rel = fabs((double)oracle_exp2_cubic(f) - exact) / exact;
        if (rel > mx) { mx = rel; arg = f; }
        sum += rel;
    }
    J->max_rel = mx;
    J->sum_rel = sum;
    J->count = (uint64_t)(J->hi - J->lo);
    J->argmax = arg;
    return NULL;
}

/*
 * Relative error of the fp32 Horner cubic versus exp2 in double.
 * mode 0: every fp32 value in [0, 1) (bit patterns 0 .. 0x3F7FFFFF);
 * mode 1: the uniform grid f = i / 2^24, i = 0 .. 2^24 - 1.
 */
int oracle_exp2_cubic_sweep(int mode, int n_threads, double* max_rel, double* mean_rel, float* argmax) {
    const uint32_t end = mode == 0 ? 0x3F800000u : (1u << 24);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 64) n_threads = 64;
    sweep_job_t jobs[64];
    pthread_t th[64];
    int ok[64];
    const uint32_t chunk = (end + (uint32_t)n_threads - 1) / (uint32_t)n_threads;
    for (int t = 0; t < n_threads; ++t) {
        uint32_t lo = (uint32_t)t * chunk, hi = lo + chunk;
        if (lo > end) lo = end;
        if (hi > end) hi = end;
        memset(&jobs[t], 0, sizeof jobs[t]);
        jobs[t].lo = lo; jobs[t].hi = hi; jobs[t].grid = mode;
        ok[t] = pthread_create(&th[t], NULL, sweep_worker, &jobs[t]) == 0;
        if (!ok[t]) sweep_worker(&jobs[t]);
    }
    double mx = 0.0, sum = 0.0;
    uint64_t cnt = 0;
    float arg = 0.0f;
    for (int t = 0; t < n_threads; ++t) {
        if (ok[t]) pthread_join(th[t], NULL);
        if (jobs[t].max_rel > mx) { mx = jobs[t].max_rel; arg = jobs[t].argmax; }
        sum += jobs[t].sum_rel;
        cnt += jobs[t].count;
    }
    *max_rel = mx;
    *mean_rel = cnt ? sum / (double)cnt : 0.0;
    *argmax = arg;
    return 0;
}
