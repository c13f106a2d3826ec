/*
 * Seeded synthetic inputs for frame-aligned block-sparse attention.
 *
 * This file is the ONE piece shared by the fp64 oracle and the CUDA path: it
 * produces input tensors and nothing else.  It holds none of the attention
 * arithmetic (no dot products, norms, softmax or masks).
 *
 * Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014).  Output i of the stream with
 * key K is mix(K + (i+1)*GAMMA), which is exactly the i-th output of the
 * sequential SplitMix64 generator seeded with K, so any element can be drawn
 * independently (and in parallel).  Normals come from the Box-Muller
 * transform (cosine branch) in fp64, then are rounded to fp32 (round to
 * nearest even) and to bf16 (round to nearest even).
 *
 * Streams are keyed by (seed, tag, b, h); every tensor [B,H,L,D] draws one
 * stream per (b, h) and element e = l*D + d uses outputs 2e and 2e+1.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <string.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Key of the stream (seed, tag, b, h). */
uint64_t synth_stream_key(uint64_t seed, uint32_t tag, uint32_t b, uint32_t h) {
    uint64_t k = sm_mix(seed + SM_GAMMA);
    k = sm_mix(k ^ ((uint64_t)tag * 0xD1B54A32D192ED03ULL));
    k = sm_mix(k ^ (((uint64_t)b << 32) | (uint64_t)h));
    return k;
}

/* i-th output (0-based) of the SplitMix64 sequence started from state `key`. */
uint64_t synth_splitmix64_at(uint64_t key, uint64_t i) {
    return sm_mix(key + (i + 1) * SM_GAMMA);
}

static inline double u01_open_closed(uint64_t x) { /* (0, 1] */
    return (double)((x >> 11) + 1) * 0x1.0p-53;
}
static inline double u01_closed_open(uint64_t x) { /* [0, 1) */
    return (double)(x >> 11) * 0x1.0p-53;
}

static inline double normal_at(uint64_t key, uint64_t e) {
    const double two_pi = 6.283185307179586476925286766559;
    double u1 = u01_open_closed(synth_splitmix64_at(key, 2 * e));
    double u2 = u01_closed_open(synth_splitmix64_at(key, 2 * e + 1));
    return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

/* fp32 -> bf16, round to nearest even (inputs are finite). */
static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ---- one (b, h) stream of n values, optionally scaled per row of D ---- */

typedef struct {
    uint64_t key;
    int64_t e0, e1;          /* element range [e0, e1) inside the stream */
    int D;
    const double *row_scale; /* per row of the stream (nullable) */
    uint16_t *out_bf16;      /* indexed by element */
    double *out_f64;         /* indexed by element (nullable) */
    int kind;                /* 0 normal->bf16, 1 normal f64, 2 uniform f64 */
} job_t;

static void run_job(const job_t *j) {
    for (int64_t e = j->e0; e < j->e1; ++e) {
        if (j->kind == 2) {
            j->out_f64[e] = u01_closed_open(synth_splitmix64_at(j->key, (uint64_t)e));
            continue;
        }
        double x = normal_at(j->key, (uint64_t)e);
        if (j->kind == 1) { j->out_f64[e] = x; continue; }
        if (j->row_scale) x *= j->row_scale[e / j->D];
        j->out_bf16[e] = f32_to_bf16_rne((float)x);
    }
}

static void *thread_main(void *arg) { run_job((const job_t *)arg); return NULL; }

static void run_parallel(job_t base, int64_t n, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < 65536 || nthreads == 1) { base.e0 = 0; base.e1 = n; run_job(&base); return; }
    pthread_t th[256];
    job_t jobs[256];
    int64_t chunk = (n + nthreads - 1) / nthreads;
    int ok[256] = {0};
    int used = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].e0 = (int64_t)t * chunk;
        jobs[t].e1 = jobs[t].e0 + chunk < n ? jobs[t].e0 + chunk : n;
        if (jobs[t].e0 >= jobs[t].e1) break;
        used = t + 1;
        if (pthread_create(&th[t], NULL, thread_main, &jobs[t]) == 0) ok[t] = 1;
        else run_job(&jobs[t]);
    }
    for (int t = 0; t < used; ++t)
        if (ok[t]) pthread_join(th[t], NULL);
}

/* A [B,H,L,D] bf16 tensor: stream (seed, tag, b, h) for each (b, h).
 * row_scale (nullable) is a [B,H,L] fp64 multiplier applied before rounding. */
void synth_tensor_bf16(uint64_t seed, uint32_t tag, int32_t B, int32_t H, int64_t L, int32_t D,
                       const double *row_scale, uint16_t *out, int32_t nthreads) {
    for (int32_t b = 0; b < B; ++b)
        for (int32_t h = 0; h < H; ++h) {
            int64_t bh = (int64_t)b * H + h;
            job_t j;
            memset(&j, 0, sizeof j);
            j.key = synth_stream_key(seed, tag, (uint32_t)b, (uint32_t)h);
            j.D = D;
            j.row_scale = row_scale ? row_scale + bh * L : NULL;
            j.out_bf16 = out + bh * L * D;
            j.kind = 0;
            run_parallel(j, L * (int64_t)D, nthreads);
        }
}

/* n values of the (seed, tag, b, h) stream: kind 1 = standard normal, kind 2 = uniform [0,1). */
void synth_stream_f64(uint64_t seed, uint32_t tag, uint32_t b, uint32_t h, int64_t n, int32_t kind,
                      double *out) {
    job_t j;
    memset(&j, 0, sizeof j);
    j.key = synth_stream_key(seed, tag, b, h);
    j.D = 1;
    j.out_f64 = out;
    j.kind = kind == 2 ? 2 : 1;
    run_parallel(j, n, 1);
}
