/*
 * synth.c - seeded synthetic inputs shared by the parity tests, the oracle
 * runs and the benchmark.
 *
 * This file holds none of the arithmetic of the kernels or of the oracle: it
 * only draws numbers.  Every value is a pure function of (seed, tag, element
 * index), so any subset of rows can be regenerated on its own and the bulk
 * generation can be split over threads without changing a single bit.
 *
 *   - SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): output i of a stream is mix(s0 + (i+1)*gamma).
 *   - uniform in (0, 1]: the top 53 bits plus one, times 2^-53.
 *   - normals by the Box-Muller transform (Box and Muller, 1958): the uniform
 *     pair (2j, 2j+1) gives normals 2j (cosine branch) and 2j+1 (sine branch).
 *   - fp32 -> bf16 by round-to-nearest-even on the bit pattern.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define SM_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t sm_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* Start state of stream `tag` under `seed`. */
static inline uint64_t sm_stream(uint64_t seed, uint64_t tag) {
    return sm_mix(seed ^ sm_mix(tag + SM_GAMMA));
}

static inline uint64_t sm_at(uint64_t s0, uint64_t i) {
    return sm_mix(s0 + (i + 1ULL) * SM_GAMMA);
}

/* Raw 64-bit word i of stream (seed, tag). */
uint64_t synth_u64(uint64_t seed, uint64_t tag, uint64_t i) {
    return sm_at(sm_stream(seed, tag), i);
}

static inline double sm_unit(uint64_t z) { /* (0, 1] */
    return (double)((z >> 11) + 1ULL) * (1.0 / 9007199254740992.0);
}

static inline double sm_normal(uint64_t s0, uint64_t i) {
    const double two_pi = 6.283185307179586476925286766559;
    uint64_t j = i >> 1;
    double u1 = sm_unit(sm_at(s0, 2 * j));
    double u2 = sm_unit(sm_at(s0, 2 * j + 1));
    double r = sqrt(-2.0 * log(u1));
    return (i & 1) ? r * sin(two_pi * u2) : r * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* ---- bulk generation, split over threads ------------------------------ */

typedef struct {
    uint64_t s0;
    int64_t row0, rows, cols;     /* rows [row0, row0+rows) of a [*, cols] matrix */
    double mean, std;
    const float* row_scale;       /* optional, indexed by local row */
    void* out;
    int is_bf16;
    int64_t r_begin, r_end;       /* this worker's local rows */
} job_t;

static void* run_job(void* p) {
    job_t* j = (job_t*)p;
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        double rs = j->row_scale ? (double)j->row_scale[r] : 1.0;
        uint64_t base = (uint64_t)(j->row0 + r) * (uint64_t)j->cols;
        for (int64_t c = 0; c < j->cols; ++c) {
            double v = (j->mean + j->std * sm_normal(j->s0, base + (uint64_t)c)) * rs;
            float f = (float)v;
            if (j->is_bf16)
                ((uint16_t*)j->out)[r * j->cols + c] = f32_to_bf16_rne(f);
            else
                ((float*)j->out)[r * j->cols + c] = f;
        }
    }
    return NULL;
}

static void run_rows(job_t proto, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (proto.rows < (int64_t)nthreads) nthreads = proto.rows > 0 ? (int)proto.rows : 1;
    pthread_t th[256];
    int spawned[256];
    job_t jobs[256];
    int64_t per = (proto.rows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].r_begin = (int64_t)t * per < proto.rows ? (int64_t)t * per : proto.rows;
        jobs[t].r_end = jobs[t].r_begin + per < proto.rows ? jobs[t].r_begin + per : proto.rows;
        spawned[t] = 0;
        if (t > 0 && jobs[t].r_begin < jobs[t].r_end) {
            if (pthread_create(&th[t], NULL, run_job, &jobs[t]) == 0) spawned[t] = 1;
            else run_job(&jobs[t]); /* could not spawn: do it on this thread */
        }
    }
    run_job(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (spawned[t]) pthread_join(th[t], NULL);
}

/*
 * Rows [row0, row0+rows) of a [*, cols] matrix whose element (r, c) is
 * mean + std * normal(r*cols + c), times row_scale[r - row0] when given,
 * rounded to fp32 and then to bf16.  `out` is [rows, cols], contiguous.
 */
void synth_normal_bf16(uint64_t seed, uint64_t tag, int64_t row0, int64_t rows, int64_t cols,
                       double mean, double std, const float* row_scale, uint16_t* out, int nthreads) {
    job_t j;
    memset(&j, 0, sizeof j);
    j.s0 = sm_stream(seed, tag);
    j.row0 = row0; j.rows = rows; j.cols = cols;
    j.mean = mean; j.std = std; j.row_scale = row_scale;
    j.out = out; j.is_bf16 = 1;
    run_rows(j, nthreads);
}

/* Same draw, rounded to fp32 only. */
void synth_normal_f32(uint64_t seed, uint64_t tag, int64_t row0, int64_t rows, int64_t cols,
                      double mean, double std, const float* row_scale, float* out, int nthreads) {
    job_t j;
    memset(&j, 0, sizeof j);
    j.s0 = sm_stream(seed, tag);
    j.row0 = row0; j.rows = rows; j.cols = cols;
    j.mean = mean; j.std = std; j.row_scale = row_scale;
    j.out = out; j.is_bf16 = 0;
    run_rows(j, nthreads);
}

/* Uniform integers in [lo, hi] (Lemire's multiply-high map; bias < 2^-40 here). */
void synth_uniform_int(uint64_t seed, uint64_t tag, int64_t n, int64_t lo, int64_t hi, int64_t* out) {
    uint64_t s0 = sm_stream(seed, tag);
    uint64_t span = (uint64_t)(hi - lo) + 1ULL;
    for (int64_t i = 0; i < n; ++i) {
        unsigned __int128 m = (unsigned __int128)sm_at(s0, (uint64_t)i) * span;
        out[i] = lo + (int64_t)(uint64_t)(m >> 64);
    }
}

/* A seeded permutation of 0..n-1 (Fisher-Yates, last position first). */
void synth_permutation(uint64_t seed, uint64_t tag, int64_t n, int64_t* out) {
    uint64_t s0 = sm_stream(seed, tag);
    for (int64_t i = 0; i < n; ++i) out[i] = i;
    for (int64_t i = n - 1; i > 0; --i) {
        unsigned __int128 m = (unsigned __int128)sm_at(s0, (uint64_t)(n - 1 - i)) * (uint64_t)(i + 1);
        int64_t k = (int64_t)(uint64_t)(m >> 64);
        int64_t t = out[i]; out[i] = out[k]; out[k] = t;
    }
}

/* Fill n bf16 slots with one bit pattern (NaN tails, 0xFFFF canaries). */
void synth_fill_u16(uint16_t* out, int64_t n, uint16_t bits) {
    for (int64_t i = 0; i < n; ++i) out[i] = bits;
}
