/*
 * Seeded synthetic-input generator shared by the CPU oracle and the CUDA path.
 *
 * This file holds no arithmetic of the DiT block itself: it only turns
 * (seed, stream, index) into reproducible Gaussian samples, rounded to the
 * storage type the GPU receives.  Both sides of every parity test draw their
 * inputs from here, so neither depends on the other for data.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used in counter mode: sample i of a stream
 * is the SplitMix64 finaliser applied to key + (i+1)*golden, where the key is
 * derived from (seed, stream) by the same finaliser.  Pairs of 53-bit
 * uniforms become standard normals by the Box-Muller transform (Box & Muller,
 * 1958), evaluated in double precision.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stddef.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed + GOLDEN) ^ (stream * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL));
}

static inline uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1) * GOLDEN); }

/* standard normal number `j` of the stream (two per Box-Muller pair) */
static inline double normal_at(uint64_t key, uint64_t j) {
    uint64_t pair = j >> 1;
    uint64_t a = draw(key, 2 * pair), b = draw(key, 2 * pair + 1);
    double u1 = ((double)(a >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0, 1] */
    double u2 = (double)(b >> 11) * (1.0 / 9007199254740992.0);         /* [0, 1) */
    double r = sqrt(-2.0 * log(u1));
    double th = 6.283185307179586476925 * u2;
    return (j & 1) ? r * sin(th) : r * cos(th);
}

/* float -> bfloat16 bits, round to nearest even (NaN kept quiet) */
static inline uint16_t f32_to_bf16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

typedef struct {
    uint64_t key, begin, end;
    double mean, std;
    int kind; /* 0 = bf16 bits, 1 = float32, 2 = float64 */
    void *out;
} job_t;

static void *worker(void *p) {
    job_t *j = (job_t *)p;
    for (uint64_t i = j->begin; i < j->end; ++i) {
        double v = j->mean + j->std * normal_at(j->key, i);
        if (j->kind == 0) ((uint16_t *)j->out)[i] = f32_to_bf16_bits((float)v);
        else if (j->kind == 1) ((float *)j->out)[i] = (float)v;
        else ((double *)j->out)[i] = v;
    }
    return NULL;
}

static void run(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, int kind, void *out,
                int threads) {
    if (threads < 1) threads = 1;
    if (threads > 256) threads = 256;
    if (n < (1u << 16)) threads = 1;
    pthread_t tid[256];
    job_t jobs[256];
    uint64_t key = stream_key(seed, stream);
    uint64_t chunk = (n + threads - 1) / threads;
    chunk = (chunk + 1) & ~1ULL; /* keep Box-Muller pairs inside one job */
    int launched = 0;
    for (int t = 0; t < threads; ++t) {
        uint64_t b = (uint64_t)t * chunk, e = b + chunk;
        if (b >= n) break;
        if (e > n) e = n;
        jobs[t] = (job_t){key, b, e, mean, std, kind, out};
        if (threads == 1 || pthread_create(&tid[t], NULL, worker, &jobs[t]) != 0) {
            worker(&jobs[t]);
            tid[t] = 0;
        }
        launched = t + 1;
    }
    for (int t = 0; t < launched; ++t)
        if (tid[t]) pthread_join(tid[t], NULL);
}

/* n samples of N(mean, std^2) from stream `stream` of `seed`, as bf16 bits (RN-even from float) */
void h3s_normal_bf16(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, uint16_t *out,
                     int threads) {
    run(seed, stream, n, mean, std, 0, out, threads);
}

void h3s_normal_f32(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, float *out,
                    int threads) {
    run(seed, stream, n, mean, std, 1, out, threads);
}

void h3s_normal_f64(uint64_t seed, uint64_t stream, uint64_t n, double mean, double std, double *out,
                    int threads) {
    run(seed, stream, n, mean, std, 2, out, threads);
}

/* raw 64-bit draws, exposed so tests can check the generator against its definition */
void h3s_raw_u64(uint64_t seed, uint64_t stream, uint64_t n, uint64_t *out) {
    uint64_t key = stream_key(seed, stream);
    for (uint64_t i = 0; i < n; ++i) out[i] = draw(key, i);
}
