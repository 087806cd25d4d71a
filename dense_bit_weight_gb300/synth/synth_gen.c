/*
 * synth_gen.c -- seeded synthetic operands (random draws and their encoding
 * as bf16 bits / packed words).  Holds none of the GEMM's arithmetic.
 *
 * Generator: splitmix64 (Steele, Lea, Flood, OOPSLA 2014) used counter-style.
 * Sequence (seed, stream) has key = mix(seed*G + stream*H + 1) and draw i is
 * mix(key + (i+1)*G), G = 0x9E3779B97F4A7C15, H = 0xD1B54A32D192ED03, where
 * mix is the splitmix64 finaliser.  Normal number e uses draws 2*(e/2) and
 * 2*(e/2)+1 through Box-Muller (Box & Muller 1958): u1 in (0,1] from the
 * first, u2 in [0,1) from the second, r = sqrt(-2 ln u1), element 2j gets
 * r*cos(2 pi u2) and element 2j+1 gets r*sin(2 pi u2).
 * Values are rounded to bf16 through fp32, round-to-nearest-even each step.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define G_GOLD 0x9E3779B97F4A7C15ULL
#define H_KEY 0xD1B54A32D192ED03ULL

static uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static uint64_t key_of(uint64_t seed, uint64_t stream)
{
    return mix64(seed * G_GOLD + stream * H_KEY + 1ULL);
}

static uint64_t draw(uint64_t key, uint64_t i) { return mix64(key + (i + 1ULL) * G_GOLD); }

static uint16_t f64_to_bf16_via_f32(double x)
{
    float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t bias = ((u >> 16) & 1u) + 0x7FFFu;
    return (uint16_t)((u + bias) >> 16);
}

static double normal_at(uint64_t key, uint64_t e)
{
    uint64_t j = e / 2;
    uint64_t d1 = draw(key, 2 * j), d2 = draw(key, 2 * j + 1);
    double u1 = ((double)(d1 >> 11) + 1.0) * 0x1.0p-53;
    double u2 = (double)(d2 >> 11) * 0x1.0p-53;
    double r = sqrt(-2.0 * log(u1));
    double t = 2.0 * 3.14159265358979323846 * u2;
    return (e & 1) ? r * sin(t) : r * cos(t);
}

enum { K_BF16_NORMAL, K_BF16_UNIFORM, K_INT_UNIFORM, K_U32 };

typedef struct {
    int kind;
    uint64_t key, start, begin, end;
    double a, b;       /* std | lo,hi */
    int64_t ilo, ispan;
    void *out;
} job_t;

static void *worker(void *p)
{
    job_t *j = (job_t *)p;
    for (uint64_t e = j->begin; e < j->end; ++e) {
        uint64_t g = j->start + e;
        switch (j->kind) {
        case K_BF16_NORMAL:
            ((uint16_t *)j->out)[e] = f64_to_bf16_via_f32(normal_at(j->key, g) * j->a);
            break;
        case K_BF16_UNIFORM: {
            double u = (double)(draw(j->key, g) >> 11) * 0x1.0p-53;
            ((uint16_t *)j->out)[e] = f64_to_bf16_via_f32(j->a + (j->b - j->a) * u);
            break;
        }
        case K_INT_UNIFORM: {
            uint64_t hi32 = draw(j->key, g) >> 32;
            ((int64_t *)j->out)[e] = j->ilo + (int64_t)((hi32 * (uint64_t)j->ispan) >> 32);
            break;
        }
        case K_U32:
            ((uint32_t *)j->out)[e] = (uint32_t)(draw(j->key, g) >> 32);
            break;
        }
    }
    return NULL;
}

static void run(job_t proto, uint64_t count)
{
    long nt = sysconf(_SC_NPROCESSORS_ONLN);
    if (nt < 1) nt = 1;
    if (nt > 64) nt = 64;
    if (count < (1u << 16)) nt = 1;
    pthread_t th[64];
    job_t jobs[64];
    for (long t = 0; t < nt; ++t) {
        jobs[t] = proto;
        jobs[t].begin = count * (uint64_t)t / (uint64_t)nt;
        jobs[t].end = count * (uint64_t)(t + 1) / (uint64_t)nt;
        if (pthread_create(&th[t], NULL, worker, &jobs[t]) != 0) {
            worker(&jobs[t]);
            th[t] = 0;
        }
    }
    for (long t = 0; t < nt; ++t)
        if (th[t]) pthread_join(th[t], NULL);
}

void synth_bf16_normal(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                       double std_dev, uint16_t *out)
{
    job_t j = {K_BF16_NORMAL, key_of(seed, stream), start, 0, 0, std_dev, 0, 0, 0, out};
    run(j, count);
}

void synth_bf16_uniform(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                        double lo, double hi, uint16_t *out)
{
    job_t j = {K_BF16_UNIFORM, key_of(seed, stream), start, 0, 0, lo, hi, 0, 0, out};
    run(j, count);
}

void synth_int_uniform(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                       int64_t lo, int64_t hi, int64_t *out)
{
    job_t j = {K_INT_UNIFORM, key_of(seed, stream), start, 0, 0, 0, 0, lo, hi - lo + 1, out};
    run(j, count);
}

void synth_u32(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count, uint32_t *out)
{
    job_t j = {K_U32, key_of(seed, stream), start, 0, 0, 0, 0, 0, 0, out};
    run(j, count);
}

void synth_normal_f64(uint64_t seed, uint64_t stream, uint64_t start, uint64_t count,
                      double *out)
{
    uint64_t key = key_of(seed, stream);
    for (uint64_t e = 0; e < count; ++e) out[e] = normal_at(key, start + e);
}
