/*
 * Seeded synthetic inputs shared by the oracle, the tests and the benchmark.
 *
 * This file holds NO arithmetic of the MoE method: only a counter-based random
 * generator and the value distributions the workloads call for (uniform bytes,
 * uniform small integers, normals rounded to fp32 or bf16, a random
 * permutation).  Neither the oracle nor the CUDA library includes it; both
 * only consume the buffers it fills.
 *
 * Generator: SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014), used in counter mode: value i of a stream
 * with key K is mix(K + (i + 1) * GAMMA), where mix is SplitMix64's output
 * finaliser.  Every value depends only on (key, i), so any slice of any tensor
 * can be regenerated on its own and the fill parallelises trivially.
 *
 * Normals: Box-Muller in double precision, then rounded to nearest-even fp32
 * (C cast) or bf16 (bit rounding below).
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#define K3S_GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t k3s_mix(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

static inline uint64_t k3s_at(uint64_t key, uint64_t i)
{
    return k3s_mix(key + (i + 1) * K3S_GAMMA);
}

/* Key of the stream for tensor `tag` under base seed `base`. */
uint64_t k3s_key(uint64_t base, uint64_t tag)
{
    return k3s_mix(base ^ k3s_mix(tag + K3S_GAMMA));
}

/* Raw 64-bit value i of stream `key` (exported for tests of the generator). */
uint64_t k3s_u64(uint64_t key, uint64_t i) { return k3s_at(key, i); }

/* n uniform bytes: byte j is byte (j % 8) of value j / 8. */
void k3s_bytes(uint8_t *out, size_t n, uint64_t key)
{
    const size_t nw = n / 8;
#pragma omp parallel for schedule(static)
    for (long long w = 0; w < (long long)nw; w++) {
        uint64_t v = k3s_at(key, (uint64_t)w);
        for (int b = 0; b < 8; b++) out[(size_t)w * 8 + b] = (uint8_t)(v >> (8 * b));
    }
    if (n % 8) {
        uint64_t v = k3s_at(key, (uint64_t)nw);
        for (size_t j = nw * 8; j < n; j++) out[j] = (uint8_t)(v >> (8 * (j - nw * 8)));
    }
}

/* n integers uniform in [lo, hi] (inclusive), one stream value each, mapped by
 * the high 64 bits of a 64x64 product (Lemire's multiply-shift; the bias is
 * below 2^-59 for ranges this small). */
void k3s_uniform_u8(uint8_t *out, size_t n, uint64_t key, int lo, int hi)
{
    const uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < (long long)n; j++) {
        uint64_t v = k3s_at(key, (uint64_t)j);
        uint64_t hi64 = (uint64_t)(((unsigned __int128)v * span) >> 64);
        out[j] = (uint8_t)(lo + (int)hi64);
    }
}

static inline double k3s_unit_open(uint64_t v)   /* (0, 1] */
{
    return ((double)(v >> 11) + 1.0) * (1.0 / 9007199254740992.0);
}
static inline double k3s_unit(uint64_t v)        /* [0, 1) */
{
    return (double)(v >> 11) * (1.0 / 9007199254740992.0);
}

/* Normal j uses stream values 2*(j/2) and 2*(j/2)+1; even j takes the cosine
 * branch, odd j the sine branch. */
static inline double k3s_normal_at(uint64_t key, uint64_t j)
{
    const uint64_t p = j / 2;
    const double u1 = k3s_unit_open(k3s_at(key, 2 * p));
    const double u2 = k3s_unit(k3s_at(key, 2 * p + 1));
    const double r = sqrt(-2.0 * log(u1));
    const double t = 6.283185307179586476925286766559 * u2;
    return (j & 1) ? r * sin(t) : r * cos(t);
}

void k3s_normal_f64(double *out, size_t n, uint64_t key, double mean, double std)
{
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < (long long)n; j++)
        out[j] = mean + std * k3s_normal_at(key, (uint64_t)j);
}

void k3s_normal_f32(float *out, size_t n, uint64_t key, double mean, double std)
{
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < (long long)n; j++)
        out[j] = (float)(mean + std * k3s_normal_at(key, (uint64_t)j));
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t k3s_bf16_rne(float f)
{
    union { float f; uint32_t u; } c;
    c.f = f;
    uint32_t u = c.u;
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* Normals rounded first to fp32, then to bf16 (both round to nearest even). */
void k3s_normal_bf16(uint16_t *out, size_t n, uint64_t key, double mean, double std)
{
#pragma omp parallel for schedule(static)
    for (long long j = 0; j < (long long)n; j++)
        out[j] = k3s_bf16_rne((float)(mean + std * k3s_normal_at(key, (uint64_t)j)));
}

/* Uniform random permutation of 0..n-1 (Fisher-Yates driven by the stream). */
void k3s_permutation(int32_t *out, int n, uint64_t key)
{
    for (int i = 0; i < n; i++) out[i] = i;
    for (int i = n - 1; i > 0; i--) {
        uint64_t v = k3s_at(key, (uint64_t)(n - 1 - i));
        int j = (int)(((unsigned __int128)v * (uint64_t)(i + 1)) >> 64);
        int32_t t = out[i]; out[i] = out[j]; out[j] = t;
    }
}
