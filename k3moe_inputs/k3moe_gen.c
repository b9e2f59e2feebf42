/*
 * k3moe_gen.c -- seeded synthetic inputs for the routed-expert layer.
 *
 * This module draws the inputs (activations, router weights, routing bias,
 * MXFP4 expert codes and scales, dense shared-expert weights) and nothing
 * else: it holds none of the layer's arithmetic.  Both the CPU oracle and
 * the GPU path are fed from it.
 *
 * Every value is a pure function of (seed, stream, index): a counter-based
 * generator built from the splitmix64 output mixer (Steele, Lea and Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014).  Any slice
 * of any tensor can be regenerated on its own, in any order, by any number of
 * threads, with the same bits.
 *
 * Normals use the Box-Muller transform.  Its logarithm and cosine are
 * evaluated here with plain series in IEEE double arithmetic (build with
 * -ffp-contract=off), so the draws are bit-identical on x86-64 and AArch64
 * and do not depend on the platform libm.
 */
#include <stdint.h>
#include <stddef.h>
#include <math.h>

#define K3G_GOLDEN 0x9E3779B97F4A7C15ull

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* The generator: 64 random bits for element i of stream `stream` under `seed`. */
uint64_t k3g_hash(uint64_t seed, uint64_t stream, uint64_t i)
{
    const uint64_t key = mix64(seed * K3G_GOLDEN + mix64(stream + 0x632BE59BD9B4E019ull));
    return mix64(key + (i + 1) * K3G_GOLDEN);
}

/* Uniform double in [0, 1) with 53 random bits. */
double k3g_uniform(uint64_t seed, uint64_t stream, uint64_t i)
{
    return (double)(k3g_hash(seed, stream, i) >> 11) * 0x1.0p-53;
}

/* Natural log for finite u > 0: u = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * then ln m = 2 atanh(t), t = (m-1)/(m+1) in (-0.172, 0.172), summed as an odd
 * series. */
double k3g_log(double u)
{
    int e;
    double m = frexp(u, &e);
    if (m < 0.70710678118654752440) {
        m *= 2.0;
        e -= 1;
    }
    const double t = (m - 1.0) / (m + 1.0);
    const double t2 = t * t;
    double term = t, sum = 0.0;
    for (int n = 1; n < 64; n += 2) {
        const double add = term / (double)n;
        sum += add;
        if (add == 0.0 || (add < 0 ? -add : add) < 1e-30)
            break;
        term *= t2;
    }
    return 2.0 * sum + (double)e * 0.69314718055994530942;
}

/* sin and cos of phi in [0, pi/2) by Taylor series. */
static void sincos_quarter(double phi, double *s, double *c)
{
    const double p2 = phi * phi;
    double ts = phi, tc = 1.0, ss = 0.0, sc = 0.0;
    for (int n = 0; n < 30; n++) {
        ss += ts;
        sc += tc;
        ts *= -p2 / (double)((2 * n + 2) * (2 * n + 3));
        tc *= -p2 / (double)((2 * n + 1) * (2 * n + 2));
    }
    *s = ss;
    *c = sc;
}

/* cos(2 pi v) for v in [0, 1), reduced to a quarter turn. */
static double cos_turn(double v)
{
    const double v4 = v * 4.0;
    const int q = (int)v4;                   /* 0..3 */
    const double phi = (v4 - (double)q) * 1.57079632679489661923;
    double s, c;
    sincos_quarter(phi, &s, &c);
    switch (q & 3) {
    case 0: return c;
    case 1: return -s;
    case 2: return -c;
    default: return s;
    }
}

/* Standard normal draw number i (Box-Muller on uniforms 2i and 2i+1). */
double k3g_normal(uint64_t seed, uint64_t stream, uint64_t i)
{
    const double u1 = 1.0 - k3g_uniform(seed, stream, 2 * i);   /* (0, 1] */
    const double u2 = k3g_uniform(seed, stream, 2 * i + 1);     /* [0, 1) */
    const double r = sqrt(-2.0 * k3g_log(u1));
    return r * cos_turn(u2);
}

/* float -> bfloat16, round to nearest even (NaN kept quiet). */
uint16_t k3g_f32_to_bf16(float f)
{
    union { float f; uint32_t u; } v = { f };
    if ((v.u & 0x7F800000u) == 0x7F800000u && (v.u & 0x007FFFFFu))
        return (uint16_t)((v.u >> 16) | 0x0040u);
    const uint32_t lsb = (v.u >> 16) & 1u;
    return (uint16_t)((v.u + 0x7FFFu + lsb) >> 16);
}

/* out[j] = bf16(sigma * N(seed, stream, offset + j)), j < n. */
void k3g_bf16_normal(uint16_t *out, size_t n, uint64_t seed, uint64_t stream,
                     uint64_t offset, double sigma)
{
#pragma omp parallel for schedule(static) if (n > 65536)
    for (size_t j = 0; j < n; j++)
        out[j] = k3g_f32_to_bf16((float)(sigma * k3g_normal(seed, stream, offset + j)));
}

/* Uniform random bytes: byte j is byte (j % 8) of hash(offset/8 + j/8).
 * `offset` must be a multiple of 8 so slices line up with whole draws. */
void k3g_bytes(uint8_t *out, size_t n, uint64_t seed, uint64_t stream, uint64_t offset)
{
    const uint64_t base = offset >> 3;
    const size_t nw = n >> 3;
#pragma omp parallel for schedule(static) if (nw > 65536)
    for (size_t w = 0; w < nw; w++) {
        uint64_t h = k3g_hash(seed, stream, base + w);
        for (int b = 0; b < 8; b++)
            out[w * 8 + (size_t)b] = (uint8_t)(h >> (8 * b));
    }
    if (n & 7) {
        uint64_t h = k3g_hash(seed, stream, base + nw);
        for (size_t b = 0; b < (n & 7); b++)
            out[nw * 8 + b] = (uint8_t)(h >> (8 * b));
    }
}

/* Uniform integers in [lo, hi] as bytes (E8M0 scale bytes). */
void k3g_uniform_bytes(uint8_t *out, size_t n, uint64_t seed, uint64_t stream,
                       uint64_t offset, int lo, int hi)
{
    const uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static) if (n > 65536)
    for (size_t j = 0; j < n; j++)
        out[j] = (uint8_t)(lo + (int)(k3g_hash(seed, stream, offset + j) % span));
}

/* A seeded permutation of 0..n-1 (Fisher-Yates from the top). */
void k3g_permutation(int32_t *perm, int32_t n, uint64_t seed, uint64_t stream)
{
    for (int32_t i = 0; i < n; i++)
        perm[i] = i;
    for (int32_t i = n - 1; i > 0; i--) {
        const int32_t j = (int32_t)(k3g_hash(seed, stream, (uint64_t)i) % (uint64_t)(i + 1));
        const int32_t t = perm[i];
        perm[i] = perm[j];
        perm[j] = t;
    }
}

/* Zipf-shaped routing bias: the expert of rank r (1-based, ranks assigned by a
 * seeded permutation) gets bias = scale * ln(r^-s) = -scale * s * ln r. */
void k3g_zipf_bias(float *bias, int32_t n, uint64_t seed, uint64_t stream,
                   double s, double scale)
{
    int32_t perm[4096];
    if (n > 4096)
        return;
    k3g_permutation(perm, n, seed, stream);
    for (int32_t r = 1; r <= n; r++)
        bias[perm[r - 1]] = (float)(-scale * s * k3g_log((double)r));
}
