/*
 * Seeded synthetic input generator shared by the fp64 oracle and the CUDA path.
 *
 * This file holds no arithmetic of the attention method: it only turns
 * (seed, stream, element index) into uniform or normal samples.  Both sides of
 * every parity test read the bytes it writes, so it must give the same bits on
 * every host (x86_64 here, aarch64 on the GPU machine).  To that end:
 *   - the bit source is counter-based SplitMix64 (Steele, Lea, Flood,
 *     "Fast splittable pseudorandom number generators", OOPSLA 2014): sample i
 *     of a stream is mix64(key + (i+1)*golden_gamma), so any slice can be drawn
 *     without drawing what precedes it;
 *   - normals come from the Box-Muller transform, with log, sin and cos written
 *     here from their Taylor / atanh series using only IEEE-754 +, -, *, / and
 *     sqrt in double precision (correctly rounded on both hosts), compiled with
 *     -ffp-contract=off so that no multiply-add gets fused differently;
 *   - float and bfloat16 outputs are produced by round-to-nearest-even.
 */
#include <stdint.h>
#include <string.h>
#include <math.h>

#define GOLDEN_GAMMA 0x9e3779b97f4a7c15ULL

static inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
    return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return mix64(mix64(seed * GOLDEN_GAMMA + 0x6a09e667f3bcc909ULL) ^ mix64(stream + 0xbb67ae8584caa73bULL));
}

static inline uint64_t draw_bits(uint64_t key, uint64_t i) {
    return mix64(key + (i + 1) * GOLDEN_GAMMA);
}

/* uniform double strictly inside (0, 1): midpoint of one of 2^53 cells */
static inline double unit_open(uint64_t bits) {
    return ((double)(bits >> 11) + 0.5) * (1.0 / 9007199254740992.0);
}

/* natural log of u in (0, 1]: u = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * log m = 2 atanh(f), f = (m-1)/(m+1), |f| < 0.1716, series to f^25. */
static double gen_log(double u) {
    int e;
    double m = frexp(u, &e);               /* exact: m in [0.5, 1) */
    if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
    double f = (m - 1.0) / (m + 1.0);
    double f2 = f * f;
    double term = f, sum = 0.0;
    for (int k = 1; k <= 25; k += 2) {
        sum += term / (double)k;
        term *= f2;
    }
    return 2.0 * sum + (double)e * 0.69314718055994530942;
}

/* cos and sin of 2*pi*v for v in (0, 1): reduce v to the nearest quarter turn
 * (exact in binary), then Taylor series on |x| <= pi/4. */
static void gen_sincos_turns(double v, double* c, double* s) {
    double q = floor(v * 4.0 + 0.5);         /* 0..4 */
    double r = v - q * 0.25;                 /* exact, |r| <= 1/8 */
    double x = r * 6.28318530717958647692;
    double x2 = x * x;
    double sn = 0.0, cs = 0.0, ts = x, tc = 1.0;
    for (int k = 1; k <= 21; k += 2) {       /* x^k/k! and x^(k-1)/(k-1)! */
        sn += ts;
        cs += tc;
        ts *= -x2 / (double)((k + 1) * (k + 2));
        tc *= -x2 / (double)(k * (k + 1));
    }
    int quad = ((int)q) & 3;
    switch (quad) {
        case 0: *c = cs;  *s = sn;  break;
        case 1: *c = -sn; *s = cs;  break;
        case 2: *c = -cs; *s = -sn; break;
        default: *c = sn; *s = -cs; break;
    }
}

static inline double normal_at(uint64_t key, uint64_t idx) {
    uint64_t pair = idx >> 1;
    double u1 = unit_open(draw_bits(key, 2 * pair));
    double u2 = unit_open(draw_bits(key, 2 * pair + 1));
    double r = sqrt(-2.0 * gen_log(u1));
    double c, s;
    gen_sincos_turns(u2, &c, &s);
    return (idx & 1) ? r * s : r * c;
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7fffu + lsb;
    return (uint16_t)(b >> 16);
}

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, float* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = (float)normal_at(key, offset + (uint64_t)i);
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint16_t* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16_rne((float)normal_at(key, offset + (uint64_t)i));
}

void synth_uniform_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double lo, double hi, float* out) {
    uint64_t key = stream_key(seed, stream);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i)
        out[i] = (float)(lo + (hi - lo) * unit_open(draw_bits(key, offset + (uint64_t)i)));
}

/* raw 64-bit draws, for the generator's own tests */
void synth_bits(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t* out) {
    uint64_t key = stream_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = draw_bits(key, offset + (uint64_t)i);
}

/* the generator's own log / sincos, exposed so tests can compare them with libm */
double synth_log(double u) { return gen_log(u); }
void synth_sincos_turns(double v, double* c, double* s) { gen_sincos_turns(v, c, s); }
