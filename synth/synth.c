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
 *     here from their Taylor / atanh series (Horner form, coefficients made by
 *     IEEE divisions) using only IEEE-754 +, -, *, / and sqrt in double
 *     precision (correctly rounded on both hosts), compiled with
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

/* Series coefficients, filled once by IEEE divisions (same bits on every host):
 * LOGC[i] = 1/(2i+1) for the atanh series, SINC[i] = (-1)^i/(2i+1)!,
 * COSC[i] = (-1)^i/(2i)!. */
#define NLOG 13
#define NTRIG 11
static double LOGC[NLOG], SINC[NTRIG], COSC[NTRIG];
static int coef_ready = 0;

static void init_coefficients(void) {
    if (coef_ready) return;
    for (int i = 0; i < NLOG; ++i) LOGC[i] = 1.0 / (double)(2 * i + 1);
    double f = 1.0;                       /* running factorial */
    for (int k = 0; k < 2 * NTRIG; ++k) {
        if (k > 0) f *= (double)k;
        double c = ((k / 2) % 2 ? -1.0 : 1.0) / f;
        if (k % 2) SINC[k / 2] = c; else COSC[k / 2] = c;
    }
    coef_ready = 1;
}

/* natural log of u in (0, 1]: u = m * 2^e with m in [sqrt(1/2), sqrt(2)),
 * log m = 2 atanh(f), f = (m-1)/(m+1), |f| < 0.1716, series to f^25 (Horner). */
static double gen_log(double u) {
    int e;
    double m = frexp(u, &e);               /* exact: m in [0.5, 1) */
    if (m < 0.70710678118654752440) { m *= 2.0; e -= 1; }
    double f = (m - 1.0) / (m + 1.0);
    double f2 = f * f;
    double p = LOGC[NLOG - 1];
    for (int i = NLOG - 2; i >= 0; --i) p = p * f2 + LOGC[i];
    return 2.0 * f * p + (double)e * 0.69314718055994530942;
}

/* cos and sin of 2*pi*v for v in (0, 1): reduce v to the nearest quarter turn
 * (exact in binary), then Taylor series (Horner) on |x| <= pi/4. */
static void gen_sincos_turns(double v, double* c, double* s) {
    double q = floor(v * 4.0 + 0.5);         /* 0..4 */
    double r = v - q * 0.25;                 /* exact, |r| <= 1/8 */
    double x = r * 6.28318530717958647692;
    double x2 = x * x;
    double sp = SINC[NTRIG - 1], cp = COSC[NTRIG - 1];
    for (int i = NTRIG - 2; i >= 0; --i) {
        sp = sp * x2 + SINC[i];
        cp = cp * x2 + COSC[i];
    }
    double sn = x * sp, cs = cp;
    int quad = ((int)q) & 3;
    switch (quad) {
        case 0: *c = cs;  *s = sn;  break;
        case 1: *c = -sn; *s = cs;  break;
        case 2: *c = -cs; *s = -sn; break;
        default: *c = sn; *s = -cs; break;
    }
}

/* the two normals of pair p: z0 = r cos(2 pi u2), z1 = r sin(2 pi u2) */
static inline void normal_pair(uint64_t key, uint64_t pair, double* z0, double* z1) {
    double u1 = unit_open(draw_bits(key, 2 * pair));
    double u2 = unit_open(draw_bits(key, 2 * pair + 1));
    double r = sqrt(-2.0 * gen_log(u1));
    double c, s;
    gen_sincos_turns(u2, &c, &s);
    *z0 = r * c;
    *z1 = r * s;
}

static inline uint16_t f32_to_bf16_rne(float f) {
    uint32_t b;
    memcpy(&b, &f, 4);
    uint32_t lsb = (b >> 16) & 1u;
    b += 0x7fffu + lsb;
    return (uint16_t)(b >> 16);
}

/* element i of a normal stream is z0 of pair i/2 when i is even, z1 when odd;
 * the loop runs over pairs so each pair is computed once */
#define NORMAL_LOOP(STORE)                                                         \
    uint64_t key = stream_key(seed, stream);                                       \
    init_coefficients();                                                           \
    if (n <= 0) return;                                                            \
    uint64_t p0 = offset >> 1, p1 = (offset + (uint64_t)n - 1) >> 1;               \
    _Pragma("omp parallel for schedule(static)")                                   \
    for (int64_t pi = (int64_t)p0; pi <= (int64_t)p1; ++pi) {                      \
        double z[2];                                                               \
        normal_pair(key, (uint64_t)pi, &z[0], &z[1]);                              \
        for (int t = 0; t < 2; ++t) {                                              \
            int64_t i = 2 * pi + t - (int64_t)offset;                              \
            if (i >= 0 && i < n) STORE;                                            \
        }                                                                          \
    }

void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, float* out) {
    NORMAL_LOOP(out[i] = (float)z[t])
}

void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint16_t* out) {
    NORMAL_LOOP(out[i] = f32_to_bf16_rne((float)z[t]))
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
double synth_log(double u) { init_coefficients(); return gen_log(u); }
void synth_sincos_turns(double v, double* c, double* s) { init_coefficients(); gen_sincos_turns(v, c, s); }
