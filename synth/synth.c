/*
 * Seeded synthetic inputs for the paged KV-cache decode step.
 *
 * This module is shared by the test harness, the benchmark and the oracle
 * harness.  It holds NONE of the method's arithmetic: it only draws random
 * numbers (values, lengths, permutations) from a counter-based generator, so
 * that any slice of any input can be regenerated on its own.
 *
 * Generator: splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014).  The i-th output of the stream with key k
 * is mix64(k + (i + 1) * GOLDEN), which is exactly the i-th output of a
 * splitmix64 generator seeded with k, but reachable in O(1).  A stream key is
 * derived from (seed, stream id) with the same mixer.
 *
 * Normal deviates: Box-Muller (Box and Muller, 1958) in double precision on a
 * pair of open-interval uniforms, cosine branch for even indices and sine
 * branch for odd ones.  "N(0,1) in bf16" is that double rounded to the nearest
 * bfloat16, ties to even.
 *
 * Plain portable C: no intrinsics, no inline assembly; the same results on
 * x86-64 and aarch64 up to libm's last-place differences in log/sin/cos,
 * which reach a bf16 value only when a draw sits on a rounding boundary.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t synth_key(uint64_t seed, uint64_t stream)
{
    return mix64(mix64(seed + GOLDEN) ^ mix64(stream * 0xD1B54A32D192ED03ULL + 0x632BE59BD9B4E019ULL));
}

uint64_t synth_u64(uint64_t key, uint64_t i)
{
    return mix64(key + (i + 1) * GOLDEN);
}

/* uniform in (0, 1]: 53 random bits, never zero (log-safe) */
static inline double u01(uint64_t x)
{
    return (double)((x >> 11) + 1) * 0x1p-53;
}

double synth_uniform(uint64_t key, uint64_t i)
{
    return u01(synth_u64(key, i));
}

double synth_normal(uint64_t key, uint64_t i)
{
    const uint64_t pair = i >> 1;
    const double u1 = u01(synth_u64(key, 2 * pair));
    const double u2 = u01(synth_u64(key, 2 * pair + 1));
    const double r = sqrt(-2.0 * log(u1));
    const double th = 6.283185307179586476925286766559 * u2;
    return (i & 1) ? r * sin(th) : r * cos(th);
}

/* double -> bfloat16 bits, round to nearest, ties to even (finite inputs;
 * NaN maps to the canonical quiet NaN 0x7FC0). Operates on the IEEE-754
 * binary64 encoding directly so that no intermediate float rounding occurs. */
uint16_t synth_bf16_from_double(double x)
{
    uint64_t b;
    memcpy(&b, &x, 8);
    const uint16_t sign = (uint16_t)((b >> 48) & 0x8000);
    const uint64_t mag = b & 0x7FFFFFFFFFFFFFFFULL;
    if (mag > 0x7FF0000000000000ULL) return 0x7FC0;          /* NaN */
    if (mag == 0x7FF0000000000000ULL) return sign | 0x7F80;  /* inf */
    double a = fabs(x);
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);          /* a = f * 2^e2, f in [0.5, 1) */
    int e = e2 - 1;               /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;       /* subnormal bf16 share the 2^-133 quantum */
    const double quantum = ldexp(1.0, e - 7);
    const double q = rint(a / quantum);  /* exact scaling; rint = ties-to-even */
    double r = q * quantum;
    if (r >= 0x1p128) return sign | 0x7F80;                  /* overflow -> inf */
    float f = (float)r;           /* exactly representable in bf16, hence in float */
    uint32_t fb;
    memcpy(&fb, &f, 4);
    return sign | (uint16_t)((fb >> 16) & 0x7FFF);
}

/* out[j] = bf16(N(0,1)) for draw index offset + j, j < n */
void synth_fill_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint16_t *out)
{
    const uint64_t key = synth_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = synth_bf16_from_double(synth_normal(key, offset + (uint64_t)j));
}

void synth_fill_normal_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double *out)
{
    const uint64_t key = synth_key(seed, stream);
#pragma omp parallel for schedule(static)
    for (int64_t j = 0; j < n; ++j) out[j] = synth_normal(key, offset + (uint64_t)j);
}

void synth_fill_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, double *out)
{
    const uint64_t key = synth_key(seed, stream);
    for (int64_t j = 0; j < n; ++j) out[j] = synth_uniform(key, offset + (uint64_t)j);
}

void synth_fill_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t *out)
{
    const uint64_t key = synth_key(seed, stream);
    for (int64_t j = 0; j < n; ++j) out[j] = synth_u64(key, offset + (uint64_t)j);
}

/* Fisher-Yates (Durstenfeld) shuffle of [0, n): step i (from n-1 down to 1)
 * swaps position i with j = u64(i) mod (i + 1). The modulo bias is below
 * n / 2^64 and irrelevant for test inputs. */
void synth_permutation(uint64_t seed, uint64_t stream, int64_t n, int32_t *out)
{
    const uint64_t key = synth_key(seed, stream);
    for (int64_t i = 0; i < n; ++i) out[i] = (int32_t)i;
    for (int64_t i = n - 1; i > 0; --i) {
        const int64_t j = (int64_t)(synth_u64(key, (uint64_t)i) % (uint64_t)(i + 1));
        const int32_t t = out[i];
        out[i] = out[j];
        out[j] = t;
    }
}
