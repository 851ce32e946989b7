/* synth.c -- seeded, counter-based generators for the synthetic decode workloads.
 *
 * This module only makes input bytes. It holds none of the decode step's arithmetic and is shared
 * by both sides of every comparison: the oracle and the CUDA path each receive the same bytes.
 *
 * Generator (fully specified so that any implementation reproduces it):
 *   mix64(z)        = SplitMix64 output function:
 *                     z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                     z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                     return z ^ (z >> 31)
 *   GAMMA           = 0x9E3779B97F4A7C15
 *   base(seed, sid) = mix64(seed * GAMMA + mix64(sid))            (sid: one id per tensor)
 *   word(n)         = mix64(base + (n + 1) * GAMMA)                (the n-th SplitMix64 output)
 *   uniform(n)      = ((word(n) >> 11) + 0.5) * 2^-53               in (0, 1)
 *   normal pair k   = Box-Muller on u1 = uniform(2k), u2 = uniform(2k+1):
 *                     r = sqrt(-2 ln u1); z0 = r cos(2 pi u2); z1 = r sin(2 pi u2)
 *                     element 2k takes z0, element 2k+1 takes z1
 *   nibble byte n   = low nibble = word(n) >> 60, high nibble = (word(n) >> 56) & 15
 *   integer n in [0, hi) = floor(uniform(n) * hi)
 * Values are rounded to bf16 / fp16 to nearest, ties to even, straight from double.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t base_of(uint64_t seed, uint64_t sid) { return mix64(seed * GAMMA + mix64(sid)); }
static inline uint64_t word_at(uint64_t base, uint64_t n) { return mix64(base + (n + 1) * GAMMA); }
static inline double uniform_at(uint64_t base, uint64_t n) {
  return ((double)(word_at(base, n) >> 11) + 0.5) * 0x1.0p-53;
}

static inline double normal_at(uint64_t base, uint64_t i) {
  uint64_t k = i >> 1;
  double u1 = uniform_at(base, 2 * k), u2 = uniform_at(base, 2 * k + 1);
  double r = sqrt(-2.0 * log(u1));
  double ang = 6.283185307179586476925 * u2;
  return (i & 1) ? r * sin(ang) : r * cos(ang);
}

/* nearest bf16, ties to even, from double */
static uint16_t to_bf16(double v) {
  if (isnan(v)) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7F80;
  int e;
  frexp(a, &e);
  double q = rint(ldexp(a, 8 - e));
  if (q == 256.0) { q = 128.0; e += 1; }
  int biased = e - 1 + 127;
  if (biased >= 255) return sign | 0x7F80;
  if (biased <= 0) return sign | (uint16_t)rint(ldexp(a, 133));
  return sign | (uint16_t)((biased << 7) | ((int)q - 128));
}

/* nearest fp16 (binary16), ties to even, from double */
static uint16_t to_fp16(double v) {
  if (isnan(v)) return 0x7E00;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  if (isinf(a)) return sign | 0x7C00;
  int e;
  frexp(a, &e);
  double q = rint(ldexp(a, 11 - e));          /* 11-bit significand in [1024, 2048] */
  if (q == 2048.0) { q = 1024.0; e += 1; }
  int biased = e - 1 + 15;
  if (biased >= 31) return sign | 0x7C00;
  if (biased <= 0) return sign | (uint16_t)rint(ldexp(a, 24));  /* subnormal: multiples of 2^-24 */
  return sign | (uint16_t)((biased << 10) | ((int)q - 1024));
}

void synth_normal_bf16(uint64_t seed, uint64_t sid, int64_t n, double mean, double std,
                       uint16_t* out) {
  uint64_t b = base_of(seed, sid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = to_bf16(mean + std * normal_at(b, (uint64_t)i));
}

/* |N(0, std)| rounded to fp16 (fmt 0) or bf16 (fmt 1): int4 group scales */
void synth_abs_normal_16(uint64_t seed, uint64_t sid, int64_t n, double std, int fmt,
                         uint16_t* out) {
  uint64_t b = base_of(seed, sid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double v = fabs(std * normal_at(b, (uint64_t)i));
    out[i] = fmt ? to_bf16(v) : to_fp16(v);
  }
}

void synth_nibbles(uint64_t seed, uint64_t sid, int64_t n_bytes, uint8_t* out) {
  uint64_t b = base_of(seed, sid);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n_bytes; ++i) {
    uint64_t w = word_at(b, (uint64_t)i);
    out[i] = (uint8_t)((w >> 60) | (((w >> 56) & 15) << 4));
  }
}

void synth_uniform_int(uint64_t seed, uint64_t sid, int64_t n, int32_t hi, int32_t* out) {
  uint64_t b = base_of(seed, sid);
  for (int64_t i = 0; i < n; ++i) {
    int32_t v = (int32_t)floor(uniform_at(b, (uint64_t)i) * (double)hi);
    out[i] = v < hi ? v : hi - 1;
  }
}

/* raw words and normals, for tests of the generator itself */
void synth_words(uint64_t seed, uint64_t sid, int64_t n, uint64_t* out) {
  uint64_t b = base_of(seed, sid);
  for (int64_t i = 0; i < n; ++i) out[i] = word_at(b, (uint64_t)i);
}
void synth_normals(uint64_t seed, uint64_t sid, int64_t n, double* out) {
  uint64_t b = base_of(seed, sid);
  for (int64_t i = 0; i < n; ++i) out[i] = normal_at(b, (uint64_t)i);
}

/* plain SplitMix64 from a given state (for checking mix64 against published outputs) and the
 * per-tensor base state, so that word(n) can be checked to be the n-th output from that base */
void synth_splitmix(uint64_t state, int64_t n, uint64_t* out) {
  for (int64_t i = 0; i < n; ++i) { state += GAMMA; out[i] = mix64(state); }
}
uint64_t synth_base(uint64_t seed, uint64_t sid) { return base_of(seed, sid); }
