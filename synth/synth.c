/*
 * Seeded synthetic inputs for the MoE FFN layer: the one module that both the
 * fp64 oracle and the CUDA library consume.  It holds none of the layer's
 * arithmetic; it only turns (seed, tensor id, element index) into numbers.
 *
 * Definition (counter based, so any slice can be produced on its own):
 *   mix64(z)       : the SplitMix64 finaliser
 *                    z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                    z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31
 *   key(seed, id)  = mix64(seed ^ mix64(id + 0x632BE59BD9B4E019))
 *   bits(i)        = mix64(key + (i + 1) * 0x9E3779B97F4A7C15)
 *                    (the i-th SplitMix64 output of a stream started at key)
 *   U(i)           = ((bits(i) >> 11) + 0.5) * 2^-53          in (0, 1)
 *   N(2j), N(2j+1) = Box-Muller on U(2j), U(2j+1):
 *                    r = sqrt(-2 ln U(2j)); N(2j) = r cos(2 pi U(2j+1)),
 *                    N(2j+1) = r sin(2 pi U(2j+1))
 *
 * Element i of a tensor is element i of its row-major flattening.  Values are
 * rounded straight from double to the storage type (bf16 round-to-nearest-even,
 * or int8 by nearbyint and clipping), never through float.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SYNTH_PI 3.14159265358979323846

static inline uint64_t mix64(uint64_t z) {
  z ^= z >> 30; z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27; z *= 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t id) {
  return mix64(seed ^ mix64(id + 0x632BE59BD9B4E019ull));
}

static inline double unif(uint64_t key, uint64_t i) {
  uint64_t b = mix64(key + (i + 1) * 0x9E3779B97F4A7C15ull);
  return ((double)(b >> 11) + 0.5) * 0x1.0p-53;
}

static inline double normal(uint64_t key, uint64_t i) {
  uint64_t j = i >> 1;
  double u1 = unif(key, 2 * j), u2 = unif(key, 2 * j + 1);
  double r = sqrt(-2.0 * log(u1));
  return (i & 1) ? r * sin(2.0 * SYNTH_PI * u2) : r * cos(2.0 * SYNTH_PI * u2);
}

/* double -> bf16 bits, round to nearest, ties to even, directly from double. */
static uint16_t to_bf16(double v) {
  if (v != v) return 0x7FC0;
  uint16_t sign = signbit(v) ? 0x8000 : 0;
  double a = fabs(v);
  if (a == 0.0) return sign;
  double r;
  if (a < 0x1.0p-126) {
    r = nearbyint(a * 0x1.0p133) * 0x1.0p-133;   /* subnormal grid */
  } else {
    int e; double m = frexp(a, &e);              /* a = m 2^e, m in [0.5,1) */
    r = ldexp(nearbyint(ldexp(m, 8)), e - 8);    /* 8 significant bits */
  }
  if (r > 0x1.FEp127) return sign | 0x7F80;      /* overflow to inf */
  float f = (float)r;                            /* exact */
  uint32_t u; memcpy(&u, &f, 4);
  return sign | (uint16_t)(u >> 16);
}

/* out[i] = bf16(scale * N(offset + i)), i < n */
void synth_normal_bf16(uint64_t seed, uint64_t id, double scale,
                       uint16_t *out, int64_t offset, int64_t n) {
  uint64_t key = stream_key(seed, id);
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = to_bf16(scale * normal(key, (uint64_t)(offset + i)));
}

/* out[i] = scale * N(offset + i) in double (used to check the generator) */
void synth_normal_f64(uint64_t seed, uint64_t id, double scale,
                      double *out, int64_t offset, int64_t n) {
  uint64_t key = stream_key(seed, id);
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = scale * normal(key, (uint64_t)(offset + i));
}

/* out[i] = clip(nearbyint(scale * N(offset + i)), lo, hi) as int8 */
void synth_int8(uint64_t seed, uint64_t id, double scale, int lo, int hi,
                int8_t *out, int64_t offset, int64_t n) {
  uint64_t key = stream_key(seed, id);
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double q = nearbyint(scale * normal(key, (uint64_t)(offset + i)));
    if (q < lo) q = lo;
    if (q > hi) q = hi;
    out[i] = (int8_t)q;
  }
}

/* out[i] = (float)(lo + (hi - lo) * U(offset + i)) */
void synth_uniform_f32(uint64_t seed, uint64_t id, double lo, double hi,
                       float *out, int64_t offset, int64_t n) {
  uint64_t key = stream_key(seed, id);
  #pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = (float)(lo + (hi - lo) * unif(key, (uint64_t)(offset + i)));
}

/* raw 64-bit stream words, for checking the generator against its definition */
void synth_bits(uint64_t seed, uint64_t id, uint64_t *out, int64_t offset, int64_t n) {
  uint64_t key = stream_key(seed, id);
  for (int64_t i = 0; i < n; ++i) out[i] = mix64(key + ((uint64_t)(offset + i) + 1) * 0x9E3779B97F4A7C15ull);
}
