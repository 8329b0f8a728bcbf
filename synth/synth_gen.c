/* Seeded synthetic-input generator (counter-based SplitMix64 + Box-Muller).
 * Random numbers and bf16 packing only; none of the NVFP4 arithmetic. */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline uint64_t mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Draw i of stream `seed`. */
static inline uint64_t draw(uint64_t seed, uint64_t i) {
  return mix((seed << 32) + (i + 1) * 0x9E3779B97F4A7C15ull);
}

static inline double unif(uint64_t seed, uint64_t i) {
  return ((double)(draw(seed, i) >> 11) + 1.0) * 0x1p-53;
}

static inline uint16_t f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);
}

/* Elements start .. start+n-1 of the normal tensor of stream `seed`. */
void syn_normal_bf16(uint64_t seed, int64_t start, int64_t n, double std, double outlier_p,
                     double outlier_mult, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; j++) {
    uint64_t e = (uint64_t)(start + j);
    double u1 = unif(seed, 3 * e), u2 = unif(seed, 3 * e + 1);
    double v = sqrt(-2.0 * log(u1)) * cos(2.0 * 3.14159265358979323846 * u2) * std;
    if (outlier_p > 0.0 && unif(seed, 3 * e + 2) <= outlier_p) v *= outlier_mult;
    out[j] = f32_to_bf16((float)v);
  }
}

void syn_uniform(uint64_t seed, int64_t start, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < n; j++) out[j] = unif(seed, (uint64_t)(start + j));
}
