/*
 * Seeded synthetic inputs shared by the tests, the benchmark and the oracle
 * checks.  This file holds no RoPE arithmetic: it only draws numbers.
 *
 *  - SplitMix64, used counter-style: value k of stream `seed` is the SplitMix64
 *    output mix of (seed + (k+1) * golden-gamma) (Steele, Lea & Flood,
 *    "Fast Splittable Pseudorandom Number Generators", OOPSLA 2014).  Being a
 *    pure function of (seed, k), the stream is identical whatever the thread
 *    count, on x86-64 and aarch64 alike.
 *  - Uniform doubles in (0, 1): the top 53 bits of a draw, offset by half a
 *    quantum so that log() never sees 0.
 *  - Standard normals: the Box-Muller transform (Box & Muller, 1958) on the
 *    draw pair (2i, 2i+1) gives elements 2i and 2i+1.
 */
#include <math.h>
#include <stdint.h>

static inline uint64_t splitmix64_at(uint64_t seed, uint64_t k) {
  uint64_t z = seed + (k + 1u) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

static inline double unit_open(uint64_t z) {
  return ((double)(z >> 11) + 0.5) * 0x1.0p-53;
}

/* n standard-normal draws, stored as float32. */
void wl_normal_f32(uint64_t seed, int64_t n, float* out) {
  const double two_pi = 6.283185307179586476925286766559;
  int64_t pairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < pairs; ++p) {
    double u1 = unit_open(splitmix64_at(seed, (uint64_t)(2 * p)));
    double u2 = unit_open(splitmix64_at(seed, (uint64_t)(2 * p + 1)));
    double r = sqrt(-2.0 * log(u1));
    double a = two_pi * u2;
    out[2 * p] = (float)(r * cos(a));
    if (2 * p + 1 < n) out[2 * p + 1] = (float)(r * sin(a));
  }
}

/* n uniform doubles in (0, 1). */
void wl_uniform_f64(uint64_t seed, int64_t n, double* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = unit_open(splitmix64_at(seed, (uint64_t)i));
}

/* n integers uniform in [lo, hi). */
void wl_uniform_int(uint64_t seed, int64_t n, int64_t lo, int64_t hi, int64_t* out) {
  double span = (double)(hi - lo);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    int64_t v = lo + (int64_t)floor(unit_open(splitmix64_at(seed, (uint64_t)i)) * span);
    out[i] = v < hi ? v : hi - 1;
  }
}
