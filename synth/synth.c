/*
 * Seeded synthetic input generator (data only).
 *
 * This file holds none of the MoE layer's arithmetic: it only fills arrays with
 * pseudo-random numbers of the distributions the workloads name (normal,
 * uniform, integer uniform).  Both the CPU oracle and the GPU library receive
 * the arrays it writes; neither side calls it for anything else.
 *
 * Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
 * number generators", OOPSLA 2014) used as a counter-based hash.  Element i of
 * a stream with key K is derived from the SplitMix64 output for state
 * K + (i + 1) * golden_gamma, so every element depends only on (K, i): the
 * result is independent of thread count and of how the array is chunked.
 *
 * Normals come from the Box-Muller transform (Box and Muller, 1958): one
 * 64-bit hash gives two 32-bit uniforms u1, u2 in (0, 1) and two normals
 * sqrt(-2 ln u1) * (cos 2 pi u2, sin 2 pi u2), computed in double precision.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define GOLDEN_GAMMA 0x9E3779B97F4A7C15ull

static inline uint64_t splitmix64_at(uint64_t key, uint64_t i) {
  uint64_t z = key + (i + 1u) * GOLDEN_GAMMA;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

/* Stream key for (seed, tensor id): hashing keeps streams of nearby ids apart. */
uint64_t synth_stream_key(uint64_t seed, uint64_t tensor_id) {
  return splitmix64_at(splitmix64_at(seed, 0x5EEDull), tensor_id);
}

/* u in (0, 1) from 32 random bits: (b + 0.5) / 2^32. */
static inline double unit_open(uint32_t b) { return ((double)b + 0.5) * (1.0 / 4294967296.0); }

/* float -> bf16 bits, round to nearest even (inputs are finite). */
static inline uint16_t f32_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

static inline void normal_pair(uint64_t key, uint64_t j, double* z0, double* z1) {
  uint64_t h = splitmix64_at(key, j);
  double u1 = unit_open((uint32_t)(h >> 32));
  double u2 = unit_open((uint32_t)h);
  double r = sqrt(-2.0 * log(u1));
  double th = 6.283185307179586476925 * u2;
  *z0 = r * cos(th);
  *z1 = r * sin(th);
}

/* out[i] = mean + std * N(0,1), i in [0, n); element i is fixed by (key, i). */
void synth_normal_f32(uint64_t key, int64_t n, double mean, double std, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (n + 1) / 2; ++j) {
    double z0, z1;
    normal_pair(key, (uint64_t)j, &z0, &z1);
    out[2 * j] = (float)(mean + std * z0);
    if (2 * j + 1 < n) out[2 * j + 1] = (float)(mean + std * z1);
  }
}

/* Same draw as synth_normal_f32, rounded to bf16 (round to nearest even). */
void synth_normal_bf16(uint64_t key, int64_t n, double mean, double std, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t j = 0; j < (n + 1) / 2; ++j) {
    double z0, z1;
    normal_pair(key, (uint64_t)j, &z0, &z1);
    out[2 * j] = f32_to_bf16_bits((float)(mean + std * z0));
    if (2 * j + 1 < n) out[2 * j + 1] = f32_to_bf16_bits((float)(mean + std * z1));
  }
}

/* out[i] = lo + (hi - lo) * U(0,1). */
void synth_uniform_f32(uint64_t key, int64_t n, double lo, double hi, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t h = splitmix64_at(key, (uint64_t)i);
    out[i] = (float)(lo + (hi - lo) * unit_open((uint32_t)(h >> 32)));
  }
}

void synth_uniform_bf16(uint64_t key, int64_t n, double lo, double hi, uint16_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t h = splitmix64_at(key, (uint64_t)i);
    out[i] = f32_to_bf16_bits((float)(lo + (hi - lo) * unit_open((uint32_t)(h >> 32))));
  }
}

/* Integers uniform on [lo, hi] (inclusive), as int8. Multiply-shift range
 * reduction (Lemire 2019) on the top 32 bits. */
void synth_uniform_int8(uint64_t key, int64_t n, int32_t lo, int32_t hi, int8_t* out) {
  uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t h = splitmix64_at(key, (uint64_t)i);
    out[i] = (int8_t)(lo + (int32_t)(((h >> 32) * span) >> 32));
  }
}
