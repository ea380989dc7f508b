/*
 * Seeded synthetic inputs for the OPT-style generation workloads.
 *
 * Test and benchmark infrastructure. Both the CPU oracle and the CUDA library
 * receive the bytes written here; nothing in this file computes any part of
 * the generation method itself (no LayerNorm, attention, GEMM or LoRA math).
 *
 * Generator: counter-based SplitMix64 (Steele, Lea & Flood, "Fast Splittable
 * Pseudorandom Number Generators", OOPSLA 2014; the 64-bit finaliser constants
 * are the published ones).  Draw n of stream `key` is mix(key + (n+1)*gamma),
 * i.e. exactly the n-th output of a SplitMix64 generator whose state starts at
 * `key`, so any element can be computed independently of the others.
 *
 * Normal variates: Box-Muller transform (Box & Muller, 1958) on draws 2p and
 * 2p+1 for the pair p: u1 in (0,1], u2 in [0,1), r = sqrt(-2 ln u1),
 * z[2p] = r cos(2 pi u2), z[2p+1] = r sin(2 pi u2); value = mean + std * z,
 * computed in double, rounded to fp32, then (for bf16 outputs) rounded to
 * bf16 with round-to-nearest-even.
 *
 * Uniform integers in [lo, hi): lo + ((draw >> 32) * (hi - lo)) >> 32.
 *
 * Every element depends only on (seed, tensor_id, index), so the results do
 * not depend on the number of OpenMP threads.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define SM64_GAMMA 0x9e3779b97f4a7c15ULL

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

/* Stream key for one tensor of one seed. */
static inline uint64_t stream_key(uint64_t seed, uint64_t tensor_id) {
  return sm64_mix(sm64_mix(seed + SM64_GAMMA) ^ (tensor_id * SM64_GAMMA));
}

static inline uint64_t draw(uint64_t key, uint64_t n) {
  return sm64_mix(key + (n + 1) * SM64_GAMMA);
}

/* fp32 -> bf16 bits, round to nearest even (inputs here are finite). */
static inline uint16_t f32_to_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

static inline void normal_pair(uint64_t key, int64_t p, double mean, double std,
                               float *z0, float *z1) {
  const double inv53 = 1.0 / 9007199254740992.0; /* 2^-53 */
  uint64_t a = draw(key, (uint64_t)(2 * p));
  uint64_t b = draw(key, (uint64_t)(2 * p + 1));
  double u1 = ((double)(a >> 11) + 1.0) * inv53; /* (0, 1] */
  double u2 = (double)(b >> 11) * inv53;         /* [0, 1) */
  double r = sqrt(-2.0 * log(u1));
  double t = 6.283185307179586476925286766559 * u2;
  *z0 = (float)(mean + std * (r * cos(t)));
  *z1 = (float)(mean + std * (r * sin(t)));
}

void synth_normal_f32(float *out, int64_t n, uint64_t seed, uint64_t tensor_id,
                      double mean, double std) {
  const uint64_t key = stream_key(seed, tensor_id);
  const int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < npairs; ++p) {
    float z0, z1;
    normal_pair(key, p, mean, std, &z0, &z1);
    out[2 * p] = z0;
    if (2 * p + 1 < n) out[2 * p + 1] = z1;
  }
}

void synth_normal_bf16(uint16_t *out, int64_t n, uint64_t seed,
                       uint64_t tensor_id, double mean, double std) {
  const uint64_t key = stream_key(seed, tensor_id);
  const int64_t npairs = (n + 1) / 2;
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < npairs; ++p) {
    float z0, z1;
    normal_pair(key, p, mean, std, &z0, &z1);
    out[2 * p] = f32_to_bf16_rne(z0);
    if (2 * p + 1 < n) out[2 * p + 1] = f32_to_bf16_rne(z1);
  }
}

void synth_uniform_i32(int32_t *out, int64_t n, uint64_t seed,
                       uint64_t tensor_id, int32_t lo, int32_t hi) {
  const uint64_t key = stream_key(seed, tensor_id);
  const uint64_t span = (uint64_t)((int64_t)hi - (int64_t)lo);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    uint64_t d = draw(key, (uint64_t)i);
    out[i] = (int32_t)((int64_t)lo + (int64_t)(((d >> 32) * span) >> 32));
  }
}

/* Raw stream access, for the generator's own known-answer tests. */
uint64_t synth_raw_draw(uint64_t seed, uint64_t tensor_id, uint64_t n) {
  return draw(stream_key(seed, tensor_id), n);
}

uint64_t synth_splitmix64_next(uint64_t *state) {
  *state += SM64_GAMMA;
  return sm64_mix(*state);
}

uint16_t synth_f32_to_bf16(float f) { return f32_to_bf16_rne(f); }
