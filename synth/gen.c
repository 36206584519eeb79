/*
 * Seeded synthetic input generator (test and benchmark infrastructure).
 *
 * Holds none of the MoE block's arithmetic: it only draws numbers.  Both the
 * CPU oracle and the CUDA path consume what it writes, so neither depends on
 * the other for its inputs.
 *
 * Generator: SplitMix64 used as a counter-based generator (Steele, Lea and
 * Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014).
 * Element n of stream s under seed S is mix64(key(S, s) + (n + 1) * GAMMA),
 * where mix64 is the SplitMix64 output finaliser and
 * key(S, s) = mix64(S * GAMMA ^ (s * STREAM_MULT)).  Every element is a pure
 * function of (S, s, n), so the output does not depend on the thread count or
 * on the sizes of other tensors.
 *
 * Normals: Box-Muller (Box and Muller 1958) from the two 32-bit halves of one
 * 64-bit draw, cosine branch only, computed in double.
 *
 * bf16: round-to-nearest-even of the fp32 value (the value is first rounded
 * from double to fp32).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>

#define GAMMA 0x9E3779B97F4A7C15ULL
#define STREAM_MULT 0xD1B54A32D192ED03ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t stream_key(uint64_t seed, uint64_t stream) {
  return mix64(seed * GAMMA ^ (stream * STREAM_MULT));
}

static inline uint64_t draw(uint64_t key, uint64_t n) {
  return mix64(key + (n + 1) * GAMMA);
}

static inline double normal_of(uint64_t z) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = ((double)(z >> 32) + 0.5) * (1.0 / 4294967296.0);
  double u2 = ((double)(z & 0xFFFFFFFFULL) + 0.5) * (1.0 / 4294967296.0);
  return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

static inline uint16_t f32_to_bf16_rne(float f) {
  union { float f; uint32_t u; } v;
  v.f = f;
  uint32_t u = v.u;
  if ((u & 0x7F800000u) == 0x7F800000u) {  /* inf / nan: keep, quiet nan */
    return (uint16_t)((u >> 16) | ((u & 0x007FFFFFu) ? 0x40u : 0u));
  }
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7FFFu + lsb;
  return (uint16_t)(u >> 16);
}

/* out[i] = bf16(std * N(0,1)) for i in [0, n): element index offset + i. */
void synth_normal_bf16(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double std, uint16_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    double v = std * normal_of(draw(key, offset + (uint64_t)i));
    out[i] = f32_to_bf16_rne((float)v);
  }
}

/* out[i] = fp32(std * N(0,1)). */
void synth_normal_f32(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                      double std, float* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    out[i] = (float)(std * normal_of(draw(key, offset + (uint64_t)i)));
  }
}

/* out[i] = uniform in [0, 1) with 53 random bits. */
void synth_uniform_f64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n,
                       double* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    out[i] = (double)(draw(key, offset + (uint64_t)i) >> 11) * (1.0 / 9007199254740992.0);
  }
}

/* Raw 64-bit draws (for permutations). */
void synth_u64(uint64_t seed, uint64_t stream, uint64_t offset, int64_t n, uint64_t* out) {
  uint64_t key = stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = draw(key, offset + (uint64_t)i);
}

/* bf16 -> fp32 widening (exact), for host-side consumers. */
void synth_bf16_to_f32(const uint16_t* in, int64_t n, float* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) {
    union { uint32_t u; float f; } v;
    v.u = ((uint32_t)in[i]) << 16;
    out[i] = v.f;
  }
}
