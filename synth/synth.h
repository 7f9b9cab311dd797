/*
 * synth.h -- seeded, counter-based synthetic input generator.
 *
 * This module produces the inputs of the optimizer step (replica gradients,
 * parameters, optimizer state) for the tests, the benchmark and the CPU
 * oracle.  It holds none of the optimizer's arithmetic: no reduction, no
 * scaling by a loss scale, no rounding of fp32 to a 16-bit type (inputs in a
 * 16-bit type are made by TRUNCATING the bit pattern, an integer operation),
 * no norm, no Adam.  The same definition compiles for the host (plain C) and
 * for the device (CUDA), so a value drawn on the GPU is bit-identical to the
 * one drawn on the CPU for the same (seed, stream, step, replica, index).
 *
 * Definition
 *   mix(z)    : the splitmix64 output function (Steele, Lea & Flood, "Fast
 *               splittable pseudorandom number generators", OOPSLA 2014;
 *               constants as published in Vigna's splitmix64.c):
 *                 z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9
 *                 z = (z ^ (z >> 27)) * 0x94D049BB133111EB
 *                 z =  z ^ (z >> 31)
 *   key       : a chain of mix() over seed, stream, step and replica, each
 *               offset by a multiple of the golden gamma 0x9E3779B97F4A7C15.
 *   bits(i)   : mix(key + gamma * (i + 1)) for element index i.
 *   normal(i) : Irwin-Hall sum of the four 16-bit fields of bits(i), centred
 *               (an integer in [-131070, 131070], variance (2^32-1)/3), times a
 *               per-tensor fp32 factor = sigma / sqrt((2^32-1)/3).  The int to
 *               float conversion is exact (|c| < 2^24); the one fp32 multiply
 *               is round-to-nearest on both sides.  Tails are truncated at
 *               +-2*sqrt(3)*sigma, an approximation of a normal law.
 *   uniform(i): the top 24 bits of bits(i) times 2^-24 times scale, in [0, scale).
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>

#ifdef __CUDACC__
#define SYNTH_HD static __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#define SYNTH_GAMMA 0x9E3779B97F4A7C15ULL

/* Stream identifiers: which tensor of the step an input belongs to. */
enum {
  SYNTH_STREAM_GRAD = 1,   /* replica gradients                        */
  SYNTH_STREAM_PARAM = 2,  /* model parameters (initial master weights) */
  SYNTH_STREAM_EXP_AVG = 3,
  SYNTH_STREAM_EXP_AVG_SQ = 4,
  SYNTH_STREAM_AUX = 5
};

SYNTH_HD uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYNTH_HD uint64_t synth_key(uint64_t seed, uint32_t stream, uint32_t step,
                            uint32_t replica) {
  uint64_t k = synth_mix64(seed + SYNTH_GAMMA);
  k = synth_mix64(k + SYNTH_GAMMA * (1ULL + (uint64_t)stream));
  k = synth_mix64(k + SYNTH_GAMMA * (1ULL + (uint64_t)step));
  k = synth_mix64(k + SYNTH_GAMMA * (1ULL + (uint64_t)replica));
  return k;
}

SYNTH_HD uint64_t synth_bits(uint64_t key, uint64_t index) {
  return synth_mix64(key + SYNTH_GAMMA * (index + 1ULL));
}

/* Centred Irwin-Hall(4) over the four 16-bit fields: an integer in [-131070, 131070]. */
SYNTH_HD int32_t synth_ih4(uint64_t b) {
  int32_t s = (int32_t)(b & 0xFFFFu) + (int32_t)((b >> 16) & 0xFFFFu) +
              (int32_t)((b >> 32) & 0xFFFFu) + (int32_t)((b >> 48) & 0xFFFFu);
  return s - 131070;
}

SYNTH_HD float synth_fmul(float a, float b) {
#ifdef __CUDA_ARCH__
  return __fmul_rn(a, b); /* never contracted into an FMA by the caller */
#else
  return a * b;
#endif
}

SYNTH_HD float synth_normal(uint64_t key, uint64_t index, float factor) {
  return synth_fmul((float)synth_ih4(synth_bits(key, index)), factor);
}

SYNTH_HD float synth_uniform(uint64_t key, uint64_t index, float scale) {
  uint32_t top = (uint32_t)(synth_bits(key, index) >> 40); /* 24 bits */
  return synth_fmul(synth_fmul((float)top, 5.9604644775390625e-08f), scale);
}

/* ---- bit casts ---------------------------------------------------------- */
SYNTH_HD uint32_t synth_f32_to_bits(float x) {
#ifdef __CUDA_ARCH__
  return __float_as_uint(x);
#else
  union { float f; uint32_t u; } c;
  c.f = x;
  return c.u;
#endif
}
SYNTH_HD float synth_bits_to_f32(uint32_t u) {
#ifdef __CUDA_ARCH__
  return __uint_as_float(u);
#else
  union { float f; uint32_t u; } c;
  c.u = u;
  return c.f;
#endif
}

/*
 * Truncation (round toward zero) of a finite fp32 value to bfloat16: keep the
 * top 16 bits.  An input-shaping step of this generator only.
 */
SYNTH_HD uint16_t synth_bf16_trunc_bits(float x) {
  return (uint16_t)(synth_f32_to_bits(x) >> 16);
}
/* The fp32 value equal to that truncated bfloat16. */
SYNTH_HD float synth_bf16_trunc_value(float x) {
  return synth_bits_to_f32(synth_f32_to_bits(x) & 0xFFFF0000u);
}

/*
 * Truncation (round toward zero) of a finite fp32 value to IEEE binary16,
 * by integer operations: normal range keeps the top 10 mantissa bits, the
 * subnormal range keeps the multiples of 2^-24, magnitudes of 2^16 and above
 * saturate to 65504.  An input-shaping step of this generator only.
 */
SYNTH_HD uint16_t synth_f16_trunc_bits(float x) {
  uint32_t u = synth_f32_to_bits(x);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  int32_t e = (int32_t)((u >> 23) & 0xFFu) - 127;
  uint32_t m = u & 0x7FFFFFu;
  if (((u >> 23) & 0xFFu) == 0) return sign; /* zero / fp32 subnormal -> 0 */
  if (e > 15) return (uint16_t)(sign | 0x7BFFu);
  if (e >= -14) return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(m >> 13));
  {
    int32_t shift = -1 - e; /* 14 .. */
    if (shift >= 24) return sign;
    return (uint16_t)(sign | (uint16_t)((m | 0x800000u) >> shift));
  }
}
/* The fp32 value equal to that truncated binary16. */
SYNTH_HD float synth_f16_trunc_value(float x) {
  uint32_t u = synth_f32_to_bits(x);
  int32_t e = (int32_t)((u >> 23) & 0xFFu) - 127;
  if (((u >> 23) & 0xFFu) == 0) return synth_bits_to_f32(u & 0x80000000u);
  if (e > 15) return synth_bits_to_f32((u & 0x80000000u) | 0x477FE000u); /* 65504 */
  if (e >= -14) return synth_bits_to_f32(u & 0xFFFFE000u);
  {
    int32_t drop = 13 + (-14 - e); /* mantissa bits below 2^-24 */
    if (drop >= 24) return synth_bits_to_f32(u & 0x80000000u);
    return synth_bits_to_f32(u & ~((1u << drop) - 1u));
  }
}

#endif /* SYNTH_H */
