/*
 * synth.h -- counter-based generator for the seeded synthetic MoE-layer inputs.
 *
 * This module produces INPUTS only (activations, router weights, biases, packed
 * int4 expert weights and their gs64 scales).  It holds none of the layer's
 * arithmetic and is the one piece shared by the oracle and the CUDA path.
 *
 * Every value is a pure function of (seed, layer, tensor id, expert, index):
 *
 *   mix64(z)      SplitMix64 output function (Steele, Lea & Flood, "Fast
 *                 splittable pseudorandom number generators", OOPSLA 2014):
 *                 z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
 *                 z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31.
 *   stream(...)   = mix64(mix64(mix64(seed*G + 0x5EED) ^ (layer<<32 | tensor)) + expert*G)
 *   draw(s, i)    = mix64(s + (i+1)*G),   G = 0x9E3779B97F4A7C15 (SplitMix64 increment)
 *
 * Derived values (all integer or exactly-rounded f32 arithmetic, so host and
 * device produce identical bits):
 *   packed int4 byte b   = bits 56..63 of draw(s, b): low nibble = bits 56..59,
 *                          high nibble = bits 60..63 (two's-complement nibbles,
 *                          uniform on [-8, 7]; even K index in the low nibble)
 *   gs64 scale j         = fl32(0.005f + fl32(0.015f * u)),  u = (draw(s,j) >> 40) * 2^-24
 *                          (two separate roundings, never an FMA)
 *   normal i             = Box-Muller in f64 on draws 2i and 2i+1, times sigma,
 *                          then rounded to f32 (and to bf16 by RNE where asked)
 *
 * The header is plain C99; when compiled by nvcc the functions are also
 * available on the device.
 */
#ifndef SYNTH_H
#define SYNTH_H

#include <stdint.h>

#if defined(__CUDACC__)
#define SYNTH_HD __host__ __device__ __forceinline__
#else
#define SYNTH_HD static inline
#endif

#define SYNTH_GOLDEN 0x9E3779B97F4A7C15ULL

/* Tensor ids used in stream(). */
enum {
  SYNTH_T_X = 1,        /* activations x[T][H]; "expert" = rejection attempt  */
  SYNTH_T_WR = 2,       /* router weights Wr[H][E]                            */
  SYNTH_T_BIAS = 3,     /* router bias b[E]                                   */
  SYNTH_T_W1Q = 4,
  SYNTH_T_W1S = 5,
  SYNTH_T_W3Q = 6,
  SYNTH_T_W3S = 7,
  SYNTH_T_W2Q = 8,
  SYNTH_T_W2S = 9
};

/* Expert id used for the always-on shared expert's weight streams. */
#define SYNTH_SHARED_EXPERT 0xFFFFFFFFu

SYNTH_HD uint64_t synth_mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

SYNTH_HD uint64_t synth_stream(uint64_t seed, uint32_t layer, uint32_t tensor,
                               uint32_t expert) {
  uint64_t s = synth_mix64(seed * SYNTH_GOLDEN + 0x5EEDULL);
  s = synth_mix64(s ^ (((uint64_t)layer << 32) | (uint64_t)tensor));
  s = synth_mix64(s + (uint64_t)expert * SYNTH_GOLDEN);
  return s;
}

SYNTH_HD uint64_t synth_draw(uint64_t stream, uint64_t i) {
  return synth_mix64(stream + (i + 1ULL) * SYNTH_GOLDEN);
}

SYNTH_HD uint8_t synth_int4_byte(uint64_t stream, uint64_t b) {
  return (uint8_t)(synth_draw(stream, b) >> 56);
}

/* 24-bit uniform on [0, 1): exact in f32. */
SYNTH_HD float synth_u24(uint64_t stream, uint64_t j) {
  return (float)(uint32_t)(synth_draw(stream, j) >> 40) * (1.0f / 16777216.0f);
}

#endif /* SYNTH_H */
