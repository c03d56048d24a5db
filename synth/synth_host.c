/*
 * synth_host.c -- host fills for the counter-based generator in synth.h.
 *
 * Build with -ffp-contract=off: the gs64 scale is defined with two separate
 * f32 roundings, and an FMA would change its bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "synth.h"

#define SYNTH_API __attribute__((visibility("default")))

SYNTH_API void synth_fill_int4(uint64_t seed, uint32_t layer, uint32_t tensor,
                               uint32_t expert, uint64_t start, uint64_t n_bytes,
                               uint8_t *out) {
  uint64_t s = synth_stream(seed, layer, tensor, expert);
  for (uint64_t i = 0; i < n_bytes; ++i) out[i] = synth_int4_byte(s, start + i);
}

SYNTH_API void synth_fill_scales(uint64_t seed, uint32_t layer, uint32_t tensor,
                                 uint32_t expert, uint64_t start, uint64_t n,
                                 float *out) {
  uint64_t s = synth_stream(seed, layer, tensor, expert);
  for (uint64_t i = 0; i < n; ++i) {
    volatile float t = 0.015f * synth_u24(s, start + i);
    out[i] = 0.005f + t;
  }
}

static double synth_normal(uint64_t s, uint64_t i) {
  uint64_t h1 = synth_draw(s, 2 * i), h2 = synth_draw(s, 2 * i + 1);
  double u1 = ((double)(h1 >> 11) + 1.0) * (1.0 / 9007199254740992.0); /* (0,1] */
  double u2 = (double)(h2 >> 11) * (1.0 / 9007199254740992.0);         /* [0,1) */
  return sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2);
}

SYNTH_API void synth_fill_normal_f32(uint64_t seed, uint32_t layer, uint32_t tensor,
                                     uint32_t expert, uint64_t start, uint64_t n,
                                     double sigma, float *out) {
  uint64_t s = synth_stream(seed, layer, tensor, expert);
  for (uint64_t i = 0; i < n; ++i) out[i] = (float)(sigma * synth_normal(s, start + i));
}

/* f32 -> bf16, round to nearest even (inputs here are finite). */
static uint16_t synth_bf16_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

SYNTH_API void synth_fill_normal_bf16(uint64_t seed, uint32_t layer, uint32_t tensor,
                                      uint32_t expert, uint64_t start, uint64_t n,
                                      double sigma, uint16_t *out) {
  uint64_t s = synth_stream(seed, layer, tensor, expert);
  for (uint64_t i = 0; i < n; ++i)
    out[i] = synth_bf16_rne((float)(sigma * synth_normal(s, start + i)));
}

SYNTH_API uint64_t synth_draw_at(uint64_t seed, uint32_t layer, uint32_t tensor,
                                 uint32_t expert, uint64_t i) {
  return synth_draw(synth_stream(seed, layer, tensor, expert), i);
}
