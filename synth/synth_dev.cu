// synth_dev.cu -- device fills for the counter-based generator in synth.h.
//
// Used to create the large packed-int4 expert weights and their gs64 scales
// directly in HBM (a 256-expert layer holds 5.5 GB of them).  The bits are the
// ones synth_host.c produces: integer hashing, and the scale's two roundings
// taken with explicit round-to-nearest intrinsics so no FMA is formed.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth.h"

namespace {

// Fills n_experts consecutive per-expert blocks of `per_expert` packed bytes.
// Each thread writes 16 bytes with one vector store.
__global__ void fill_int4_kernel(uint64_t seed, uint32_t layer, uint32_t tensor,
                                 uint32_t expert0, uint64_t per_expert,
                                 uint32_t n_experts, uint8_t *out) {
  const uint64_t chunks_per_expert = per_expert / 16;
  const uint64_t total = chunks_per_expert * n_experts;
  for (uint64_t c = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; c < total;
       c += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t e = (uint32_t)(c / chunks_per_expert);
    const uint64_t b0 = (c - (uint64_t)e * chunks_per_expert) * 16;
    const uint32_t eid = (expert0 == SYNTH_SHARED_EXPERT) ? expert0 : expert0 + e;
    const uint64_t s = synth_stream(seed, layer, tensor, eid);
    uint32_t w[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t v = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) v |= (uint32_t)synth_int4_byte(s, b0 + 4 * q + j) << (8 * j);
      w[q] = v;
    }
    *reinterpret_cast<uint4 *>(out + (uint64_t)e * per_expert + b0) =
        make_uint4(w[0], w[1], w[2], w[3]);
  }
}

__global__ void fill_scales_kernel(uint64_t seed, uint32_t layer, uint32_t tensor,
                                   uint32_t expert0, uint64_t per_expert,
                                   uint32_t n_experts, float *out) {
  const uint64_t total = per_expert * n_experts;
  for (uint64_t i = blockIdx.x * (uint64_t)blockDim.x + threadIdx.x; i < total;
       i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t e = (uint32_t)(i / per_expert);
    const uint64_t j = i - (uint64_t)e * per_expert;
    const uint32_t eid = (expert0 == SYNTH_SHARED_EXPERT) ? expert0 : expert0 + e;
    const uint64_t s = synth_stream(seed, layer, tensor, eid);
    out[i] = __fadd_rn(0.005f, __fmul_rn(0.015f, synth_u24(s, j)));
  }
}

}  // namespace

extern "C" {

// Returns 0, or a cudaError_t value.  per_expert must be a multiple of 16 and
// `out` 16-byte aligned.  expert0 == SYNTH_SHARED_EXPERT fills the shared
// expert (n_experts must then be 1).
__attribute__((visibility("default"))) int synth_dev_fill_int4(
    uint64_t seed, uint32_t layer, uint32_t tensor, uint32_t expert0,
    uint64_t per_expert, uint32_t n_experts, void *out, void *stream) {
  if (per_expert % 16 != 0 || ((uintptr_t)out & 15) != 0) return (int)cudaErrorInvalidValue;
  if (per_expert == 0 || n_experts == 0) return 0;
  fill_int4_kernel<<<152 * 8, 256, 0, (cudaStream_t)stream>>>(
      seed, layer, tensor, expert0, per_expert, n_experts, (uint8_t *)out);
  return (int)cudaGetLastError();
}

__attribute__((visibility("default"))) int synth_dev_fill_scales(
    uint64_t seed, uint32_t layer, uint32_t tensor, uint32_t expert0,
    uint64_t per_expert, uint32_t n_experts, void *out, void *stream) {
  if (per_expert == 0 || n_experts == 0) return 0;
  fill_scales_kernel<<<152 * 8, 256, 0, (cudaStream_t)stream>>>(
      seed, layer, tensor, expert0, per_expert, n_experts, (float *)out);
  return (int)cudaGetLastError();
}

}  // extern "C"
