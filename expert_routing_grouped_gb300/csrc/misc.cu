// misc.cu -- small kernels around the layer: the router-weight transpose done
// once at init, and the f32 RMS pre-norm used between stacked layers.
#include "moe_internal.cuh"

namespace moe {
namespace {

// dst[E][H] = src[H][E]^T, 32x32 tiles through shared memory.
__global__ void transpose_kernel(const float *__restrict__ src, float *__restrict__ dst, int H,
                                 int E) {
  __shared__ float tile[32][33];
  const int e0 = blockIdx.x * 32, h0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int hh = h0 + i, ee = e0 + threadIdx.x;
    if (hh < H && ee < E) tile[i][threadIdx.x] = src[(size_t)hh * E + ee];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int ee = e0 + i, hh = h0 + threadIdx.x;
    if (hh < H && ee < E) dst[(size_t)ee * H + hh] = tile[threadIdx.x][i];
  }
}

// out[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps)); the norm is computed in f32
// (the pages keep norms in f32: colibrì engine teardown, text-matrix.pages.dev,
// "System map").  One 1024-thread block per token, 16-byte loads, a fixed
// reduction order.
__global__ void __launch_bounds__(1024) rmsnorm_bf16_kernel(const float *__restrict__ x, int H,
                                                            float eps,
                                                            __nv_bfloat16 *__restrict__ out) {
  pdl_enter();
  __shared__ float part[32];
  const int t = blockIdx.x;
  const float4 *row = reinterpret_cast<const float4 *>(x + (size_t)t * H);
  const int n4 = H / 4;
  float4 v[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int i = threadIdx.x + r * 1024;
    v[r] = (i < n4) ? row[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  rmsnorm_row_bf16(row, v, H, eps, out + (size_t)t * H, part);
}

// Library weight layout, written once at init from the canonical layout.
//  * Nibbles: each 32-bit word holds K indices 8w..8w+7.  Canonical order puts
//    index 8w+j at bits 4j..4j+3 as two's complement; the library stores the
//    even indices 8w+0,2,4,6 at bits 0-3, 4-7, 8-11, 12-15 and the odd ones at
//    bits 16-19, 20-23, 24-27, 28-31, each as offset binary (value + 8), so a
//    single AND/OR with 0x000F000F / 0x43004300 on the word shifted by 4i gives
//    the bf16 pair (128 + q + 8) for indices (8w+2i, 8w+2i+1).
//  * W1/W3 rows are interleaved in 128-row blocks: block b holds features
//    64b..64b+63; its 32-row quadrant Q holds W1 rows of features 64b+16Q+0..15
//    then W3 rows of the same 16 features.  Scales follow the same row order.
__device__ __forceinline__ uint32_t repack_word(uint32_t w) {
  uint32_t out = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t nib = ((w >> (4 * j)) & 0xFu) ^ 0x8u;
    const int pos = (j & 1) ? 4 + (j >> 1) : (j >> 1);
    out |= nib << (4 * pos);
  }
  return out;
}

// W1 and W3 of n_exp experts ([n_exp][I][kb] bytes each) into the interleaved
// [n_exp][2I][kb] array, nibbles repacked; kb = bytes per row (multiple of 4).
__global__ void repack_w13_kernel(const uint8_t *__restrict__ w1, const uint8_t *__restrict__ w3,
                                  uint8_t *__restrict__ dst, long long n_exp, int I, int kb) {
  const long long words_per_row = kb / 4;
  const long long total = n_exp * 2LL * I * words_per_row;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const long long wi = i % words_per_row;
    long long r = i / words_per_row;                 // source row over [n_exp][2][I]
    const int f = (int)(r % I);
    r /= I;
    const int which = (int)(r % 2);
    const long long e = r / 2;
    const uint8_t *src = (which ? w3 : w1) + ((size_t)e * I + f) * kb;
    const uint32_t w = reinterpret_cast<const uint32_t *>(src)[wi];
    uint8_t *drow = dst + ((size_t)e * 2 * I + w13_row_of(f, which)) * kb;
    reinterpret_cast<uint32_t *>(drow)[wi] = repack_word(w);
  }
}

// Scales of W1/W3 into the interleaved row order ([n_exp][2I][groups]).
__global__ void repack_w13_scales_kernel(const float *__restrict__ s1, const float *__restrict__ s3,
                                         float *__restrict__ dst, long long n_exp, int I,
                                         int groups) {
  const long long total = n_exp * 2LL * I * groups;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(i % groups);
    long long r = i / groups;
    const int f = (int)(r % I);
    r /= I;
    const int which = (int)(r % 2);
    const long long e = r / 2;
    const float v = (which ? s3 : s1)[((size_t)e * I + f) * groups + g];
    dst[((size_t)e * 2 * I + w13_row_of(f, which)) * groups + g] = v;
  }
}

// Per-row power-of-two factor of the tensor-core path's fp16 weights:
// out[r] = 2^(8 - e) with max_g |s[r][g]| < 2^e, so every |q * s * out[r]| < 2^11
// and the row's largest scale sits in [2^7, 2^8): well inside fp16's range
// whatever the model's scale magnitudes.  One warp per row.
__global__ void row_pow2_kernel(const float *__restrict__ s, long long n_rows, int groups,
                                float *__restrict__ out) {
  const long long nw = (long long)gridDim.x * blockDim.x / 32;
  const int lane = threadIdx.x & 31;
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; r < n_rows; r += nw) {
    float m = 0.f;
    for (int g = lane; g < groups; g += 32) m = fmaxf(m, fabsf(s[r * groups + g]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) {
      const int eb = (__float_as_int(m) >> 23) & 0xFF;
      const int e = m > 0.f ? (eb > 0 ? eb : 1) - 126 : 8;
      const int f = max(-126, min(126, 8 - e));
      out[r] = __int_as_float((f + 127) << 23);
    }
  }
}

// Largest Euclidean row norm of W1 (norms[0]) and of W3 (norms[1]) over the
// interleaved W13 rows [n_rows][kb] (offset-binary nibbles) and their scales
// [n_rows][kb/32]; norms are raised with an integer max (non-negative floats
// order as their bits), so the result does not depend on the order of rows.
// One warp per row.
__global__ void w13_norm_kernel(const uint8_t *__restrict__ q, const float *__restrict__ s,
                                long long n_rows, int kb, float *__restrict__ norms) {
  const long long nw = (long long)gridDim.x * blockDim.x / 32;
  const int lane = threadIdx.x & 31;
  const int groups = kb / 32;
  for (long long r = (blockIdx.x * (long long)blockDim.x + threadIdx.x) / 32; r < n_rows; r += nw) {
    float acc = 0.f;
    for (int g = lane; g < groups; g += 32) {
      const uint32_t *wq = reinterpret_cast<const uint32_t *>(q + r * kb + (size_t)g * 32);
      int sq = 0;
      for (int i = 0; i < 8; ++i) {
        const uint32_t w = wq[i];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int v = (int)((w >> (4 * j)) & 0xFu) - 8;
          sq += v * v;
        }
      }
      const float sc = s[r * groups + g];
      acc = fmaf((float)sq * sc, sc, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      const int is_w3 = (r & 31) >= 16;   // the interleaved layout's quadrant halves
      atomicMax(reinterpret_cast<int *>(norms) + is_w3, __float_as_int(sqrtf(acc)));
    }
  }
}

// In-place nibble repack of a plain [rows][kb] array (W2).
__global__ void repack_words_kernel(uint32_t *__restrict__ w, long long n_words) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_words;
       i += (long long)gridDim.x * blockDim.x)
    w[i] = repack_word(w[i]);
}

}  // namespace

cudaError_t launch_repack_w13(const uint8_t *w1, const uint8_t *w3, uint8_t *dst, long long n_exp,
                              int I, int kb, cudaStream_t s) {
  return launch_k(false, repack_w13_kernel, dim3(152 * 8), dim3(256), 0, s, w1, w3, dst, n_exp, I,
                  kb);
}

cudaError_t launch_repack_w13_scales(const float *s1, const float *s3, float *dst, long long n_exp,
                                     int I, int groups, cudaStream_t s) {
  return launch_k(false, repack_w13_scales_kernel, dim3(152 * 8), dim3(256), 0, s, s1, s3, dst,
                  n_exp, I, groups);
}

cudaError_t launch_repack_words(uint8_t *w, long long n_bytes, cudaStream_t s) {
  return launch_k(false, repack_words_kernel, dim3(152 * 8), dim3(256), 0, s,
                  reinterpret_cast<uint32_t *>(w), n_bytes / 4);
}

cudaError_t launch_row_pow2(const float *s, long long n_rows, int groups, float *out,
                            cudaStream_t st) {
  return launch_k(false, row_pow2_kernel, dim3(152 * 4), dim3(256), 0, st, s, n_rows, groups, out);
}

cudaError_t launch_w13_norm(const uint8_t *q, const float *s, long long n_rows, int kb,
                            float *norms, cudaStream_t st) {
  return launch_k(false, w13_norm_kernel, dim3(152 * 4), dim3(256), 0, st, q, s, n_rows, kb, norms);
}

cudaError_t launch_transpose_router(const float *src, float *dst, int H, int E, cudaStream_t s) {
  const dim3 grid((E + 31) / 32, (H + 31) / 32), block(32, 8);
  return launch_k(false, transpose_kernel, grid, block, 0, s, src, dst, H, E);
}

cudaError_t launch_rmsnorm_bf16(const float *x, int T, int H, float eps, uint16_t *out,
                                cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_k(false, rmsnorm_bf16_kernel, dim3(T), dim3(1024), 0, s, x, H, eps,
                  reinterpret_cast<__nv_bfloat16 *>(out));
}

}  // namespace moe
