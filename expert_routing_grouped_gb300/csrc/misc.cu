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
// "System map").  One block per token; fixed reduction order.
__global__ void __launch_bounds__(256) rmsnorm_bf16_kernel(const float *__restrict__ x, int H,
                                                           float eps,
                                                           __nv_bfloat16 *__restrict__ out) {
  __shared__ float part[8];
  const int t = blockIdx.x;
  const float *row = x + (size_t)t * H;
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) ss = fmaf(row[i], row[i], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += part[w];
  const float r = 1.0f / sqrtf(tot / (float)H + eps);
  for (int i = threadIdx.x; i < H; i += blockDim.x)
    out[(size_t)t * H + i] = __float2bfloat16_rn(row[i] * r);
}

}  // namespace

cudaError_t launch_transpose_router(const float *src, float *dst, int H, int E, cudaStream_t s) {
  const dim3 grid((E + 31) / 32, (H + 31) / 32), block(32, 8);
  transpose_kernel<<<grid, block, 0, s>>>(src, dst, H, E);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bf16(const float *x, int T, int H, float eps, uint16_t *out,
                                cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  rmsnorm_bf16_kernel<<<T, 256, 0, s>>>(x, H, eps, reinterpret_cast<__nv_bfloat16 *>(out));
  return cudaGetLastError();
}

}  // namespace moe
