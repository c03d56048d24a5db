// gemv.cu -- steps 4-5 of the layer for small T (decode and MTP-verify
// batches): int4 gs64 dequant GEMV, f32 throughout.
//
// At small T the layer is bound by streaming the activated experts' packed
// weights from HBM (the pages' expert tier moves ~19 MB per expert: colibrì
// engine teardown, text-matrix.pages.dev, "System map").  Only experts that
// received tokens are read (Colibri C + cuBLASLt tutorial, cf-1.com, §3.3
// Step 4: skip empty experts).
//
//   gemv_w13:  h[p][n] = silu(W1[n] . x_t) * (W3[n] . x_t) for every grouped
//              position p of every active expert (and the shared expert),
//              silu(g) = g / (1 + e^-g).
//   gemv_w2:   out[t][o] = sum_j w[t][j] * (W2_{idx[t][j]}[o] . h[inv(t,j)])
//              + W2_shared[o] . h_shared[t], summed in slot order then the
//              shared expert -- the combine of tutorial §3.3 Step 5, fused,
//              one owner per output element, no atomics.
//
// Weights are read with 128-bit non-allocating loads; a lane's 16 bytes are 32
// consecutive weights, all inside one 64-wide scale group.
#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Exact int4 -> f32 for the 8 weights of one word of the library layout
// (K indices 8w+0,2,4,6 at bits 0-15, 8w+1,3,5,7 at bits 16-31, offset binary).
// A nibble at bits 4p..4p+3 (p <= 4) is OR-ed into the mantissa of 2^(23-4p),
// whose unit in the last place is then exactly 1, and the float minus
// (2^(23-4p) + 8) is the signed value.  Nibbles above bit 19 are shifted down
// by 12 first.  q[j] is the weight of K index 8w+j.
__device__ __forceinline__ void dequant8(uint32_t w, float q[8]) {
  const uint32_t v = w >> 12;
  q[0] = __uint_as_float((w & 0x0000000Fu) | 0x4B000000u) - 8388616.0f;  // 2^23 + 8
  q[2] = __uint_as_float((w & 0x000000F0u) | 0x49000000u) - 524296.0f;   // 2^19 + 8
  q[4] = __uint_as_float((w & 0x00000F00u) | 0x47000000u) - 32776.0f;    // 2^15 + 8
  q[6] = __uint_as_float((w & 0x0000F000u) | 0x45000000u) - 2056.0f;     // 2^11 + 8
  q[1] = __uint_as_float((w & 0x000F0000u) | 0x43000000u) - 136.0f;      // 2^7 + 8
  q[3] = __uint_as_float((v & 0x00000F00u) | 0x47000000u) - 32776.0f;
  q[5] = __uint_as_float((v & 0x0000F000u) | 0x45000000u) - 2056.0f;
  q[7] = __uint_as_float((v & 0x000F0000u) | 0x43000000u) - 136.0f;
}

// 32 activations starting at element k0 of row `row`, as f32.
__device__ __forceinline__ void load_x32(const void *x, int x_is_bf16, size_t row_off, int k0,
                                         float xv[32]) {
  if (x_is_bf16) {
    const uint4 *p = reinterpret_cast<const uint4 *>(
        reinterpret_cast<const __nv_bfloat16 *>(x) + row_off + k0);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 u = __ldg(p + i);
      const uint32_t ws[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        xv[8 * i + 2 * j] = __uint_as_float(ws[j] << 16);
        xv[8 * i + 2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
      }
    }
  } else {
    const float4 *p = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) +
                                                       row_off + k0);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = __ldg(p + i);
      xv[4 * i] = f.x;
      xv[4 * i + 1] = f.y;
      xv[4 * i + 2] = f.z;
      xv[4 * i + 3] = f.w;
    }
  }
}

__device__ __forceinline__ float dot32(const uint4 wq, const float xv[32]) {
  const uint32_t ws[4] = {wq.x, wq.y, wq.z, wq.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float q[8];
    dequant8(ws[i], q);
#pragma unroll
    for (int j = 0; j < 8; ++j) acc = fmaf(q[j], xv[8 * i + j], acc);
  }
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------------------
// W1/W3 + SwiGLU.  Block = 8 warps; an item is (active expert, 8 row pairs),
// one row pair (W1 row n, W3 row n) per warp, full K per warp.  Tokens of the
// expert are taken kGemvTokens at a time.
constexpr int W13_WARPS = 8;

__global__ void __launch_bounds__(256) gemv_w13_kernel(
    const void *__restrict__ x, int x_is_bf16, int T, int H, int k, int E, int I, int Is,
    int h_stride, ExpertWeights ex, ExpertWeights sh, const int32_t *__restrict__ active,
    const int32_t *__restrict__ n_active_p, const int32_t *__restrict__ offsets,
    const int32_t *__restrict__ perm, float *__restrict__ hbuf) {
  const int n_active = *n_active_p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int slabs_r = I / W13_WARPS, slabs_s = Is / W13_WARPS;
  // Routed experts first, then (if present, as the last active entry) the shared one.
  const int has_shared = (n_active > 0 && active[n_active - 1] == E) ? 1 : 0;
  const int n_routed = n_active - has_shared;
  const int items = n_routed * slabs_r + has_shared * slabs_s;
  const int A = T * k;
  const int chunks = H / 32;      // 16-byte chunks per row

  for (int item = blockIdx.x; item < items; item += gridDim.x) {
    int e, n;
    const uint8_t *q13;
    const float *s13;
    int p0, cnt;
    if (item < n_routed * slabs_r) {
      e = active[item / slabs_r];
      n = (item % slabs_r) * W13_WARPS + warp;
      q13 = ex.w13q + (size_t)e * 2 * I * (H / 2);
      s13 = ex.w13s + (size_t)e * 2 * I * (H / 64);
      p0 = offsets[e];
      cnt = offsets[e + 1] - p0;
    } else {
      e = E;
      n = (item - n_routed * slabs_r) * W13_WARPS + warp;
      q13 = sh.w13q;
      s13 = sh.w13s;
      p0 = A;
      cnt = T;
    }
    const size_t row1 = w13_row_of(n, 0), row3 = w13_row_of(n, 1);
    const uint8_t *r1 = q13 + row1 * (H / 2);
    const uint8_t *r3 = q13 + row3 * (H / 2);
    const float *rs1 = s13 + row1 * (H / 64);
    const float *rs3 = s13 + row3 * (H / 64);
    for (int b0 = 0; b0 < cnt; b0 += kGemvTokens) {
      const int nb = min(kGemvTokens, cnt - b0);
      size_t xoff[kGemvTokens];
#pragma unroll
      for (int i = 0; i < kGemvTokens; ++i) {
        const int p = p0 + b0 + min(i, nb - 1);
        const int t = (e < E) ? perm[p] / k : (p - A);
        xoff[i] = (size_t)t * H;
      }
      float g[kGemvTokens] = {}, u[kGemvTokens] = {};
      for (int c = lane; c < chunks; c += 32) {
        const uint4 w1 = ld_stream(r1 + (size_t)c * 16);
        const uint4 w3 = ld_stream(r3 + (size_t)c * 16);
        const float sc1 = __ldg(rs1 + (c >> 1)), sc3 = __ldg(rs3 + (c >> 1));
#pragma unroll
        for (int i = 0; i < kGemvTokens; ++i) {
          if (i < nb) {
            float xv[32];
            load_x32(x, x_is_bf16, xoff[i], c * 32, xv);
            g[i] = fmaf(sc1, dot32(w1, xv), g[i]);
            u[i] = fmaf(sc3, dot32(w3, xv), u[i]);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kGemvTokens; ++i) {
        if (i < nb) {
          const float gg = warp_sum(g[i]);
          const float uu = warp_sum(u[i]);
          if (lane == 0) {
            const float silu = gg / (1.0f + expf(-gg));
            hbuf[(size_t)(p0 + b0 + i) * h_stride + n] = silu * uu;
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// W2 + combine.  Block = 8 warps, one output row o per warp, all tokens.
__global__ void __launch_bounds__(256) gemv_w2_combine_kernel(
    int T, int H, int k, int E, int I, int Is, int n_shared, int h_stride, ExpertWeights ex,
    ExpertWeights sh, const int32_t *__restrict__ idx, const float *__restrict__ wts,
    const int32_t *__restrict__ inv, const float *__restrict__ hbuf, float *__restrict__ out,
    int accumulate) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int A = T * k;
  for (int o = blockIdx.x * 8 + warp; o < H; o += gridDim.x * 8) {
    for (int t = 0; t < T; ++t) {
      float acc = 0.f;
      for (int j = 0; j < k; ++j) {
        const int e = idx[t * k + j];
        const int p = inv[t * k + j];
        const uint8_t *r2 = ex.w2q + ((size_t)e * H + o) * (I / 2);
        const float *rs2 = ex.w2s + ((size_t)e * H + o) * (I / 64);
        const float *hp = hbuf + (size_t)p * h_stride;
        float part = 0.f;
        for (int c = lane; c < I / 32; c += 32) {
          const uint4 wq = ld_stream(r2 + (size_t)c * 16);
          float hv[32];
          load_x32(hp, 0, 0, c * 32, hv);
          part = fmaf(__ldg(rs2 + (c >> 1)), dot32(wq, hv), part);
        }
        acc = fmaf(wts[t * k + j], warp_sum(part), acc);
      }
      if (n_shared) {
        const uint8_t *r2 = sh.w2q + (size_t)o * (Is / 2);
        const float *rs2 = sh.w2s + (size_t)o * (Is / 64);
        const float *hp = hbuf + (size_t)(A + t) * h_stride;
        float part = 0.f;
        for (int c = lane; c < Is / 32; c += 32) {
          const uint4 wq = ld_stream(r2 + (size_t)c * 16);
          float hv[32];
          load_x32(hp, 0, 0, c * 32, hv);
          part = fmaf(__ldg(rs2 + (c >> 1)), dot32(wq, hv), part);
        }
        acc += warp_sum(part);
      }
      if (lane == 0) {
        float *dst = out + (size_t)t * H + o;
        *dst = accumulate ? *dst + acc : acc;
      }
    }
  }
}

}  // namespace

cudaError_t launch_gemv_w13(const moe_handle *h, const void *x, int T, cudaStream_t st) {
  const int blocks = h->num_sms * 4;
  const int h_stride = h->I > h->Is ? h->I : h->Is;
  gemv_w13_kernel<<<blocks, 256, 0, st>>>(x, h->L.x_dtype == 1, T, h->H, h->k, h->E, h->I,
                                          h->S ? h->Is : W13_WARPS, h_stride, h->ex, h->sh,
                                          h->ws.active, h->ws.n_active, h->ws.offsets,
                                          h->ws.perm, h->ws.h);
  return cudaGetLastError();
}

cudaError_t launch_gemv_w2_combine(const moe_handle *h, int T, float *out, bool accumulate,
                                   cudaStream_t st) {
  const int h_stride = h->I > h->Is ? h->I : h->Is;
  int blocks = (h->H + 7) / 8;
  if (blocks > h->num_sms * 4) blocks = h->num_sms * 4;
  gemv_w2_combine_kernel<<<blocks, 256, 0, st>>>(T, h->H, h->k, h->E, h->I, h->Is, h->S,
                                                 h_stride, h->ex, h->sh, h->ws.idx, h->ws.w,
                                                 h->ws.inv, h->ws.h, out, accumulate ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace moe
