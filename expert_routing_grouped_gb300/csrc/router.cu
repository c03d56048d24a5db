// router.cu -- step 1-2 of the layer: f32 router logits, then top-k selection
// with renormalised weights.
//
// The router stays f32 (colibrì engine teardown, text-matrix.pages.dev,
// "System map": norm/router/bias are kept in f32 because they are small and
// sensitive).  Scoring is softmax (Colibri C + cuBLASLt tutorial, cf-1.com,
// §2.1 step 2) or sigmoid with a noaux_tc selection bias (n_group = 1, or
// group-limited with n_group > 1), scaled by routed_scaling_factor (teardown
// "Three key engineering decisions" (1)); softmax without renormalisation and
// an adaptive top-p trim are the variants the tuning guide names.
//
// Logits carry f32 rounding (plain f32 FMA here; for large T with bf16
// activations, tensor cores over three bf16 planes of the f32 weights, see
// ggemm_tc.cu) so the selection matches an exact reference whenever the top
// keys are separated by more than f32 rounding.  No TF32.
// Every reduction runs in a fixed order, so results are bitwise reproducible.
#include <algorithm>
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

// The router's selection rule, passed to the kernels by value.
struct RouteRule {
  int mode;         // 0 softmax, 1 sigmoid + noaux_tc, 2 softmax without renormalisation
  int n_group;      // > 1: group-limited selection (mode 1)
  int topk_group;   // groups kept
  float top_p;      // in (0, 1): adaptive top-p trim
  float rsf;
};

RouteRule route_rule(const moe_handle *h) {
  return RouteRule{h->L.router_mode, h->L.n_group, h->L.topk_group, h->L.top_p,
                   h->L.routed_scaling_factor};
}

__device__ __forceinline__ float load_x(const void *x, int x_is_bf16, size_t i) {
  if (x_is_bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(x)[i]);
  return reinterpret_cast<const float *>(x)[i];
}

// ---------------------------------------------------------------------------
// Small T (decode, MTP verify): split-K GEMV.  Block = 8 warps, one expert per
// warp; blockIdx.y selects a contiguous H range.  x of the range is staged in
// shared memory as f32.  Writes z_part[split][t][e].
//
// Every load of a thread is issued before its first use (x in 16-byte vectors;
// the router row in batches of kMaxRowVec float4 per lane), so the block pays
// one memory latency per phase rather than one per element.
constexpr int kMaxRowVec = 12;

template <int NT>
__device__ __forceinline__ void stage_x(const void *__restrict__ x, int x_is_bf16, int T, int H,
                                        int h0, int hps, float *xs) {
  constexpr int B = 4;   // vectors a thread loads before it converts and stores any
  if (x_is_bf16) {
    const int nv = hps / 8;                       // 8 bf16 per 16 bytes
    for (int i0 = threadIdx.x; i0 < NT * nv; i0 += B * blockDim.x) {
      uint4 u[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int i = i0 + b * blockDim.x;
        const int t = i / nv, c = i - t * nv;
        u[b] = make_uint4(0u, 0u, 0u, 0u);
        if (i < NT * nv && t < T)
          u[b] = __ldg(reinterpret_cast<const uint4 *>(
                           reinterpret_cast<const __nv_bfloat16 *>(x) + (size_t)t * H + h0) +
                       c);
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int i = i0 + b * blockDim.x;
        if (i < NT * nv) {
          const int t = i / nv, c = i - t * nv;
          const float4 lo = make_float4(__uint_as_float(u[b].x << 16),
                                        __uint_as_float(u[b].x & 0xFFFF0000u),
                                        __uint_as_float(u[b].y << 16),
                                        __uint_as_float(u[b].y & 0xFFFF0000u));
          const float4 hi = make_float4(__uint_as_float(u[b].z << 16),
                                        __uint_as_float(u[b].z & 0xFFFF0000u),
                                        __uint_as_float(u[b].w << 16),
                                        __uint_as_float(u[b].w & 0xFFFF0000u));
          reinterpret_cast<float4 *>(xs + t * hps)[2 * c] = lo;
          reinterpret_cast<float4 *>(xs + t * hps)[2 * c + 1] = hi;
        }
      }
    }
  } else {
    const int nv = hps / 4;
    for (int i0 = threadIdx.x; i0 < NT * nv; i0 += B * blockDim.x) {
      float4 v[B];
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int i = i0 + b * blockDim.x;
        const int t = i / nv, c = i - t * nv;
        v[b] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (i < NT * nv && t < T)
          v[b] = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) +
                                                        (size_t)t * H + h0) +
                       c);
      }
#pragma unroll
      for (int b = 0; b < B; ++b) {
        const int i = i0 + b * blockDim.x;
        if (i < NT * nv) {
          const int t = i / nv, c = i - t * nv;
          reinterpret_cast<float4 *>(xs + t * hps)[c] = v[b];
        }
      }
    }
  }
}

// The first batch of a warp's router-row loads, issued before the block stages
// x so the two memory round trips overlap.
__device__ __forceinline__ void row_prefetch(const float *__restrict__ wrow, int hps,
                                             float4 wv[kMaxRowVec]) {
  const int lane = threadIdx.x & 31;
  const int nv = hps / 128;
#pragma unroll
  for (int v = 0; v < kMaxRowVec; ++v)
    if (v < nv) wv[v] = __ldg(reinterpret_cast<const float4 *>(wrow + v * 128 + lane * 4));
}

// acc[t] = sum over this warp's H range of x[t][h] * wr_t[e][h], lanes reduced;
// wv holds the row's first kMaxRowVec float4 per lane (row_prefetch).
template <int NT>
__device__ __forceinline__ void row_dot(const float *__restrict__ wrow, const float *xs, int hps,
                                        float4 wv[kMaxRowVec], float acc[NT]) {
  const int lane = threadIdx.x & 31;
  const int nv = hps / 128;                       // float4 per lane
#pragma unroll
  for (int t = 0; t < NT; ++t) acc[t] = 0.f;
  for (int v0 = 0; v0 < nv; v0 += kMaxRowVec) {
    if (v0 > 0) {
#pragma unroll
      for (int v = 0; v < kMaxRowVec; ++v)
        if (v0 + v < nv)
          wv[v] = __ldg(reinterpret_cast<const float4 *>(wrow + (v0 + v) * 128 + lane * 4));
    }
#pragma unroll
    for (int v = 0; v < kMaxRowVec; ++v) {
      if (v0 + v < nv) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float4 xv =
              *reinterpret_cast<const float4 *>(xs + t * hps + (v0 + v) * 128 + lane * 4);
          acc[t] = fmaf(xv.x, wv[v].x, acc[t]);
          acc[t] = fmaf(xv.y, wv[v].y, acc[t]);
          acc[t] = fmaf(xv.z, wv[v].z, acc[t]);
          acc[t] = fmaf(xv.w, wv[v].w, acc[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < NT; ++t) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], o);
  }
}

template <int NT>
__global__ void __launch_bounds__(256) router_gemv_kernel(
    const void *__restrict__ x, int x_is_bf16, int T, int H, int E,
    const float *__restrict__ wr_t, int h_per_split, float *__restrict__ z_part,
    int zstride) {
  pdl_enter();
  extern __shared__ float xs[];   // [NT][h_per_split]
  const int split = blockIdx.y;
  const int h0 = split * h_per_split;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  float4 wv[kMaxRowVec];
  if (e < E) row_prefetch(wr_t + (size_t)e * H + h0, h_per_split, wv);
  stage_x<NT>(x, x_is_bf16, T, H, h0, h_per_split, xs);
  __syncthreads();
  if (e >= E) return;
  float acc[NT];
  row_dot<NT>(wr_t + (size_t)e * H + h0, xs, h_per_split, wv, acc);
  if (lane == 0) {
#pragma unroll
    for (int t = 0; t < NT; ++t)
      if (t < T) z_part[((size_t)split * zstride + t) * E + e] = acc[t];
  }
}

// ---------------------------------------------------------------------------
// Large T: tiled SIMT SGEMM, z[t][e] = sum_h x[t][h] * wr_t[e][h].
// Block tile 64 tokens x 64 experts, K step 16, 256 threads, 4x4 per thread.
constexpr int RG_BT = 64, RG_BE = 64, RG_BK = 16;

__global__ void __launch_bounds__(256) router_gemm_kernel(
    const void *__restrict__ x, int x_is_bf16, int T, int H, int E,
    const float *__restrict__ wr_t, float *__restrict__ z) {
  pdl_enter();
  __shared__ float xs[RG_BK][RG_BT + 4];
  __shared__ float ws[RG_BK][RG_BE + 4];
  const int t0 = blockIdx.y * RG_BT, e0 = blockIdx.x * RG_BE;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  // Split-K: this CTA's share of the H / RG_BK steps (gridDim.z splits), its
  // partial logits written to z[blockIdx.z][T][E].
  const int steps = H / RG_BK;
  const int ks0 = (int)((long long)steps * blockIdx.z / gridDim.z);
  const int ks1 = (int)((long long)steps * (blockIdx.z + 1) / gridDim.z);
  z += (size_t)blockIdx.z * T * E;
  float acc[4][4] = {};
  for (int k0 = ks0 * RG_BK; k0 < ks1 * RG_BK; k0 += RG_BK) {
    // 64 x 16 elements of each operand, 4 per thread.
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int i = threadIdx.x + r * 256;
      const int row = i >> 4, kk = i & 15;
      const int t = t0 + row, e = e0 + row;
      xs[kk][row] = (t < T) ? load_x(x, x_is_bf16, (size_t)t * H + k0 + kk) : 0.f;
      ws[kk][row] = (e < E) ? __ldg(wr_t + (size_t)e * H + k0 + kk) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < RG_BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = t0 + ty * 4 + i;
    if (t >= T) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = e0 + tx * 4 + j;
      if (e < E) z[(size_t)t * E + e] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------------------
// Top-k of one token by one warp; expert e lives in lane e % 32, slot e / 32.
// Keys: softmax modes, l = z + b; sigmoid mode, s = sigmoid(z), key = s + b.
// With groups (sigmoid mode, n_group > 1), each group's score is the sum of
// its two largest keys, and the keys of experts outside the topk_group best
// groups (ties to the lower group) drop to -inf before the selection.
// k rounds of a warp argmax (larger key first, lower id on ties) give the
// slots in descending key order.  Weights, times rsf: mode 0
// w_j = exp(l_j - l_0) / sum_sel exp(l_i - l_0); mode 2 the same numerator
// over the sum across all E experts; mode 1 w_j = s_j / sum_sel s_i.  Top-p
// keeps slot j while the shares of the slots before it sum below top_p (slot
// 0 always), gives the dropped slots id -1 and weight 0, and (modes 0 and 1)
// renormalises over the kept slots.  Split partial logits are summed in
// split order.  Every sum runs in a fixed order.

// Selection key and score of one expert from its logit zz and bias b.
__device__ __forceinline__ void key_of(float zz, float b, int mode, float &key, float &val) {
  if (mode != 1) {
    key = zz + b;
    val = key;
  } else {
    const float sc = 1.0f / (1.0f + expf(-zz));
    val = sc;
    key = sc + b;
  }
}

template <int EPL>
__device__ __forceinline__ void topk_select(float key[EPL], float val[EPL], int t, int E, int k,
                                            const RouteRule r, int32_t *__restrict__ idx_out,
                                            float *__restrict__ w_out);

template <int EPL>
__device__ __forceinline__ void topk_token(const float *__restrict__ z_part, int splits,
                                           int zstride, int t, int E, int k, const RouteRule r,
                                           const float *__restrict__ bias,
                                           int32_t *__restrict__ idx_out,
                                           float *__restrict__ w_out) {
  const int lane = threadIdx.x & 31;
  float key[EPL], val[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    key[i] = -INFINITY;
    val[i] = 0.f;
    if (e < E) {
      // Issue all split loads before summing (in split order).
      float part[kRouterSplitMax];
#pragma unroll
      for (int s = 0; s < kRouterSplitMax; ++s)
        part[s] = (s < splits) ? z_part[((size_t)s * zstride + t) * E + e] : 0.f;
      float zz = 0.f;
#pragma unroll
      for (int s = 0; s < kRouterSplitMax; ++s)
        if (s < splits) zz += part[s];
      key_of(zz, bias ? bias[e] : 0.f, r.mode, key[i], val[i]);
    }
  }
  topk_select<EPL>(key, val, t, E, k, r, idx_out, w_out);
}

// Group-limited selection (n_group > 1): lane g of the warp computes group g's
// score, the sum of its two largest keys; the keys of experts outside the
// topk_group best groups (ties to the lower group) drop to -inf.
template <int EPL>
__device__ __forceinline__ void group_mask(float key[EPL], int E, const RouteRule r) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int gsz = E / r.n_group;
  float my_gs = -INFINITY;
  for (int g = 0; g < r.n_group; ++g) {
    float a = -INFINITY, b2 = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e >= g * gsz && e < (g + 1) * gsz) {
        const float v = key[i];
        if (v > a) {
          b2 = a;
          a = v;
        } else if (v > b2) {
          b2 = v;
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {   // merge two top-2 lists
      const float oa = __shfl_xor_sync(full, a, o), ob = __shfl_xor_sync(full, b2, o);
      b2 = fmaxf(fminf(a, oa), fmaxf(b2, ob));
      a = fmaxf(a, oa);
    }
    if (lane == g) my_gs = a + b2;
  }
  int gkept = 0;   // lane g: group g is eligible
  for (int j = 0; j < r.topk_group; ++j) {
    float bv = gkept ? -INFINITY : my_gs;
    int bg = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(full, bv, o);
      const int og = __shfl_xor_sync(full, bg, o);
      if (ov > bv || (ov == bv && og < bg)) {
        bv = ov;
        bg = og;
      }
    }
    if (lane == bg) gkept = 1;
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    const int g = (e < E) ? e / gsz : 0;
    if (!__shfl_sync(full, gkept, g)) key[i] = -INFINITY;
  }
}

// The same selection as argmax_rounds for up to 8 candidates per lane, with
// each round's warp argmax done by the hardware reductions: the keys become
// order-preserving 32-bit integers (a NaN, and the padding past E, lowest;
// -0 as +0), each lane sorts its own
// (key, id, score) triples once, and a round is the warp maximum of the lanes'
// first keys (redux.sync max), then the lowest id among the lanes that hold
// it (redux.sync min) -- larger key first, lower id on ties.  The winning
// lane drops its first triple.  Lane j < k ends with slot j's expert and
// score.
__device__ __forceinline__ uint32_t order_bits(float f) {
  const uint32_t u = __float_as_uint(f);
  if (f != f) return 0u;
  if (f == 0.f) return 0x80000000u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
template <int EPL>
__device__ __forceinline__ void topk_redux(const float key[EPL], const float val[EPL], int E,
                                           int k, int &my_idx, float &my_val) {
  static_assert(EPL <= 8, "at most 8 candidates per lane");
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  uint32_t lb[8];   // this lane's candidates, first in order first
  int li[8];
  float lv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    lb[i] = (i < EPL && lane + 32 * i < E) ? order_bits(key[i % EPL]) : 0u;
    li[i] = i < EPL ? lane + 32 * i : 0x7fffffff;
    lv[i] = i < EPL ? val[i % EPL] : 0.f;
  }
  // bitonic sort of the 8 triples: larger key first, lower id on ties
#pragma unroll
  for (int size = 2; size <= 8; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const int a = ((i & size) == 0) ? i : j, b = ((i & size) == 0) ? j : i;
          const bool swap = lb[b] > lb[a] || (lb[b] == lb[a] && li[b] < li[a]);
          const uint32_t tb = lb[a];
          const int ti = li[a];
          const float tv = lv[a];
          lb[a] = swap ? lb[b] : lb[a];
          li[a] = swap ? li[b] : li[a];
          lv[a] = swap ? lv[b] : lv[a];
          lb[b] = swap ? tb : lb[b];
          li[b] = swap ? ti : li[b];
          lv[b] = swap ? tv : lv[b];
        }
      }
  my_idx = -1;
  my_val = 0.f;
#pragma unroll 8
  for (int j = 0; j < k; ++j) {
    const uint32_t m = __reduce_max_sync(full, lb[0]);
    const int win = (int)__reduce_min_sync(full, lb[0] == m ? (uint32_t)li[0] : 0x7fffffffu);
    const float v = __shfl_sync(full, lv[0], win & 31);
    if (lane == j) {
      my_idx = win;
      my_val = v;
    }
    const bool pop = li[0] == win;
#pragma unroll
    for (int i = 0; i < 7; ++i) {
      lb[i] = pop ? lb[i + 1] : lb[i];
      li[i] = pop ? li[i + 1] : li[i];
      lv[i] = pop ? lv[i + 1] : lv[i];
    }
    lb[7] = pop ? 0u : lb[7];
    li[7] = pop ? 0x7fffffff : li[7];
  }
}

// k rounds of a warp argmax (larger key first, lower id on ties): lane j < k
// ends with slot j's expert and score.
template <int EPL>
__device__ __forceinline__ void argmax_rounds(float key[EPL], const float val[EPL], int k,
                                              int &my_idx, float &my_val) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  my_idx = -1;
  my_val = 0.f;
  for (int j = 0; j < k; ++j) {
    float bk = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (key[i] > bk) {   // ascending i: first maximum has the lowest id
        bk = key[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ok = __shfl_xor_sync(full, bk, o);
      const int oe = __shfl_xor_sync(full, be, o);
      if (ok > bk || (ok == bk && oe < be)) {
        bk = ok;
        be = oe;
      }
    }
    // Owner removes the winner and broadcasts its value.
    float v = 0.f;
    if ((be & 31) == lane) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i == be) {
          v = val[i];
          key[i] = -INFINITY;
        }
    }
    v = __shfl_sync(full, v, be & 31);
    if (lane == j) {
      my_idx = be;
      my_val = v;
    }
  }
}

// Weights of the k slots (lane j < k holds slot j's expert and score), the
// top-p trim, and the writes of token t's ids and weights.  val holds every
// expert's score (mode 2 divides by the sum over all of them).  sidx (or
// nullptr) also receives the ids.
template <int EPL>
__device__ __forceinline__ void slot_weights(int my_idx, float my_val, const float val[EPL], int t,
                                             int E, int k, const RouteRule r,
                                             int32_t *__restrict__ idx_out,
                                             float *__restrict__ w_out, int *sidx) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  // Numerators, and the sum over the selection in slot order.
  const float top = __shfl_sync(full, my_val, 0);
  float num = 0.f;
  if (lane < k) num = (r.mode != 1) ? expf(my_val - top) : my_val;
  float den = 0.f;
#pragma unroll 8
  for (int j = 0; j < k; ++j) den += __shfl_sync(full, num, j);
  // Mode 2 divides by the sum over all experts (xor-butterfly: the same bits
  // on every lane).
  float all = 0.f;
  if (r.mode == 2) {
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (lane + 32 * i < E) all += expf(val[i] - top);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) all += __shfl_xor_sync(full, all, o);
  }
  int kept = k;
  float norm = den;
  if (r.top_p > 0.f && r.top_p < 1.f) {
    float cum = 0.f;
    for (int j = 1; j < k; ++j) {
      cum += __shfl_sync(full, num, j - 1) / den;
      if (kept == k && cum >= r.top_p) kept = j;
    }
    norm = 0.f;
    for (int j = 0; j < kept; ++j) norm += __shfl_sync(full, num, j);
  }
  if (lane < k) {
    const bool keep = lane < kept;
    idx_out[(size_t)t * k + lane] = keep ? my_idx : -1;
    w_out[(size_t)t * k + lane] = keep ? num / (r.mode == 2 ? all : norm) * r.rsf : 0.f;
    if (sidx) sidx[t * k + lane] = keep ? my_idx : -1;
  }
}

// The selection of topk_token from the token's keys and scores (expert e in
// lane e % 32, slot e / 32; -inf keys past E).
template <int EPL>
__device__ __forceinline__ void topk_select(float key[EPL], float val[EPL], int t, int E, int k,
                                            const RouteRule r, int32_t *__restrict__ idx_out,
                                            float *__restrict__ w_out) {
  if (r.n_group > 1) group_mask<EPL>(key, E, r);
  int my_idx;
  float my_val;
  if constexpr (EPL <= 8)
    topk_redux<EPL>(key, val, E, k, my_idx, my_val);
  else
    argmax_rounds<EPL>(key, val, k, my_idx, my_val);
  slot_weights<EPL>(my_idx, my_val, val, t, E, k, r, idx_out, w_out, nullptr);
}

template <int EPL>
__global__ void __launch_bounds__(256, 1) router_topk_kernel(
    const float *__restrict__ z_part, int splits, int zstride, int T, int E, int k,
    const RouteRule r, const float *__restrict__ bias, int32_t *__restrict__ idx_out,
    float *__restrict__ w_out) {
  pdl_enter();
  z_part = after_wait(z_part);
  idx_out = after_wait(idx_out);
  w_out = after_wait(w_out);
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  topk_token<EPL>(z_part, splits, zstride, t, E, k, r, bias, idx_out, w_out);
}

// ---------------------------------------------------------------------------
// T <= kRouteTokens in one launch: the split-K router GEMV of
// router_gemv_kernel, then self-resetting atomic tickets (nothing waits): for
// T > 1 the last split CTA of each 8-expert block sums that block's partials
// into keys and scores, and the last block to finish loads them; for T = 1
// the last CTA of the grid sums every partial itself.  That CTA takes the
// top-k of each token and groups the T*k assignments by expert -- the stable
// counting sort of dispatch.cu, written out from ranks.  It also clears the
// status word.
template <int EPL, int NT>
__global__ void __launch_bounds__(256) route_small_kernel(
    const void *__restrict__ x, int x_is_bf16, int T, int H, int E, int k, const RouteRule r,
    const float *__restrict__ wr_t, const float *__restrict__ bias, int h_per_split,
    float *__restrict__ z_part, int32_t *__restrict__ ticket, float *__restrict__ route_kv,
    int n_shared,
    int32_t *__restrict__ idx, float *__restrict__ w, int32_t *__restrict__ counts,
    int32_t *__restrict__ offsets, int32_t *__restrict__ perm, int32_t *__restrict__ inv,
    int32_t *__restrict__ active, int32_t *__restrict__ n_active, int32_t *__restrict__ tiles,
    int32_t *__restrict__ n_tiles, int32_t *__restrict__ status,
    unsigned long long *__restrict__ usage) {
  extern __shared__ float xs[];   // [NT][h_per_split]
  __shared__ int last;
  pdl_enter();
  const int split = blockIdx.y;
  const int h0 = split * h_per_split;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  float4 wv[kMaxRowVec];
  if (e < E) row_prefetch(wr_t + (size_t)e * H + h0, h_per_split, wv);
  stage_x<NT>(x, x_is_bf16, T, H, h0, h_per_split, xs);
  __syncthreads();
  if (e < E) {
    float acc[NT];
    row_dot<NT>(wr_t + (size_t)e * H + h0, xs, h_per_split, wv, acc);
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if (t < T) z_part[((size_t)split * NT + t) * E + e] = acc[t];
    }
  }
  // Last-CTA-done.  For more than one token, two levels: the last split CTA
  // of each 8-expert block sums the block's partials in split order (read
  // through L2: other CTAs wrote them) and writes its keys and scores, and the
  // last block to finish takes the top-k and groups.  For one token the extra
  // round trip costs more than it saves: the last CTA of the whole grid sums
  // every partial itself.  The tickets reset themselves for the next call;
  // nothing waits.
  const int splits = gridDim.y;
  float *kg = route_kv, *vg = route_kv + kRouteTokens * E;   // [T][E] keys, scores
  __threadfence();
  __syncthreads();
  if (T > 1) {
    if (threadIdx.x == 0) {
      last = (atomicAdd(ticket + 1 + blockIdx.x, 1) == splits - 1);
      if (last) ticket[1 + blockIdx.x] = 0;
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    if ((int)threadIdx.x < T * 8) {
      const int t = threadIdx.x >> 3, eb = blockIdx.x * 8 + (threadIdx.x & 7);
      if (eb < E) {
        const float b = bias ? __ldg(bias + eb) : 0.f;
        float part[kRouterSplitMax];
#pragma unroll
        for (int sp = 0; sp < kRouterSplitMax; ++sp)
          part[sp] = sp < splits ? __ldcg(z_part + ((size_t)sp * NT + t) * E + eb) : 0.f;
        float zz = 0.f;
#pragma unroll
        for (int sp = 0; sp < kRouterSplitMax; ++sp)
          if (sp < splits) zz += part[sp];
        key_of(zz, b, r.mode, kg[t * E + eb], vg[t * E + eb]);
      }
    }
    __threadfence();
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int n = T > 1 ? (int)gridDim.x : (int)(gridDim.x * gridDim.y);
    last = (atomicAdd(ticket, 1) == n - 1);
    if (last) *ticket = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x == 0) *status = kStatusOk;
  // Every (token, expert) key and score into shared memory; a batch's loads
  // are all issued before its stores or sums.
  float *ks = xs, *vs = xs + T * E;
  if (T > 1) {
    constexpr int U = 8;
    for (int i0 = threadIdx.x; i0 < T * E; i0 += U * blockDim.x) {
      float a[U], b[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * blockDim.x;
        a[u] = i < T * E ? __ldcg(kg + i) : 0.f;
        b[u] = i < T * E ? __ldcg(vg + i) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * blockDim.x;
        if (i < T * E) {
          ks[i] = a[u];
          vs[i] = b[u];
        }
      }
    }
  } else {
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
      const float b = bias ? __ldg(bias + e) : 0.f;
      float part[kRouterSplitMax];
#pragma unroll
      for (int sp = 0; sp < kRouterSplitMax; ++sp)
        part[sp] = sp < splits ? __ldcg(z_part + (size_t)sp * NT * E + e) : 0.f;
      float zz = 0.f;
#pragma unroll
      for (int sp = 0; sp < kRouterSplitMax; ++sp)
        if (sp < splits) zz += part[sp];
      key_of(zz, b, r.mode, ks[e], vs[e]);
    }
  }
  __syncthreads();
  // Top-k, weights and the top-p trim: warp t for token t (T <= 8 warps).
  const int A = T * k;
  int *sidx = reinterpret_cast<int *>(vs + T * E);   // [A] ids after the top-p trim
  int *sg = sidx + A;                                // [A] 2 id + (first of its expert)
  if (warp < T) {
    float key[EPL], val[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? ks[warp * E + e] : -INFINITY;
      val[i] = e < E ? vs[warp * E + e] : 0.f;
    }
    if (r.n_group > 1) group_mask<EPL>(key, E, r);
    int my_idx;
    float my_val;
    if constexpr (EPL <= 8)
      topk_redux<EPL>(key, val, E, k, my_idx, my_val);
    else
      argmax_rounds<EPL>(key, val, k, my_idx, my_val);
    slot_weights<EPL>(my_idx, my_val, val, warp, E, k, r, idx, w, sidx);
  }
  __syncthreads();
  // Stable grouping of the A = T*k assignments by expert, the result of the
  // counting sort written out from ranks: assignment a goes to position
  // (assignments to smaller experts) + (earlier assignments to its expert).
  // Slots top-p dropped (-1) are left out; any other id outside [0, E) sets
  // the bad-expert status and is left out too.
  for (int a = threadIdx.x; a < A; a += blockDim.x) {
    const int ea = sidx[a];
    const bool ok = ea >= 0 && ea < E;
    int before = 0, same = 0;
#pragma unroll 8
    for (int b = 0; b < A; ++b) {
      const int eb = sidx[b];
      before += ((uint32_t)eb < (uint32_t)ea) ? 1 : 0;   // ids below 0 do not count
      same += (b < a && eb == ea) ? 1 : 0;
    }
    sg[a] = 2 * ea + ((ok && same == 0) ? 1 : 0);
    if (ok) {
      perm[before + same] = a;
      inv[a] = before + same;
    } else {
      inv[a] = -1;
      if (ea != -1) atomicExch(status, kStatusBadExpert);
    }
  }
  __syncthreads();
  // Per expert: its count, its first position, its place in the active list
  // (ascending ids, the shared expert last, one token block each); expert
  // E - 1 also writes the totals.
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int c = 0, below = 0, dist = 0;
#pragma unroll 8
    for (int b = 0; b < A; ++b) {
      const int v = sg[b];
      const int eb = v >> 1;
      const int lt = ((uint32_t)eb < (uint32_t)e) ? 1 : 0;   // ids below 0 do not count
      c += (eb == e) ? 1 : 0;
      below += lt;
      dist += lt & v;
    }
    counts[e] = c;
    offsets[e] = below;
    if (usage && c) usage[e] += (unsigned long long)c;
    if (c > 0) {
      active[dist] = e;
      tiles[dist] = e << 16;
    }
    if (e == E - 1) {
      offsets[E] = below + c;
      int na = dist + (c > 0 ? 1 : 0);
      if (n_shared) {
        active[na] = E;
        tiles[na] = E << 16;
        ++na;
      }
      *n_active = na;
      n_tiles[0] = na;
    }
  }
}

// Split-K partitions of the GEMV router over H (T <= 4 on the route-only
// path; any T <= kRouteTokens in the fused routing launch).
int gemv_splits(int E, int H, int num_sms) {
  const int blocks_e = (E + 7) / 8;
  int s = 1;
  // Split H until the grid covers the SMs once (two blocks fit per SM, so the
  // grid stays one wave and the last block to finish -- which does the top-k
  // and the grouping -- starts early), keeping 128-float slices.
  while (s < kRouterSplitMax && blocks_e * s < num_sms && (H % (2 * s * 128)) == 0) s *= 2;
  return s;
}

int router_splits(int T, int E, int H, int num_sms) {
  return T > 4 ? 1 : gemv_splits(E, H, num_sms);
}

// Split-K partitions of the batched routers (T > 4): a grid of `base` CTAs
// (expert tiles x token tiles) is split over K until it covers the SMs, for
// batches of up to kRouterSplitTokens tokens (the partials' buffer holds
// kRouterSplitMax of those), each split keeping at least `min_steps` K steps.
int batched_router_splits(int T, int base, int k_steps, int min_steps, int num_sms) {
  int s = 1;
  if (T > kRouterSplitTokens) return 1;
  while (s < kRouterSplitMax && base * s < num_sms && k_steps / (2 * s) >= min_steps) s *= 2;
  return s;
}

}  // namespace

cudaError_t launch_route_small(const moe_handle *h, const void *x, int T,
                               unsigned long long *usage, cudaStream_t st) {
  const int E = h->E, H = h->H, k = h->k;
  const int splits = gemv_splits(E, H, h->num_sms);
  const int hps = H / splits;
  const int nt = T <= 4 ? 4 : kRouteTokens;
  // x staging for the GEMV; then the last CTA's keys and scores and its two
  // grouping arrays.
  const size_t smem = (size_t)std::max(nt * hps, 2 * T * E + 2 * T * k) * sizeof(float);
  const int epl = (E + 31) / 32;
  const dim3 grid((E + 7) / 8, splits);
  const moe::Workspace &w = h->ws;
  cudaError_t err = cudaSuccess;
#define MOE_RS2(N, NTT)                                                                         \
  do {                                                                                          \
    if (smem > 48 * 1024) {                                                                     \
      err = cudaFuncSetAttribute(route_small_kernel<N, NTT>,                                    \
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,       \
                                             (int)smem);                                        \
      if (err != cudaSuccess) return err;                                                       \
    }                                                                                           \
    err = launch_k(false, route_small_kernel<N, NTT>, grid, dim3(256), smem, st, x,            \
                   h->L.x_dtype == 1, T, H, E, k, route_rule(h), h->wr_t, h->bias, hps,         \
                   w.z_part, w.ticket, w.route_kv, h->S, w.idx, w.w, w.counts, w.offsets,       \
                   w.perm, w.inv, w.active, w.n_active, w.tiles, w.n_tiles, w.status, usage);   \
  } while (0)
#define MOE_RS(N)                                                                               \
  do {                                                                                          \
    if (nt == 4) MOE_RS2(N, 4);                                                                 \
    else MOE_RS2(N, kRouteTokens);                                                              \
  } while (0)
  if (epl <= 1) MOE_RS(1);
  else if (epl <= 2) MOE_RS(2);
  else if (epl <= 4) MOE_RS(4);
  else if (epl <= 8) MOE_RS(8);
  else if (epl <= 16) MOE_RS(16);
  else MOE_RS(32);
#undef MOE_RS
#undef MOE_RS2
  return err;
}

cudaError_t launch_router(const moe_handle *h, const void *x, int T, cudaStream_t st) {
  const int E = h->E, H = h->H, k = h->k;
  const int xb = h->L.x_dtype == 1;
  int splits = router_splits(T, E, H, h->num_sms);
  cudaError_t err = cudaSuccess;
  if (T <= 4) {
    const int hps = H / splits;
    const dim3 grid((E + 7) / 8, splits);
    const size_t smem = (size_t)4 * hps * sizeof(float);
    if (smem > 48 * 1024) {
      err = cudaFuncSetAttribute(router_gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
      if (err != cudaSuccess) return err;
    }
    err = launch_k(false, router_gemv_kernel<4>, grid, dim3(256), smem, st, x, xb, T, H, E,
                   h->wr_t, hps, h->ws.z_part, kGemvTokens);
  } else if (xb && tc_path_available()) {
    // bf16 activations: tensor cores on the three bf16 planes of the f32 weights
    // (tiles of 128 experts x 64 tokens, 64-K blocks, at least 2 per split).
    splits = batched_router_splits(T, ((E + 127) / 128) * ((T + 63) / 64), H / 64, 2, h->num_sms);
    err = launch_router_tc(h, x, T, h->ws.z_part, splits, st);
  } else {
    const dim3 grid((E + RG_BE - 1) / RG_BE, (T + RG_BT - 1) / RG_BT);
    splits = batched_router_splits(T, (int)(grid.x * grid.y), H / RG_BK, 4, h->num_sms);
    err = launch_k(false, router_gemm_kernel, dim3(grid.x, grid.y, splits), dim3(256), 0, st, x,
                   xb, T, H, E, h->wr_t, h->ws.z_part);
  }
  if (err != cudaSuccess) return err;
  const int zstride = (T <= 4) ? kGemvTokens : T;
  const int epl = (E + 31) / 32;
  const dim3 g2((T + 7) / 8);
#define MOE_TOPK(N)                                                                          \
  err = launch_k(h->pdl, router_topk_kernel<N>, g2, dim3(256), 0, st, h->ws.z_part, splits,   \
                 zstride, T, E, k, route_rule(h), h->bias, h->ws.idx, h->ws.w)
  if (epl <= 1) MOE_TOPK(1);
  else if (epl <= 2) MOE_TOPK(2);
  else if (epl <= 4) MOE_TOPK(4);
  else if (epl <= 8) MOE_TOPK(8);
  else if (epl <= 16) MOE_TOPK(16);
  else MOE_TOPK(32);
#undef MOE_TOPK
  return err;
}

}  // namespace moe

// ---------------------------------------------------------------------------
// Allocation-free routing (moe_route_noalloc).  The pages have no counterpart;
// this serves callers that cannot call cudaMalloc (see include/moe.h).  It
// launches the same router kernels as above, but their logit scratch lives in
// the file-scope array below instead of a handle's workspace.

namespace moe {
namespace {

constexpr size_t kRouteScratchFloats = size_t(1) << 20;   // 4 MiB per device
static __device__ __align__(256) float g_route_scratch[kRouteScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float *g_scratch_ptr[kMaxDevices] = {};
int g_scratch_sms[kMaxDevices] = {};

// Device address of the scratch array for the current device (looked up once
// per device with that device current).  Returns cudaSuccess or the error.
cudaError_t scratch_for_current_device(float **ptr, int *num_sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    int sms = 0;
    err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    g_scratch_ptr[dev] = static_cast<float *>(p);
    g_scratch_sms[dev] = sms;
  }
  *ptr = g_scratch_ptr[dev];
  *num_sms = g_scratch_sms[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace moe

extern "C" __attribute__((visibility("default"))) int moe_route_noalloc(
    const void *x, int T, int hidden, int num_experts, int top_k, int x_dtype, int router_mode,
    float routed_scaling_factor, const float *router_w_eh, const float *router_bias,
    int32_t *idx, float *w, moe_stream_t stream) {
  using namespace moe;
  if (num_experts < 1 || num_experts > kMaxExperts || top_k < 1 || top_k > num_experts ||
      top_k > kMaxTopK || router_mode < 0 || router_mode > 2 ||
      !(routed_scaling_factor > 0.f))
    return MOE_ERR_ROUTING;
  if (T < 0 || hidden < 512 || hidden % 512 || (x_dtype != 0 && x_dtype != 1))
    return MOE_ERR_ARG;
  if (router_mode == 1 && !router_bias) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !router_w_eh || !idx || !w) return MOE_ERR_ARG;
  // x and the router rows are read with 16-byte vector loads.
  if (((uintptr_t)x | (uintptr_t)router_w_eh) & 15) return MOE_ERR_ARG;
  const int E = num_experts, H = hidden;
  // Scratch needed: split partials [splits][4][E] for T <= 4, logits [T][E] above.
  if (T > 4 && (size_t)T * E > kRouteScratchFloats) return MOE_ERR_NOMEM;
  float *z = nullptr;
  int sms = 0;
  if (scratch_for_current_device(&z, &sms) != cudaSuccess) return MOE_ERR_DEVICE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int xb = x_dtype == 1;
  int splits = 1;
  if (T <= 4) {
    splits = router_splits(T, E, H, sms);
    if ((size_t)splits * kGemvTokens * E > kRouteScratchFloats) return MOE_ERR_NOMEM;
    const int hps = H / splits;
    const size_t smem = (size_t)4 * hps * sizeof(float);
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(router_gemv_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MOE_ERR_DEVICE;
    if (launch_k(false, router_gemv_kernel<4>, dim3((E + 7) / 8, splits), dim3(256), smem, st, x,
                 xb, T, H, E, router_w_eh, hps, z, kGemvTokens) != cudaSuccess)
      return MOE_ERR_DEVICE;
  } else {
    if (launch_k(false, router_gemm_kernel, dim3((E + RG_BE - 1) / RG_BE, (T + RG_BT - 1) / RG_BT),
                 dim3(256), 0, st, x, xb, T, H, E, router_w_eh, z) != cudaSuccess)
      return MOE_ERR_DEVICE;
  }
  const int zstride = (T <= 4) ? kGemvTokens : T;
  const int epl = (E + 31) / 32;
  const dim3 g2((T + 7) / 8);
  cudaError_t err = cudaSuccess;
#define MOE_TOPK_NA(N)                                                                      \
  err = launch_k(false, router_topk_kernel<N>, g2, dim3(256), 0, st, z, splits, zstride, T, E, \
                 top_k, RouteRule{router_mode, 0, 0, 0.f, routed_scaling_factor}, router_bias, \
                 idx, w)
  if (epl <= 1) MOE_TOPK_NA(1);
  else if (epl <= 2) MOE_TOPK_NA(2);
  else if (epl <= 4) MOE_TOPK_NA(4);
  else if (epl <= 8) MOE_TOPK_NA(8);
  else if (epl <= 16) MOE_TOPK_NA(16);
  else MOE_TOPK_NA(32);
#undef MOE_TOPK_NA
  return err == cudaSuccess ? MOE_OK : MOE_ERR_DEVICE;
}
