// router.cu -- step 1-2 of the layer: f32 router logits, then top-k selection
// with renormalised weights.
//
// The router stays f32 (colibrì engine teardown, text-matrix.pages.dev,
// "System map": norm/router/bias are kept in f32 because they are small and
// sensitive).  Scoring is softmax (Colibri C + cuBLASLt tutorial, cf-1.com,
// §2.1 step 2) or sigmoid with a noaux_tc selection bias, n_group = 1, scaled
// by routed_scaling_factor (teardown "Three key engineering decisions" (1)).
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
  if (x_is_bf16) {
    const int nv = hps / 8;                       // 8 bf16 per 16 bytes
    for (int i = threadIdx.x; i < NT * nv; i += blockDim.x) {
      const int t = i / nv, c = i - t * nv;
      float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
      if (t < T) {
        const uint4 u = __ldg(reinterpret_cast<const uint4 *>(
                                  reinterpret_cast<const __nv_bfloat16 *>(x) + (size_t)t * H + h0) +
                              c);
        lo = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                         __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
        hi = make_float4(__uint_as_float(u.z << 16), __uint_as_float(u.z & 0xFFFF0000u),
                         __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xFFFF0000u));
      }
      reinterpret_cast<float4 *>(xs + t * hps)[2 * c] = lo;
      reinterpret_cast<float4 *>(xs + t * hps)[2 * c + 1] = hi;
    }
  } else {
    const int nv = hps / 4;
    for (int i = threadIdx.x; i < NT * nv; i += blockDim.x) {
      const int t = i / nv, c = i - t * nv;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < T)
        v = __ldg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) +
                                                   (size_t)t * H + h0) +
                  c);
      reinterpret_cast<float4 *>(xs + t * hps)[c] = v;
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
  float acc[4][4] = {};
  for (int k0 = 0; k0 < H; k0 += RG_BK) {
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

// The selection of topk_token from the token's keys and scores (expert e in
// lane e % 32, slot e / 32; -inf keys past E).
template <int EPL>
__device__ __forceinline__ void topk_select(float key[EPL], float val[EPL], int t, int E, int k,
                                            const RouteRule r, int32_t *__restrict__ idx_out,
                                            float *__restrict__ w_out) {
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  if (r.n_group > 1) {
    // Lane g holds group g's score: the sum of its two largest keys.
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
  int my_idx = -1;
  float my_val = 0.f;
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
  // Numerators, and the sum over the selection in slot order.
  const float top = __shfl_sync(full, my_val, 0);
  float num = 0.f;
  if (lane < k) num = (r.mode != 1) ? expf(my_val - top) : my_val;
  float den = 0.f;
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
  }
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
// T <= 4 in one launch: the split-K router GEMV of router_gemv_kernel, then the
// last CTA to finish (an atomic ticket, reset by that CTA for the next call;
// nothing waits) reads every partial through L2, takes the top-k of each token
// and groups the T*k <= 128 assignments by expert with the same stable
// counting sort as dispatch.cu.  Also clears the status word first.
template <int EPL, int NT>
__global__ void __launch_bounds__(256) route_small_kernel(
    const void *__restrict__ x, int x_is_bf16, int T, int H, int E, int k, const RouteRule r,
    const float *__restrict__ wr_t, const float *__restrict__ bias, int h_per_split,
    float *__restrict__ z_part, int32_t *__restrict__ ticket, int n_shared,
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
  // Last-CTA-done: publish the partials, take a ticket.
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int n = gridDim.x * gridDim.y;
    last = (atomicAdd(ticket, 1) == n - 1);
    if (last) *ticket = 0;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();
  if (threadIdx.x == 0) *status = kStatusOk;
  // Logits of every (token, expert) from the split partials (summed in split
  // order, read through L2: other CTAs wrote them), their keys and scores into
  // shared memory -- all threads at once, so the partials cost one round trip.
  float *ks = xs, *vs = xs + T * E;
  const int splits = gridDim.y;
#pragma unroll 4
  for (int i = threadIdx.x; i < T * E; i += blockDim.x) {
    const int t = i / E, e = i - t * E;
    float zz = 0.f;
    for (int s = 0; s < splits; ++s) zz += __ldcg(z_part + ((size_t)s * NT + t) * E + e);
    key_of(zz, bias ? bias[e] : 0.f, r.mode, ks[i], vs[i]);
  }
  __syncthreads();
  // Top-k: warp t selects for token t.
  if (warp < T) {
    float key[EPL], val[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      key[i] = e < E ? ks[warp * E + e] : -INFINITY;
      val[i] = e < E ? vs[warp * E + e] : 0.f;
    }
    topk_select<EPL>(key, val, warp, E, k, r, idx, w);
  }
  __syncthreads();
  // Stable counting sort of the A = T*k assignments (A <= 128, E <= 1024).
  __shared__ int cnt[kMaxExperts];
  __shared__ int base[kMaxExperts];
  __shared__ int wsum[8];
  const int A = T * k;
  for (int i = threadIdx.x; i < E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  for (int a = threadIdx.x; a < A; a += blockDim.x) {
    const int ea = __ldcg(idx + a);
    if (ea >= 0 && ea < E) atomicAdd(&cnt[ea], 1);
    else if (ea != -1) atomicExch(status, kStatusBadExpert);   // -1: a slot top-p dropped
  }
  __syncthreads();
  // Exclusive scan of cnt over E: each thread owns a contiguous run of experts.
  const int per = (E + blockDim.x - 1) / blockDim.x;
  const int e0 = threadIdx.x * per;
  int run = 0;
  for (int i = 0; i < per; ++i)
    if (e0 + i < E) run += cnt[e0 + i];
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  int wbase = 0;
  for (int i = 0; i < warp; ++i) wbase += wsum[i];
  int pos = wbase + incl - run;
  for (int i = 0; i < per; ++i) {
    const int ee = e0 + i;
    if (ee < E) {
      counts[ee] = cnt[ee];
      if (usage && cnt[ee]) usage[ee] += (unsigned long long)cnt[ee];
      offsets[ee] = pos;
      base[ee] = pos;
      pos += cnt[ee];
    }
  }
  if (threadIdx.x == blockDim.x - 1) offsets[E] = pos;
  __syncthreads();
  // Scatter in ascending assignment order (warp 0, 32 assignments at a time).
  if (warp == 0) {
    const unsigned lt = (1u << lane) - 1u;
    for (int c0 = 0; c0 < A; c0 += 32) {
      const int a = c0 + lane;
      int ea = (a < A) ? __ldcg(idx + a) : E;
      if (ea < 0 || ea >= E) ea = E;
      if (a < A && ea == E) inv[a] = -1;
      const unsigned peers = __match_any_sync(0xffffffffu, ea);
      const int rank = __popc(peers & lt);
      if (ea < E) {
        const int p = base[ea] + rank;
        perm[p] = a;
        inv[a] = p;
      }
      __syncwarp();
      if (ea < E && (peers & lt) == 0) base[ea] += __popc(peers);
      __syncwarp();
    }
  }
  // Active experts (ascending, shared expert last) and one token block each:
  // the same per-thread runs, scanned over the non-empty flags.
  __syncthreads();
  int nz = 0;
  for (int i = 0; i < per; ++i)
    if (e0 + i < E && cnt[e0 + i] > 0) ++nz;
  int inz = nz;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, inz, o);
    if (lane >= o) inz += n;
  }
  if (lane == 31) wsum[warp] = inz;
  __syncthreads();
  int nbase = 0, ntot = 0;
  for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
    if (i < warp) nbase += wsum[i];
    ntot += wsum[i];
  }
  int apos = nbase + inz - nz;
  for (int i = 0; i < per; ++i) {
    const int ee = e0 + i;
    if (ee < E && cnt[ee] > 0) {
      active[apos] = ee;
      tiles[apos] = ee << 16;
      ++apos;
    }
  }
  if (threadIdx.x == 0) {
    int na = ntot, nt = ntot;
    if (n_shared) {
      active[na++] = E;
      tiles[nt++] = E << 16;
    }
    *n_active = na;
    n_tiles[0] = nt;
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

}  // namespace

cudaError_t launch_route_small(const moe_handle *h, const void *x, int T,
                               unsigned long long *usage, cudaStream_t st) {
  const int E = h->E, H = h->H, k = h->k;
  const int splits = gemv_splits(E, H, h->num_sms);
  const int hps = H / splits;
  const int nt = T <= 4 ? 4 : kRouteTokens;
  // x staging for the GEMV, then the keys and scores of the last CTA's top-k.
  const size_t smem = (size_t)std::max(nt * hps, 2 * T * E) * sizeof(float);
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
                   w.z_part, w.ticket, h->S, w.idx, w.w, w.counts, w.offsets, w.perm, w.inv,     \
                   w.active, w.n_active, w.tiles, w.n_tiles, w.status, usage);                  \
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
  return err != cudaSuccess ? err : cudaGetLastError();
}

cudaError_t launch_router(const moe_handle *h, const void *x, int T, cudaStream_t st) {
  const int E = h->E, H = h->H, k = h->k;
  const int xb = h->L.x_dtype == 1;
  const int splits = router_splits(T, E, H, h->num_sms);
  if (T <= 4) {
    const int hps = H / splits;
    const dim3 grid((E + 7) / 8, splits);
    const size_t smem = (size_t)4 * hps * sizeof(float);
    if (smem > 48 * 1024) {
      cudaError_t err = cudaFuncSetAttribute(router_gemv_kernel<4>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (err != cudaSuccess) return err;
    }
    router_gemv_kernel<4><<<grid, 256, smem, st>>>(x, xb, T, H, E, h->wr_t, hps, h->ws.z_part,
                                                   kGemvTokens);
  } else if (xb && tc_path_available()) {
    // bf16 activations: tensor cores on the three bf16 planes of the f32 weights.
    cudaError_t err = launch_router_tc(h, x, T, h->ws.z_part, st);
    if (err != cudaSuccess) return err;
  } else {
    const dim3 grid((E + RG_BE - 1) / RG_BE, (T + RG_BT - 1) / RG_BT);
    router_gemm_kernel<<<grid, 256, 0, st>>>(x, xb, T, H, E, h->wr_t, h->ws.z_part);
  }
  cudaError_t err = cudaGetLastError();
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
  return err != cudaSuccess ? err : cudaGetLastError();
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
    router_gemv_kernel<4><<<dim3((E + 7) / 8, splits), 256, smem, st>>>(x, xb, T, H, E,
                                                                        router_w_eh, hps, z,
                                                                        kGemvTokens);
  } else {
    router_gemm_kernel<<<dim3((E + RG_BE - 1) / RG_BE, (T + RG_BT - 1) / RG_BT), 256, 0, st>>>(
        x, xb, T, H, E, router_w_eh, z);
  }
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_DEVICE;
  const int zstride = (T <= 4) ? kGemvTokens : T;
  const int epl = (E + 31) / 32;
  const dim3 g2((T + 7) / 8);
#define MOE_TOPK_NA(N)                                                                      \
  router_topk_kernel<N><<<g2, 256, 0, st>>>(z, splits, zstride, T, E, top_k,               \
                                            RouteRule{router_mode, 0, 0, 0.f,               \
                                                      routed_scaling_factor},               \
                                            router_bias, idx, w)
  if (epl <= 1) MOE_TOPK_NA(1);
  else if (epl <= 2) MOE_TOPK_NA(2);
  else if (epl <= 4) MOE_TOPK_NA(4);
  else if (epl <= 8) MOE_TOPK_NA(8);
  else if (epl <= 16) MOE_TOPK_NA(16);
  else MOE_TOPK_NA(32);
#undef MOE_TOPK_NA
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_DEVICE;
}
