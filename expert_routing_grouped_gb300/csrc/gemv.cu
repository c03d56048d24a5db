// gemv.cu -- steps 4-5 of the layer for small T (decode and MTP-verify
// batches): int4 gs64 dequant GEMV with exact products and f32 accumulation.
//
// At small T the layer is bound by streaming the activated experts' packed
// weights from HBM (the pages' expert tier moves ~19 MB per expert: colibrì
// engine teardown, text-matrix.pages.dev, "System map").  Only experts that
// received tokens are read (Colibri C + cuBLASLt tutorial, cf-1.com, §3.3
// Step 4: skip empty experts).
//
//   W13:  h[p][n] = silu(W1[n] . x_t) * (W3[n] . x_t) for every grouped
//         position p of every active expert (and of the shared expert),
//         silu(g) = g / (1 + e^-g).
//   W2:   y[p][o] = w_p * (W2[o] . h[p]); the combine kernel then sums each
//         token's rows in slot order, then the shared expert (tutorial §3.3
//         Step 5), one owner per output element, no atomics.
//
// An item is 32 consecutive weight rows of one active expert (W13: 16
// features' W1 and W3 rows, interleaved; W2: 32 output rows); each of the 8
// warps streams 4 of those rows over the full K with 128-bit non-allocating
// loads (a lane's 16 bytes = 32 weights inside one 64-wide scale group).  The
// expert's activation rows sit in shared memory (staged when the expert
// changes, XOR-swizzled against bank conflicts) and are reused across the 4
// rows.  CTAs take contiguous item ranges, so one activation stage serves
// many items.
// Two kernels: the bf16-pair kernel (W13 on bf16 x, and W2 on h, which W13
// leaves as two exact bf16 planes) multiplies bf16 codes by bf16 activations
// with fma.rn.f32.bf16; W13 on f32 x decodes the codes to f32 and uses packed
// f32x2 arithmetic.
#include "moe_internal.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kRowsPerItem = 32;
constexpr int kWarps = 8;
constexpr int kRowsPerWarp = kRowsPerItem / kWarps;   // 4
constexpr int kActSmemBytes = 96 * 1024;

// Weights are read once per call: no L1 allocation, and an evict-first L2
// policy (pol) so that they do not push out what is worth keeping there (the
// workspace, and the next layer's router and shared expert when prefetched).
__device__ __forceinline__ uint4 ld_stream(const void *p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}

// Exact int4 -> f32 pairs for the 8 weights of one word of the library layout
// (K indices 8w+0,2,4,6 at bits 0-15, 8w+1,3,5,7 at bits 16-31, offset
// binary).  A nibble at bits 4p..4p+3 (p <= 4) is OR-ed into the mantissa of
// 2^(23-4p), whose unit in the last place is then exactly 1; subtracting
// 2^(23-4p) + 8 leaves the signed value.  Nibbles above bit 19 are shifted
// down by 12 first.  q[i] = (weight 8w+2i, weight 8w+2i+1).
__device__ __forceinline__ void dequant8(uint32_t w, float2 q[4]) {
  const uint32_t v = w >> 12;
  q[0] = __fadd2_rn(make_float2(__uint_as_float((w & 0x0000000Fu) | 0x4B000000u),
                                __uint_as_float((w & 0x000F0000u) | 0x43000000u)),
                    make_float2(-8388616.0f, -136.0f));
  q[1] = __fadd2_rn(make_float2(__uint_as_float((w & 0x000000F0u) | 0x49000000u),
                                __uint_as_float((v & 0x00000F00u) | 0x47000000u)),
                    make_float2(-524296.0f, -32776.0f));
  q[2] = __fadd2_rn(make_float2(__uint_as_float((w & 0x00000F00u) | 0x47000000u),
                                __uint_as_float((v & 0x0000F000u) | 0x45000000u)),
                    make_float2(-32776.0f, -2056.0f));
  q[3] = __fadd2_rn(make_float2(__uint_as_float((w & 0x0000F000u) | 0x45000000u),
                                __uint_as_float((v & 0x000F0000u) | 0x43000000u)),
                    make_float2(-2056.0f, -136.0f));
}

// h as two exact bf16 planes: row p's hi plane at planes + 2p * stride, its lo
// plane at (2p + 1) * stride.
__device__ __forceinline__ void store_h_planes(__nv_bfloat16 *planes, int stride, int p, int f,
                                               float h) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(h);
  planes[(size_t)(2 * p) * stride + f] = hi;
  planes[(size_t)(2 * p + 1) * stride + f] = __float2bfloat16_rn(h - __bfloat162float(hi));
}

// One item: 32 consecutive weight rows (group g) of one active expert e.
struct Item {
  const uint8_t *wq;   // the expert's packed rows
  const float *ws;     // the expert's scales
  int e, g, p0, cnt, K;
};

__device__ __forceinline__ Item item_at(int item, int n_routed, int items_r, int E, int A, int T,
                                        int K_r, int K_s, int rows_r, const uint8_t *wq_r,
                                        const float *ws_r, const uint8_t *wq_s, const float *ws_s,
                                        const int32_t *active, const int32_t *offsets) {
  Item it;
  if (item < n_routed * items_r) {
    it.K = K_r;
    it.e = active[item / items_r];
    it.g = item % items_r;
    it.wq = wq_r + (size_t)it.e * rows_r * (K_r / 2);
    it.ws = ws_r + (size_t)it.e * rows_r * (K_r / 64);
    it.p0 = offsets[it.e];
    it.cnt = offsets[it.e + 1] - it.p0;
  } else {
    it.K = K_s;
    it.e = E;
    it.g = item - n_routed * items_r;
    it.wq = wq_s;
    it.ws = ws_s;
    it.p0 = A;
    it.cnt = T;
  }
  return it;
}

// The weights and scales of chunk c of an item's four rows for this warp.
__device__ __forceinline__ void load_chunk(const Item &it, const int rr[kRowsPerWarp], int c,
                                           uint4 wv[kRowsPerWarp], float sc[kRowsPerWarp],
                                           uint64_t pol) {
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) {
    const size_t row = (size_t)it.g * kRowsPerItem + rr[i];
    wv[i] = ld_stream(it.wq + row * (it.K / 2) + (size_t)c * 16, pol);
    sc[i] = __ldg(it.ws + row * (it.K / 64) + (c >> 1));
  }
}

// W13 + SwiGLU for f32 activations (x of an f32-input layer): h is written as
// the exact bf16 planes hi = bf16(h), lo = bf16(h - hi) that W2 reads.
// Each lane keeps the next chunk's weights in flight while it works on the
// current one; the last chunk of an item prefetches the first chunk of the
// next item (when the item has one token batch).
template <int NT>
__global__ void __launch_bounds__(256) gemv_kernel(
    const void *__restrict__ act, int act_is_bf16, int act_stride, int T, int k, int E,
    int K_r, int K_s, int rows_r, int rows_s, const uint8_t *__restrict__ wq_r, const float *__restrict__ ws_r,
    const uint8_t *__restrict__ wq_s, const float *__restrict__ ws_s,
    const int32_t *__restrict__ active, const int32_t *__restrict__ n_active_p,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    __nv_bfloat16 *__restrict__ out_h, int out_stride) {
  pdl_enter();
  act = after_wait(act);
  active = after_wait(active);
  n_active_p = after_wait(n_active_p);
  offsets = after_wait(offsets);
  perm = after_wait(perm);
  out_h = after_wait(out_h);
  extern __shared__ float act_s[];   // [NT][K] activations of the current expert pass
  const int n_active = *n_active_p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first_policy();
  const int has_shared = (n_active > 0 && active[n_active - 1] == E) ? 1 : 0;
  const int n_routed = n_active - has_shared;
  const int items_r = rows_r / kRowsPerItem, items_s = rows_s / kRowsPerItem;
  const int items = n_routed * items_r + has_shared * items_s;
  const int A = T * k;
  const int i0 = (int)((long long)items * blockIdx.x / gridDim.x);
  const int i1 = (int)((long long)items * (blockIdx.x + 1) / gridDim.x);
  int staged_e = -1, staged_b = -1;
  const int sw = lane & 7;             // swizzle of every chunk this lane reads

  // Rows of this warp inside an item: W1 of features 2w, 2w+1 and W3 of the
  // same (rows 2w, 2w+1, 16+2w, 17+2w of the 32-row group).
  const int rr[kRowsPerWarp] = {2 * warp, 2 * warp + 1, 16 + 2 * warp, 17 + 2 * warp};

  bool pre = false;                    // wv/sc already hold this item's first chunk
  uint4 wv[kRowsPerWarp];
  float sc[kRowsPerWarp];
  for (int item = i0; item < i1; ++item) {
    const Item it = item_at(item, n_routed, items_r, E, A, T, K_r, K_s, rows_r, wq_r, ws_r, wq_s,
                            ws_s, active, offsets);
    const int e = it.e, g = it.g, p0 = it.p0, cnt = it.cnt, K = it.K;
    const int chunks = K / 32;   // 16-byte chunks per row
    for (int b0 = 0; b0 < cnt; b0 += NT) {
      const int nb = min(NT, cnt - b0);
      if (!pre || b0 > 0) {
        if (lane < chunks) load_chunk(it, rr, lane, wv, sc, pol);
      }
      pre = false;
      if (e != staged_e || b0 != staged_b) {
        __syncthreads();   // previous readers are done
        for (int i = threadIdx.x; i < NT * (K / 4); i += blockDim.x) {
          const int tkn = i / (K / 4), c4 = i - tkn * (K / 4);
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (tkn < nb) {
            const int p = p0 + b0 + tkn;
            const int src = (e < E) ? perm[p] / k : p - A;   // the token's x row
            if (act_is_bf16) {
              const uint2 u = __ldcg(reinterpret_cast<const uint2 *>(
                                        reinterpret_cast<const __nv_bfloat16 *>(act) +
                                        (size_t)src * act_stride) +
                                    c4);
              v = make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u),
                              __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xFFFF0000u));
            } else {
              v = __ldcg(reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(act) +
                                                         (size_t)src * act_stride) +
                        c4);
            }
          }
          // float4 j of 32-float chunk c is stored at slot j ^ (c & 7) of the
          // chunk: lanes reading the same j of chunks c..c+7 hit 8 bank groups.
          const int cc = c4 >> 3, jj = c4 & 7;
          reinterpret_cast<float4 *>(act_s + (size_t)tkn * K)[cc * 8 + (jj ^ (cc & 7))] = v;
        }
        __syncthreads();
        staged_e = e;
        staged_b = b0;
      }
      float acc[kRowsPerWarp][NT];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[i][t] = 0.f;
      for (int c = lane; c < chunks; c += 32) {
        uint4 wn[kRowsPerWarp];
        float sn[kRowsPerWarp];
        const int cn = c + 32;
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          wn[i] = make_uint4(0, 0, 0, 0);
          sn[i] = 0.f;
        }
        if (cn < chunks) {
          load_chunk(it, rr, cn, wn, sn, pol);
        } else if (b0 + NT >= cnt && item + 1 < i1) {
          const Item nx = item_at(item + 1, n_routed, items_r, E, A, T, K_r, K_s, rows_r, wq_r,
                                  ws_r, wq_s, ws_s, active, offsets);
          if (lane < nx.K / 32) {
            load_chunk(nx, rr, lane, wn, sn, pol);
            pre = true;
          }
        }
        // activations of this chunk (32 K) for each token, as f32 pairs
        float2 xa[NT][16];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const float4 *xp = reinterpret_cast<const float4 *>(act_s + (size_t)t * K + c * 32);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 f = xp[j ^ sw];   // c & 7 == lane & 7
            xa[t][2 * j] = make_float2(f.x, f.y);
            xa[t][2 * j + 1] = make_float2(f.z, f.w);
          }
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const uint32_t words[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
          float2 part[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) part[t] = make_float2(0.f, 0.f);
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
            float2 q[4];
            dequant8(words[wi], q);
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
              for (int t = 0; t < NT; ++t) part[t] = __ffma2_rn(q[j], xa[t][4 * wi + j], part[t]);
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[i][t] = fmaf(sc[i], part[t].x + part[t].y, acc[i][t]);
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          wv[i] = wn[i];
          sc[i] = sn[i];
        }
      }
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc[i][t] += __shfl_xor_sync(0xffffffffu, acc[i][t], o);
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nb) {
            const int p = p0 + b0 + t;
            // 32-row group g = 128-row block g/4, quadrant g%4: features
            // 64 (g/4) + 16 (g%4) + 2w + {0, 1}
            const int f0 = (g >> 2) * 64 + (g & 3) * 16 + 2 * warp;
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float gg = acc[j][t], uu = acc[2 + j][t];
              store_h_planes(out_h, out_stride, p, f0 + j, gg / (1.0f + expf(-gg)) * uu);
            }
          }
        }
      }
    }
  }
}

// ----------------------------------------------------------------------------
// The bf16-pair GEMV.  A pair of int4 codes becomes a bf16 pair (136 + q_even,
// 136 + q_odd) in one lop3; fma.rn.f32.bf16 multiplies it by bf16 activations
// exactly and accumulates in f32.  136 times the chunk's activation sum (f32,
// computed once per token when the expert's activations are staged) is taken
// off per 32-weight chunk, before the gs64 scale:
//   W[n] . a = sum_chunks s_chunk * (sum_i (136 + q_i) a_i - 136 * sum_i a_i).
// The activations come in PL bf16 planes whose sum is the operand: W13 reads
// x itself (one plane; bf16 x is exact), W2 reads h as the exact split
// h = hi + lo, hi = bf16(h), lo = bf16(h - hi) (16 significant bits, about
// 8e-6 relative), which the W13 epilogue writes.
//   MODE 0 (W13): rows 2w, 2w+1, 16+2w, 17+2w of a 32-row group are W1 / W3
//                 of features 2w, 2w+1; h = silu(g) * u, written as planes.
//   MODE 1 (W2):  rows 4w..4w+3; y[p][o] = routing weight * (W2[o] . h[p]).
// Each lane prefetches the next chunk's weights and scales before it uses the
// current ones (at an item's last chunk, the next item's first).
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t w) {
  uint32_t d;
  // (w & 0x000F000F) | 0x43004300: two offset-binary nibbles into bf16 128 + n.
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(d) : "r"(w));
  return d;
}

__device__ __forceinline__ void mfma_pair(float &acc0, float &acc1, uint32_t q2, uint32_t x2) {
  asm("{\n\t.reg .b16 ql, qh, xl, xh;\n\t"
      "mov.b32 {ql, qh}, %2;\n\t"
      "mov.b32 {xl, xh}, %3;\n\t"
      "fma.rn.f32.bf16 %0, ql, xl, %0;\n\t"
      "fma.rn.f32.bf16 %1, qh, xh, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1)
      : "r"(q2), "r"(x2));
}

template <int NT, int PL, int MODE>
__global__ void __launch_bounds__(256) gemv_bf16_kernel(
    const __nv_bfloat16 *__restrict__ act, int act_stride, int T, int k, int E, int K_r, int K_s,
    int rows_r, int rows_s, const uint8_t *__restrict__ wq_r, const float *__restrict__ ws_r,
    const uint8_t *__restrict__ wq_s, const float *__restrict__ ws_s,
    const int32_t *__restrict__ active, const int32_t *__restrict__ n_active_p,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    const float *__restrict__ wts, float *__restrict__ out_y, __nv_bfloat16 *__restrict__ out_h,
    int out_stride, const __grid_constant__ L2Prefetch pf) {
  static_assert(PL == 1 || PL == 2, "one or two activation planes");
  if (MODE == 1) l2_prefetch_share(pf);   // init-time weights: no wait needed
  // W13 runs the shared expert's items before it waits for the routing kernel
  // it is chained to: they need only x, which was complete before that kernel
  // (the first of the call, launched plainly) started, and they write only the
  // shared expert's rows of h, which nothing reads before W2.  So the shared
  // expert's weights stream while the routing kernel runs; the routed items
  // follow the wait.  W2 waits first.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint4 smem_v[];
  // [PL][NT][K/8] 16-byte groups of bf16 activations: group j of 32-wide chunk
  // c at slot j ^ ((c >> 1) & 3), so 8 lanes reading the same j of chunks
  // c..c+7 hit 8 different 16-byte bank groups; then [NT][K/32] f32 chunk sums
  // over the planes.  K is the larger of the routed and shared lengths.
  const int Kmax = K_r > K_s ? K_r : K_s;
  uint4 *xs = smem_v;
  float *xsum = reinterpret_cast<float *>(smem_v + (size_t)PL * NT * (Kmax / 8));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint64_t pol = l2_evict_first_policy();
  const int items_r = rows_r / kRowsPerItem, items_s = rows_s / kRowsPerItem;
  const int A = T * k;
  const bool early = MODE == 0 && items_s > 0;
  int staged_e = -1, staged_b = -1;
  int rr[kRowsPerWarp];
  if (MODE == 0) {
    rr[0] = 2 * warp;
    rr[1] = 2 * warp + 1;
    rr[2] = 16 + 2 * warp;
    rr[3] = 17 + 2 * warp;
  } else {
#pragma unroll
    for (int i = 0; i < kRowsPerWarp; ++i) rr[i] = kRowsPerWarp * warp + i;
  }

  bool pre = false;                    // wv/sc already hold this item's first chunk
  uint4 wv[kRowsPerWarp];
  float sc[kRowsPerWarp];
  // The work is dealt as contiguous ranges of one sequence of the n routed
  // and shared items, with the shared items spread through it (shared item s
  // at position floor(s n / items_s)): about items_s CTAs then take one
  // shared item each in phase 0, while the routing kernel runs, and as many
  // fewer routed items in phase 1, instead of a few CTAs taking them all.
  // Both parts of a range stay contiguous.  Before the wait the routed count
  // is not known; the deal assumes the usual one, min(E, T k) distinct
  // experts.  When the routing turns out otherwise (repeated experts, a
  // top-p trim) phase 1 deals the routed items evenly instead.
  const long long r_guess = (long long)min(E, T * k) * items_r;
  const long long n_guess = r_guess + items_s;
  const long long g_lo = n_guess * blockIdx.x / gridDim.x;
  const long long g_hi = n_guess * (blockIdx.x + 1) / gridDim.x;
  const long long s_lo = (g_lo * items_s + n_guess - 1) / n_guess;   // shared items before g_lo
  const long long s_hi = (g_hi * items_s + n_guess - 1) / n_guess;
  for (int phase = early ? 0 : 1; phase < 2; ++phase) {
  // Phase 0: the shared expert's items (item_at with no routed experts maps
  // item i to the shared expert's 32-row group i).  Phase 1: after the wait,
  // the routed items (and, in W2, the shared expert's after them).
  int n_routed = 0, items = items_s;
  int i0 = (int)s_lo, i1 = (int)s_hi;
  if (phase == 1) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    act = after_wait(act);
    active = after_wait(active);
    n_active_p = after_wait(n_active_p);
    offsets = after_wait(offsets);
    perm = after_wait(perm);
    wts = after_wait(wts);
    out_y = after_wait(out_y);
    out_h = after_wait(out_h);
    const int n_active = *n_active_p;
    const int has_shared = (n_active > 0 && active[n_active - 1] == E) ? 1 : 0;
    n_routed = n_active - has_shared;
    items = n_routed * items_r + (early ? 0 : has_shared * items_s);
    if (early && items == r_guess) {
      i0 = (int)(g_lo - s_lo);
      i1 = (int)(g_hi - s_hi);
    } else {
      i0 = (int)((long long)items * blockIdx.x / gridDim.x);
      i1 = (int)((long long)items * (blockIdx.x + 1) / gridDim.x);
    }
  }
  pre = false;
  for (int item = i0; item < i1; ++item) {
    const Item it = item_at(item, n_routed, items_r, E, A, T, K_r, K_s, rows_r, wq_r, ws_r, wq_s,
                            ws_s, active, offsets);
    const int e = it.e, g = it.g, p0 = it.p0, cnt = it.cnt, K = it.K;
    const int chunks = K / 32;
    for (int b0 = 0; b0 < cnt; b0 += NT) {
      const int nb = min(NT, cnt - b0);
      if (!pre || b0 > 0) {
        if (lane < chunks) load_chunk(it, rr, lane, wv, sc, pol);
      }
      pre = false;
      if (e != staged_e || b0 != staged_b) {
        __syncthreads();   // previous readers are done
        // One thread per (token, chunk): 64 bytes per plane in, swizzled out,
        // the chunk sum over the planes.
        for (int i = threadIdx.x; i < NT * chunks; i += blockDim.x) {
          const int tkn = i / chunks, c = i - tkn * chunks;
          float sum = 0.f;
#pragma unroll
          for (int pl = 0; pl < PL; ++pl) {
            uint4 v[4] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0),
                          make_uint4(0, 0, 0, 0)};
            if (tkn < nb) {
              const int p = p0 + b0 + tkn;
              // W13 reads the token's x row; W2 reads the grouped position's planes.
              const size_t row = MODE == 0 ? (size_t)((e < E) ? perm[p] / k : p - A)
                                           : (size_t)(2 * p + pl);
              const uint4 *src = reinterpret_cast<const uint4 *>(act + row * act_stride) + c * 4;
#pragma unroll
              for (int j = 0; j < 4; ++j) v[j] = __ldcg(src + j);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
                for (int m = 0; m < 4; ++m)
                  sum += __uint_as_float(u[m] << 16) + __uint_as_float(u[m] & 0xFFFF0000u);
              }
            }
            uint4 *dst = xs + ((size_t)pl * NT + tkn) * (K / 8) + c * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j ^ ((c >> 1) & 3)] = v[j];
          }
          xsum[tkn * chunks + c] = sum;
        }
        __syncthreads();
        staged_e = e;
        staged_b = b0;
      }
      float acc[kRowsPerWarp][NT];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t) acc[i][t] = 0.f;
      for (int c = lane; c < chunks; c += 32) {
        // prefetch the next chunk of the same rows, or the next item's first
        uint4 wn[kRowsPerWarp];
        float sn[kRowsPerWarp];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          wn[i] = make_uint4(0, 0, 0, 0);
          sn[i] = 0.f;
        }
        const int cn = c + 32;
        if (cn < chunks) {
          load_chunk(it, rr, cn, wn, sn, pol);
        } else if (b0 + NT >= cnt && item + 1 < i1) {
          const Item nx = item_at(item + 1, n_routed, items_r, E, A, T, K_r, K_s, rows_r, wq_r,
                                  ws_r, wq_s, ws_s, active, offsets);
          if (lane < nx.K / 32) {
            load_chunk(nx, rr, lane, wn, sn, pol);
            pre = true;
          }
        }
        uint32_t xw[PL][NT][16];
        float xc[NT];
#pragma unroll
        for (int pl = 0; pl < PL; ++pl)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const uint4 *src = xs + ((size_t)pl * NT + t) * (K / 8) + c * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 u = src[j ^ ((c >> 1) & 3)];
              xw[pl][t][4 * j] = u.x;
              xw[pl][t][4 * j + 1] = u.y;
              xw[pl][t][4 * j + 2] = u.z;
              xw[pl][t][4 * j + 3] = u.w;
            }
          }
#pragma unroll
        for (int t = 0; t < NT; ++t) xc[t] = 136.0f * xsum[t * chunks + c];
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          const uint32_t words[4] = {wv[i].x, wv[i].y, wv[i].z, wv[i].w};
          float pe[NT], po[NT];
#pragma unroll
          for (int t = 0; t < NT; ++t) pe[t] = po[t] = 0.f;
#pragma unroll
          for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
              const uint32_t q2 = nib_pair_bf16(words[wi] >> (4 * pp));
#pragma unroll
              for (int t = 0; t < NT; ++t)
#pragma unroll
                for (int pl = 0; pl < PL; ++pl) mfma_pair(pe[t], po[t], q2, xw[pl][t][4 * wi + pp]);
            }
          }
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[i][t] = fmaf(sc[i], (pe[t] + po[t]) - xc[t], acc[i][t]);
        }
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) {
          wv[i] = wn[i];
          sc[i] = sn[i];
        }
      }
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) acc[i][t] += __shfl_xor_sync(0xffffffffu, acc[i][t], o);
      if (lane == 0) {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (t < nb) {
            const int p = p0 + b0 + t;
            if (MODE == 0) {
              // 32-row group g = 128-row block g/4, quadrant g%4: features
              // 64 (g/4) + 16 (g%4) + 2w + {0, 1}
              const int f0 = (g >> 2) * 64 + (g & 3) * 16 + 2 * warp;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const float gg = acc[j][t], uu = acc[2 + j][t];
                store_h_planes(out_h, out_stride, p, f0 + j, gg / (1.0f + expf(-gg)) * uu);
              }
            } else {
              const float wt = (e < E) ? __ldcg(wts + __ldcg(perm + p)) : 1.0f;
#pragma unroll
              for (int i = 0; i < kRowsPerWarp; ++i)
                out_y[(size_t)p * out_stride + g * kRowsPerItem + rr[i]] = wt * acc[i][t];
            }
          }
        }
      }
    }
  }
  }   // phase
}

// ----------------------------------------------------------------------------
// The single-token W2 GEMV on warp-level MMAs (T = 1: the decode regime).
// The weights stream exactly as in the bf16-pair kernel (32-row items, 16-byte
// non-allocating loads, one chunk prefetched ahead), and its exactness is
// kept: bf16 (136 + q) codes times h's exact bf16 planes, f32 accumulation
// inside each 64-wide group, 136 x (the group's sum of h) taken off and the
// group scale applied per group.  Each iteration stores its 32 rows x 1024 K
// and their scales into a shared tile; after one CTA barrier every warp
// multiplies its 128-K slice of both 16-row tiles with mma.sync.m16n8k16
// (bf16 in, f32 accumulate): one instruction covers 16 x 16 weights and both
// planes, which are its B columns 0 (hi) and 1 (lo), so the sum of the two
// accumulator columns is the product with h.  The eight warps' partial tiles
// of an item are summed in warp order (the same sum every run).  Every tile
// iteration ends at a CTA barrier that ties each warp to the slowest one's
// loads, so the kernel serves items of at most four iterations (K <= 4096);
// at K = 6144 (W13) and 14336 (a Mixtral-shaped W2) the SIMT kernel is
// faster.
// Fragment layout (PTX ISA, mma.m16n8k16 for 16-bit types), lane = 4 g + q:
// A rows g and g + 8, B column g, accumulator rows g, g + 8 and columns 2q,
// 2q + 1.  Inside a 64-wide group the K order is permuted alike for A and B:
// in step s, slots 2q, 2q + 1 hold K = 16q + 2s, +1 and slots 2q + 8, 2q + 9
// hold K = 16q + 8 + 2s, +1.  A lane's A values are then the 32-bit words 2q
// and 2q + 1 of its rows' 32-byte group (pair s = the nibbles at bits 4s and
// 16 + 4s), and its B values the 16 activations K = 16q .. 16q + 15.
constexpr int kTileK = 1024;                   // K per iteration (32 chunks)
constexpr int kWPitch = kTileK / 2 + 32;       // bytes per staged weight row (an odd multiple of 32)
constexpr int kSPitch = kTileK / 64 + 1;       // floats per staged scale row

__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared memory of the MMA kernel: h's two planes and their chunk sums, two
// weight tiles, two scale tiles, the partial tiles.
size_t w2_mma_smem(int K) {
  return (size_t)2 * K * 2 + (size_t)K / 8 + 2 * kRowsPerItem * kWPitch +
         2 * kRowsPerItem * kSPitch * 4 + kWarps * 2 * 32 * 8;
}

__global__ void __launch_bounds__(256, 2) gemv_w2_mma_kernel(
    const __nv_bfloat16 *__restrict__ act, int act_stride, int k, int E, int K_r, int K_s,
    int rows_r, int rows_s, const uint8_t *__restrict__ wq_r, const float *__restrict__ ws_r,
    const uint8_t *__restrict__ wq_s, const float *__restrict__ ws_s,
    const int32_t *__restrict__ active, const int32_t *__restrict__ n_active_p,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    const float *__restrict__ wts, float *__restrict__ out_y, int out_stride,
    const __grid_constant__ L2Prefetch pf) {
  constexpr int PL = 2;   // h's planes = B columns 0 and 1
  constexpr int T = 1;
  l2_prefetch_share(pf);  // init-time weights: no wait needed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint4 smem_v[];
  const int Kmax = K_r > K_s ? K_r : K_s;
  uint4 *xs = smem_v;                                                      // [PL][K/8], swizzled
  float *xsum = reinterpret_cast<float *>(smem_v + (size_t)PL * (Kmax / 8));  // [K/32]
  uint8_t *wbuf = reinterpret_cast<uint8_t *>(xsum + Kmax / 32);          // [2][32][kWPitch]
  float *sbuf = reinterpret_cast<float *>(wbuf + 2 * kRowsPerItem * kWPitch);  // [2][32][kSPitch]
  float2 *part = reinterpret_cast<float2 *>(sbuf + 2 * kRowsPerItem * kSPitch);  // [8][2][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const uint64_t pol = l2_evict_first_policy();
  const int items_r = rows_r / kRowsPerItem, items_s = rows_s / kRowsPerItem;
  const int A = T * k;
  int staged_e = -1;
  int rr[kRowsPerWarp];   // this warp's rows of an item in the tile
#pragma unroll
  for (int i = 0; i < kRowsPerWarp; ++i) rr[i] = kRowsPerWarp * warp + i;
  bool pre = false;                    // wv/sc already hold this item's first chunk
  uint4 wv[kRowsPerWarp];
  float sc[kRowsPerWarp];
  uint32_t tile = 0;                   // tiles written so far (buffer = tile & 1)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  act = after_wait(act);
  active = after_wait(active);
  n_active_p = after_wait(n_active_p);
  offsets = after_wait(offsets);
  perm = after_wait(perm);
  wts = after_wait(wts);
  out_y = after_wait(out_y);
  // [routed items, the shared expert's], contiguous ranges per CTA
  const int n_active = *n_active_p;
  const int has_shared = (n_active > 0 && active[n_active - 1] == E) ? 1 : 0;
  const int n_routed = n_active - has_shared;
  const int items = n_routed * items_r + has_shared * items_s;
  const int i0 = (int)((long long)items * blockIdx.x / gridDim.x);
  const int i1 = (int)((long long)items * (blockIdx.x + 1) / gridDim.x);
  for (int item = i0; item < i1; ++item) {
    const Item it = item_at(item, n_routed, items_r, E, A, T, K_r, K_s, rows_r, wq_r, ws_r, wq_s,
                            ws_s, active, offsets);
    const int e = it.e, gi = it.g, p0 = it.p0, K = it.K;
    const int chunks = K / 32;
    if (!pre) {
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        wv[i] = make_uint4(0, 0, 0, 0);
        sc[i] = 0.f;
      }
      if (lane < chunks) load_chunk(it, rr, lane, wv, sc, pol);
    }
    pre = false;
    if (e != staged_e) {
      __syncthreads();   // previous readers are done
      // One thread per chunk: 64 bytes per plane in, swizzled out, the
      // chunk sum over the planes.
      for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
        float sum = 0.f;
#pragma unroll
        for (int pl = 0; pl < PL; ++pl) {
          const size_t row = (size_t)(2 * p0 + pl);   // the position's plane pl
          const uint4 *src = reinterpret_cast<const uint4 *>(act + row * act_stride) + c * 4;
          uint4 v[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) v[j] = __ldcg(src + j);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
            for (int m = 0; m < 4; ++m)
              sum += __uint_as_float(u[m] << 16) + __uint_as_float(u[m] & 0xFFFF0000u);
          }
          uint4 *dst = xs + (size_t)pl * (K / 8) + c * 4;
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j ^ ((c >> 1) & 3)] = v[j];
        }
        xsum[c] = sum;
      }
      __syncthreads();
      staged_e = e;
    }
    float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    const int niter = (K + kTileK - 1) / kTileK;
    for (int itn = 0; itn < niter; ++itn, ++tile) {
      // prefetch the next iteration's chunk of the same rows, or the next
      // item's first
      uint4 wn[kRowsPerWarp];
      float sn[kRowsPerWarp];
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        wn[i] = make_uint4(0, 0, 0, 0);
        sn[i] = 0.f;
      }
      const int cn = (itn + 1) * 32 + lane;
      if (itn + 1 < niter) {
        if (cn < chunks) load_chunk(it, rr, cn, wn, sn, pol);
      } else if (item + 1 < i1) {
        const Item nx = item_at(item + 1, n_routed, items_r, E, A, T, K_r, K_s, rows_r, wq_r,
                                ws_r, wq_s, ws_s, active, offsets);
        if (lane < nx.K / 32) load_chunk(nx, rr, lane, wn, sn, pol);
        pre = true;
      }
      // this iteration's rows and scales into tile buffer tile & 1 (its
      // readers two tiles ago passed the barrier of the tile in between)
      uint8_t *wt = wbuf + (size_t)(tile & 1) * kRowsPerItem * kWPitch;
      float *st = sbuf + (size_t)(tile & 1) * kRowsPerItem * kSPitch;
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i)
        *reinterpret_cast<uint4 *>(wt + rr[i] * kWPitch + lane * 16) = wv[i];
      if ((lane & 1) == 0) {
#pragma unroll
        for (int i = 0; i < kRowsPerWarp; ++i) st[rr[i] * kSPitch + (lane >> 1)] = sc[i];
      }
      __syncthreads();
      // this warp's groups 2w, 2w + 1 of the iteration, both tiles
      const int G = min(kTileK, K - itn * kTileK) / 64;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int gl = 2 * warp + j;
        if (gl >= G) break;
        const int gk = itn * (kTileK / 64) + gl;   // group index in K
        uint32_t b0[4] = {0u, 0u, 0u, 0u}, b1[4] = {0u, 0u, 0u, 0u};
        if (g < PL) {
          const int c = 2 * gk + (q >> 1), j0 = 2 * (q & 1), sw = (c >> 1) & 3;
          const uint4 *src = xs + (size_t)g * (K / 8) + c * 4;
          const uint4 u0 = src[j0 ^ sw], u1 = src[(j0 + 1) ^ sw];
          b0[0] = u0.x; b0[1] = u0.y; b0[2] = u0.z; b0[3] = u0.w;
          b1[0] = u1.x; b1[1] = u1.y; b1[2] = u1.z; b1[3] = u1.w;
        }
        __syncwarp();   // the MMAs below are warp-collective
        const float xc = 136.0f * (xsum[2 * gk] + xsum[2 * gk + 1]);
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          // tile t: item rows 16t + g and 16t + g + 8
          const int rl = 16 * t + g, rh = rl + 8;
          const uint2 wl = *reinterpret_cast<const uint2 *>(wt + rl * kWPitch + gl * 32 + q * 8);
          const uint2 wh = *reinterpret_cast<const uint2 *>(wt + rh * kWPitch + gl * 32 + q * 8);
          const float sl = st[rl * kSPitch + gl], sh = st[rh * kSPitch + gl];
          float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4)
            mma16816(d, nib_pair_bf16(wl.x >> (4 * s4)), nib_pair_bf16(wh.x >> (4 * s4)),
                     nib_pair_bf16(wl.y >> (4 * s4)), nib_pair_bf16(wh.y >> (4 * s4)), b0[s4],
                     b1[s4]);
          // columns 0 and 1 (lanes q = 0): h's two planes
          acc[t][0] = fmaf(sl, (d[0] + d[1]) - xc, acc[t][0]);
          acc[t][1] = fmaf(sh, (d[2] + d[3]) - xc, acc[t][1]);
        }
      }
#pragma unroll
      for (int i = 0; i < kRowsPerWarp; ++i) {
        wv[i] = wn[i];
        sc[i] = sn[i];
      }
    }
    // The item's partial tiles; warp t sums tile t over the warps and
    // writes it (lanes q = 0 hold columns 0 and 1).
#pragma unroll
    for (int t = 0; t < 2; ++t) part[(warp * 2 + t) * 32 + lane] = make_float2(acc[t][0], acc[t][1]);
    __syncthreads();
    if (warp < 2 && q == 0) {
      const int t = warp;
      float r0 = 0.f, r1 = 0.f;
      for (int v = 0; v < kWarps; ++v) {   // warp order: the same sum every run
        const float2 pv = part[(v * 2 + t) * 32 + lane];
        r0 += pv.x;
        r1 += pv.y;
      }
      const int p = p0;
      const float w8 = (e < E) ? __ldcg(wts + __ldcg(perm + p)) : 1.0f;
      out_y[(size_t)p * out_stride + gi * kRowsPerItem + 16 * t + g] = w8 * r0;
      out_y[(size_t)p * out_stride + gi * kRowsPerItem + 16 * t + g + 8] = w8 * r1;
    }
  }
}

// 8 bytes global -> registers, not kept in L1, evict-first in L2.
__device__ __forceinline__ uint2 ld_stream8(const void *p, uint64_t pol) {
  uint2 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
               : "=r"(r.x), "=r"(r.y)
               : "l"(p), "l"(pol));
  return r;
}

// The single-token W2 GEMV with K split over the warps (T = 1, K = 512 G:
// G 64-wide groups per warp).  The products, the exactness and the fragment
// layout are those of gemv_w2_mma_kernel; the weights take another road.
// An item is 32 rows of one expert; warp w takes its groups w G .. w G + G - 1
// of both 16-row tiles, and each lane loads exactly its A fragments from
// global memory, 8 bytes of rows g and g + 8 per group (the four lanes of a
// row read one full 32-byte sector), with no shared tile and no barrier
// between loads and MMAs.  The two tiles of an item are the units of a
// two-deep register pipeline: the loads of the next unit are in flight while
// a unit is multiplied.  At an item's end the eight warps' partial tiles go
// through shared memory (double-buffered) and one CTA barrier; warps 0 and 1
// sum them in warp order (the same sum every run) and write y.  An expert's
// slot -- its id, rows, position and routing weight -- is read once, one
// item ahead of its first item, and h is staged once per expert.
template <int G>
__global__ void __launch_bounds__(256, 2) gemv_w2_ks_kernel(
    const __nv_bfloat16 *__restrict__ act, int act_stride, int k, int E, int K_r, int K_s,
    int rows_r, int rows_s, const uint8_t *__restrict__ wq_r, const float *__restrict__ ws_r,
    const uint8_t *__restrict__ wq_s, const float *__restrict__ ws_s,
    const int32_t *__restrict__ active, const int32_t *__restrict__ n_active_p,
    const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
    const float *__restrict__ wts, float *__restrict__ out_y, int out_stride,
    const __grid_constant__ L2Prefetch pf) {
  constexpr int PL = 2;   // h's planes = B columns 0 and 1
  constexpr int K = 512 * G;
  constexpr int T = 1;
  l2_prefetch_share(pf);  // init-time weights: no wait needed
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ uint4 smem_v[];
  uint4 *xs = smem_v;                                                  // [PL][K/8], swizzled
  float *xsum = reinterpret_cast<float *>(smem_v + PL * (K / 8));      // [K/32]
  float2 *part = reinterpret_cast<float2 *>(xsum + K / 32);            // [2][8][2][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const uint64_t pol = l2_evict_first_policy();
  const int items_r = rows_r / kRowsPerItem, items_s = rows_s / kRowsPerItem;
  const int A = T * k;
  // While the up-projection pass finishes, thread 0 reads the routing's
  // outputs (written long before, but read here before the wait: they may in
  // principle be a previous call's) and prefetches this CTA's first item into
  // L2.  A hint only: everything below reads them again after the wait.
  if (threadIdx.x == 0) {
    const int na = __ldcg(n_active_p);
    const int hs = (rows_s > 0 && na > 0) ? 1 : 0;
    const int nr = na - hs;
    const int its = nr * items_r + hs * items_s;
    const int f = (int)((long long)its * blockIdx.x / gridDim.x);
    const int l = (int)((long long)its * (blockIdx.x + 1) / gridDim.x);
    if (f < l && nr >= 0 && nr <= E) {
      const bool routed = f < nr * items_r;
      const int e = routed ? __ldcg(active + f / items_r) : E;
      const int gi = routed ? f % items_r : f - nr * items_r;
      if ((routed ? (e >= 0 && e < E) : items_s > 0) && gi >= 0 &&
          gi < (routed ? items_r : items_s)) {
        const uint8_t *w = routed ? wq_r + (size_t)e * rows_r * (K / 2) : wq_s;
        const float *sc = routed ? ws_r + (size_t)e * rows_r * (K / 64) : ws_s;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                         w + (size_t)gi * kRowsPerItem * (K / 2)),
                     "r"((uint32_t)(kRowsPerItem * (K / 2)))
                     : "memory");
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(
                         sc + (size_t)gi * kRowsPerItem * (K / 64)),
                     "r"((uint32_t)(kRowsPerItem * (K / 64) * 4))
                     : "memory");
      }
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  act = after_wait(act);
  active = after_wait(active);
  n_active_p = after_wait(n_active_p);
  offsets = after_wait(offsets);
  perm = after_wait(perm);
  wts = after_wait(wts);
  out_y = after_wait(out_y);
  // [routed items, the shared expert's], contiguous ranges per CTA (the
  // routing lists the shared expert last whenever there is one)
  const int n_active = *n_active_p;
  const int has_shared = (rows_s > 0 && n_active > 0) ? 1 : 0;
  const int n_routed = n_active - has_shared;
  const int routed_items = n_routed * items_r;
  const int items = routed_items + has_shared * items_s;
  const int i0 = (int)((long long)items * blockIdx.x / gridDim.x);
  const int i1 = (int)((long long)items * (blockIdx.x + 1) / gridDim.x);
  // An expert's slot: routed slots a < n_routed hold items_r items each, the
  // shared slot n_routed the rest.
  struct Slot {
    int a, e, p0;
    const uint8_t *wq;
    const float *ws;
  };
  auto slot_of = [&](int a) {
    Slot sl;
    sl.a = a;
    if (a < n_routed) {
      sl.e = active[a];
      sl.wq = wq_r + (size_t)sl.e * rows_r * (K / 2);
      sl.ws = ws_r + (size_t)sl.e * rows_r * (K / 64);
      sl.p0 = offsets[sl.e];
    } else {
      sl.e = E;
      sl.wq = wq_s;
      sl.ws = ws_s;
      sl.p0 = A;
    }
    return sl;
  };
  auto slot_index = [&](int item) { return item < routed_items ? item / items_r : n_routed; };
  auto group_of = [&](int item) {
    return item < routed_items ? item % items_r : item - routed_items;
  };
  // per-unit registers: rows g and g + 8 of the unit's tile, this warp's groups
  uint2 wl0[G], wh0[G], wl1[G], wh1[G];
  float sl0[G], sh0[G], sl1[G], sh1[G];
  auto load_unit = [&](uint2 (&wl)[G], uint2 (&wh)[G], float (&sl)[G], float (&sh)[G],
                       const Slot &sl_, int gi, int t) {
    const size_t r0 = (size_t)gi * kRowsPerItem + 16 * t + g;
    const uint8_t *p0 = sl_.wq + r0 * (K / 2) + warp * G * 32 + q * 8;
    const uint8_t *p1 = p0 + (size_t)8 * (K / 2);
#pragma unroll
    for (int j = 0; j < G; ++j) {
      wl[j] = ld_stream8(p0 + j * 32, pol);
      wh[j] = ld_stream8(p1 + j * 32, pol);
    }
    const float *s0 = sl_.ws + r0 * (K / 64) + warp * G;
    const float *s1 = s0 + 8 * (K / 64);
    if constexpr (G == 4) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(s0));
      const float4 b = __ldg(reinterpret_cast<const float4 *>(s1));
      sl[0] = a.x; sl[1] = a.y; sl[2] = a.z; sl[3] = a.w;
      sh[0] = b.x; sh[1] = b.y; sh[2] = b.z; sh[3] = b.w;
    } else {
      const float2 a = __ldg(reinterpret_cast<const float2 *>(s0));
      const float2 b = __ldg(reinterpret_cast<const float2 *>(s1));
      sl[0] = a.x; sl[1] = a.y;
      sh[0] = b.x; sh[1] = b.y;
    }
  };
  // One unit's MMAs: this warp's groups of one 16-row tile; h's planes are
  // the B columns 0 (hi) and 1 (lo).  Lanes q = 0 end with the rows' sums.
  auto mul_unit = [&](const uint2 (&wl)[G], const uint2 (&wh)[G], const float (&sl)[G],
                      const float (&sh)[G], float &acc0, float &acc1) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const int gk = warp * G + j;   // group index in K
      uint32_t b0[4] = {0u, 0u, 0u, 0u}, b1[4] = {0u, 0u, 0u, 0u};
      if (g < PL) {
        const int c = 2 * gk + (q >> 1), j0 = 2 * (q & 1), sw = (c >> 1) & 3;
        const uint4 *src = xs + (size_t)g * (K / 8) + c * 4;
        const uint4 u0 = src[j0 ^ sw], u1 = src[(j0 + 1) ^ sw];
        b0[0] = u0.x; b0[1] = u0.y; b0[2] = u0.z; b0[3] = u0.w;
        b1[0] = u1.x; b1[1] = u1.y; b1[2] = u1.z; b1[3] = u1.w;
      }
      __syncwarp();   // the MMAs below are warp-collective
      const float xc = 136.0f * (xsum[2 * gk] + xsum[2 * gk + 1]);
      float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4)
        mma16816(d, nib_pair_bf16(wl[j].x >> (4 * s4)), nib_pair_bf16(wh[j].x >> (4 * s4)),
                 nib_pair_bf16(wl[j].y >> (4 * s4)), nib_pair_bf16(wh[j].y >> (4 * s4)), b0[s4],
                 b1[s4]);
      acc0 = fmaf(sl[j], (d[0] + d[1]) - xc, acc0);
      acc1 = fmaf(sh[j], (d[2] + d[3]) - xc, acc1);
    }
  };
  if (i0 < i1) {
    Slot cur = slot_of(slot_index(i0));
    Slot nxt = cur;
    int staged = -1, par = 0;
    load_unit(wl0, wh0, sl0, sh0, cur, group_of(i0), 0);
    load_unit(wl1, wh1, sl1, sh1, cur, group_of(i0), 1);
    float w8 = 1.f;   // routing weights of cur and nxt (warps 0 and 1)
    if (warp < 2 && cur.e < E) w8 = __ldcg(wts + __ldcg(perm + cur.p0));
    float w8n = w8;
    for (int item = i0; item < i1; ++item, par ^= 1) {
      const int gi = group_of(item);
      // the next item's slot, read one item ahead when the expert changes
      const bool more = item + 1 < i1;
      const int na = more ? slot_index(item + 1) : cur.a;
      if (na != nxt.a) {
        nxt = slot_of(na);
        if (warp < 2) w8n = nxt.e < E ? __ldcg(wts + __ldcg(perm + nxt.p0)) : 1.f;
      }
      if (cur.a != staged) {
        __syncthreads();   // previous readers of xs are done
        // One thread per chunk: 64 bytes per plane in, swizzled out, the
        // chunk sum over the planes.
        for (int c = threadIdx.x; c < K / 32; c += blockDim.x) {
          float sum = 0.f;
#pragma unroll
          for (int pl = 0; pl < PL; ++pl) {
            const size_t row = (size_t)(2 * cur.p0 + pl);   // the position's plane pl
            const uint4 *src = reinterpret_cast<const uint4 *>(act + row * act_stride) + c * 4;
            uint4 v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = __ldcg(src + j);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint32_t u[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
              for (int m = 0; m < 4; ++m)
                sum += __uint_as_float(u[m] << 16) + __uint_as_float(u[m] & 0xFFFF0000u);
            }
            uint4 *dst = xs + (size_t)pl * (K / 8) + c * 4;
#pragma unroll
            for (int j = 0; j < 4; ++j) dst[j ^ ((c >> 1) & 3)] = v[j];
          }
          xsum[c] = sum;
        }
        __syncthreads();
        staged = cur.a;
      }
      float acc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
      mul_unit(wl0, wh0, sl0, sh0, acc[0][0], acc[0][1]);
      if (more) load_unit(wl0, wh0, sl0, sh0, nxt, group_of(item + 1), 0);
      mul_unit(wl1, wh1, sl1, sh1, acc[1][0], acc[1][1]);
      if (more) load_unit(wl1, wh1, sl1, sh1, nxt, group_of(item + 1), 1);
      // The item's partial tiles; warp t sums tile t over the warps and
      // writes it (lanes q = 0 hold columns 0 and 1).
      float2 *pp = part + par * (kWarps * 2 * 32);
#pragma unroll
      for (int t = 0; t < 2; ++t) pp[(warp * 2 + t) * 32 + lane] = make_float2(acc[t][0], acc[t][1]);
      __syncthreads();
      if (warp < 2 && q == 0) {
        const int t = warp;
        float r0 = 0.f, r1 = 0.f;
        for (int v = 0; v < kWarps; ++v) {   // warp order: the same sum every run
          const float2 pv = pp[(v * 2 + t) * 32 + lane];
          r0 += pv.x;
          r1 += pv.y;
        }
        out_y[(size_t)cur.p0 * out_stride + gi * kRowsPerItem + 16 * t + g] = w8 * r0;
        out_y[(size_t)cur.p0 * out_stride + gi * kRowsPerItem + 16 * t + g + 8] = w8 * r1;
      }
      if (more && nxt.a != cur.a) {
        cur = nxt;
        w8 = w8n;
      }
    }
  }
}

template <int G>
cudaError_t launch_w2_ks(const moe_handle *h, cudaStream_t st) {
  constexpr int K = 512 * G;
  const size_t smem = (size_t)2 * K * 2 + K / 8 + (size_t)2 * kWarps * 2 * 32 * 8;
  int per_sm = 1;
  const cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &per_sm, gemv_w2_ks_kernel<G>, kWarps * 32, smem);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  return launch_k(h->pdl, gemv_w2_ks_kernel<G>, dim3(h->num_sms * per_sm), dim3(kWarps * 32),
                  smem, st, h->ws.hpl, K, h->k, h->E, h->I, K, h->H, h->S ? h->H : 0,
                  h->ex.w2q, h->ex.w2s, h->sh.w2q, h->sh.w2s, h->ws.active, h->ws.n_active,
                  h->ws.offsets, h->ws.perm, h->ws.w, h->ws.y, h->H, next_layer_prefetch(h));
}

cudaError_t launch_w2_mma(const moe_handle *h, cudaStream_t st) {
  const int h_stride = h->I > h->Is ? h->I : h->Is;
  const int K_s = h->S ? h->Is : h->I;
  const size_t smem = w2_mma_smem(h_stride);
  static bool attr = false;
  if (!attr) {
    cudaError_t err = cudaFuncSetAttribute(gemv_w2_mma_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (err != cudaSuccess) return err;
    attr = true;
  }
  // Exactly the resident CTAs: items are dealt as contiguous per-CTA ranges.
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_w2_mma_kernel, kWarps * 32,
                                                    smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return launch_k(h->pdl, gemv_w2_mma_kernel, dim3(h->num_sms * per_sm), dim3(kWarps * 32), smem,
                  st, h->ws.hpl, h_stride, h->k, h->E, h->I, K_s, h->H, h->S ? h->H : 0, h->ex.w2q,
                  h->ex.w2s, h->sh.w2q, h->sh.w2s, h->ws.active, h->ws.n_active, h->ws.offsets,
                  h->ws.perm, h->ws.w, h->ws.y, h->H, next_layer_prefetch(h));
}

template <int NT, int PL, int MODE>
cudaError_t launch_bf16(const moe_handle *h, const __nv_bfloat16 *act, int act_stride, int T,
                        int K_r, int K_s, int rows_r, int rows_s, const uint8_t *wq_r,
                        const float *ws_r, const uint8_t *wq_s, const float *ws_s, float *out_y,
                        __nv_bfloat16 *out_h, int out_stride, cudaStream_t st) {
  const int Kmax = K_r > K_s ? K_r : K_s;
  const size_t smem = (size_t)PL * NT * (Kmax / 8) * 16 + (size_t)NT * (Kmax / 32) * 4;
  static bool attr = false;
  if (!attr) {
    cudaError_t err = cudaFuncSetAttribute(gemv_bf16_kernel<NT, PL, MODE>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kActSmemBytes);
    if (err != cudaSuccess) return err;
    attr = true;
  }
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_bf16_kernel<NT, PL, MODE>,
                                                    kWarps * 32, smem) != cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  return launch_k(h->pdl, gemv_bf16_kernel<NT, PL, MODE>, dim3(h->num_sms * per_sm),
                  dim3(kWarps * 32), smem, st, act, act_stride, T, h->k, h->E, K_r, K_s, rows_r,
                  rows_s, wq_r, ws_r, wq_s, ws_s, h->ws.active, h->ws.n_active, h->ws.offsets,
                  h->ws.perm, h->ws.w, out_y, out_h, out_stride,
                  MODE == 1 ? next_layer_prefetch(h) : L2Prefetch{});
}

template <int NT>
cudaError_t launch_nt(const moe_handle *h, const void *act, int act_bf16, int T,
                      cudaStream_t st) {
  const int K = h->H;
  const size_t smem = (size_t)NT * K * sizeof(float);
  static bool attr = false;
  if (!attr) {
    cudaError_t err = cudaFuncSetAttribute(
        gemv_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kActSmemBytes);
    if (err != cudaSuccess) return err;
    attr = true;
  }
  // Exactly the resident CTAs: items are split into contiguous per-CTA ranges,
  // so a CTA that waited for a slot would add a second wave.
  int per_sm = 1;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<NT>, kWarps * 32, smem) !=
          cudaSuccess ||
      per_sm < 1)
    per_sm = 1;
  const int h_stride = h->I > h->Is ? h->I : h->Is;
  return launch_k(h->pdl, gemv_kernel<NT>, dim3(h->num_sms * per_sm), dim3(kWarps * 32), smem, st,
                  act, act_bf16, h->H, T, h->k, h->E, K, K, 2 * h->I, h->S ? 2 * h->Is : 0,
                  h->ex.w13q, h->ex.w13s, h->sh.w13q, h->sh.w13s, h->ws.active, h->ws.n_active,
                  h->ws.offsets, h->ws.perm, h->ws.hpl, h_stride);
}

}  // namespace

// Shared memory of the bf16-pair kernel: PL planes of NT tokens' activations
// and their chunk sums.
static size_t bf16_smem(int NT, int PL, int K) {
  return (size_t)PL * NT * (K / 8) * 16 + (size_t)NT * (K / 32) * 4;
}

cudaError_t launch_gemv_w13(const moe_handle *h, const void *x, int T, cudaStream_t st) {
  const int H = h->H, h_stride = h->I > h->Is ? h->I : h->Is;
  if (h->L.x_dtype == 1 && bf16_smem(4, 1, H) <= (size_t)kActSmemBytes) {
    const __nv_bfloat16 *xb = reinterpret_cast<const __nv_bfloat16 *>(x);
#define MOE_W13(NT)                                                                             \
  return launch_bf16<NT, 1, 0>(h, xb, H, T, H, H, 2 * h->I, h->S ? 2 * h->Is : 0, h->ex.w13q,   \
                               h->ex.w13s, h->sh.w13q, h->sh.w13s, nullptr, h->ws.hpl, h_stride, \
                               st)
    if (T >= 3) MOE_W13(4);
    if (T == 2) MOE_W13(2);
    MOE_W13(1);
#undef MOE_W13
  }
  // f32 activations: tokens per pass up to 4, as many as fit 96 KB.
  const int fit = kActSmemBytes / (H * 4);
  if (fit >= 4 && T >= 3) return launch_nt<4>(h, x, h->L.x_dtype == 1, T, st);
  if (fit >= 2 && T >= 2) return launch_nt<2>(h, x, h->L.x_dtype == 1, T, st);
  return launch_nt<1>(h, x, h->L.x_dtype == 1, T, st);
}

cudaError_t launch_gemv_w2(const moe_handle *h, int T, cudaStream_t st) {
  const int h_stride = h->I > h->Is ? h->I : h->Is;
  // T = 1: the K-split MMA kernel where routed and shared experts share a K
  // of 1024 or 2048 (its register pipeline holds one item per lane); else the
  // tiled MMA kernel when an item takes few tile iterations (K <= 4096: each
  // iteration ends at a CTA barrier; at K = 6144 (W13) and 14336 (a
  // Mixtral-shaped W2) the SIMT kernel measured faster).
  const int K_s = h->S ? h->Is : h->I;
  if (T == 1 && K_s == h->I && h->I == 2048) return launch_w2_ks<4>(h, st);
  if (T == 1 && K_s == h->I && h->I == 1024) return launch_w2_ks<2>(h, st);
  if (T == 1 && h_stride <= 4096 && w2_mma_smem(h_stride) <= 113 * 1024) return launch_w2_mma(h, st);
#define MOE_W2(NT)                                                                             \
  return launch_bf16<NT, 2, 1>(h, h->ws.hpl, h_stride, T, h->I, h->S ? h->Is : h->I, h->H,     \
                               h->S ? h->H : 0, h->ex.w2q, h->ex.w2s, h->sh.w2q, h->sh.w2s,     \
                               h->ws.y, nullptr, h->H, st)
  if (T >= 2 && bf16_smem(2, 2, h_stride) <= (size_t)kActSmemBytes) MOE_W2(2);
  MOE_W2(1);
#undef MOE_W2
}

}  // namespace moe
