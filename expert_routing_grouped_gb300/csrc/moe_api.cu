// moe_api.cu -- the C ABI declared in include/moe.h.
//
// moe_init validates the layout, makes ONE device allocation that holds the
// library's copy of the weights and a workspace sized for max_tokens (the
// pages pre-allocate one pool at init and only do pointer arithmetic per call:
// pure-C Colibri tutorial, trdm.cn, §2.2 and §3.2; Colibri C + cuBLASLt
// tutorial, cf-1.com, §2.2 "Unified Memory Pool"), and copies the weights in.
// moe_forward only launches kernels on the caller's stream.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "moe_internal.cuh"

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Carver {
  char *base;
  size_t off = 0;
  template <class T>
  T *take(size_t n) {
    off = align_up(off, kAlign);
    T *p = base ? reinterpret_cast<T *>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
};

int validate_layout(const moe_layout *L) {
  if (!L) return MOE_ERR_ARG;
  if (L->num_experts < 1 || L->num_experts > moe::kMaxExperts) return MOE_ERR_ROUTING;
  if (L->top_k < 1 || L->top_k > L->num_experts || L->top_k > moe::kMaxTopK) return MOE_ERR_ROUTING;
  if (L->router_mode < 0 || L->router_mode > 2) return MOE_ERR_ROUTING;
  if (L->n_group < 0 || L->n_group > 32 || !(L->top_p >= 0.f)) return MOE_ERR_ROUTING;
  if (L->n_group > 1) {
    const int gsz = L->num_experts / L->n_group;
    if (L->router_mode != 1 || L->num_experts % L->n_group || gsz < 2 || L->topk_group < 1 ||
        L->topk_group > L->n_group || L->top_k > L->topk_group * gsz)
      return MOE_ERR_ROUTING;
  }
  if (!(L->routed_scaling_factor > 0.f)) return MOE_ERR_ROUTING;
  if (L->hidden < 512 || L->hidden % 512) return MOE_ERR_ARG;
  if (L->intermediate < 1024 || L->intermediate % 1024) return MOE_ERR_ARG;
  if (L->n_shared != 0 && L->n_shared != 1) return MOE_ERR_ARG;
  if (L->n_shared && (L->shared_intermediate < 1024 || L->shared_intermediate % 1024))
    return MOE_ERR_ARG;
  if (L->x_dtype != 0 && L->x_dtype != 1) return MOE_ERR_ARG;
  if (L->max_tokens < 1 || (long long)L->max_tokens * L->top_k > (1LL << 26)) return MOE_ERR_ARG;
  return MOE_OK;
}

int validate_weights(const moe_layout *L, const moe_weights *W) {
  if (!W) return MOE_ERR_ARG;
  if (!W->router_w || !W->w1_q || !W->w1_s || !W->w3_q || !W->w3_s || !W->w2_q || !W->w2_s)
    return MOE_ERR_ARG;
  if (L->router_mode == 1 && !W->router_bias) return MOE_ERR_ARG;
  if (L->n_shared && (!W->sw1_q || !W->sw1_s || !W->sw3_q || !W->sw3_s || !W->sw2_q || !W->sw2_s))
    return MOE_ERR_ARG;
  return MOE_OK;
}

// Test hook: MOE_FAULT_ALLOC_AT=n makes the n-th device allocation of a
// moe_init call report failure, to exercise the clean-up path.
bool fault_alloc(int n) {
  const char *v = getenv("MOE_FAULT_ALLOC_AT");
  return v && atoi(v) == n;
}

void carve(moe_handle *h, Carver &c) {
  const size_t E = h->E, H = h->H, I = h->I, Is = h->Is, S = h->S, k = h->k;
  const size_t maxT = h->L.max_tokens, A = maxT * k, rows = A + S * maxT;
  const size_t Imax = I > Is ? I : Is;
  h->wr_t = c.take<float>(E * H);
  h->wr_planes = c.take<__nv_bfloat16>(3 * E * H);
  h->bias = c.take<float>(E);
  h->hnorm = c.take<float>(2);
  h->ex.w13q = c.take<uint8_t>(E * 2 * I * H / 2);
  h->ex.w2q = c.take<uint8_t>(E * H * I / 2);
  h->ex.w13s = c.take<float>(E * 2 * I * H / 64);
  h->ex.w2s = c.take<float>(E * H * I / 64);
  h->ex.w13e = c.take<float>(E * 2 * I);
  h->ex.w2e = c.take<float>(E * H);
  if (S) {
    h->sh.w13q = c.take<uint8_t>(2 * Is * H / 2);
    h->sh.w2q = c.take<uint8_t>(H * Is / 2);
    h->sh.w13s = c.take<float>(2 * Is * H / 64);
    h->sh.w2s = c.take<float>(H * Is / 64);
    h->sh.w13e = c.take<float>(2 * Is);
    h->sh.w2e = c.take<float>(H);
  }
  moe::Workspace &w = h->ws;
  // router partial logits: up to kRouterSplitMax splits of the small-T GEMV
  // router, and of the batched routers up to kRouterSplitTokens tokens
  const size_t zrows = std::max({maxT, (size_t)moe::kRouterSplitMax * moe::kRouteTokens,
                                 (size_t)moe::kRouterSplitMax *
                                     std::min(maxT, (size_t)moe::kRouterSplitTokens)});
  w.z_part = c.take<float>(zrows * E);
  w.idx = c.take<int32_t>(A);
  w.w = c.take<float>(A);
  w.counts = c.take<int32_t>(E);
  w.offsets = c.take<int32_t>(E + 1);
  w.perm = c.take<int32_t>(A);
  w.inv = c.take<int32_t>(A);
  w.active = c.take<int32_t>(E + 1);
  w.n_active = c.take<int32_t>(1);
  w.tiles = c.take<int32_t>(A / moe::kTileTokens + E + maxT / moe::kTileTokens + 2);
  w.n_tiles = c.take<int32_t>(2);
  w.status = c.take<int32_t>(1);
  w.ticket = c.take<int32_t>(1 + (E + 7) / 8);
  w.route_kv = c.take<float>(2 * (size_t)moe::kRouteTokens * E);
  w.usage = c.take<unsigned long long>(E);
  w.hpl = c.take<__nv_bfloat16>(2 * rows * Imax);
  w.hb = c.take<__half>(rows * Imax);
  w.y = c.take<float>(rows * H);
  w.xp = c.take<__half>(rows * H);
  w.wperm = c.take<float>(rows);
  w.xcol = c.take<float>(rows);
  w.hcol = c.take<float>(rows);
  const size_t rows_x = (size_t)moe::kExactTokens * (h->k + S);
  w.xe = c.take<__nv_bfloat16>(2 * rows_x * H);
  w.he = c.take<__nv_bfloat16>(2 * rows_x * Imax);
  // Decode tensor-core kernel: row blocks of the larger pass (W13: 2I or 2Is
  // rows per expert, W2: H) over the most experts a decode batch activates,
  // and one partial-sum slot per (CTA, row block) segment and pipeline.
  const size_t n_r = std::min<size_t>(E, (size_t)moe::kExactTokens * k);
  const size_t rb13 = n_r * (2 * I / 128) + S * (2 * Is / 128);
  const size_t rb2 = (n_r + S) * (H / 128);
  h->dec_rb_max = (int)std::max(rb13, rb2);
  const size_t slots = ((size_t)h->num_sms + h->dec_rb_max) * moe::kDecPipes;
  w.dec_partial = c.take<float>(slots * 128 * moe::kDecTokens);
  w.dec_ticket = c.take<int32_t>(2 * (size_t)h->dec_rb_max);
  w.x_stage = c.take<char>(maxT * H * h->x_elem);
  w.out_stage = c.take<float>(maxT * H);
}

// Copies one expert set (E routed experts, or the shared one) from the
// canonical layout into the library layout, staging through a bounded device
// buffer so host and device sources are handled alike.
int copy_expert_set(const moe::ExpertWeights &dst, const uint8_t *w1q, const float *w1s,
                    const uint8_t *w3q, const float *w3s, const uint8_t *w2q, const float *w2s,
                    size_t n_exp, size_t H, size_t I, char *stage, size_t stage_bytes) {
  const size_t qrow = H / 2, srow = H / 64;                 // W1/W3 row bytes / groups
  const size_t per_exp = 2 * I * qrow + 2 * I * srow * 4;   // staged bytes per expert (W1+W3)
  size_t chunk = stage_bytes / per_exp;
  if (chunk < 1) return MOE_ERR_NOMEM;
  if (chunk > n_exp) chunk = n_exp;
  for (size_t e0 = 0; e0 < n_exp; e0 += chunk) {
    const size_t ne = (e0 + chunk <= n_exp) ? chunk : n_exp - e0;
    uint8_t *t1 = reinterpret_cast<uint8_t *>(stage);
    uint8_t *t3 = t1 + ne * I * qrow;
    float *ts1 = reinterpret_cast<float *>(t3 + ne * I * qrow);
    float *ts3 = ts1 + ne * I * srow;
    if (cudaMemcpy(t1, w1q + e0 * I * qrow, ne * I * qrow, cudaMemcpyDefault) != cudaSuccess ||
        cudaMemcpy(t3, w3q + e0 * I * qrow, ne * I * qrow, cudaMemcpyDefault) != cudaSuccess ||
        cudaMemcpy(ts1, w1s + e0 * I * srow, ne * I * srow * 4, cudaMemcpyDefault) != cudaSuccess ||
        cudaMemcpy(ts3, w3s + e0 * I * srow, ne * I * srow * 4, cudaMemcpyDefault) != cudaSuccess)
      return MOE_ERR_DEVICE;
    if (moe::launch_repack_w13(t1, t3, const_cast<uint8_t *>(dst.w13q) + e0 * 2 * I * qrow,
                               (long long)ne, (int)I, (int)qrow, 0) != cudaSuccess ||
        moe::launch_repack_w13_scales(ts1, ts3, const_cast<float *>(dst.w13s) + e0 * 2 * I * srow,
                                      (long long)ne, (int)I, (int)srow, 0) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return MOE_ERR_DEVICE;
  }
  // W2 [n_exp][H][I/2]: plain copy, then repack the nibbles in place.
  if (cudaMemcpy(const_cast<uint8_t *>(dst.w2q), w2q, n_exp * H * I / 2, cudaMemcpyDefault) !=
          cudaSuccess ||
      cudaMemcpy(const_cast<float *>(dst.w2s), w2s, n_exp * H * (I / 64) * 4, cudaMemcpyDefault) !=
          cudaSuccess ||
      moe::launch_repack_words(const_cast<uint8_t *>(dst.w2q), (long long)(n_exp * H * I / 2), 0) !=
          cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return MOE_ERR_DEVICE;
  return MOE_OK;
}

// The tensor-core path's fp16 range control, from the repacked weights: the
// per-row power-of-two factors of W13 and W2, and the largest W1 / W3 row
// norms (raised into hnorm, which the caller zeroes first).
int tc_weight_factors(const moe::ExpertWeights &ew, size_t n_exp, size_t H, size_t I,
                      float *hnorm) {
  if (moe::launch_row_pow2(ew.w13s, (long long)(n_exp * 2 * I), (int)(H / 64),
                           const_cast<float *>(ew.w13e), 0) != cudaSuccess ||
      moe::launch_row_pow2(ew.w2s, (long long)(n_exp * H), (int)(I / 64),
                           const_cast<float *>(ew.w2e), 0) != cudaSuccess ||
      moe::launch_w13_norm(ew.w13q, ew.w13s, (long long)(n_exp * 2 * I), (int)(H / 2), hnorm,
                           0) != cudaSuccess)
    return MOE_ERR_DEVICE;
  return MOE_OK;
}

int copy_weights(moe_handle *h, const moe_weights *W) {
  const size_t E = h->E, H = h->H, I = h->I, Is = h->Is;
  // One staging buffer: at least one expert's W1+W3, at most 512 MB.
  const size_t Imax = I > Is ? I : Is;
  const size_t per_exp = 2 * Imax * (H / 2) + 2 * Imax * (H / 64) * 4;
  size_t stage_bytes = (size_t)512 << 20;
  if (stage_bytes < per_exp) stage_bytes = per_exp;
  if (stage_bytes > per_exp * E) stage_bytes = per_exp * (E > 1 ? E : 1);
  char *stage = nullptr;
  if (fault_alloc(2) || cudaMalloc(&stage, stage_bytes) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NOMEM;
  }
  int rc = copy_expert_set(h->ex, W->w1_q, W->w1_s, W->w3_q, W->w3_s, W->w2_q, W->w2_s, E, H, I,
                           stage, stage_bytes);
  if (rc == MOE_OK && h->S)
    rc = copy_expert_set(h->sh, W->sw1_q, W->sw1_s, W->sw3_q, W->sw3_s, W->sw2_q, W->sw2_s, 1, H,
                         Is, stage, stage_bytes);
  if (rc == MOE_OK && cudaMemset(h->hnorm, 0, 2 * sizeof(float)) != cudaSuccess) rc = MOE_ERR_DEVICE;
  if (rc == MOE_OK) rc = tc_weight_factors(h->ex, E, H, I, h->hnorm);
  if (rc == MOE_OK && h->S) rc = tc_weight_factors(h->sh, 1, H, Is, h->hnorm);
  if (rc == MOE_OK) {
    if (W->router_bias) {
      if (cudaMemcpy(h->bias, W->router_bias, E * 4, cudaMemcpyDefault) != cudaSuccess)
        rc = MOE_ERR_DEVICE;
    } else if (cudaMemset(h->bias, 0, E * 4) != cudaSuccess) {
      rc = MOE_ERR_DEVICE;
    }
  }
  // Router: canonical [H][E] -> [E][H] through the staging buffer.
  if (rc == MOE_OK) {
    float *tmp = reinterpret_cast<float *>(stage);
    if (E * H * 4 > stage_bytes) {
      rc = MOE_ERR_NOMEM;
    } else if (cudaMemcpy(tmp, W->router_w, E * H * 4, cudaMemcpyDefault) != cudaSuccess ||
               moe::launch_transpose_router(tmp, h->wr_t, (int)H, (int)E, 0) != cudaSuccess ||
               moe::launch_split_planes(h->wr_t, h->wr_planes, (long long)(E * H), 0) !=
                   cudaSuccess ||
               cudaDeviceSynchronize() != cudaSuccess) {
      rc = MOE_ERR_DEVICE;
    }
  }
  cudaFree(stage);
  return rc;
}

}  // namespace

namespace moe {
L2Prefetch next_layer_prefetch(const moe_handle *h) {
  L2Prefetch pf{};
  const moe_handle *nx = h->next;
  if (!nx) return pf;
  auto add = [&pf](const void *p, size_t bytes) {
    if (p && bytes >= 16 && pf.n < L2Prefetch::kMax) {
      pf.ptr[pf.n] = static_cast<const char *>(p);
      pf.bytes[pf.n] = bytes & ~static_cast<size_t>(15);
      ++pf.n;
    }
  };
  const size_t E = nx->E, H = nx->H, Is = nx->Is;
  add(nx->wr_t, E * H * 4);
  if (nx->S) {
    add(nx->sh.w13q, 2 * Is * H / 2);
    add(nx->sh.w13s, 2 * Is * (H / 64) * 4);
    add(nx->sh.w2q, H * Is / 2);
    add(nx->sh.w2s, H * (Is / 64) * 4);
  }
  return pf;
}
}  // namespace moe

namespace {

int choose_regime(const moe_handle *h, int T) {
  if (h->regime_opt == 1) return 1;
  if (h->regime_opt == 2) return 2;
  if (h->regime_opt == 3) return T <= moe::kExactTokens ? 3 : 1;
  if (!moe::tc_path_available() || T <= h->small_t_max) return 1;
  return T <= moe::kExactTokens ? 3 : 2;
}

// Records the boundary after a stage when tracing is on.
void mark(moe_handle *h, const char *name, cudaStream_t st) {
  if (!h->profile || h->n_ev > moe_handle::kMaxStages) return;
  if (h->n_ev > 0) h->stage_names[h->n_ev - 1] = name;
  cudaEventRecord(h->ev[h->n_ev++], st);
}

int run_forward(moe_handle *h, const void *x, int T, float *out, bool accumulate,
                cudaStream_t st) {
  int regime = choose_regime(h, T);
  unsigned long long *usage = h->count_usage ? h->ws.usage : nullptr;
  h->n_ev = 0;
  cudaError_t err = cudaSuccess;
  mark(h, nullptr, st);
  if (T <= moe::kRouteTokens) {
    // One launch routes and groups (and clears the status word).
    err = moe::launch_route_small(h, x, T, usage, st);
    h->launches += 1;
    mark(h, "route", st);
  } else {
    err = cudaMemsetAsync(h->ws.status, 0, sizeof(int32_t), st);
    if (err == cudaSuccess) err = moe::launch_router(h, x, T, st);
    h->launches += 2;
    mark(h, "router", st);
    if (err == cudaSuccess) err = moe::launch_dispatch(h, T, moe::kTileTokens, usage, st);
    h->launches += 3;   // ranks, scan, scatter
    mark(h, "dispatch", st);
  }
  if (err == cudaSuccess) {
    if (regime == 1) {
      err = moe::launch_gemv_w13(h, x, T, st);
      h->launches += 1;
      mark(h, "w13", st);
      if (err == cudaSuccess) err = moe::launch_gemv_w2(h, T, st);
      h->launches += 1;
      mark(h, "w2", st);
      if (err == cudaSuccess) err = moe::launch_combine(h, T, out, accumulate, st);
      h->launches += 1;
      mark(h, "combine", st);
    } else if (regime == 3) {
      err = moe::launch_decode_tc(h, x, T, out, accumulate, st);
    } else {
      err = moe::launch_tc_path(h, x, T, out, accumulate, st);
    }
  }
  h->last_T = T;
  h->last_regime = regime;
  h->last_stream = st;
  return err == cudaSuccess ? MOE_OK : MOE_ERR_DEVICE;
}

// device: x and out are device pointers the kernels access directly.
int check_call(moe_handle *h, const void *x, int T, const void *out, bool device = true) {
  if (!h || T < 0) return MOE_ERR_ARG;
  if (T > h->L.max_tokens) return MOE_ERR_NOMEM;
  if (T > 0 && (!x || !out)) return MOE_ERR_ARG;
  // x is read and out written with 16-byte vector accesses.
  if (device && T > 0 && (((uintptr_t)x | (uintptr_t)out) & 15)) return MOE_ERR_ARG;
  return MOE_OK;
}

}  // namespace

extern "C" {

__attribute__((visibility("default"))) int moe_init(const moe_layout *layout,
                                                    const moe_weights *weights,
                                                    moe_handle **out) {
  if (!out) return MOE_ERR_ARG;
  *out = nullptr;
  int rc = validate_layout(layout);
  if (rc) return rc;
  rc = validate_weights(layout, weights);
  if (rc) return rc;
  moe_handle *h = new (std::nothrow) moe_handle();
  if (!h) return MOE_ERR_NOMEM;
  h->L = *layout;
  h->E = layout->num_experts;
  h->k = layout->top_k;
  h->H = layout->hidden;
  h->I = layout->intermediate;
  h->S = layout->n_shared;
  h->Is = layout->n_shared ? layout->shared_intermediate : 0;
  h->x_elem = layout->x_dtype == 1 ? 2 : 4;
  h->regime_opt = 0;
  h->small_t_max = 1;
  h->pdl = 1;
  h->wait_ns = 2000000000ull;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    delete h;
    return MOE_ERR_DEVICE;
  }
  Carver sizer{nullptr};
  carve(h, sizer);
  h->pool_bytes = align_up(sizer.off, kAlign);
  if (fault_alloc(1) || cudaMalloc(&h->pool, h->pool_bytes) != cudaSuccess) {
    cudaGetLastError();
    h->pool = nullptr;
    delete h;
    return MOE_ERR_NOMEM;
  }
  Carver c{static_cast<char *>(h->pool)};
  carve(h, c);
  rc = copy_weights(h, weights);
  if (rc == MOE_OK && (cudaMemset(h->ws.status, 0, 4) != cudaSuccess ||
                       cudaMemset(h->ws.ticket, 0, (1 + (h->E + 7) / 8) * 4) != cudaSuccess ||
                       cudaMemset(h->ws.usage, 0, (size_t)h->E * 8) != cudaSuccess ||
                       cudaMemset(h->ws.dec_ticket, 0, 2 * (size_t)h->dec_rb_max * 4) != cudaSuccess))
    rc = MOE_ERR_DEVICE;
  if (rc != MOE_OK) {
    cudaFree(h->pool);
    delete h;
    return rc;
  }
  *out = h;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_forward(moe_handle *h, const void *x, int T,
                                                       float *out, moe_stream_t stream) {
  int rc = check_call(h, x, T, out);
  if (rc || T == 0) return rc;
  return run_forward(h, x, T, out, false, reinterpret_cast<cudaStream_t>(stream));
}

__attribute__((visibility("default"))) int moe_route(moe_handle *h, const void *x, int T,
                                                     moe_stream_t stream) {
  int rc = check_call(h, x, T, x);
  if (rc || T == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemsetAsync(h->ws.status, 0, sizeof(int32_t), st);
  if (err == cudaSuccess) err = moe::launch_router(h, x, T, st);
  if (err == cudaSuccess) err = moe::launch_dispatch(h, T, moe::kTileTokens, nullptr, st);
  h->last_T = T;
  h->last_regime = 0;
  h->last_stream = st;
  return err == cudaSuccess ? MOE_OK : MOE_ERR_DEVICE;
}

__attribute__((visibility("default"))) int moe_forward_residual(moe_handle *h, const void *x,
                                                                int T, float *resid,
                                                                moe_stream_t stream) {
  int rc = check_call(h, x, T, resid);
  if (rc || T == 0) return rc;
  return run_forward(h, x, T, resid, true, reinterpret_cast<cudaStream_t>(stream));
}

__attribute__((visibility("default"))) int moe_forward_residual_norm(
    moe_handle *h, const void *x, int T, float *resid, float eps, uint16_t *norm_out,
    moe_stream_t stream) {
  int rc = check_call(h, x, T, resid);
  if (rc) return rc;
  if (!(eps >= 0.f)) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  // norm_out is written with 16-byte accesses and must not overlap resid,
  // which the same kernel reads and writes (it may be x: x is no longer read
  // when the combine runs).
  const uintptr_t nb = reinterpret_cast<uintptr_t>(norm_out),
                  rb = reinterpret_cast<uintptr_t>(resid);
  const size_t nlen = (size_t)T * h->H * sizeof(uint16_t), rlen = (size_t)T * h->H * sizeof(float);
  if (!norm_out || (nb & 15) || (nb < rb + rlen && rb < nb + nlen)) return MOE_ERR_ARG;
  h->norm_out = norm_out;
  h->norm_eps = eps;
  rc = run_forward(h, x, T, resid, true, reinterpret_cast<cudaStream_t>(stream));
  h->norm_out = nullptr;
  return rc;
}

__attribute__((visibility("default"))) int moe_forward_host(moe_handle *h, const void *x_host,
                                                            int T, float *out_host,
                                                            moe_stream_t stream) {
  int rc = check_call(h, x_host, T, out_host, false);
  if (rc || T == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const size_t xb = (size_t)T * h->H * h->x_elem, ob = (size_t)T * h->H * sizeof(float);
  if (cudaMemcpyAsync(h->ws.x_stage, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return MOE_ERR_DEVICE;
  // A pinned, 16-byte aligned output buffer that the GPU can address (on a
  // Grace host, over NVLink-C2C) is written by the combine kernel itself: its
  // stores carry the device-to-host transfer, and no copy follows the layer.
  // Any other buffer gets the result through the staging copy.
  float *out_dev = h->ws.out_stage;
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, out_host) == cudaSuccess && at.type == cudaMemoryTypeHost &&
      at.devicePointer && (reinterpret_cast<uintptr_t>(at.devicePointer) & 15) == 0)
    out_dev = static_cast<float *>(at.devicePointer);
  rc = run_forward(h, h->ws.x_stage, T, out_dev, false, st);
  if (rc) return rc;
  if (out_dev == h->ws.out_stage &&
      cudaMemcpyAsync(out_host, h->ws.out_stage, ob, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MOE_ERR_DEVICE;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_DEVICE;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_rmsnorm_bf16(const float *x, int T, int H,
                                                            float eps, uint16_t *out,
                                                            moe_stream_t stream) {
  if (T < 0 || H <= 0 || H % 8 || !(eps >= 0.f)) return MOE_ERR_ARG;
  if (T == 0) return MOE_OK;
  if (!x || !out || ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(out)) & 15))
    return MOE_ERR_ARG;
  return moe::launch_rmsnorm_bf16(x, T, H, eps, out, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? MOE_OK
             : MOE_ERR_DEVICE;
}

__attribute__((visibility("default"))) int moe_set_option(moe_handle *h, int option, int value) {
  if (!h) return MOE_ERR_ARG;
  if (option == MOE_OPT_REGIME) {
    if (value < 0 || value > 3) return MOE_ERR_ARG;
    h->regime_opt = value;
    return MOE_OK;
  }
  if (option == MOE_OPT_SMALL_T_MAX) {
    if (value < 0) return MOE_ERR_ARG;
    h->small_t_max = value;
    return MOE_OK;
  }
  if (option == MOE_OPT_PROFILE) {
    if (value != 0 && value != 1) return MOE_ERR_ARG;
    if (value && !h->ev[0]) {
      for (int i = 0; i <= moe_handle::kMaxStages; ++i)
        if (cudaEventCreate(&h->ev[i]) != cudaSuccess) return MOE_ERR_DEVICE;
    }
    h->profile = value;
    h->n_ev = 0;
    return MOE_OK;
  }
  if (option == MOE_OPT_PDL) {
    if (value != 0 && value != 1) return MOE_ERR_ARG;
    h->pdl = value;
    return MOE_OK;
  }
  if (option == MOE_OPT_WAIT_LIMIT_US) {
    if (value < 0) return MOE_ERR_ARG;
    h->wait_ns = value == 0 ? 0ull : (unsigned long long)value * 1000ull;
    return MOE_OK;
  }
  if (option == MOE_OPT_USAGE) {
    if (value != 0 && value != 1) return MOE_ERR_ARG;
    h->count_usage = value;
    return MOE_OK;
  }
  return MOE_ERR_ARG;
}

__attribute__((visibility("default"))) int moe_usage_read(moe_handle *h, int64_t *host_counts,
                                                          int n_experts) {
  if (!h || !host_counts || n_experts != h->E) return MOE_ERR_ARG;
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess ||
      cudaMemcpy(host_counts, h->ws.usage, (size_t)h->E * 8, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_DEVICE;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_usage_reset(moe_handle *h) {
  if (!h) return MOE_ERR_ARG;
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess ||
      cudaMemset(h->ws.usage, 0, (size_t)h->E * 8) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess)
    return MOE_ERR_DEVICE;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_set_next_layer(moe_handle *h,
                                                              const moe_handle *next) {
  if (!h || next == h) return MOE_ERR_ARG;
  h->next = next;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_debug_view(moe_handle *h, moe_debug *d) {
  if (!h || !d) return MOE_ERR_ARG;
  d->T = h->last_T;
  d->idx = h->ws.idx;
  d->w = h->ws.w;
  d->counts = h->ws.counts;
  d->offsets = h->ws.offsets;
  d->perm = h->ws.perm;
  d->inv = h->ws.inv;
  d->status = h->ws.status;
  d->regime = h->last_regime;
  d->launches = h->launches;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_debug_read(moe_handle *h, int field,
                                                          void *host_dst, size_t bytes) {
  if (!h || !host_dst) return MOE_ERR_ARG;
  const size_t A = (size_t)h->last_T * h->k;
  const void *src = nullptr;
  size_t need = 0;
  switch (field) {
    case MOE_DBG_IDX: src = h->ws.idx; need = A * 4; break;
    case MOE_DBG_W: src = h->ws.w; need = A * 4; break;
    case MOE_DBG_COUNTS: src = h->ws.counts; need = (size_t)h->E * 4; break;
    case MOE_DBG_OFFSETS: src = h->ws.offsets; need = (size_t)(h->E + 1) * 4; break;
    case MOE_DBG_PERM: src = h->ws.perm; need = A * 4; break;
    case MOE_DBG_INV: src = h->ws.inv; need = A * 4; break;
    default: return MOE_ERR_ARG;
  }
  if (bytes != need) return MOE_ERR_ARG;
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess) return MOE_ERR_DEVICE;
  if (need && cudaMemcpy(host_dst, src, need, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_DEVICE;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_stage_times(moe_handle *h, float *ms,
                                                           const char **names, int max, int *n) {
  if (!h || !ms || !n || max < 0) return MOE_ERR_ARG;
  *n = 0;
  if (!h->profile || h->n_ev < 2) return MOE_OK;
  if (cudaEventSynchronize(h->ev[h->n_ev - 1]) != cudaSuccess) return MOE_ERR_DEVICE;
  const int stages = h->n_ev - 1;
  for (int i = 0; i < stages && i < max; ++i) {
    if (cudaEventElapsedTime(&ms[i], h->ev[i], h->ev[i + 1]) != cudaSuccess) return MOE_ERR_DEVICE;
    if (names) names[i] = h->stage_names[i];
  }
  *n = stages < max ? stages : max;
  return MOE_OK;
}

__attribute__((visibility("default"))) int moe_status(moe_handle *h, int32_t *status) {
  if (!h || !status) return MOE_ERR_ARG;
  if (cudaStreamSynchronize(h->last_stream) != cudaSuccess) return MOE_ERR_DEVICE;
  if (cudaMemcpy(status, h->ws.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_DEVICE;
  return MOE_OK;
}

__attribute__((visibility("default"))) size_t moe_device_bytes(const moe_handle *h) {
  return h ? h->pool_bytes : 0;
}

__attribute__((visibility("default"))) void moe_free(moe_handle *h) {
  if (!h) return;
  if (h->pool) cudaFree(h->pool);
  for (int i = 0; i <= moe_handle::kMaxStages; ++i)
    if (h->ev[i]) cudaEventDestroy(h->ev[i]);
  delete h;
}

__attribute__((visibility("default"))) const char *moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_NOMEM: return "out of memory, or T > max_tokens";
    case MOE_ERR_ROUTING: return "invalid routing layout";
    case MOE_ERR_DEVICE: return "CUDA error or device status";
    case MOE_ERR_ARG: return "invalid argument";
    case MOE_ERR_IO: return "usage-history file error";
    case MOE_ERR_ENGINE: return "usage history of another engine or shape";
    default: return "unknown error";
  }
}

}  // extern "C"
