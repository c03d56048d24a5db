/*
 * moe_oracle.c -- plain f64 definition of one MoE-layer forward.
 *
 * TEST INFRASTRUCTURE ONLY (see moe_oracle.h).  Single-threaded, no blocking,
 * no fusion: each step is written as the pages state it, in their order, so it
 * can be checked by eye.  Readings of points the pages leave open are marked
 * "Reading:".
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define OR_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- inputs -- */

static double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* x[t][h] as f64 (exact from f32 or bf16). */
static double x_at(const oracle_layout *L, const void *x, int t, int h) {
  size_t i = (size_t)t * (size_t)L->hidden + (size_t)h;
  if (L->x_dtype == 1) return bf16_to_f64(((const uint16_t *)x)[i]);
  return (double)((const float *)x)[i];
}

static int check_layout(const oracle_layout *L) {
  if (!L) return -4;
  if (L->num_experts < 1 || L->top_k < 1 || L->top_k > L->num_experts) return -2;
  if (L->router_mode < 0 || L->router_mode > 2) return -2;
  if (L->n_group < 0 || !(L->top_p >= 0.0)) return -2;
  if (L->n_group > 1) {
    const int gsize = L->num_experts / L->n_group;
    if (L->router_mode != 1 || L->num_experts % L->n_group || gsize < 2) return -2;
    if (L->topk_group < 1 || L->topk_group > L->n_group) return -2;
    if (L->top_k > L->topk_group * gsize) return -2;
  }
  if (L->hidden <= 0 || L->intermediate <= 0) return -4;
  if (L->hidden % 64 || L->intermediate % 64) return -4;
  if (L->n_shared != 0 && L->n_shared != 1) return -4;
  if (L->n_shared && (L->shared_intermediate <= 0 || L->shared_intermediate % 64)) return -4;
  if (L->x_dtype != 0 && L->x_dtype != 1) return -4;
  return 0;
}

/* ------------------------------------------------------- step 1: router -- */

/* z[t][e] = sum over h (ascending) of x[t][h] * Wr[h][e]; Wr is [hidden,
 * num_experts] (pure-C Colibri tutorial, trdm.cn, §3.1) and stays f32 (colibrì
 * engine teardown, text-matrix.pages.dev, "System map": norm/router/bias f32). */
OR_API int oracle_router_logits(const oracle_layout *L, const oracle_weights *W,
                                const void *x, int T, double *z) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (T < 0 || (T > 0 && (!W || !W->router_w || !x || !z))) return -4;
  const int H = L->hidden, E = L->num_experts;
  /* Each z[t][e] accumulates its products in ascending h; walking h in the
   * outer loop only makes the Wr reads contiguous. */
  for (int t = 0; t < T; ++t) {
    double *zt = z + (size_t)t * E;
    for (int e = 0; e < E; ++e) zt[e] = 0.0;
    for (int h = 0; h < H; ++h) {
      const double xv = x_at(L, x, t, h);
      const float *wr = W->router_w + (size_t)h * E;
      for (int e = 0; e < E; ++e) zt[e] += xv * (double)wr[e];
    }
  }
  return 0;
}

/* ----------------------------------------------- step 2: top-k + weights -- */

static double sigmoid(double v) { return 1.0 / (1.0 + exp(-v)); }

typedef struct {
  double key;
  int e;
} keyed;

/* Reading: ties go to the lowest expert index; slots are ordered by
 * descending key, then ascending index.  A full sort, not a heap. */
static int keyed_cmp(const void *a, const void *b) {
  const keyed *p = (const keyed *)a, *q = (const keyed *)b;
  if (p->key > q->key) return -1;
  if (p->key < q->key) return 1;
  return (p->e > q->e) - (p->e < q->e);
}

/*
 * Softmax modes (tutorial cf-1.com §2.1 step 2: "linear layer + softmax ->
 * top-2 ids and weights"): logits l = z + b (b an additive logit bias, zero
 * when absent); p = softmax(l) over all E; select the k largest (softmax is
 * monotone, so the key is l itself).  Mode 0: w_j = p[idx_j] / sum_sel p * rsf
 * (Reading: renormalised over the selection).  Mode 2: w_j = p[idx_j] * rsf,
 * the unrenormalised variant.
 *
 * Sigmoid + noaux_tc (teardown "Three key engineering decisions" (1)):
 * s = sigmoid(z); key = s + b (the selection bias enters selection only);
 * select the k largest keys; w_j = s[idx_j] / sum_sel s * rsf.  With
 * n_group <= 1 every expert is eligible.  With n_group > 1 (Reading: the
 * published group-limited noaux_tc): the experts form n_group contiguous groups
 * of E / n_group; a group's score is the sum of its two largest keys; the
 * topk_group groups with the largest scores (ties to the lower group) stay
 * eligible, and the k experts are chosen among their members only.
 *
 * Adaptive expert top-p (colibri tuning guide, gitcode.com, knob table:
 * "--topp", a lossy trim of the expert set).  Reading: with the slots in
 * selection order and q_j = (slot j's weight before rsf) / (sum over the
 * selection), slot j is kept while the cumulative share of the slots before
 * it, C_j = q_0 + ... + q_{j-1}, is below top_p (slot 0 always).  Dropped
 * slots get id -1 and weight 0.  Modes 0 and 1 renormalise the kept weights
 * over the kept slots; mode 2 keeps its unrenormalised weights.
 */
static int groups_on(const oracle_layout *L) { return L->n_group > 1; }
static int top_p_on(const oracle_layout *L) { return L->top_p > 0.0 && L->top_p < 1.0; }

OR_API int oracle_route_from_logits(const oracle_layout *L, const float *router_bias,
                                    const double *z, int T, int32_t *idx, double *w,
                                    double *key, double *gap) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (T < 0 || (T > 0 && (!z || !idx || !w))) return -4;
  if (L->router_mode == 1 && !router_bias) return -4;
  const int E = L->num_experts, k = L->top_k;
  const int G = groups_on(L) ? L->n_group : 1, gsize = E / G;
  keyed *ks = (keyed *)malloc(sizeof(keyed) * (size_t)E);
  keyed *gs = (keyed *)malloc(sizeof(keyed) * (size_t)G);
  double *val = (double *)malloc(sizeof(double) * (size_t)E);
  int *eligible = (int *)malloc(sizeof(int) * (size_t)E);
  double *kk = (double *)malloc(sizeof(double) * (size_t)E);   /* keys in expert order */
  if (!ks || !gs || !val || !eligible || !kk) {
    free(ks);
    free(gs);
    free(val);
    free(eligible);
    free(kk);
    return -1;
  }
  for (int t = 0; t < T; ++t) {
    const double *zt = z + (size_t)t * E;
    if (L->router_mode != 1) {
      /* p = softmax(z + b) over all experts. */
      double m = -INFINITY;
      for (int e = 0; e < E; ++e) {
        kk[e] = zt[e] + (router_bias ? (double)router_bias[e] : 0.0);
        if (kk[e] > m) m = kk[e];
      }
      double sum = 0.0;
      for (int e = 0; e < E; ++e) {
        val[e] = exp(kk[e] - m);
        sum += val[e];
      }
      for (int e = 0; e < E; ++e) val[e] /= sum;
    } else {
      for (int e = 0; e < E; ++e) {
        val[e] = sigmoid(zt[e]);
        kk[e] = val[e] + (double)router_bias[e];
      }
    }
    if (key)
      for (int e = 0; e < E; ++e) key[(size_t)t * E + e] = kk[e];
    double g = INFINITY;   /* decision margin */

    /* Group-limited eligibility. */
    for (int e = 0; e < E; ++e) eligible[e] = 1;
    if (groups_on(L)) {
      for (int gi = 0; gi < G; ++gi) {
        for (int j = 0; j < gsize; ++j) {
          ks[j].key = kk[gi * gsize + j];
          ks[j].e = gi * gsize + j;
        }
        qsort(ks, (size_t)gsize, sizeof(keyed), keyed_cmp);
        gs[gi].key = ks[0].key + ks[1].key;
        gs[gi].e = gi;
      }
      qsort(gs, (size_t)G, sizeof(keyed), keyed_cmp);
      for (int e = 0; e < E; ++e) eligible[e] = 0;
      for (int j = 0; j < L->topk_group; ++j)
        for (int i = 0; i < gsize; ++i) eligible[gs[j].e * gsize + i] = 1;
      if (L->topk_group < G) {
        for (int j = 0; j < L->topk_group; ++j) {
          const double d = gs[j].key - gs[j + 1].key;
          if (d < g) g = d;
        }
      }
    }

    /* Top-k over the eligible experts. */
    int n = 0;
    for (int e = 0; e < E; ++e)
      if (eligible[e]) {
        ks[n].key = kk[e];
        ks[n].e = e;
        ++n;
      }
    qsort(ks, (size_t)n, sizeof(keyed), keyed_cmp);
    const int top = (k < n) ? k + 1 : n;
    for (int j = 0; j + 1 < top; ++j) {
      const double d = ks[j].key - ks[j + 1].key;
      if (d < g) g = d;
    }

    /* Weights, then the top-p trim. */
    double sel = 0.0;
    for (int j = 0; j < k; ++j) sel += val[ks[j].e];
    int kept = k;
    if (top_p_on(L)) {
      double cum = 0.0;
      for (int j = 1; j < k; ++j) {
        cum += val[ks[j - 1].e] / sel;
        const double d = fabs(cum - L->top_p);
        if (d < g) g = d;
        if (kept == k && cum >= L->top_p) kept = j;
      }
    }
    double norm = 0.0;
    for (int j = 0; j < kept; ++j) norm += val[ks[j].e];
    for (int j = 0; j < k; ++j) {
      const size_t a = (size_t)t * k + j;
      if (j >= kept) {
        idx[a] = -1;
        w[a] = 0.0;
      } else {
        idx[a] = ks[j].e;
        w[a] = (L->router_mode == 2 ? val[ks[j].e] : val[ks[j].e] / norm) *
               L->routed_scaling_factor;
      }
    }
    if (gap) gap[t] = g;
  }
  free(ks);
  free(gs);
  free(val);
  free(eligible);
  free(kk);
  return 0;
}

OR_API int oracle_route(const oracle_layout *L, const oracle_weights *W, const void *x,
                        int T, int32_t *idx, double *w, double *key, double *gap) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (T == 0) return 0;
  if (!W) return -4;
  double *z = (double *)malloc(sizeof(double) * (size_t)T * (size_t)L->num_experts);
  if (!z) return -1;
  rc = oracle_router_logits(L, W, x, T, z);
  if (!rc) rc = oracle_route_from_logits(L, W->router_bias, z, T, idx, w, key, gap);
  free(z);
  return rc;
}

/* --------------------------------------------- step 3: group by expert -- */

/* Counting sort (tutorial cf-1.com §3.3 Step 3): counts per expert, prefix
 * sum into offsets[E+1], then scatter.  The assignment of token t's slot j is
 * a = t*k + j; scanning a in ascending order keeps each expert's group in
 * ascending token order (Reading: stable; the §2.2 example, routes
 * [0,2,1,0,2,1] -> e0 <- {t0,t3}, e1 <- {t2,t5}, e2 <- {t1,t4}, is consistent).
 * inv[a] is the position of assignment a in the grouped order. */
OR_API int oracle_dispatch(const int32_t *idx, int T, int k, int E, int32_t *counts,
                           int32_t *offsets, int32_t *perm, int32_t *inv) {
  if (T < 0 || k < 1 || E < 1 || !counts || !offsets) return -4;
  if (T > 0 && (!idx || !perm || !inv)) return -4;
  const int A = T * k;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (int a = 0; a < A; ++a) {
    if (idx[a] == -1) continue;   /* a slot dropped by the top-p trim */
    if (idx[a] < 0 || idx[a] >= E) return -2;
    counts[idx[a]] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t *fill = (int32_t *)calloc((size_t)E, sizeof(int32_t));
  if (!fill) return -1;
  for (int a = 0; a < A; ++a) {
    int e = idx[a];
    if (e == -1) {
      inv[a] = -1;
      continue;
    }
    int pos = offsets[e] + fill[e]++;
    perm[pos] = a;
    inv[a] = pos;
  }
  free(fill);
  return 0;
}

/* ------------------------------------------------- step 4: expert FFNs -- */

/* One packed byte holds two consecutive K indices, the even one in the low
 * nibble; a nibble is a two's-complement int4 in [-8, 7].  Weight k of the row
 * is q_k * s[k/64]: one f32 scale per 64 weights along K (gs64, teardown
 * "Three key engineering decisions" (1)).  Exact in f64. */
OR_API int oracle_dequant_row(const uint8_t *q, const float *s, int K, double *out) {
  if (!q || !s || !out || K <= 0 || K % 64) return -4;
  for (int kk = 0; kk < K; ++kk) {
    uint8_t byte = q[kk / 2];
    int nib = (kk % 2 == 0) ? (byte & 0xF) : (byte >> 4);
    int v = (nib >= 8) ? nib - 16 : nib;
    out[kk] = (double)v * (double)s[kk / 64];
  }
  return 0;
}

/* SwiGLU expert (tutorial cf-1.com §2.1 step 4, "W1, W2, W3"):
 *   g = W1 x, u = W3 x, h = silu(g) * u with silu(g) = g / (1 + e^-g),
 *   y = W2 h.
 * W1, W3 are [I][H]; W2 is [H][I].  All n rows of x share one pass over each
 * weight row (the per-expert mini-batch of the pages). */
OR_API int oracle_expert_ffn(int H, int I, const uint8_t *w1q, const float *w1s,
                             const uint8_t *w3q, const float *w3s, const uint8_t *w2q,
                             const float *w2s, const double *x, int n, double *y) {
  if (H <= 0 || I <= 0 || H % 64 || I % 64 || n < 0) return -4;
  if (n == 0) return 0;
  if (!w1q || !w1s || !w3q || !w3s || !w2q || !w2s || !x || !y) return -4;
  double *row1 = (double *)malloc(sizeof(double) * (size_t)H);
  double *row3 = (double *)malloc(sizeof(double) * (size_t)H);
  double *row2 = (double *)malloc(sizeof(double) * (size_t)I);
  double *h = (double *)malloc(sizeof(double) * (size_t)n * (size_t)I);
  if (!row1 || !row3 || !row2 || !h) {
    free(row1);
    free(row3);
    free(row2);
    free(h);
    return -1;
  }
  for (int i = 0; i < I; ++i) {
    oracle_dequant_row(w1q + (size_t)i * (H / 2), w1s + (size_t)i * (H / 64), H, row1);
    oracle_dequant_row(w3q + (size_t)i * (H / 2), w3s + (size_t)i * (H / 64), H, row3);
    for (int r = 0; r < n; ++r) {
      const double *xr = x + (size_t)r * H;
      double g = 0.0, u = 0.0;
      for (int c = 0; c < H; ++c) {
        g += row1[c] * xr[c];
        u += row3[c] * xr[c];
      }
      h[(size_t)r * I + i] = g / (1.0 + exp(-g)) * u;
    }
  }
  for (int o = 0; o < H; ++o) {
    oracle_dequant_row(w2q + (size_t)o * (I / 2), w2s + (size_t)o * (I / 64), I, row2);
    for (int r = 0; r < n; ++r) {
      const double *hr = h + (size_t)r * I;
      double acc = 0.0;
      for (int c = 0; c < I; ++c) acc += row2[c] * hr[c];
      y[(size_t)r * H + o] = acc;
    }
  }
  free(row1);
  free(row3);
  free(row2);
  free(h);
  return 0;
}

/* ------------------------------------------------ stack pre-norm (f64) -- */

OR_API int oracle_rmsnorm(const float *x, int T, int H, double eps, double *out) {
  if (T < 0 || H <= 0 || eps < 0.0 || (T > 0 && (!x || !out))) return -4;
  for (int t = 0; t < T; ++t) {
    double ss = 0.0;
    for (int h = 0; h < H; ++h) ss += (double)x[(size_t)t * H + h] * (double)x[(size_t)t * H + h];
    double r = 1.0 / sqrt(ss / (double)H + eps);
    for (int h = 0; h < H; ++h) out[(size_t)t * H + h] = (double)x[(size_t)t * H + h] * r;
  }
  return 0;
}

/* ---------------------------------------------------- the whole layer -- */

OR_API int oracle_moe_forward(const oracle_layout *L, const oracle_weights *W,
                              const void *x, int T, double *out, int32_t *idx_out,
                              double *w_out) {
  int rc = check_layout(L);
  if (rc) return rc;
  if (T < 0) return -4;
  if (T == 0) return 0;
  if (!W || !x || !out) return -4;
  if (L->n_shared && (!W->sw1_q || !W->sw1_s || !W->sw3_q || !W->sw3_s || !W->sw2_q || !W->sw2_s))
    return -4;
  const int E = L->num_experts, k = L->top_k, H = L->hidden, I = L->intermediate;
  const int A = T * k;
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)A);
  double *w = (double *)malloc(sizeof(double) * (size_t)A);
  int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
  int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * (size_t)(E + 1));
  int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * (size_t)A);
  int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * (size_t)A);
  double *xg = (double *)malloc(sizeof(double) * (size_t)A * H);  /* grouped inputs  */
  double *yg = (double *)malloc(sizeof(double) * (size_t)A * H);  /* grouped outputs */
  double *xs = (double *)malloc(sizeof(double) * (size_t)T * H);
  double *ys = (double *)malloc(sizeof(double) * (size_t)T * H);
  if (!idx || !w || !counts || !offsets || !perm || !inv || !xg || !yg || !xs || !ys) {
    rc = -1;
    goto done;
  }

  /* Steps 1-2. */
  rc = oracle_route(L, W, x, T, idx, w, NULL, NULL);
  if (rc) goto done;

  /* Step 3. */
  rc = oracle_dispatch(idx, T, k, E, counts, offsets, perm, inv);
  if (rc) goto done;

  /* Step 4: gather each expert's group and run its FFN; skip empty experts
   * (tutorial cf-1.com §3.3 Step 4: "if expert_counts[i] == 0, skip"). */
  for (int p = 0; p < offsets[E]; ++p) {   /* the real assignments */
    int t = perm[p] / k;
    for (int c = 0; c < H; ++c) xg[(size_t)p * H + c] = x_at(L, x, t, c);
  }
  for (int e = 0; e < E; ++e) {
    if (counts[e] == 0) continue;
    if (!W->w1_q || !W->w1_q[e] || !W->w1_s[e] || !W->w3_q[e] || !W->w3_s[e] || !W->w2_q[e] ||
        !W->w2_s[e]) {
      rc = -4;
      goto done;
    }
    rc = oracle_expert_ffn(H, I, W->w1_q[e], W->w1_s[e], W->w3_q[e], W->w3_s[e], W->w2_q[e],
                           W->w2_s[e], xg + (size_t)offsets[e] * H, counts[e],
                           yg + (size_t)offsets[e] * H);
    if (rc) goto done;
  }
  /* The shared expert sees every token (teardown "System map", tier 1:
   * the shared expert is resident and applied on every layer). */
  if (L->n_shared) {
    for (int t = 0; t < T; ++t)
      for (int c = 0; c < H; ++c) xs[(size_t)t * H + c] = x_at(L, x, t, c);
    rc = oracle_expert_ffn(H, L->shared_intermediate, W->sw1_q, W->sw1_s, W->sw3_q, W->sw3_s,
                           W->sw2_q, W->sw2_s, xs, T, ys);
    if (rc) goto done;
  }

  /* Step 5: out[t] = sum over j ascending of w[t][j] * y[(t,j)], then the
   * shared expert's output with weight 1 (Reading: the shared expert is not
   * scaled by the routing weights or by rsf). */
  for (int t = 0; t < T; ++t)
    for (int c = 0; c < H; ++c) {
      double acc = 0.0;
      for (int j = 0; j < k; ++j) {
        int a = t * k + j;
        if (inv[a] < 0) continue;   /* dropped by the top-p trim */
        acc += w[a] * yg[(size_t)inv[a] * H + c];
      }
      if (L->n_shared) acc += ys[(size_t)t * H + c];
      out[(size_t)t * H + c] = acc;
    }
  if (idx_out) memcpy(idx_out, idx, sizeof(int32_t) * (size_t)A);
  if (w_out) memcpy(w_out, w, sizeof(double) * (size_t)A);

done:
  free(idx);
  free(w);
  free(counts);
  free(offsets);
  free(perm);
  free(inv);
  free(xg);
  free(yg);
  free(xs);
  free(ys);
  return rc;
}
