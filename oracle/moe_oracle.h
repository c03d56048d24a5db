/*
 * moe_oracle.h -- plain, slow, f64 CPU definition of one MoE-layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  This oracle exists to check the CUDA path; only
 * the test suite, the package smoke check and the benchmark's CPU-baseline leg
 * may load it.  It shares no code with the CUDA library (the one shared piece
 * is the seeded input generator in synth/, which holds none of the layer's
 * arithmetic).
 *
 * The layer, in the order the pages give it ("Colibri" C + cuBLASLt tutorial,
 * cf-1.com, §2.1 five-step list and §3.3 Steps 2-5):
 *   1. router logits  z = x . Wr            (router kept in f32: colibrì engine
 *                                            teardown, text-matrix.pages.dev, "System map")
 *   2. top-k ids and weights                (softmax, or sigmoid + noaux_tc with
 *                                            n_group = 1 times routed_scaling_factor:
 *                                            colibrì engine teardown, "Three key engineering
 *                                            decisions" (1))
 *   3. group assignments by expert          (counting sort: counts, prefix sum,
 *                                            scatter; tutorial §3.3 Step 3)
 *   4. per-expert SwiGLU FFN over its group (W1, W3 then W2; skip empty experts;
 *                                            tutorial §3.3 Step 4), int4 weights with
 *                                            one f32 scale per 64 along K (gs64,
 *                                            teardown "Three key engineering decisions")
 *   5. weighted sum back to token order     (tutorial §3.3 Step 5), plus the always-
 *                                            applied shared expert (teardown "System map",
 *                                            tier 1)
 *
 * Layouts (canonical, host memory):
 *   x          [T][H]   f32 (x_dtype 0) or bf16 bits (x_dtype 1)
 *   router_w   [H][E]   f32, rows indexed by h (pure-C Colibri tutorial,
 *                        trdm.cn, §3.1: router is [hidden_size, num_experts])
 *   router_bias[E]      f32 or NULL
 *   W1, W3     [I][H/2] packed int4 (even K index in the low nibble), scales [I][H/64] f32
 *   W2         [H][I/2] packed int4, scales [H][I/64] f32
 * Per-expert pointer arrays may hold NULL for experts that no token selects.
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
  int32_t num_experts;          /* E                                      */
  int32_t top_k;                /* k                                      */
  int32_t hidden;               /* H (multiple of 64)                     */
  int32_t intermediate;         /* I (multiple of 64)                     */
  int32_t n_shared;             /* 0 or 1                                 */
  int32_t shared_intermediate;  /* I of the shared expert                 */
  int32_t router_mode;          /* 0 softmax, 1 sigmoid + noaux_tc,
                                   2 softmax without renormalisation      */
  int32_t x_dtype;              /* 0 f32, 1 bf16                          */
  double routed_scaling_factor; /* rsf                                    */
  int32_t n_group;              /* 0 or 1: no groups; > 1: grouped noaux_tc
                                   (sigmoid mode only), E % n_group == 0   */
  int32_t topk_group;           /* groups kept when n_group > 1           */
  double top_p;                 /* adaptive expert top-p; 0 or >= 1: off  */
} oracle_layout;

typedef struct {
  const float *router_w;
  const float *router_bias;
  const uint8_t *const *w1_q;
  const float *const *w1_s;
  const uint8_t *const *w3_q;
  const float *const *w3_s;
  const uint8_t *const *w2_q;
  const float *const *w2_s;
  const uint8_t *sw1_q, *sw3_q, *sw2_q;
  const float *sw1_s, *sw3_s, *sw2_s;
} oracle_weights;

/* Step 1: z[T][E] in f64. */
int oracle_router_logits(const oracle_layout *L, const oracle_weights *W,
                         const void *x, int T, double *z);

/* Steps 1-2: idx[T][k], w[T][k]; key[T][E] and gap[T] optional (may be NULL).
 * gap[t] is the token's decision margin: the smallest difference between
 * adjacent keys among the top-(k+1) sorted eligible keys (all of them when
 * fewer), and, where they apply, between adjacent group scores among the
 * top-(topk_group+1), and between the top-p threshold and each cumulative
 * share it is compared with.  With top-p on, a dropped slot holds id -1 and
 * weight 0. */
int oracle_route(const oracle_layout *L, const oracle_weights *W, const void *x,
                 int T, int32_t *idx, double *w, double *key, double *gap);

/* Steps 2 only, from given logits z[T][E] (f64). */
int oracle_route_from_logits(const oracle_layout *L, const float *router_bias,
                             const double *z, int T, int32_t *idx, double *w,
                             double *key, double *gap);

/* Step 3: counts[E], offsets[E+1], perm[T*k], inv[T*k].  An id of -1 (a slot
 * the top-p trim dropped) is no assignment: not counted, inv = -1, and perm
 * lists only the offsets[E] real assignments. */
int oracle_dispatch(const int32_t *idx, int T, int k, int E, int32_t *counts,
                    int32_t *offsets, int32_t *perm, int32_t *inv);

/* gs64 dequantisation of one row of K packed int4 weights, exact in f64. */
int oracle_dequant_row(const uint8_t *q, const float *s, int K, double *out);

/* Step 4 for one expert and n rows: y[n][H] = W2 . (silu(W1 x) * (W3 x)). */
int oracle_expert_ffn(int H, int I, const uint8_t *w1q, const float *w1s,
                      const uint8_t *w3q, const float *w3s, const uint8_t *w2q,
                      const float *w2s, const double *x, int n, double *y);

/* Pre-norm of the layer stack: out[t] = x[t] / sqrt(mean_h x[t][h]^2 + eps),
 * no learned gain.  The pages' forward normalises (RMSNorm) before the MoE
 * layer (Colibri C + cuBLASLt tutorial, cf-1.com, §2.1 step 1); the norm is
 * kept in f32 on the GPU (colibrì engine teardown, "System map"). */
int oracle_rmsnorm(const float *x, int T, int H, double eps, double *out);

/* The whole layer.  out[T][H] f64; idx/w may be NULL. */
int oracle_moe_forward(const oracle_layout *L, const oracle_weights *W,
                       const void *x, int T, double *out, int32_t *idx, double *w);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ORACLE_H */
