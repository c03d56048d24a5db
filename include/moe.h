/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE-layer forward library, libmoe.so.
 *
 * One call runs one Mixture-of-Experts layer over T tokens on one GPU:
 *
 *   1. router   z = x . Wr (f32), then softmax top-k, or sigmoid scores with a
 *               noaux_tc selection bias (n_group = 1); the k selected weights
 *               are renormalised and multiplied by routed_scaling_factor.
 *               (colibrì engine teardown, text-matrix.pages.dev, "Three key
 *               engineering decisions" (1): sigmoid + noaux_tc with
 *               routed_scaling_factor; "System map": router, norm and bias f32.
 *               Colibri C + cuBLASLt tutorial, cf-1.com, §2.1 step 2: linear
 *               layer + softmax -> top-k ids and weights.)
 *               Variants: softmax weights left unrenormalised (router_mode 2,
 *               w_j = p_j * rsf with p the softmax over all E); group-limited
 *               noaux_tc (n_group > 1: E/n_group contiguous experts per group,
 *               a group scored by the sum of its two largest keys, the
 *               topk_group best groups eligible, ties to the lower group); and
 *               the adaptive expert top-p trim of the colibri tuning guide
 *               (gitcode.com, knob table, "--topp"; lossy): with slots in
 *               selection order and q_j each slot's share of the selected
 *               weights, slot j is kept while q_0 + ... + q_{j-1} < top_p
 *               (slot 0 always); a dropped slot gets id -1 and weight 0 and is
 *               not dispatched; modes 0 and 1 renormalise over the kept slots.
 *   2. dispatch a counting sort that groups the T*k assignments by expert:
 *               per-expert counts, prefix-sum offsets, a permutation, and no
 *               allocation (tutorial cf-1.com §3.3 Step 3; pure-C Colibri
 *               tutorial, trdm.cn, §2.2: a pre-allocated pool, only pointer
 *               arithmetic at run time).
 *   3. experts  SwiGLU FFN per expert over its group, y = W2 (silu(W1 x) * W3 x),
 *               with int4 weights carrying one f32 scale per 64 weights along K
 *               (gs64; teardown "Three key engineering decisions" (1)), plus an
 *               always-applied shared expert (teardown "System map", tier 1).
 *               Empty experts are skipped (tutorial cf-1.com §3.3 Step 4).
 *   4. combine  out[t] = sum_j w[t][j] * y(t, j) + y_shared(t), in a fixed order,
 *               without atomics (tutorial cf-1.com §3.3 Step 5).
 *
 * The API follows the pages' engine interface -- init with a maximum batch,
 * forward, free; batch 0 is a dry run; negative return codes; one instance per
 * thread (pure-C Colibri tutorial, trdm.cn, §4.2 and §5.1-5.2) -- with the
 * layout and the CUDA stream made explicit.
 *
 * Canonical weight layout (what moe_init reads; host or device memory):
 *   router_w     [H][E]     f32, row h holds the E logits' weights
 *   router_bias  [E]        f32: softmax mode, an additive logit offset (may be
 *                           NULL); sigmoid mode, the noaux_tc selection bias
 *                           (required; it enters selection only)
 *   w1_q, w3_q   [E][I][H/2] packed int4: byte b of a row holds K indices 2b
 *                           (low nibble) and 2b+1 (high nibble); a nibble is a
 *                           two's-complement value in [-8, 7]
 *   w1_s, w3_s   [E][I][H/64] f32 gs64 scales: weight k of a row is q_k * s[k/64]
 *   w2_q         [E][H][I/2] packed int4, w2_s [E][H][I/64] f32
 *   sw*_q/_s     the shared expert's W1/W3 [Is][H/2],[Is][H/64] and W2
 *                [H][Is/2],[H][Is/64]; NULL when n_shared == 0
 * Experts are contiguous by id (tutorial cf-1.com §3.1: base + id * size).
 *
 * Numerics.  Routing, dispatch and the decode expert paths (T <= 8 by default:
 * the SIMT GEMV path for one token, the exact tensor-core path for 2-8) compute
 * in f32: exact int4 codes, f32 (or exactly split bf16 hi/lo) operands, f32
 * group scales and accumulation.  The large-T expert path feeds the tensor
 * cores with bf16(q * s) weights and bf16 activations and accumulates in f32.
 * The output is f32.  Results are bitwise identical from run to run.
 *
 * Return codes (extending the pages' 0 / -1 / -2 / -3):
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_NOMEM (-1)    /* out of memory at init, or T > max_tokens        */
#define MOE_ERR_ROUTING (-2)  /* invalid routing layout: top_k < 1 or > E,
                                 E > 1024, unknown router_mode, a group rule
                                 that does not fit, top_p < 0 or NaN            */
#define MOE_ERR_DEVICE (-3)   /* CUDA error, or a nonzero device status word     */
#define MOE_ERR_ARG (-4)      /* NULL pointer, a size not a multiple of 64,
                                 unsupported dtype, bad option                  */
#define MOE_ERR_IO (-5)       /* a usage-history file could not be opened,
                                 written or parsed                              */
#define MOE_ERR_ENGINE (-6)   /* a usage history written by another engine, or
                                 for other dimensions                           */

/* A CUDA stream (cudaStream_t); NULL is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef struct moe_layout {
  int32_t num_experts;           /* E, 1..1024                                   */
  int32_t top_k;                 /* k, 1..min(E, 32)                             */
  int32_t hidden;                /* H, a multiple of 512                         */
  int32_t intermediate;          /* I, a multiple of 1024 (routed experts)       */
  int32_t n_shared;              /* 0 or 1                                       */
  int32_t shared_intermediate;   /* I of the shared expert (multiple of 1024)    */
  int32_t router_mode;           /* 0 softmax, 1 sigmoid + noaux_tc, 2 softmax
                                    without renormalisation                      */
  float routed_scaling_factor;   /* rsf (1.0 for plain softmax routers)          */
  int32_t x_dtype;               /* 0 f32, 1 bf16                                */
  int32_t max_tokens;            /* largest T a forward call may pass (>= 1)     */
  /* Router variants; all zero gives the plain rules above. */
  int32_t n_group;               /* 0 or 1: every expert eligible; 2..32: group-
                                    limited noaux_tc (router_mode 1 only)        */
  int32_t topk_group;            /* groups kept, 1..n_group (n_group > 1)        */
  float top_p;                   /* adaptive expert top-p in (0, 1); 0 (or >= 1)
                                    off                                          */
} moe_layout;

typedef struct moe_weights {
  const float *router_w;
  const float *router_bias;
  const uint8_t *w1_q;
  const float *w1_s;
  const uint8_t *w3_q;
  const float *w3_s;
  const uint8_t *w2_q;
  const float *w2_s;
  const uint8_t *sw1_q;
  const float *sw1_s;
  const uint8_t *sw3_q;
  const float *sw3_s;
  const uint8_t *sw2_q;
  const float *sw2_s;
} moe_weights;

typedef struct moe_handle moe_handle;

/* Device pointers into the handle's workspace, valid until the next forward
 * on the handle.  They describe the last forward call. */
typedef struct moe_debug {
  int32_t T;               /* tokens of the last call                           */
  const int32_t *idx;      /* [T][k] selected experts, slots by descending key  */
  const float *w;          /* [T][k] renormalised weights times rsf             */
  const int32_t *counts;   /* [E] assignments per expert                        */
  const int32_t *offsets;  /* [E+1] exclusive prefix sum of counts             */
  const int32_t *perm;     /* [T*k] grouped position -> assignment t*k+j; the
                              first offsets[E] entries are meaningful          */
  const int32_t *inv;      /* [T*k] assignment -> grouped position (-1 for a
                              slot the top-p trim dropped)                     */
  const int32_t *status;   /* one int32 device status word (0 = ok)             */
  int32_t regime;          /* 1 GEMV path, 2 tensor-core path, 3 exact TC path  */
  int64_t launches;        /* kernels launched by this handle since moe_init    */
} moe_debug;

/*
 * Validates the layout, allocates all device memory the handle will ever use
 * (repacked weights and a workspace sized for max_tokens), and copies the
 * weights in.  Weight pointers may be host or device memory; they are not
 * retained.  On failure *out is NULL and nothing is leaked.
 * Returns MOE_OK, MOE_ERR_NOMEM, MOE_ERR_ROUTING, MOE_ERR_ARG or MOE_ERR_DEVICE.
 */
int moe_init(const moe_layout *layout, const moe_weights *weights, moe_handle **out);

/*
 * out[T][H] (f32, device) = MoE(x), x [T][H] device (f32 or bf16 per layout).
 * Asynchronous on `stream`; no allocation, no host synchronisation.
 * T == 0 validates the arguments and launches nothing (dry run; x and out may
 * then be NULL).  T > max_tokens returns MOE_ERR_NOMEM.  x and out must be
 * 16-byte aligned (the kernels use 16-byte vector accesses); a misaligned
 * pointer returns MOE_ERR_ARG before anything is launched.  A handle serves
 * one stream at a time and is not thread-safe.  moe_route and
 * moe_forward_residual take the same checks.
 */
int moe_forward(moe_handle *h, const void *x, int T, float *out, moe_stream_t stream);

/* Steps 1-2 only: routes x [T][H] (device) and groups the assignments by
 * expert, leaving idx, w, counts, offsets, perm and inv in the workspace (read
 * them with moe_debug_view / moe_debug_read).  Lets a caller learn which
 * experts the next call will stream before running it. */
int moe_route(moe_handle *h, const void *x, int T, moe_stream_t stream);

/* As moe_forward, but adds the layer output into resid[T][H] (f32, device):
 * resid += MoE(x).  The residual add is fused into the combine step. */
int moe_forward_residual(moe_handle *h, const void *x, int T, float *resid,
                         moe_stream_t stream);

/*
 * End-to-end call with HOST buffers: copies x (host) into the handle's
 * workspace, runs the layer, delivers the result to out (host), and waits for
 * the stream.  When out is pinned host memory with a device address and
 * 16-byte aligned (cudaPointerGetAttributes reports it as host memory), the
 * combine step writes the result into it directly (on a Grace host, over
 * NVLink-C2C) and no copy follows; any other out buffer receives a copy from
 * the workspace.  The results are the same either way.  Pinned x gives the
 * fastest input copy.
 */
int moe_forward_host(moe_handle *h, const void *x_host, int T, float *out_host,
                     moe_stream_t stream);

/*
 * As moe_forward_residual, and then norm_out[t] = bf16(rmsnorm(resid[t]))
 * from the updated resid, bit for bit what moe_rmsnorm_bf16(resid, T, H, eps,
 * norm_out) would give: the next stacked layer's pre-norm, computed by the
 * kernel that adds the layer output into resid (one launch in place of two;
 * norm before each MoE layer: tutorial cf-1.com §2.1 step 1).  norm_out
 * [T][H] bf16 bits, device, 16-byte aligned: the input of a next layer
 * whose x_dtype is bf16.  It may be x (x is no longer read when it is
 * written) but must not overlap resid.  eps >= 0.
 * Returns as moe_forward_residual; MOE_ERR_ARG also for a null, misaligned
 * or overlapping norm_out or a bad eps.
 */
int moe_forward_residual_norm(moe_handle *h, const void *x, int T, float *resid, float eps,
                              uint16_t *norm_out, moe_stream_t stream);

/*
 * Pre-norm between stacked layers: out_bf16[t] = bf16(x[t] / sqrt(mean(x[t]^2) + eps)),
 * computed in f32 with no learned gain (the pages normalise with RMSNorm before
 * the MoE layer: tutorial cf-1.com §2.1 step 1; the norm stays f32: teardown
 * "System map").  x [T][H] f32 device, out [T][H] bf16 bits device, both
 * 16-byte aligned; H a multiple of 8.
 */
int moe_rmsnorm_bf16(const float *x, int T, int H, float eps, uint16_t *out,
                     moe_stream_t stream);

/* Chooses the expert path: 0 automatic (T <= small_t_max -> the SIMT GEMV
 * path, T <= 8 -> the exact tensor-core path, else tensor cores), 1 always
 * the SIMT GEMV path, 2 always the tensor-core path (fp16 weights and
 * operands with exact power-of-two range control), 3 the exact tensor-core path (T <= 8 only, else the GEMV path:
 * exact int4 codes, f32 operands as bf16 hi/lo pairs, f32 group scales and
 * accumulation -- the GEMV path's numerics, on four MMA pipelines per SM). */
#define MOE_OPT_REGIME 1
/* Largest T that the automatic choice sends to the GEMV path (default 1). */
#define MOE_OPT_SMALL_T_MAX 2
/* 1: record a CUDA event on the forward's stream at every stage boundary
 * (read the stage times with moe_stage_times); 0 (default): no events. */
#define MOE_OPT_PROFILE 3
/* 1: every moe_forward / moe_forward_residual / moe_forward_host call adds its
 * per-expert assignment counts into the handle's 64-bit usage counters (read
 * them with moe_usage_read); the dispatch kernel does the adding, so the option
 * costs no launch.  moe_route (a look-ahead) never counts.  0 (default): off. */
#define MOE_OPT_USAGE 4
/* 1 (default): launch every kernel of a call after the first with
 * programmatic dependent launch -- it may be scheduled while its predecessor
 * on the stream is still running, and waits (griddepcontrol) for it to finish
 * before touching memory, so launch latency and start-up overlap the
 * predecessor's tail.  The first kernel of a call is launched plainly (the
 * wait covers kernels, not the caller's copies or memsets before it).  The
 * same results bit for bit; 0: plain launches. */
#define MOE_OPT_PDL 5
/* The time limit, in microseconds, of each wait between the roles of the
 * pipelined tensor-core kernels (a copy or an MMA that a role waits for);
 * default 2000000 (2 s).  A wait that runs out sets the status word to 2 and
 * the kernel stops its roles, waits (with the full 2 s limit) for its own
 * copies and MMAs in flight, frees its tensor memory and returns, so the next
 * forward runs normally; moe_status reports the 2 and moe_forward returns
 * MOE_OK (the launch succeeded).  0 makes every wait that is not complete
 * when first tested give up at once: a way to exercise that recovery path
 * without a fault or a hang.  Negative values return MOE_ERR_ARG. */
#define MOE_OPT_WAIT_LIMIT_US 6
int moe_set_option(moe_handle *h, int option, int value);

/*
 * Next-layer prefetch (the colibri tuning guide's PILOT, gitcode.com knob
 * table and "PILOT" paragraph: while one layer runs, the engine fetches what
 * the next layer will read, ahead of its routing).  With every weight resident
 * in HBM, the GPU form of that read-ahead is an L2 prefetch of what the next
 * layer reads whatever it routes to: its router weights and its shared
 * expert.  After moe_set_next_layer(h, next), every forward on h issues
 * cp.async.bulk.prefetch.L2 for next's router and shared expert from the W2
 * pass of the GEMV and exact decode paths (T <= 8), spread over its CTAs; it
 * is a hint and changes no result.  next == NULL clears the link; a handle
 * cannot name itself (MOE_ERR_ARG).  next is not owned: clear the link (or
 * free h) before moe_free(next).  Returns MOE_OK or MOE_ERR_ARG.
 */
int moe_set_next_layer(moe_handle *h, const moe_handle *next);

/* Fills *d with device pointers describing the last forward call. */
int moe_debug_view(moe_handle *h, moe_debug *d);

/*
 * Allocation-free routing.  The pages have no counterpart to this call; it
 * exists for callers that cannot call cudaMalloc: code running inside a
 * stream-capture region, where allocation is not allowed; hot loops that must
 * not pay for the device-wide synchronisation cudaMalloc/cudaFree may cause;
 * and processes whose GPU memory is entirely owned by another allocator (a
 * framework's caching allocator, a fixed arena).  Such a caller cannot create
 * a moe_handle, because moe_init allocates.
 *
 * Runs steps 1-2 of the layer (router logits in f32, then softmax or
 * sigmoid + noaux_tc top-k with renormalised weights times rsf) with the same
 * kernels as moe_forward, and allocates nothing: the logit scratch is a fixed
 * 4 MiB array in the library's device image, which every GPU that loads the
 * library keeps until the process exits.
 *   x            [T][hidden] device, f32 (x_dtype 0) or bf16 (x_dtype 1),
 *                16-byte aligned
 *   router_w_eh  [num_experts][hidden] f32 device, 16-byte aligned: row e is
 *                expert e's router vector (the layout of a linear layer's
 *                weight; the transpose of moe_weights.router_w)
 *   router_bias  [num_experts] f32 device, or NULL (softmax mode only)
 *   idx, w       [T][top_k] device outputs, as moe_debug.idx / moe_debug.w
 * router_mode 0, 1 or 2; the group and top-p variants need a handle.
 * Limits: hidden a multiple of 512; num_experts <= 1024; top_k <= 32; for
 * T > 4, T * num_experts <= 1048576 (larger calls return MOE_ERR_NOMEM and
 * launch nothing).  T == 0 does nothing.
 * The first call on each device looks up the scratch array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls share the one scratch array, which
 * keeps the last call's contents; nothing in it needs clearing, because every
 * value a call reads was written earlier in the same call.  Calls that
 * overlap on the GPU (different streams, or concurrent host threads) race on
 * the scratch and must be serialised by the caller.
 * A misaligned x or router_w_eh returns MOE_ERR_ARG before any launch.
 * MOE_ERR_DEVICE reports only errors of this call's own launches.
 * Returns MOE_OK, MOE_ERR_NOMEM, MOE_ERR_ROUTING, MOE_ERR_ARG or MOE_ERR_DEVICE.
 */
int moe_route_noalloc(const void *x, int T, int hidden, int num_experts, int top_k, int x_dtype,
                      int router_mode, float routed_scaling_factor, const float *router_w_eh,
                      const float *router_bias, int32_t *idx, float *w, moe_stream_t stream);

/* Fields of moe_debug_read. */
#define MOE_DBG_IDX 0      /* int32 [T][k]  */
#define MOE_DBG_W 1        /* f32   [T][k]  */
#define MOE_DBG_COUNTS 2   /* int32 [E]     */
#define MOE_DBG_OFFSETS 3  /* int32 [E+1]   */
#define MOE_DBG_PERM 4     /* int32 [T*k]   */
#define MOE_DBG_INV 5      /* int32 [T*k]   */
/* Synchronises the handle's last stream and copies one field of the last
 * forward call into host memory; `bytes` must equal the field's size for the
 * last call's T (MOE_ERR_ARG otherwise). */
int moe_debug_read(moe_handle *h, int field, void *host_dst, size_t bytes);

/* Stage times of the last forward with MOE_OPT_PROFILE on (synchronises).
 * T <= 8: route (router, top-k and dispatch in one kernel), then w13, w2,
 * combine (GEMV path) or gather, w13, w2, combine (tensor-core paths).
 * T > 8: router, dispatch, then the same expert stages.  Writes up to `max`
 * values in ms and the stage count to *n; names[i] (optional) receives static
 * strings. */
int moe_stage_times(moe_handle *h, float *ms, const char **names, int max, int *n);

/* Synchronises the handle's last stream and returns its device status word
 * (0 when every kernel completed normally). */
int moe_status(moe_handle *h, int32_t *status);

/*
 * Expert usage history (colibri tuning guide, gitcode.com, "learned cache":
 * the engine records which experts each layer actually routed to and pins the
 * hottest; "usage-history format": route_trace.h).
 *
 * moe_usage_read synchronises the handle's last stream and copies its usage
 * counters, int64 [num_experts] (assignments per expert summed over the
 * counted forwards since init or the last reset), into host memory;
 * n_experts must equal the layout's.  moe_usage_reset synchronises and zeroes
 * them.  Both return MOE_OK, MOE_ERR_ARG or MOE_ERR_DEVICE.
 */
int moe_usage_read(moe_handle *h, int64_t *host_counts, int n_experts);
int moe_usage_reset(moe_handle *h);

/* Engine identity of a usage history: the FNV-1a 32-bit hash of the engine's
 * name (offset basis 2166136261, prime 16777619, one byte at a time).  The
 * tuning guide gives one value: "glm_moe_dsa" -> 3815245270.  NULL -> 0. */
uint32_t moe_engine_id(const char *name);

/*
 * Writes a usage history in the route_trace text format (colibri tuning guide,
 * "usage-history format"): plain text, one record per line, each record
 * exactly three decimal integers separated by single spaces:
 *   -1 n_layers n_experts            header: dimensions
 *   -2 1 engine_id                   header: format version 1, engine id
 *   layer expert count               one per non-zero count, layer-major,
 *                                    experts ascending
 * Only non-zero counts are written.  A history with no non-zero count is a
 * zero-byte file (no header either), so that a reader can tell "nothing
 * recorded" from the file's size.  counts is host memory, int64
 * [n_layers][n_experts], every value >= 0.  The file is created or truncated.
 * Returns MOE_OK, MOE_ERR_ARG (NULL, n_layers < 1, n_experts < 1, a negative
 * count) or MOE_ERR_IO.
 */
int moe_route_trace_write(const char *path, int n_layers, int n_experts, uint32_t engine_id,
                          const int64_t *counts);

/*
 * Reads a route_trace file and ADDS its counts into counts (host, int64
 * [n_layers][n_experts]; the caller zeroes it first for a plain read).
 * Records whose first field is negative are headers: -1 must carry these
 * dimensions, -2 this engine_id (else MOE_ERR_ENGINE and counts is left as it
 * was); other negative record types are skipped, so that later header types
 * stay readable.  engine_id 0 accepts a history from any engine (the guide
 * trusts a file the user names explicitly, and checks one the engine found by
 * itself); the dimensions are checked either way.  A file with no header (the older headerless form) is
 * accepted as it stands.  A zero-byte file is an empty history: MOE_OK, no
 * change.  A record without exactly three integer fields, or with a layer or
 * expert out of range or a negative count, is MOE_ERR_IO (counts unchanged).
 * *found_engine (optional) receives the -2 record's engine id, 0 if none.
 */
int moe_route_trace_read(const char *path, int n_layers, int n_experts, uint32_t engine_id,
                         int64_t *counts, uint32_t *found_engine);

/* Bytes of device memory the handle owns (weights + workspace). */
size_t moe_device_bytes(const moe_handle *h);

/* Releases everything the handle owns; NULL is a no-op. */
void moe_free(moe_handle *h);

/* Text for a return code. */
const char *moe_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
