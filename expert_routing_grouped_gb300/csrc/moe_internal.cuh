// moe_internal.cuh -- handle layout and kernel entry points shared by the
// library's translation units.  Device code targets sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kRouterSplitMax = 16;   // split-K partitions of the router
constexpr int kRouterSplitTokens = 1024;   // largest T whose router is split above 4 tokens
constexpr int kGemvTokens = 4;        // tokens one GEMV pass carries in registers
constexpr int kRouteTokens = 8;       // largest T of the fused routing launch
constexpr int kTileTokens = 160;      // tokens per tensor-core tile (the MMA's N)
constexpr int kExactTokens = 8;       // largest batch of the exact (f32-accumulate) tensor-core mode
constexpr int kDecPipes = 4;          // decode tensor-core kernel: MMA pipelines per CTA
constexpr int kDecTokens = kExactTokens;   // tokens per partial-sum row of that kernel

// Device status word codes (sticky until the next forward overwrites them).
enum Status : int32_t {
  kStatusOk = 0,
  kStatusBadExpert = 1,       // a routed id outside [0, E)
  kStatusTimeout = 2,         // a bounded wait gave up
  kStatusBadTile = 3,         // a tile outside its expert's range
};

// Per-expert weight views into the library's device copy.  W13 is the
// interleaved [n_experts][2I][H/2] array (see misc.cu), W2 is [n_experts][H][I/2];
// both with repacked offset-binary nibbles.  Scales are f32, gs64, in the same
// row order: w13s [n_experts][2I][H/64], w2s [n_experts][H][I/64].
// w13e / w2e: per-row power-of-two factors of the tensor-core path's fp16
// weights (fp16(q * s * e) in the MMA, the accumulator times 1/e after it).
struct ExpertWeights {
  const uint8_t *w13q, *w2q;
  const float *w13s, *w2s;
  const float *w13e, *w2e;
};

struct Workspace {
  // routing
  float *z_part;      // [splits][max_tokens][E] router partial logits
  int32_t *idx;       // [max_tokens][k]
  float *w;           // [max_tokens][k]
  // dispatch
  int32_t *counts;    // [E]
  int32_t *offsets;   // [E+1]
  int32_t *perm;      // [max_tokens*k]
  int32_t *inv;       // [max_tokens*k]
  int32_t *active;    // [E+1] ids of experts with tokens (ascending), shared = E last
  int32_t *n_active;  // [1]
  int32_t *tiles;     // [max_tiles] packed (expert, m-tile) for the tensor-core path
  int32_t *n_tiles;   // [2] tile count for W13 and W2 kernels
  int32_t *status;    // [1]
  int32_t *ticket;    // [1 + ceil(E/8)] fused small-T routing, self-resetting: [0] the
                      // last 8-expert block to finish, [1 + b] the last split of block b
  float *route_kv;    // [2][kRouteTokens][E] fused small-T routing: keys, then scores
  unsigned long long *usage;  // [E] assignments per expert over the counted forwards
  // expert activations
  __nv_bfloat16 *hpl; // [max_tokens*k + S*max_tokens][2][I_max] GEMV path: h as exact bf16
                      // planes, hi = bf16(h) then lo = bf16(h - hi)
  __half *hb;         // [max_tokens*k + S*max_tokens][I_max] fp16 h * 2^fh (tensor-core path)
  float *y;           // [max_tokens*k + S*max_tokens][H] f32 (tensor-core path)
  __half *xp;         // [max_tokens*k + S*max_tokens][H] fp16 x * 2^ex in grouped order
  float *wperm;       // [max_tokens*k + S*max_tokens] routing weight per grouped row (shared 1);
                      // on the tensor-core path times 2^-fh of the row's token
  float *xcol;        // [max_tokens*k + S*max_tokens] 2^-ex of the row's token (tensor-core path)
  float *hcol;        // [max_tokens*k + S*max_tokens] 2^fh of the row's token (tensor-core path)
  // exact tensor-core mode (T <= kExactTokens): operands as bf16 (hi, lo) plane pairs
  __nv_bfloat16 *xe;  // [2 * kExactTokens*(k+S)][H] grouped x (one plane when x is bf16)
  __nv_bfloat16 *he;  // [2 * kExactTokens*(k+S)][I_max] h planes
  float *dec_partial;  // decode kernel split-K partial sums [slots][pipeline][128][kDecTokens]
  int32_t *dec_ticket; // decode kernel arrival counters [2][dec_rb_max] (W13, W2)
  // host-call staging
  void *x_stage;      // [max_tokens][H] (x dtype)
  float *out_stage;   // [max_tokens][H]
};

// Programmatic dependent launch.  A kernel launched with launch_k(pdl = true)
// may be scheduled while the previous kernel on the stream is still running;
// it calls pdl_enter() first, which lets the next kernel be scheduled in turn
// and then waits until the previous grid has finished and its writes are
// visible -- so nothing it reads or writes can race with its predecessor,
// and only the launch latency and the CTAs' start-up overlap.  Without the
// launch attribute both instructions return at once.  The wait covers grids
// only, not copies or memsets, so the first kernel of every library call is
// launched plainly: only the library's own kernels within a call are chained.
static __device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Workspace pointers of a chained kernel are taken through after_wait() once
// pdl_enter() has returned.  A plain load through a const __restrict__
// parameter counts as invariant for the kernel's whole life, so the compiler
// may schedule it above the wait, where it reads what the previous forward
// left there; a pointer that comes out of a volatile asm placed after the wait
// carries no such guarantee, and every address derived from it depends on the
// wait.  Data the predecessor wrote is read through L2 (plain loads or
// __ldcg), not the read-only __ldg path: this grid is resident while it is
// being written.
template <typename T>
static __device__ __forceinline__ T *after_wait(T *p) {
  unsigned long long v = reinterpret_cast<unsigned long long>(p);
  asm volatile("" : "+l"(v));
  return reinterpret_cast<T *>(v);
}

// Address ranges to pull into L2 ahead of their use: the next layer's router
// and shared expert, which that layer reads whatever it routes to.  Every
// range starts on a 16-byte boundary and its length is a multiple of 16.
// The f32 RMS pre-norm of one row by a 1024-thread block:
// out_row = bf16(row / sqrt(mean(row^2) + eps)).  v[r] holds the row's float4
// number threadIdx.x + 1024 r (zero past the row's end); float4s from 2048 on
// (H > 8192) are read from row.  One definition for the stand-alone norm and
// the one fused into the combine, so the two give the same bits: a fixed
// per-thread fmaf order, then warp and block sums in a fixed order.
static __device__ __forceinline__ void rmsnorm_row_bf16(const float4 *row, const float4 (&v)[2],
                                                        int H, float eps,
                                                        __nv_bfloat16 *out_row, float *part) {
  const int n4 = H / 4;
  float ss = 0.f;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    ss = fmaf(v[r].x, v[r].x, ss);
    ss = fmaf(v[r].y, v[r].y, ss);
    ss = fmaf(v[r].z, v[r].z, ss);
    ss = fmaf(v[r].w, v[r].w, ss);
  }
  for (int i = threadIdx.x + 2048; i < n4; i += 1024) {
    const float4 f = row[i];
    ss = fmaf(f.x, f.x, fmaf(f.y, f.y, fmaf(f.z, f.z, fmaf(f.w, f.w, ss))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 32; ++w) tot += part[w];
  const float r = 1.0f / sqrtf(tot / (float)H + eps);
  __nv_bfloat162 *o2 = reinterpret_cast<__nv_bfloat162 *>(out_row);
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const int i = threadIdx.x + rr * 1024;
    if (i < n4) {
      o2[2 * i] = __floats2bfloat162_rn(v[rr].x * r, v[rr].y * r);
      o2[2 * i + 1] = __floats2bfloat162_rn(v[rr].z * r, v[rr].w * r);
    }
  }
  for (int i = threadIdx.x + 2048; i < n4; i += 1024) {
    const float4 f = row[i];
    o2[2 * i] = __floats2bfloat162_rn(f.x * r, f.y * r);
    o2[2 * i + 1] = __floats2bfloat162_rn(f.z * r, f.w * r);
  }
}

struct L2Prefetch {
  static constexpr int kMax = 5;
  const char *ptr[kMax];
  unsigned long long bytes[kMax];
  int n;
};

// Thread 0 of each CTA prefetches the CTA's 1/gridDim share of every range
// with cp.async.bulk.prefetch.L2 (a hint: nothing waits for it, and the data
// read from these addresses is the same with or without it).
static __device__ __forceinline__ void l2_prefetch_share(const L2Prefetch &pf) {
  if (threadIdx.x != 0) return;
  constexpr unsigned long long kPiece = 32768;
  for (int r = 0; r < pf.n; ++r) {
    const unsigned long long b = pf.bytes[r];
    const unsigned long long share = ((b + gridDim.x - 1) / gridDim.x + 15) & ~15ull;
    const unsigned long long lo = share * blockIdx.x;
    const unsigned long long hi = lo + share < b ? lo + share : b;
    for (unsigned long long off = lo; off < hi; off += kPiece) {
      const unsigned long long len = hi - off < kPiece ? hi - off : kPiece;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(pf.ptr[r] + off),
                   "r"((uint32_t)len)
                   : "memory");
    }
  }
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args &&...args) {
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = pdl ? &attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

}  // namespace moe

struct moe_handle {
  moe_layout L;
  int E, k, H, I, S, Is;
  size_t x_elem;                 // 4 (f32) or 2 (bf16)
  // weights (device, library-owned)
  float *wr_t;                   // [E][H] f32 router weights, transposed
  __nv_bfloat16 *wr_planes;      // [3][E][H] bf16 hi/mid/lo planes of wr_t (tensor-core router)
  float *bias;                   // [E] or nullptr
  float *hnorm;                  // [2] largest W1 / W3 row norm over all experts (bounds |h|)
  const moe_handle *next;        // moe_set_next_layer: the layer whose router and shared expert
                                 // this one's W2 pass prefetches into L2 (or nullptr)
  moe::ExpertWeights ex;         // routed experts
  moe::ExpertWeights sh;         // shared expert (single)
  moe::Workspace ws;
  void *pool;                    // one device allocation holding everything
  size_t pool_bytes;
  int regime_opt;                // MOE_OPT_REGIME
  int small_t_max;               // MOE_OPT_SMALL_T_MAX
  int pdl;                       // MOE_OPT_PDL
  int count_usage;               // MOE_OPT_USAGE
  unsigned long long wait_ns;    // MOE_OPT_WAIT_LIMIT_US, in ns (default 2 s)
  // moe_forward_residual_norm: during that call, the combine also writes
  // bf16(rmsnorm(resid)) here (else nullptr)
  uint16_t *norm_out;
  float norm_eps;
  int last_T;
  int last_regime;
  cudaStream_t last_stream;
  int num_sms;
  int dec_rb_max;                // row blocks of the larger decode matrix pass
  // tracing
  int profile;                   // MOE_OPT_PROFILE
  static constexpr int kMaxStages = 8;
  cudaEvent_t ev[kMaxStages + 1];
  int n_ev;                      // events recorded by the last forward
  const char *stage_names[kMaxStages];
  long long launches;            // kernels launched since init
};

namespace moe {

// The next layer's router and shared expert as L2 prefetch ranges (none when
// no next layer is set).
L2Prefetch next_layer_prefetch(const moe_handle *h);
// router.cu
cudaError_t launch_router(const moe_handle *h, const void *x, int T, cudaStream_t s);
// T <= kRouteTokens: router, top-k and dispatch in one launch (also clears the
// status word).
// usage (nullable): [E] counters the per-expert counts are added into.
cudaError_t launch_route_small(const moe_handle *h, const void *x, int T,
                               unsigned long long *usage, cudaStream_t s);
// dispatch.cu
cudaError_t launch_dispatch(const moe_handle *h, int T, int tile_m, unsigned long long *usage,
                            cudaStream_t s);
// gemv.cu
cudaError_t launch_gemv_w13(const moe_handle *h, const void *x, int T, cudaStream_t s);
cudaError_t launch_gemv_w2(const moe_handle *h, int T, cudaStream_t s);
// ggemm_tc.cu
bool tc_path_available();
cudaError_t launch_combine(const moe_handle *h, int T, float *out, bool accumulate,
                           cudaStream_t s);
cudaError_t launch_split_planes(const float *wr_t, __nv_bfloat16 *planes, long long n,
                                cudaStream_t s);
// splits: split-K partitions (gridDim.z); z receives [splits][T][E] partials.
cudaError_t launch_router_tc(const moe_handle *h, const void *x, int T, float *z, int splits,
                             cudaStream_t s);
// 2D tensor map over a row-major [rows][cols] array (row stride in elements),
// box [box_rows][box_cols], 128-byte swizzle or none.  False if the driver
// entry point is missing or the encoder rejects the arguments.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, size_t elem, uint64_t cols,
              uint64_t rows, uint64_t row_stride_elems, uint32_t box_cols, uint32_t box_rows,
              bool swizzle = true);
// Grouped x of a decode-sized batch as bf16 operand planes (xe) and the
// per-row routing weights (wperm).
cudaError_t launch_gather_exact(const moe_handle *h, const void *x, int T, cudaStream_t st);
// decode_tc.cu: the exact tensor-core path for T <= kExactTokens (gather,
// W13, W2, combine).
cudaError_t launch_decode_tc(const moe_handle *h, const void *x, int T, float *out,
                             bool accumulate, cudaStream_t st);
cudaError_t launch_tc_path(const moe_handle *h, const void *x, int T, float *out,
                           bool accumulate, cudaStream_t s);
// misc.cu
cudaError_t launch_rmsnorm_bf16(const float *x, int T, int H, float eps, uint16_t *out,
                                cudaStream_t s);
cudaError_t launch_transpose_router(const float *src, float *dst, int H, int E, cudaStream_t s);
cudaError_t launch_repack_w13(const uint8_t *w1, const uint8_t *w3, uint8_t *dst, long long n_exp,
                              int I, int kb, cudaStream_t s);
cudaError_t launch_repack_w13_scales(const float *s1, const float *s3, float *dst, long long n_exp,
                                     int I, int groups, cudaStream_t s);
cudaError_t launch_repack_words(uint8_t *w, long long n_bytes, cudaStream_t s);
// out[r] = the power of two that scales row r's gs64 scales [n_rows][groups]
// into [2^7, 2^8) (fp16 weights of the tensor-core path).
cudaError_t launch_row_pow2(const float *s, long long n_rows, int groups, float *out,
                            cudaStream_t s_);
// norms[0], norms[1] (raised, not reset) = the largest Euclidean norm of a W1
// row and of a W3 row of an interleaved W13 array [n_rows][kb].
cudaError_t launch_w13_norm(const uint8_t *q, const float *s, long long n_rows, int kb,
                            float *norms, cudaStream_t st);

// Row of W1 (is_w3 = 0) or W3 (1) feature f in the interleaved W13 layout.
__host__ __device__ __forceinline__ size_t w13_row_of(int f, int is_w3) {
  return (size_t)(f >> 6) * 128 + (size_t)((f & 63) >> 4) * 32 + (f & 15) + (is_w3 ? 16 : 0);
}

}  // namespace moe
